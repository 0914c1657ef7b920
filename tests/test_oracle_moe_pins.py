"""Pins of the oracle's DeepSeek FP8 block-scale MoE layer ("flashinfer-rs" page,
section "API Example: Fused MoE FP8 (cudarc)", DeepSeek FP8 block-scale mode,
built from the groupwise GEMM of the MATE page, section GEMM).  CPU only.

The layer is pinned to hand-worked closed forms, to a second composition built
here from the separately pinned grouped-GEMM oracle (the contiguous,
128-row-aligned expert layout of group_deepgemm_fp8_nt_groupwise, assembled in
Python) and to invariants of the routing (slot order, empty slots, repeated
experts).
"""
import numpy as np
import pytest
import torch

BF16_ONE = 0x3F80


def f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def ones_layer(tokens, hidden, inter, experts, x_bits):
    w1 = np.full((experts, 2 * inter, hidden), 0x38, np.uint8)  # E4M3 1.0
    w2 = np.full((experts, hidden, inter), 0x38, np.uint8)
    s1 = np.ones((experts, 2 * inter // 128, hidden // 128), np.float32)
    s2 = np.ones((experts, hidden // 128, inter // 128), np.float32)
    return np.full((tokens, hidden), x_bits, np.uint16), w1, w2, s1, s2


def test_closed_form_all_ones(oracle_mod):
    # x = 1, all weights 1, unit scales, hidden 256, inter 128.  The token's
    # 1x128 quantisation gives codes 448 with scale 1/448, so every fc1 output
    # is 256 * 448 * FP32(1/448) = 256 (to 2^-24), i.e. 256 in BF16; SwiGLU gives
    # 256 / (1 + e^-256) * 256 = 65536 exactly in FP64; its quantisation codes
    # 448 with scale FP32(65536/448), so fc2 gives 128 * 65536 = 2^23 in BF16;
    # two slots sum to 2^24, one slot gives 2^23, no slot 0.
    x, w1, w2, s1, s2 = ones_layer(4, 256, 128, 2, BF16_ONE)
    ts = np.array([[0, 1], [1, 1], [-1, 0], [-1, -1]], np.int32)
    out = f64(oracle_mod.moe_deepseek_fp8_block_scale(x, ts, w1, w2, s1, s2))
    assert np.all(out[0] == 2.0 ** 24) and np.all(out[1] == 2.0 ** 24)
    assert np.all(out[2] == 2.0 ** 23) and np.all(out[3] == 0.0)
    # x = 0.5: fc1 gives 128, SwiGLU 128 * 128 = 16384, fc2 128 * 16384 = 2^21
    x, w1, w2, s1, s2 = ones_layer(2, 256, 128, 2, 0x3F00)
    out = f64(oracle_mod.moe_deepseek_fp8_block_scale(x, ts[:2], w1, w2, s1, s2))
    assert np.all(out == 2.0 ** 22)


def random_layer(seed, tokens, hidden, inter, experts, top_k, empty=0.1):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((tokens, hidden), generator=g).bfloat16()
    x_bits = x.view(torch.int16).numpy().view(np.uint16)
    w1 = (torch.randn((experts, 2 * inter, hidden), generator=g) * 2).clamp(-448, 448) \
        .to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    w2 = (torch.randn((experts, hidden, inter), generator=g) * 2).clamp(-448, 448) \
        .to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    s1 = torch.exp2(torch.empty((experts, 2 * inter // 128, hidden // 128)).uniform_(-8, -5,
                                                                                     generator=g))
    s2 = torch.exp2(torch.empty((experts, hidden // 128, inter // 128)).uniform_(-8, -5,
                                                                                generator=g))
    ts = torch.stack([torch.randperm(experts, generator=g)[:top_k] for _ in range(tokens)])
    drop = torch.rand((tokens, top_k), generator=g) < empty
    ts[drop] = -1
    return x_bits, ts.int().numpy(), w1, w2, s1.numpy(), s2.numpy()


def moe_via_grouped_gemm(oracle_mod, x_bits, ts, w1, w2, s1, s2):
    """The same layer assembled from the grouped-GEMM oracle: every (token,
    slot) becomes one row of an expert-contiguous, 128-row-aligned layout."""
    tokens, hidden = x_bits.shape
    top_k = ts.shape[1]
    experts, two_i = w1.shape[0], w1.shape[1]
    inter = two_i // 2
    xq, xs = oracle_mod.quant_1x128(f64(x_bits))
    rows, m_indices, row_of = [], [], {}
    for e in range(experts):
        pairs = [(t, s) for t in range(tokens) for s in range(top_k) if ts[t, s] == e]
        for p in pairs:
            row_of[p] = len(m_indices)
            m_indices.append(e)
            rows.append(p[0])
        for _ in range((-len(pairs)) % 128):
            m_indices.append(-1)
            rows.append(-1)
    rows = np.array(rows)
    valid = rows >= 0
    a = np.zeros((len(rows), hidden), np.uint8)
    sa = np.zeros((len(rows), hidden // 128), np.float32)
    a[valid], sa[valid] = xq[rows[valid]], xs[rows[valid]]
    mi = np.array(m_indices, np.int32)
    h, _, written = oracle_mod.group_gemm_contiguous(a, w1, sa, s1, mi)
    h, _ = oracle_mod.round_to(h)  # BF16
    g_, u = h[:, :inter], h[:, inter:]
    act = np.where(valid[:, None], g_ / (1.0 + np.exp(-g_)) * u, 0.0)
    aq, sq = oracle_mod.quant_1x128(act)
    y, _, _ = oracle_mod.group_gemm_contiguous(aq, w2, sq, s2, mi)
    y, _ = oracle_mod.round_to(y)
    acc = np.zeros((tokens, hidden))
    for t in range(tokens):
        for s in range(top_k):
            if ts[t, s] >= 0:
                acc[t] += y[row_of[(t, s)]]
    _, bits = oracle_mod.round_to(acc)
    return bits


@pytest.mark.parametrize("seed,tokens,hidden,inter,experts,top_k", [
    (1, 9, 256, 128, 4, 2), (2, 20, 384, 256, 6, 3), (3, 5, 128, 384, 3, 3)])
def test_equals_composition_from_grouped_gemm(oracle_mod, seed, tokens, hidden, inter,
                                              experts, top_k):
    args = random_layer(seed, tokens, hidden, inter, experts, top_k)
    got = oracle_mod.moe_deepseek_fp8_block_scale(*args)
    want = moe_via_grouped_gemm(oracle_mod, *args)
    assert np.array_equal(got, want)
    assert np.any(f64(got) != 0)


def test_slot_order_and_repeated_experts(oracle_mod):
    x, ts, w1, w2, s1, s2 = random_layer(4, 8, 256, 128, 4, 3, empty=0.0)
    base = oracle_mod.moe_deepseek_fp8_block_scale(x, ts, w1, w2, s1, s2)
    # the FP64 sum over slots is exact here, so any slot order gives the same bits
    perm = oracle_mod.moe_deepseek_fp8_block_scale(x, ts[:, ::-1].copy(), w1, w2, s1, s2)
    assert np.array_equal(base, perm)
    # an empty slot contributes nothing; a repeated expert counts twice
    one = ts.copy()
    one[:, 1:] = -1
    y1 = f64(oracle_mod.moe_deepseek_fp8_block_scale(x, one, w1, w2, s1, s2))
    two = one.copy()
    two[:, 2] = one[:, 0]
    y2 = f64(oracle_mod.moe_deepseek_fp8_block_scale(x, two, w1, w2, s1, s2))
    assert np.array_equal(y2, 2 * y1)


def test_rejects_bad_expert_ids(oracle_mod):
    x, ts, w1, w2, s1, s2 = random_layer(5, 4, 256, 128, 4, 2)
    ts[1, 0] = 4
    with pytest.raises(ValueError):
        oracle_mod.moe_deepseek_fp8_block_scale(x, ts, w1, w2, s1, s2)
    ts[1, 0] = -2
    with pytest.raises(ValueError):
        oracle_mod.moe_deepseek_fp8_block_scale(x, ts, w1, w2, s1, s2)


def test_quantiser_agrees_with_the_norm_path(oracle_mod):
    # the shared 1x128 quantiser on BF16 values gives what the norm +
    # quantisation writes for its normed_out
    g = torch.Generator().manual_seed(6)
    inp = torch.randn((4, 512), generator=g).bfloat16()
    res = torch.randn((4, 512), generator=g).bfloat16()
    w = torch.ones(512).bfloat16()
    b = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    got = oracle_mod.fused_add_rmsnorm_fp8_block_quant(b(inp), b(res), b(w))
    codes, scales = oracle_mod.quant_1x128(f64(got["normed_out"]))
    assert np.array_equal(codes, got["out"]) and np.array_equal(scales, got["block_scale"])


# ------------------------------------------------ the layer's steps, one by one

def bf16_bits(x):
    return torch.tensor(np.asarray(x, np.float32)).bfloat16().view(torch.int16).numpy() \
        .view(np.uint16)


def test_swiglu_step_is_the_layers(oracle_mod):
    """The SwiGLU step the oracle exposes is the one its layer applies: the
    layer rebuilt from the pinned grouped GEMM and this step gives the same bits."""
    x, ts, w1, w2, s1, s2 = random_layer(7, 12, 256, 256, 4, 2)
    xq, xs = oracle_mod.quant_1x128(f64(x))
    want = oracle_mod.moe_deepseek_fp8_block_scale(x, ts, w1, w2, s1, s2)
    out = np.zeros((12, 256))
    for t in range(12):
        for s in range(2):
            e = ts[t, s]
            if e < 0:
                continue
            a = np.zeros((128, 256), np.uint8)
            sa = np.zeros((128, 2), np.float32)
            a[0], sa[0] = xq[t], xs[t]
            mi = np.full(128, -1, np.int32)
            mi[0] = 0
            _, hb, _ = oracle_mod.group_gemm_contiguous(a, w1[e:e + 1], sa, s1[e:e + 1], mi)
            aq, asc = oracle_mod.moe_swiglu_quant(hb[:1])
            a2 = np.zeros((128, 256), np.uint8)
            sa2 = np.zeros((128, 2), np.float32)
            a2[0], sa2[0] = aq[0], asc[0]
            _, yb, _ = oracle_mod.group_gemm_contiguous(a2, w2[e:e + 1], sa2, s2[e:e + 1], mi)
            out[t] += f64(yb[0])
    _, bits = oracle_mod.round_to(out)
    assert np.array_equal(bits, want)


def test_swiglu_step_special_cases(oracle_mod):
    rng = np.random.default_rng(8)
    up = rng.normal(size=(3, 256))
    # a zero gate or a zero up part: act = 0, scale 0 and codes 0
    h = np.concatenate([np.zeros((3, 256)), up], axis=1)
    codes, scales = oracle_mod.moe_swiglu_quant(bf16_bits(h))
    assert not codes.any() and not scales.any()
    h = np.concatenate([up, np.zeros((3, 256))], axis=1)
    codes, scales = oracle_mod.moe_swiglu_quant(bf16_bits(h))
    assert not codes.any() and not scales.any()
    # gates >= 64: e^-g < 2^-53, so silu(g) = g exactly and the step is the
    # (separately pinned) 1x128 quantisation of gate * up
    g = 64.0 * 2.0 ** rng.integers(0, 6, size=(3, 256))
    hb = bf16_bits(np.concatenate([g, up], axis=1))
    gq, uq = f64(hb[:, :256]), f64(hb[:, 256:])
    codes, scales = oracle_mod.moe_swiglu_quant(hb)
    want_c, want_s = oracle_mod.quant_1x128(gq * uq)
    assert np.array_equal(codes, want_c) and np.array_equal(scales, want_s)
    # gates <= -1024: e^-g overflows, silu(g) = -0, nothing survives
    hb = bf16_bits(np.concatenate([np.full((3, 256), -1024.0), up], axis=1))
    codes, scales = oracle_mod.moe_swiglu_quant(hb)
    assert not scales.any() and np.all((codes == 0) | (codes == 0x80))


def test_swiglu_step_sign_symmetry(oracle_mod):
    # negating the up part negates act exactly: same scales, sign bits flipped
    rng = np.random.default_rng(9)
    h = bf16_bits(rng.normal(size=(4, 512)) * 3)
    neg = h.copy()
    neg[:, 256:] ^= 0x8000
    c1, s1 = oracle_mod.moe_swiglu_quant(h)
    c2, s2 = oracle_mod.moe_swiglu_quant(neg)
    assert np.array_equal(s1, s2)
    nz = (c1 & 0x7F) != 0
    assert np.array_equal(c2[nz], c1[nz] ^ 0x80)


def test_combine_step_hand_worked_and_invariants(oracle_mod):
    # hand-worked: 1 + 2^-8 is the midpoint of BF16 1.0 (0x3F80) and 1 + 2^-7
    # (0x3F81) and rounds to the even 0x3F80; 1 + 3 * 2^-9 lies above it: 0x3F81
    y = bf16_bits(np.array([[1.0], [2.0 ** -8], [3 * 2.0 ** -9], [-1.0]]))
    row_of = np.array([[0, 1], [0, 2], [3, -1], [-1, -1], [1, 3]], np.int32)
    out = oracle_mod.moe_combine(y, row_of)
    assert out[:, 0].tolist() == [0x3F80, 0x3F81, 0xBF80, 0x0000, 0xBF7F]
    rng = np.random.default_rng(10)
    y = bf16_bits(rng.normal(size=(40, 256)))
    ro = rng.permutation(40)[:32].reshape(8, 4).astype(np.int32)
    ro[2, 1] = -1
    base = oracle_mod.moe_combine(y, ro)
    # one slot: the row itself; a row taken twice: exactly double; any slot order
    assert np.array_equal(oracle_mod.moe_combine(y, ro[:, :1]), y[ro[:, 0]])
    twice = oracle_mod.moe_combine(y, np.repeat(ro[:, :1], 2, axis=1))
    assert np.array_equal(f64(twice), 2 * f64(y[ro[:, 0]]))
    assert np.array_equal(oracle_mod.moe_combine(y, ro[:, ::-1].copy()), base)
