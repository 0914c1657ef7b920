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
