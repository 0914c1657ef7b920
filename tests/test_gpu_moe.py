"""GPU parity of the DeepSeek FP8 block-scale MoE layer (fused_moe_deepseek_fp8_block_scale,
built on the grouped GEMM) against the CPU oracle, through the C ABI.

Stage by stage.  The workspace is the caller's, so after a call the test reads each step's
output from it (layout: fused_moe_deepseek_fp8_block_scale_workspace_layout) and checks that
step against the oracle's function for it, fed the GPU's own input of that step:
  route            the layout itself: every routed slot has its own row, tagged with its
                   expert; each expert's rows are contiguous from a multiple of 128
  quantise+gather  bit-exact against the oracle's 1x128 quantiser of the token
  fc1, fc2         the grouped GEMM's tolerance against oracle.group_gemm_contiguous
                   (|gpu - ref| <= 1e-2 |ref| + 2e-3 rms(ref))
  SwiGLU+quantise  scales within 2^-17 relative; codes bit-exact, except where the exact
                   quotient act / scale lies within 2^-16 (relative) of the midpoint of the
                   two codes: the kernel evaluates silu in FP32 with the hardware exponential
                   (a relative error below 2^-17 for the gates BF16 holds below 128), the
                   oracle in FP64
  combine          bit-exact against oracle.moe_combine, except where a partial sum of the
                   token's slots (in slot order) is not an FP32 value, so that the kernel's
                   FP32 sum was rounded: there within one BF16 unit
End to end the layer is compared with |gpu - ref| <= 2e-2 |ref| + 2e-2 rms(ref): both sides
take the same discrete steps (two 1x128 quantisations, three BF16 roundings), and where an
input of a step lies at a rounding boundary the two land one step apart (one activation code
one E4M3 step apart moves one term of an inter-long dot product by up to 1/8 of that term).
The stage checks above are what pins the layer; the end-to-end bound only bounds how far such
steps carry.  Exact closed forms hold bit for bit.
"""
import numpy as np
import pytest
import torch

import workloads
from parity import assert_close

pytestmark = pytest.mark.gpu


def f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_gpu(fp8g, w, workspace=None, fill=None):
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in w.items()}
    out = torch.full((w["tokens"], w["hidden"]), -7.0, dtype=torch.bfloat16, device="cuda")
    if workspace is None and fill is not None:
        need = fp8g.moe_workspace_size(w["tokens"], w["num_experts"], w["top_k"], w["hidden"],
                                       w["inter"])
        workspace = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
    fp8g.fused_moe_deepseek_fp8_block_scale(d["input"], d["token_selected"], d["fc1"], d["fc2"],
                                            out, d["fc1_scale"], d["fc2_scale"],
                                            workspace=workspace)
    torch.cuda.synchronize()
    return bits(out)


def oracle_of(oracle_mod, w, tokens=None):
    sel = slice(None) if tokens is None else tokens
    return oracle_mod.moe_deepseek_fp8_block_scale(
        bits(w["input"])[sel], w["token_selected"].cpu().numpy()[sel], w["fc1"].cpu(),
        w["fc2"].cpu(), w["fc1_scale"].cpu(), w["fc2_scale"].cpu())


def check(got_bits, ref_bits, label):
    got, ref = f64(got_bits), f64(ref_bits)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(got - ref)
    assert np.all(err <= 2e-2 * np.abs(ref) + 2e-2 * rms), (label, float(err.max()), rms)


def test_closed_form_all_ones_exact(fp8g):
    tokens, hidden, inter, experts = 5, 256, 128, 3
    ts = torch.tensor([[0, 1], [2, 2], [-1, 1], [-1, -1], [1, 0]], dtype=torch.int32)
    w = dict(input=torch.ones((tokens, hidden)).bfloat16(), token_selected=ts,
             fc1=torch.full((experts, 2 * inter, hidden), 0x38, dtype=torch.uint8),
             fc2=torch.full((experts, hidden, inter), 0x38, dtype=torch.uint8),
             fc1_scale=torch.ones((experts, 2 * inter // 128, hidden // 128)),
             fc2_scale=torch.ones((experts, hidden // 128, inter // 128)),
             tokens=tokens, top_k=2, num_experts=experts, hidden=hidden, inter=inter)
    got = f64(run_gpu(fp8g, w))
    want = np.array([2.0 ** 24, 2.0 ** 24, 2.0 ** 23, 0.0, 2.0 ** 24])
    assert np.array_equal(got, np.repeat(want[:, None], hidden, axis=1))


@pytest.mark.parametrize("tokens,top_k,experts,hidden,inter", [
    (37, 3, 5, 256, 128), (130, 2, 4, 384, 256), (300, 8, 16, 512, 384), (1, 1, 1, 128, 128)])
def test_parity_small_layers(fp8g, oracle_mod, tokens, top_k, experts, hidden, inter):
    w = workloads.moe(tokens, top_k, experts, hidden, inter, seed=tokens + experts)
    w["token_selected"][::7, 0] = -1  # some empty slots
    got = run_gpu(fp8g, w, fill=0xFF)   # garbage-filled workspace
    check(got, oracle_of(oracle_mod, w), (tokens, top_k, experts, hidden, inter))


def test_workspace_reuse_is_deterministic(fp8g):
    w = workloads.moe(200, 4, 8, 256, 256, seed=21)
    need = fp8g.moe_workspace_size(200, 8, 4, 256, 256)
    ws = torch.full((need,), 0x5A, dtype=torch.uint8, device="cuda")
    a = run_gpu(fp8g, w, workspace=ws)
    b = run_gpu(fp8g, w, workspace=ws)
    c = run_gpu(fp8g, w, fill=0x00)
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_bad_expert_ids_are_skipped_and_flagged(fp8g, oracle_mod):
    w = workloads.moe(40, 2, 4, 256, 128, seed=22)
    fp8g.get_device_status(clear=True)
    bad = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in w.items()}
    bad["token_selected"][3, 1] = 9
    bad["token_selected"][5, 0] = -5
    got = run_gpu(fp8g, bad)
    assert fp8g.get_device_status(clear=True) & fp8g.DEVICE_BAD_M_INDICES
    skipped = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in w.items()}
    skipped["token_selected"][3, 1] = -1
    skipped["token_selected"][5, 0] = -1
    check(got, oracle_of(oracle_mod, skipped), "bad ids")


def test_moe_workload_sampled_tokens(fp8g, oracle_mod):
    w = workloads.make("moe_4096tok_top8_e64_h7168_i2048", device="cuda")
    got = run_gpu(fp8g, w)
    g = torch.Generator().manual_seed(5)
    pick = np.sort(np.concatenate([[0, w["tokens"] - 1],
                                   torch.randint(1, w["tokens"] - 1, (30,), generator=g).numpy()]))
    ref = oracle_of(oracle_mod, w, pick)
    check(got[pick], ref, "4096 tokens sampled")


def test_argument_errors(fp8g):
    w = workloads.moe(8, 2, 4, 256, 128, seed=23)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in w.items()}
    out = torch.zeros((8, 256), dtype=torch.bfloat16, device="cuda")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fused_moe_deepseek_fp8_block_scale(d["input"], d["token_selected"], d["fc1"],
                                                d["fc2"], out, d["fc1_scale"], d["fc2_scale"],
                                                workspace=small)
    assert e.value.status == fp8g.ERR_INVALID_ARGUMENT and "workspace" in str(e.value)
    torch.cuda.synchronize()
    assert not out.float().any()


# ---------------------------------------------------------------- stage by stage

def _region(ws, off, name, dtype, shape):
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    return ws[off[name]:off[name] + n].view(dtype).view(*shape).cpu()


def _stages(fp8g, w, ws):
    t, k, e, hd, it = w["tokens"], w["top_k"], w["num_experts"], w["hidden"], w["inter"]
    rows, off = fp8g.moe_workspace_layout(t, e, k, hd, it)
    u16 = lambda x: x.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    return dict(
        rows=rows,
        m_indices=_region(ws, off, "m_indices", torch.int32, (rows,)).numpy(),
        row_of=_region(ws, off, "row_of", torch.int32, (t, k)).numpy(),
        a1=_region(ws, off, "a1", torch.uint8, (rows, hd)).numpy(),
        a1_scale=_region(ws, off, "a1_scale", torch.float32, (rows, hd // 128)).numpy(),
        h=u16(_region(ws, off, "h", torch.int16, (rows, 2 * it))),
        a2=_region(ws, off, "a2", torch.uint8, (rows, it)).numpy(),
        a2_scale=_region(ws, off, "a2_scale", torch.float32, (rows, it // 128)).numpy(),
        y=u16(_region(ws, off, "y", torch.int16, (rows, hd))))


def _check_route(st, ts, experts):
    mi, ro = st["m_indices"], st["row_of"]
    valid = (ts >= 0) & (ts < experts)
    assert np.array_equal(ro >= 0, valid)
    assert np.array_equal(mi[ro[valid]], ts[valid])
    assert np.unique(ro[valid]).size == int(valid.sum())
    assert np.array_equal(np.sort(np.nonzero(mi >= 0)[0]), np.sort(ro[valid]))
    for e in np.unique(ts[valid]):
        r = np.nonzero(mi == e)[0]
        assert r[0] % 128 == 0 and r[-1] - r[0] + 1 == r.size, e  # contiguous from 128k


def _check_quant_gather(oracle_mod, st, w, ts):
    xq, xs = oracle_mod.quant_1x128(f64(bits(w["input"])))
    valid = st["row_of"] >= 0
    tok = np.broadcast_to(np.arange(ts.shape[0])[:, None], ts.shape)[valid]
    rows = st["row_of"][valid]
    assert np.array_equal(st["a1"][rows], xq[tok])
    assert np.array_equal(st["a1_scale"][rows], xs[tok])


def _check_gemm(oracle_mod, a, sa, wt, ws_, mi, got_bits, sample=None):
    routed = np.nonzero(mi >= 0)[0]
    if sample is None:
        ref, _, written = oracle_mod.group_gemm_contiguous(a, wt, sa, ws_, mi)
        assert written[routed].all()
        assert_close(f64(got_bits[routed]), ref[routed], "grouped GEMM stage")
        return
    g = np.random.default_rng(sample)
    r = routed[g.integers(0, routed.size, 65536)]
    c = g.integers(0, got_bits.shape[1], 65536)
    ref, _, written = oracle_mod.group_gemm_contiguous_at(a, wt, sa, ws_, mi, r, c)
    assert written.all()
    assert_close(f64(got_bits[r, c]), ref, "grouped GEMM stage (sampled)")


def _check_swiglu(oracle_mod, st):
    routed = np.nonzero(st["m_indices"] >= 0)[0]
    h = st["h"][routed]
    codes, scales = oracle_mod.moe_swiglu_quant(h)
    got_c, got_s = st["a2"][routed], st["a2_scale"][routed]
    rel = np.abs(got_s.astype(np.float64) - scales) / np.maximum(scales, 1e-38)
    assert np.all(rel <= 2.0 ** -17), float(rel.max())
    bad = np.nonzero(got_c != codes)
    if bad[0].size:
        inter = codes.shape[1]
        g = f64(h[:, :inter])[bad]
        act = g / (1.0 + np.exp(-g)) * f64(h[:, inter:])[bad]
        q = act / scales[bad[0], bad[1] // 128].astype(np.float64)
        table = oracle_mod.e4m3_table()
        v1, v2 = table[got_c[bad]], table[codes[bad]]
        mid = 0.5 * (v1 + v2)
        # the two codes are neighbours and the exact quotient sits at their midpoint
        step = np.abs(v1 - v2)
        assert np.all(step <= 2.0 ** (np.floor(np.log2(np.maximum(np.abs(mid), 2.0 ** -6))) - 2))
        assert np.all(np.abs(q - mid) <= 2.0 ** -16 * np.abs(q)), np.abs(q - mid).max()


def _check_combine(oracle_mod, st, got_out):
    ro, y = st["row_of"], st["y"]
    want = oracle_mod.moe_combine(y, ro)
    for t0 in range(0, ro.shape[0], 256):
        rr = ro[t0:t0 + 256]
        vals = np.where((rr >= 0)[:, :, None], f64(y[np.maximum(rr, 0)]), 0.0)
        prefix = np.cumsum(vals, axis=1)
        exact32 = (prefix.astype(np.float32).astype(np.float64) == prefix).all(axis=1)
        g, r = got_out[t0:t0 + 256], want[t0:t0 + 256]
        assert np.array_equal(g[exact32], r[exact32])
        if (~exact32).any():
            gi = g[~exact32].astype(np.int32) - r[~exact32].astype(np.int32)
            assert np.all(np.abs(gi) <= 1)


def _run_with_workspace(fp8g, w):
    need = fp8g.moe_workspace_size(w["tokens"], w["num_experts"], w["top_k"], w["hidden"],
                                   w["inter"])
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")
    out = run_gpu(fp8g, w, workspace=ws)
    return out, ws


@pytest.mark.parametrize("tokens,top_k,experts,hidden,inter", [
    (37, 3, 5, 256, 128), (300, 8, 16, 512, 384), (130, 2, 4, 384, 256)])
def test_stagewise_parity_small_layers(fp8g, oracle_mod, tokens, top_k, experts, hidden, inter):
    w = workloads.moe(tokens, top_k, experts, hidden, inter, seed=100 + tokens)
    w["token_selected"][::9, -1] = -1
    out, ws = _run_with_workspace(fp8g, w)
    st = _stages(fp8g, w, ws)
    ts = w["token_selected"].numpy()
    _check_route(st, ts, experts)
    _check_quant_gather(oracle_mod, st, w, ts)
    _check_gemm(oracle_mod, st["a1"], st["a1_scale"], w["fc1"], w["fc1_scale"], st["m_indices"],
                st["h"])
    _check_swiglu(oracle_mod, st)
    _check_gemm(oracle_mod, st["a2"], st["a2_scale"], w["fc2"], w["fc2_scale"], st["m_indices"],
                st["y"])
    _check_combine(oracle_mod, st, out)


def test_quantise_gather_at_extreme_magnitudes(fp8g, oracle_mod):
    # The 1 x 128 quantisation divides by the block scale with one reciprocal and
    # two FMA corrections where the scale lies in [2^-100, 2^100], and by the IEEE
    # division outside it.  Blocks of every token are scaled to both sides of
    # both limits (and far past them); the codes and scales stay bit-exact.
    tokens, top_k, experts, hidden, inter = 24, 2, 4, 768, 128
    w = workloads.moe(tokens, top_k, experts, hidden, inter, seed=77)
    x = w["input"].float()
    exps = [-120.0, -95.0, -85.0, 0.0, 100.0, 110.0]  # per 128-column block
    for b, e in enumerate(exps):
        x[:, b * 128:(b + 1) * 128] *= 2.0 ** e
    x[::5, 256:384] *= 2.0 ** 9   # straddle the lower limit from the other side
    w["input"] = x.bfloat16()
    assert torch.isfinite(w["input"].float()).all()
    out, ws = _run_with_workspace(fp8g, w)
    st = _stages(fp8g, w, ws)
    ts = w["token_selected"].numpy()
    _check_route(st, ts, experts)
    _check_quant_gather(oracle_mod, st, w, ts)
    s = st["a1_scale"][st["row_of"][ts >= 0]]
    assert (s < 2.0 ** -100).any() and (s > 2.0 ** 100).any() and \
        ((s > 2.0 ** -100) & (s < 2.0 ** 100)).any()


def test_stagewise_parity_4096_tokens(fp8g, oracle_mod):
    w = workloads.make("moe_4096tok_top8_e64_h7168_i2048", device="cuda")
    out, ws = _run_with_workspace(fp8g, w)
    st = _stages(fp8g, w, ws)
    del ws
    torch.cuda.empty_cache()
    ts = w["token_selected"].cpu().numpy()
    host = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in w.items()}
    _check_route(st, ts, w["num_experts"])
    _check_quant_gather(oracle_mod, st, host, ts)
    _check_gemm(oracle_mod, st["a1"], st["a1_scale"], host["fc1"], host["fc1_scale"],
                st["m_indices"], st["h"], sample=11)
    _check_swiglu(oracle_mod, st)
    _check_gemm(oracle_mod, st["a2"], st["a2_scale"], host["fc2"], host["fc2_scale"],
                st["m_indices"], st["y"], sample=12)
    _check_combine(oracle_mod, st, out)
