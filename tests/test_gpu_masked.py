"""GPU parity of the masked batched form (batch_deepgemm_fp8_nt_groupwise)."""
import numpy as np
import pytest
import torch

import workloads
from parity import as_f64, assert_close, bits16, sentinel_like, to_device, written_rows

pytestmark = pytest.mark.gpu


def _run(fp8g, w, expected_m=None):
    d = to_device(w)
    out = sentinel_like((w["num_groups"], w["max_m"], w["n"]), torch.bfloat16, "cuda")
    fp8g.fp8_batch_gemm_masked(d["a"], d["b"], d["a_scale"], d["b_scale"], d["masked_m"],
                               w["expected_m"] if expected_m is None else expected_m, out)
    torch.cuda.synchronize()
    return out


# expected_m picks the tile shape: a hint above 128 (with max_m above 128) runs
# 256-row tiles on CTA pairs, otherwise one CTA per 128-row tile
@pytest.mark.parametrize("hint", ["low", "high"])
@pytest.mark.parametrize("masked,max_m,n,k", [((0, 1, 130, 256), 256, 384, 256),
                                              ((5, 77), 100, 128, 384),
                                              ((129, 128, 3), 200, 256, 512),
                                              ((255, 40, 0, 256, 300), 300, 512, 640)])
def test_small_full_parity(fp8g, oracle_mod, masked, max_m, n, k, hint):
    mm = torch.tensor(masked, dtype=torch.int32)
    w = workloads.masked(len(masked), max_m, n, k, seed=max_m + n + k, masked_m=mm)
    out = _run(fp8g, w, expected_m=1 if hint == "low" else max_m)
    ref, _, written = oracle_mod.batch_gemm_masked(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                   w["masked_m"])
    rows = written.any(axis=2)
    assert np.array_equal(written_rows(out), rows)
    assert_close(as_f64(out)[rows], ref[rows], "masked %s %s" % (masked, hint))
    assert fp8g.get_device_status() == 0


def test_out_of_range_masked_m_is_clamped_and_flagged(fp8g, oracle_mod):
    mm = torch.tensor([300, -5, 64], dtype=torch.int32)
    w = workloads.masked(3, 256, 256, 256, seed=8, masked_m=mm)
    fp8g.get_device_status(clear=True)
    out = _run(fp8g, w)
    assert fp8g.get_device_status(clear=True) == fp8g.DEVICE_MASKED_M_CLAMPED
    ref, _, written = oracle_mod.batch_gemm_masked(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                   w["masked_m"])
    rows = written.any(axis=2)
    assert np.array_equal(written_rows(out), rows)
    assert rows[0].all() and not rows[1].any() and rows[2, :64].all()
    assert_close(as_f64(out)[rows], ref[rows], "masked clamped")


def test_moe_decode_32_groups_sampled_and_expected_m_invariance(fp8g, oracle_mod):
    w = workloads.make("masked_g32_maxm256_n4096_k7168")
    out = _run(fp8g, w)
    mm = w["masked_m"].numpy()
    rows_expected = np.arange(w["max_m"])[None, :] < mm[:, None]
    assert np.array_equal(written_rows(out), rows_expected)
    g = np.random.default_rng(15)
    gs = g.integers(0, w["num_groups"], 65536)
    rs = g.integers(0, w["max_m"], 65536)
    cs = g.integers(0, w["n"], 65536)
    ref, _, wr = oracle_mod.batch_gemm_masked_at(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                 w["masked_m"], gs, rs, cs)
    got = as_f64(out)[gs, rs, cs]
    assert_close(got[wr], ref[wr], "masked moe decode sampled")
    base = bits16(out)
    for em in (1, 256):
        other = bits16(_run(fp8g, w, expected_m=em))
        assert np.array_equal(other[rows_expected], base[rows_expected])


def test_decode_shape_full_parity_and_expected_m_invariance(fp8g, oracle_mod):
    # a few tokens per expert in 256-row buffers: every valid row checked, and
    # the expected_m hint (which picks the kernel's variant) changes no bit
    w = workloads.make("masked_g32_maxm256_n4096_k7168_decode")
    out = _run(fp8g, w)
    mm = w["masked_m"].numpy()
    rows_expected = np.arange(w["max_m"])[None, :] < mm[:, None]
    assert np.array_equal(written_rows(out), rows_expected)
    ref, _, written = oracle_mod.batch_gemm_masked(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                   w["masked_m"])
    assert np.array_equal(written.any(axis=2), rows_expected)
    assert_close(as_f64(out)[rows_expected], ref[rows_expected], "masked decode")
    base = bits16(out)
    for em in (0, 1, 64, 128, 256):
        again = _run(fp8g, w, expected_m=em)
        assert np.array_equal(written_rows(again), rows_expected), em
        assert np.array_equal(bits16(again)[rows_expected], base[rows_expected]), em
    assert fp8g.get_device_status() == 0


def test_all_groups_empty(fp8g):
    mm = torch.zeros(4, dtype=torch.int32)
    w = workloads.masked(4, 128, 256, 256, seed=9, masked_m=mm)
    out = _run(fp8g, w)
    assert not written_rows(out).any()


def test_page_signature(fp8g, oracle_mod):
    mm = torch.tensor([3, 140], dtype=torch.int32)
    w = workloads.masked(2, 160, 256, 256, seed=10, masked_m=mm)
    d = to_device(w)
    out = fp8g.batch_deepgemm_fp8_nt_groupwise(d["a"].view(torch.float8_e4m3fn),
                                               d["b"].view(torch.float8_e4m3fn), d["a_scale"],
                                               d["b_scale"], d["masked_m"], expected_m=64)
    ref, _, written = oracle_mod.batch_gemm_masked(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                   w["masked_m"])
    rows = written.any(axis=2)
    assert_close(as_f64(out)[rows], ref[rows], "masked page signature")
