"""GPU parity of the contiguous grouped form (group_deepgemm_fp8_nt_groupwise)."""
import numpy as np
import pytest
import torch

import workloads
from parity import as_f64, assert_close, sentinel_like, to_device, written_rows

pytestmark = pytest.mark.gpu


def _m_indices(counts):
    mi = []
    for e, c in enumerate(counts):
        if c:
            pad = -(-c // 128) * 128
            mi += [e] * c + [-1] * (pad - c)
    return torch.tensor(mi, dtype=torch.int32)


def _run(fp8g, w):
    d = to_device(w)
    out = sentinel_like((w["m"], w["n"]), torch.bfloat16, "cuda")
    fp8g.fp8_group_gemm_contiguous(d["a"], d["b"], d["a_scale"], d["b_scale"], d["m_indices"], out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("counts,n,k", [((3, 0, 130, 128, 1), 384, 256),
                                        ((1,), 128, 128),
                                        ((250, 5, 0, 0, 129, 64), 256, 640)])
def test_small_full_parity(fp8g, oracle_mod, counts, n, k):
    w = workloads.grouped(0, 0, len(counts), n, k, seed=sum(counts) + n,
                          m_indices=_m_indices(counts))
    out = _run(fp8g, w)
    ref, _, written = oracle_mod.group_gemm_contiguous(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                       w["m_indices"])
    rows = written.any(axis=1)
    assert np.array_equal(written_rows(out), rows)  # bit-exact on which rows are written
    assert_close(as_f64(out)[rows], ref[rows], "grouped %s" % (counts,))


def test_unaligned_total_rows(fp8g, oracle_mod):
    # M_total not a multiple of 128: the last block is partial
    mi = torch.cat([_m_indices((130,)), torch.full((20,), 1, dtype=torch.int32)])
    w = workloads.grouped(0, 0, 2, 256, 256, seed=5, m_indices=mi)
    out = _run(fp8g, w)
    ref, _, written = oracle_mod.group_gemm_contiguous(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                       w["m_indices"])
    rows = written.any(axis=1)
    assert np.array_equal(written_rows(out), rows)
    assert_close(as_f64(out)[rows], ref[rows], "grouped unaligned")


def test_all_padding_writes_nothing(fp8g):
    mi = torch.full((256,), -1, dtype=torch.int32)
    w = workloads.grouped(0, 0, 3, 256, 256, seed=6, m_indices=mi)
    out = _run(fp8g, w)
    assert not written_rows(out).any()
    assert fp8g.get_device_status(clear=True) == 0


def test_padding_rows_inside_a_block(fp8g, oracle_mod):
    # -1 rows between an expert's rows (the block still holds one expert): only
    # the expert's rows are computed and written
    mi = torch.full((384,), -1, dtype=torch.int32)
    mi[0:128:3] = 0
    mi[128:256:2] = 2
    mi[300:310] = 1
    w = workloads.grouped(0, 0, 3, 384, 384, seed=7, m_indices=mi)
    out = _run(fp8g, w)
    ref, _, written = oracle_mod.group_gemm_contiguous(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                       w["m_indices"])
    rows = written.any(axis=1)
    assert np.array_equal(written_rows(out), rows)
    assert np.array_equal(rows, (mi >= 0).numpy())
    assert_close(as_f64(out)[rows], ref[rows], "grouped interleaved padding")
    assert fp8g.get_device_status(clear=True) == 0


def test_moe_4096_tokens_top8_64_experts_sampled(fp8g, oracle_mod):
    w = workloads.make("grouped_4096tok_top8_e64_n4096_k7168")
    out = _run(fp8g, w)
    mi = w["m_indices"].numpy()
    assert np.array_equal(written_rows(out), mi != -1)
    # seeded sample plus the first and last row of every expert segment
    r, c = workloads.sample_positions(w["m"], w["n"], 65536, seed=13)
    valid = np.nonzero(mi != -1)[0]
    seg_edges = np.unique(np.concatenate([valid[np.r_[True, np.diff(valid) != 1]],
                                          valid[np.r_[np.diff(valid) != 1, True]]]))
    g = torch.Generator().manual_seed(14)
    er = torch.tensor(np.repeat(seg_edges, 64), dtype=torch.int64)
    ec = torch.randint(0, w["n"], (er.numel(),), generator=g)
    r, c = torch.cat([r, er]), torch.cat([c, ec])
    ref, _, wr = oracle_mod.group_gemm_contiguous_at(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                     w["m_indices"], r, c)
    got = as_f64(out)[r.numpy(), c.numpy()]
    assert np.array_equal(wr, mi[r.numpy()] != -1)
    assert_close(got[wr], ref[wr], "grouped moe sampled")
    assert fp8g.get_device_status() == 0


def test_broken_precondition_is_flagged_and_skipped(fp8g, oracle_mod):
    mi = _m_indices((130, 128))
    mi[5] = 1     # block 0 now mixes experts 0 and 1
    mi[300] = 7   # block 2 has an id >= num_groups
    w = workloads.grouped(0, 0, 2, 256, 256, seed=6, m_indices=mi)
    assert fp8g.get_device_status(clear=True) in (0, fp8g.DEVICE_BAD_M_INDICES)
    out = _run(fp8g, w)
    status = fp8g.get_device_status(clear=True)
    assert status == fp8g.DEVICE_BAD_M_INDICES
    written = written_rows(out)
    assert not written[:128].any() and not written[256:384].any()
    # the intact block (rows 128..255: expert 0's tail + padding) is computed
    good = _m_indices((130, 128))
    w_ok = dict(w, m_indices=good)
    ref, _, wr = oracle_mod.group_gemm_contiguous(w_ok["a"], w_ok["b"], w_ok["a_scale"],
                                                  w_ok["b_scale"], good)
    rows = np.zeros(w["m"], bool)
    rows[128:256] = wr[128:256].any(axis=1)
    assert np.array_equal(written, rows)
    assert_close(as_f64(out)[rows], ref[rows], "grouped intact block")


def test_page_signature(fp8g, oracle_mod):
    w = workloads.grouped(0, 0, 3, 256, 384, seed=7, m_indices=_m_indices((10, 200, 3)))
    d = to_device(w)
    out = fp8g.group_deepgemm_fp8_nt_groupwise(d["a"].view(torch.float8_e4m3fn),
                                               d["b"].view(torch.float8_e4m3fn),
                                               d["a_scale"], d["b_scale"], d["m_indices"])
    ref, _, written = oracle_mod.group_gemm_contiguous(w["a"], w["b"], w["a_scale"], w["b_scale"],
                                                       w["m_indices"])
    rows = written.any(axis=1)
    assert_close(as_f64(out)[rows], ref[rows], "grouped page signature")
