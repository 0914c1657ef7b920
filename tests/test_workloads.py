"""The seeded input generators: determinism and the structure of the workloads."""
import numpy as np
import torch

import workloads


def test_dense_is_deterministic_and_in_range():
    w1 = workloads.dense(64, 256, 384, seed=5)
    w2 = workloads.dense(64, 256, 384, seed=5)
    w3 = workloads.dense(64, 256, 384, seed=6)
    for key in ("a", "b", "a_scale", "b_scale"):
        assert torch.equal(w1[key], w2[key])
    assert not torch.equal(w1["a"], w3["a"])
    codes = torch.cat([w1["a"].flatten(), w1["b"].flatten()])
    assert not torch.any((codes & 0x7F) == 0x7F)  # no NaN codes
    assert w1["a_scale"].shape == (64, 3) and w1["b_scale"].shape == (2, 3)
    s = torch.cat([w1["a_scale"].flatten(), w1["b_scale"].flatten()])
    assert s.min() >= 2.0 ** -6 and s.max() <= 1.0


def test_dense_mn_major_is_the_transpose():
    wk = workloads.dense(32, 256, 256, seed=7, scale_major="K")
    wm = workloads.dense(32, 256, 256, seed=7, scale_major="MN")
    assert torch.equal(wk["a_scale"].t(), wm["a_scale"])
    assert torch.equal(wk["b_scale"].t(), wm["b_scale"])
    assert wm["a_scale"].is_contiguous()


def test_normal_codes_follow_the_distribution():
    w = workloads.dense(256, 256, 1024, seed=8)
    v = w["a"].view(torch.float8_e4m3fn).float()
    assert abs(v.mean().item()) < 0.02 and abs(v.std().item() - 1.0) < 0.05


def test_uniform4_config():
    w = workloads.make("dense_128x256x256")
    v = w["a"].view(torch.float8_e4m3fn).float()
    assert v.abs().max() <= 4.0 and v.abs().max() > 3.5
    s = w["a_scale"]
    assert s.min() >= 2.0 ** -4 and s.max() <= 4.0


def test_routing_m_indices_structure():
    gen = workloads.generator(3)
    mi = workloads.routing_m_indices(512, 8, 64, gen)
    a = mi.numpy()
    assert a.size % 128 == 0
    assert (a != -1).sum() == 512 * 8
    # expert ids ascending, each segment starts on a 128-row boundary and
    # holds its rows first, then -1 padding
    experts = [e for e in np.unique(a) if e != -1]
    prev_end = 0
    for e in experts:
        rows = np.nonzero(a == e)[0]
        assert rows[0] % 128 == 0 and rows[0] == prev_end
        assert np.array_equal(rows, np.arange(rows[0], rows[0] + rows.size))
        seg_end = rows[0] + -(-rows.size // 128) * 128
        assert np.all(a[rows[-1] + 1:seg_end] == -1)
        prev_end = seg_end
    assert prev_end == a.size


def test_masked_counts_in_range():
    w = workloads.masked(32, 256, 256, 128, seed=9)
    mm = w["masked_m"]
    assert mm.dtype == torch.int32 and mm.min() >= 0 and mm.max() <= 256
    assert w["a"].shape == (32, 256, 128) and w["b_scale"].shape == (32, 2, 1)


def test_sample_positions_cover_extra_rows():
    r, c = workloads.sample_positions(100, 256, 50, seed=1, extra_rows=(0, 99))
    assert r.numel() == 50 + 2 * 256
    assert torch.equal(c[-256:], torch.arange(256))
    assert r.max() < 100 and c.max() < 256


def test_masked_decode_config():
    w = workloads.make("masked_g32_maxm256_n4096_k7168_decode")
    mm = w["masked_m"]
    assert mm.dtype == torch.int32 and mm.shape == (32,)
    assert int(mm.min()) >= 0 and int(mm.max()) <= 16 and w["expected_m"] == 8
    assert w["a"].shape == (32, 256, 7168) and w["b"].shape == (32, 4096, 7168)
