"""Comparison helpers shared by the GPU parity tests.

Tolerance (per element, over the rows the operation defines):
    |gpu - ref| <= 1e-2 * |ref| + 2e-3 * rms(ref)
where ref is the oracle's FP64 value before rounding.  The GPU accumulates each
128-wide block in FP32 on the tensor cores and promotes with FP32 scales, then
rounds once to BF16/FP16 (at most 2^-9 relative for BF16, inside the 1e-2 term).
"""
import numpy as np
import torch

REL_TOL = 1e-2
RMS_TOL = 2e-3
SENTINEL_BITS = 0x7FC1  # a NaN pattern no kernel result can take


def as_f64(t):
    """Output tensor (bf16/f16, any device) as an FP64 numpy array."""
    return t.detach().float().cpu().double().numpy()


def bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(got, ref, what=""):
    """got: FP64 numpy array of GPU results; ref: oracle FP64 values (same shape)."""
    got = np.asarray(got, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    assert got.shape == ref.shape
    if ref.size == 0:
        return
    assert np.all(np.isfinite(got)), "%s: non-finite GPU output" % what
    rms = float(np.sqrt(np.mean(ref * ref)))
    tol = REL_TOL * np.abs(ref) + RMS_TOL * rms
    err = np.abs(got - ref)
    bad = np.nonzero(err > tol)[0]
    if bad.size:
        i = bad[np.argmax(err[bad] / tol[bad])]
        raise AssertionError(
            "%s: %d of %d elements outside tolerance; worst at flat index %d: gpu=%r ref=%r "
            "(err %.3g, tol %.3g, rms %.3g)" % (what, bad.size, ref.size, i, got[i], ref[i],
                                                err[i], tol[i], rms))


def sentinel_like(shape, dtype, device):
    out = torch.empty(shape, dtype=torch.int16, device=device)
    out.fill_(np.int16(np.uint16(SENTINEL_BITS).view(np.int16)))
    return out.view(dtype)


def written_rows(out):
    """Boolean per row (last dim reduced): True where no element holds the sentinel,
    asserting each row is either fully written or fully untouched."""
    b = bits16(out).reshape(-1, out.shape[-1])
    untouched = b == SENTINEL_BITS
    full = untouched.all(axis=1)
    none = ~untouched.any(axis=1)
    assert np.all(full | none), "a row is partly written"
    return none.reshape(out.shape[:-1])


def to_device(w, device="cuda"):
    return {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in w.items()}
