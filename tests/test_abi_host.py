"""The C-ABI library on a host without a GPU: it loads, exports every entry
point that the headers in include/ declare, and rejects bad arguments on the
host with the documented status codes, before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8g.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    from fp8_block_scaled_nt_gb300 import _build
    _build.build()
    import fp8_block_scaled_nt_gb300 as fp8g
    return fp8g


def declared_functions(headers=HEADERS):
    names = set()
    for h in headers:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_three_forms_and_helpers():
    names = declared_functions()
    for f in ("fp8_gemm_nt_groupwise", "fp8_group_gemm_contiguous", "fp8_batch_gemm_masked",
              "fused_add_rmsnorm_fp8_block_quant", "fp8g_last_error", "fp8g_get_device_status",
              "fp8g_get_stream_status", "fused_moe_deepseek_fp8_block_scale_workspace_layout",
              "fp8g_testing_set_wait_limit_ns"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    handle = lib.load()
    for name in declared_functions():
        assert hasattr(handle, name), name


def test_header_compiles_as_c():
    import subprocess
    import tempfile
    from fp8_block_scaled_nt_gb300 import _build
    inc = os.path.join(_build.cuda_home(), "include")
    src = ('#include "fp8g.h"\n#include "fp8g_testing.h"\n'
           'int main(void){ return (int)FP8G_OK; }\n')
    with tempfile.TemporaryDirectory() as d:
        p = os.path.join(d, "t.c")
        open(p, "w").write(src)
        r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                            "-I", inc, "-c", p, "-o", os.path.join(d, "t.o")],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def _dense(h, a=16, b=16, sa=16, sb=16, out=16, dt=0, os_=None, m=128, n=256, k=256, major=0,
           gran=(1, 128, 128), mma_sm=1):
    return h.fp8_gemm_nt_groupwise(a, b, sa, sb, out, dt, os_, m, n, k, major, gran[0], gran[1],
                                   gran[2], mma_sm, None)


@pytest.mark.parametrize("kwargs,status,msg", [
    (dict(k=200), 1, "k = 200"),
    (dict(k=0), 1, "k = 0"),
    (dict(n=192), 1, "n = 192"),
    (dict(m=-1), 1, "m = -1"),
    (dict(dt=7), 1, "out_dtype"),
    (dict(major=3), 1, "scale_major"),
    (dict(mma_sm=5), 1, "mma_sm"),
    (dict(gran=(1, 128, 64)), 2, "granularity"),
    (dict(a=0), 1, "null"),
    (dict(out=0), 1, "null"),
    (dict(b=24), 1, "16-byte"),
    (dict(sa=18), 1, "4-byte"),
    (dict(n=1 << 31), 2, "2^31"),
    (dict(dt=2), 1, "output_scale"),
    (dict(os_=16), 1, "output_scale"),
    (dict(dt=2, os_=18), 1, "4-byte"),
])
def test_dense_host_validation(lib, kwargs, status, msg):
    h = lib.load()
    assert _dense(h, **kwargs) == status
    assert msg in lib.last_error()


def test_empty_problem_is_ok_without_device(lib):
    h = lib.load()
    assert _dense(h, m=0, a=0, out=0, sa=0) == 0
    assert h.fp8_batch_gemm_masked(16, 16, 16, 16, 16, 1, 16, 0, 256, 256, 256, None) == 0
    assert h.fp8_group_gemm_contiguous(0, 16, 0, 16, 0, 0, 0, 256, 256, 4, None) == 0


def test_grouped_host_validation(lib):
    h = lib.load()
    assert h.fp8_group_gemm_contiguous(16, 16, 16, 16, 16, 16, 256, 256, 256, 0, None) == 1
    assert "num_groups" in lib.last_error()
    assert h.fp8_group_gemm_contiguous(16, 16, 16, 16, 0, 16, 256, 256, 256, 4, None) == 1
    assert "m_indices" in lib.last_error()
    assert h.fp8_group_gemm_contiguous(16, 16, 16, 16, 18, 16, 256, 256, 256, 4, None) == 1
    assert h.fp8_group_gemm_contiguous(16, 16, 16, 16, 16, 16, 256, 256, 100, 4, None) == 1


def test_masked_host_validation(lib):
    h = lib.load()
    assert h.fp8_batch_gemm_masked(16, 16, 16, 16, 16, -1, 16, 4, 256, 256, 256, None) == 1
    assert "expected_m" in lib.last_error()
    assert h.fp8_batch_gemm_masked(16, 16, 16, 16, 0, 1, 16, 4, 256, 256, 256, None) == 1
    assert "masked_m" in lib.last_error()
    assert h.fp8_batch_gemm_masked(16, 16, 16, 16, 16, 1, 16, -1, 256, 256, 256, None) == 1


def _norm(h, out=16, bs=16, normed=16, inp=16, res=16, w=16, eps=1e-6, rows=4, hidden=256):
    return h.fused_add_rmsnorm_fp8_block_quant(out, bs, normed, inp, res, w, eps, rows, hidden,
                                               None)


@pytest.mark.parametrize("kwargs,status,msg", [
    (dict(hidden=200), 1, "hidden = 200"),
    (dict(hidden=0), 1, "hidden = 0"),
    (dict(hidden=65536 + 128), 2, "65536"),
    (dict(rows=-1), 1, "rows = -1"),
    (dict(eps=float("nan")), 1, "eps"),
    (dict(eps=-1.0), 1, "eps"),
    (dict(out=0), 1, "null"),
    (dict(w=0), 1, "null"),
    (dict(res=24), 1, "16-byte"),
    (dict(bs=18), 1, "4-byte"),
])
def test_norm_quant_host_validation(lib, kwargs, status, msg):
    h = lib.load()
    assert _norm(h, **kwargs) == status
    assert msg in lib.last_error()


def test_norm_quant_empty_is_ok_without_device(lib):
    assert _norm(lib.load(), rows=0, out=0, inp=0) == 0


def _moe(h, inp=16, ts=16, w1=16, w2=16, out=16, s1=16, s2=16, t=8, e=4, k=2, hd=256, i=128,
         ws=256, wsb=1 << 30):
    return h.fused_moe_deepseek_fp8_block_scale(inp, ts, w1, w2, out, s1, s2, t, e, k, hd, i,
                                                ws, wsb, None)


@pytest.mark.parametrize("kwargs,status,msg", [
    (dict(hd=200), 1, "hidden_size"),
    (dict(i=100), 1, "inter_size"),
    (dict(k=5), 1, "top_k"),
    (dict(e=0), 1, "num_experts"),
    (dict(e=5000, k=2), 1, "num_experts"),
    (dict(t=-1), 1, "num_tokens"),
    (dict(ws=0), 1, "null"),
    (dict(ws=272), 1, "256-byte"),
    (dict(wsb=1000), 1, "workspace of 1000 bytes"),
])
def test_moe_host_validation(lib, kwargs, status, msg):
    h = lib.load()
    assert _moe(h, **kwargs) == status
    assert msg in lib.last_error()


def test_moe_workspace_size_and_empty_call(lib):
    # rows bound: round_up(T*K + 127*E, 128); regions 256-byte aligned
    size = lib.moe_workspace_size(8, 4, 2, 256, 128)
    rows = (8 * 2 + 127 * 4 + 127) // 128 * 128
    assert size >= rows * (256 + 2 * 256 + 128 + 2 * 256) and size % 256 == 0
    assert lib.moe_workspace_size(8, 4, 2, 200, 128) == 0  # bad shape
    assert _moe(lib.load(), t=0, inp=0, out=0, ws=0, wsb=0) == 0


def test_moe_noalloc_rejects_oversize_on_the_host(lib):
    h = lib.load()
    # 8192 tokens x top-2, hidden 1024, inter 512: far beyond the 64 MiB scratch
    assert lib.moe_workspace_size(8192, 4, 2, 1024, 512) > lib.MOE_STATIC_SCRATCH_BYTES
    rc = h.fused_moe_deepseek_fp8_block_scale_noalloc(16, 16, 16, 16, 16, 16, 16, 8192, 4, 2,
                                                      1024, 512, None)
    assert rc == 2 and "static scratch" in lib.last_error()


def _bmm(h, a=16, b=16, af=0, bf=0, sa=16, ach=0, sb=16, bch=0, out=16, dt=0, batch=2, m=100,
         n=208, k=176):
    return h.bmm_fp8(a, b, af, bf, sa, ach, sb, bch, out, dt, batch, m, n, k, None)


@pytest.mark.parametrize("kwargs,status,msg", [
    (dict(k=100), 1, "k = 100"),
    (dict(k=0), 1, "k = 0"),
    (dict(n=200), 1, "n = 200"),
    (dict(n=-16), 1, "n = -16"),
    (dict(m=-1), 1, "m = -1"),
    (dict(af=2), 1, "E4M3 or E5M2"),
    (dict(dt=2), 1, "out_dtype"),
    (dict(b=0), 1, "null"),
    (dict(out=24), 1, "16-byte"),
    (dict(sb=18), 1, "4-byte"),
    (dict(n=1 << 31), 2, "2^31"),
])
def test_bmm_host_validation(lib, kwargs, status, msg):
    h = lib.load()
    assert _bmm(h, **kwargs) == status
    assert msg in lib.last_error()


def test_bmm_accepts_multiples_of_16_and_empty_problems(lib):
    import torch
    h = lib.load()
    assert _bmm(h, m=0, a=0, out=0, sa=0) == 0
    assert _bmm(h, batch=0, a=0, b=0, out=0) == 0
    if not torch.cuda.is_available():
        # n = 208, k = 176 pass the shape checks; the call then needs a device
        assert _bmm(h) == 4 and "cudaGetDevice" in lib.last_error()
        assert _bmm(h, n=16, k=16) == 4


def test_valid_call_without_a_device_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("host has a GPU")
    h = lib.load()
    assert _dense(h) == 4  # FP8G_ERR_CUDA: no device, nothing launched
    assert "cudaGetDevice" in lib.last_error()
    flags = ctypes.c_uint(0)
    assert h.fp8g_get_device_status(ctypes.byref(flags), 0) == 4


def test_binding_rejects_bad_tensors_before_the_library(lib):
    import torch
    a = torch.zeros((128, 256), dtype=torch.float32)
    with pytest.raises(TypeError):
        lib.fp8_gemm_nt_groupwise(a, a, a, a, a)
    a8 = torch.zeros((128, 256), dtype=torch.uint8)
    with pytest.raises(ValueError):
        lib.fp8_gemm_nt_groupwise(a8, torch.zeros((256, 128), dtype=torch.uint8),
                                  torch.ones((128, 2)), torch.ones((2, 2)),
                                  torch.empty((128, 256), dtype=torch.bfloat16))
    with pytest.raises(lib.Fp8gError):
        lib.gemm_fp8_nt_groupwise(a8, a8, None, None, backend="mudnn")


def test_moe_workspace_layout_matches_the_size(lib):
    t, e, k, hd, it = 37, 5, 3, 384, 256
    rows, offs = lib.moe_workspace_layout(t, e, k, hd, it)
    assert rows == (t * k + 127 * e + 127) // 128 * 128
    sizes = dict(m_indices=4 * rows, row_of=4 * t * k, a1=rows * hd, a1_scale=4 * rows * hd // 128,
                 h=2 * rows * 2 * it, a2=rows * it, a2_scale=4 * rows * it // 128, y=2 * rows * hd)
    at = 0
    for name in lib.MOE_WORKSPACE_REGIONS:  # in order, each 256-byte aligned, no overlap
        assert offs[name] == at and at % 256 == 0, name
        at += (sizes[name] + 255) // 256 * 256
    assert at == lib.moe_workspace_size(t, e, k, hd, it)
    with pytest.raises(lib.Fp8gError):
        lib.moe_workspace_layout(t, e, k, 200, it)


def test_stream_status_without_a_device_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("host has a GPU")
    flags = ctypes.c_uint(0)
    assert lib.load().fp8g_get_stream_status(ctypes.byref(flags), 1, None) == 4


def _moe_tensors(t=8, k=2, e=4, hd=256, it=128):
    import torch
    return dict(input=torch.zeros((t, hd), dtype=torch.bfloat16),
                token_selected=torch.zeros((t, k), dtype=torch.int32),
                fc1_weights=torch.zeros((e, 2 * it, hd), dtype=torch.uint8),
                fc2_weights=torch.zeros((e, hd, it), dtype=torch.uint8),
                out=torch.zeros((t, hd), dtype=torch.bfloat16),
                fc1_scales=torch.ones((e, 2 * it // 128, hd // 128)),
                fc2_scales=torch.ones((e, hd // 128, it // 128)))


@pytest.mark.parametrize("entry", ["fused_moe_deepseek_fp8_block_scale",
                                   "fused_moe_deepseek_fp8_block_scale_noalloc"])
@pytest.mark.parametrize("bad,msg", [
    (dict(out=((4, 256), "bfloat16")), "out must be"),
    (dict(fc2_weights=((4, 256, 64), "uint8")), "fc2_weights"),
    (dict(fc1_scales=((4, 1, 2), "float32")), "fc1_scales"),
    (dict(fc2_scales=((4, 2, 1), "float64")), "fc2_scales"),
    (dict(token_selected=((7, 2), "int32")), "token_selected"),
    (dict(fc1_weights=((4, 255, 256), "uint8")), "fc1_weights"),
])
def test_moe_wrappers_reject_mismatched_tensors_before_the_library(lib, entry, bad, msg):
    """Both MoE wrappers check every tensor against the others: the C ABI gets
    only pointers and sizes, so a smaller out or weight tensor would otherwise
    be read or written past its end on the device."""
    import torch
    args = _moe_tensors()
    for name, (shape, dt) in bad.items():
        args[name] = torch.zeros(shape, dtype=getattr(torch, dt))
    with pytest.raises(ValueError) as e:
        getattr(lib, entry)(**args)
    assert msg in str(e.value)


def test_page_wrapper_leaves_the_tile_shape_to_the_library(lib, monkeypatch):
    """The page's gemm_fp8_nt_groupwise defaults mma_sm to MATE's 1; here an
    omitted mma_sm reaches the C ABI as 0 (automatic: CTA pairs on large
    problems), and an explicit value goes through unchanged."""
    import torch
    seen = []

    class FakeLib:
        def fp8_gemm_nt_groupwise(self, *args):
            seen.append(args[14])
            return 0

    monkeypatch.setattr(lib, "load", lambda: FakeLib())
    monkeypatch.setattr(lib, "_cuda_contig", lambda ts, names: torch.device("cpu"))
    monkeypatch.setattr(lib, "_stream_handle", lambda stream, dev: None)
    a = torch.zeros((256, 256), dtype=torch.uint8)
    sa, sb = torch.ones((256, 2)), torch.ones((2, 2))
    lib.gemm_fp8_nt_groupwise(a, a, sa, sb)
    lib.gemm_fp8_nt_groupwise(a, a, sa, sb, mma_sm=1)
    lib.gemm_fp8_nt_groupwise(a, a, sa, sb, mma_sm=2)
    lib.fp8_gemm_nt_groupwise(a, a, sa, sb, torch.empty((256, 256), dtype=torch.bfloat16))
    assert seen == [0, 1, 2, 0]
