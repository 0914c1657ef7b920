"""The MoE layer's allocation-free entry point (fused_moe_deepseek_fp8_block_scale_noalloc:
scratch in the library's fixed per-device array) against the workspace entry point.

Collected last on purpose: it must pass alone in a fresh process and after every other test
(whatever the earlier tests left in the static scratch).
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _layer(tokens=96, top_k=4, experts=8, hidden=1024, inter=512, seed=31):
    w = workloads.moe(tokens, top_k, experts, hidden, inter, seed=seed, device="cuda")
    w["token_selected"][::5, 1] = -1
    return w


def _with_workspace(fp8g, w):
    out = torch.full((w["tokens"], w["hidden"]), -1.0, dtype=torch.bfloat16, device="cuda")
    fp8g.fused_moe_deepseek_fp8_block_scale(w["input"], w["token_selected"], w["fc1"], w["fc2"],
                                            out, w["fc1_scale"], w["fc2_scale"])
    torch.cuda.synchronize()
    return _bits(out)


def _noalloc(fp8g, w):
    out = torch.full((w["tokens"], w["hidden"]), -1.0, dtype=torch.bfloat16, device="cuda")
    fp8g.fused_moe_deepseek_fp8_block_scale_noalloc(w["input"], w["token_selected"], w["fc1"],
                                                    w["fc2"], out, w["fc1_scale"], w["fc2_scale"])
    torch.cuda.synchronize()
    return _bits(out)


def test_noalloc_equals_workspace_entry_on_two_calls_in_a_row(fp8g):
    w = _layer()
    need = fp8g.moe_workspace_size(w["tokens"], w["num_experts"], w["top_k"], w["hidden"],
                                   w["inter"])
    assert 0 < need <= fp8g.MOE_STATIC_SCRATCH_BYTES
    want = _with_workspace(fp8g, w)
    first = _noalloc(fp8g, w)
    second = _noalloc(fp8g, w)
    assert np.array_equal(first, want)
    assert np.array_equal(second, want)
    # a different problem through the same scratch right after
    w2 = _layer(tokens=40, top_k=2, experts=4, hidden=512, inter=256, seed=32)
    assert np.array_equal(_noalloc(fp8g, w2), _with_workspace(fp8g, w2))


def test_noalloc_rejects_problems_beyond_the_static_scratch(fp8g):
    w = _layer(tokens=4, top_k=2, experts=4, hidden=1024, inter=512, seed=33)
    big_tokens = 8192  # the routed layout of 8192 tokens x top-2 needs far more than 64 MiB
    inp = torch.zeros((big_tokens, 1024), dtype=torch.bfloat16, device="cuda")
    ts = torch.zeros((big_tokens, 2), dtype=torch.int32, device="cuda")
    ts[:, 1] = 1
    out = torch.zeros((big_tokens, 1024), dtype=torch.bfloat16, device="cuda")
    assert fp8g.moe_workspace_size(big_tokens, 4, 2, 1024, 512) > fp8g.MOE_STATIC_SCRATCH_BYTES
    with pytest.raises(fp8g.Fp8gError) as e:
        fp8g.fused_moe_deepseek_fp8_block_scale_noalloc(inp, ts, w["fc1"], w["fc2"], out,
                                                        w["fc1_scale"], w["fc2_scale"])
    assert e.value.status == fp8g.ERR_UNSUPPORTED and "static scratch" in str(e.value)
    torch.cuda.synchronize()
    assert not out.float().any()
