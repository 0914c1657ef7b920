"""Seeded synthetic inputs for the FP8 groupwise-scaled NT GEMM and for the
fused add-RMSNorm + 1 x 128 FP8 quantisation that produces its activations.

This module only draws random numbers and packs them into the operand layouts
of the MATE page "FlashInfer Wrapper APIs", section GEMM; it holds none of the
GEMM's arithmetic.  Both the CUDA path and the CPU oracle are fed the same
tensors from here, so the oracle never sees anything the CUDA path produced.

E4M3 codes come from torch's ``float8_e4m3fn`` cast (round to nearest even)
after clipping to the format's finite range [-448, 448], so nothing saturates
to NaN.  Scales are ``2**U(lo, hi)`` in FP32 (log-uniform).

Random streams: a ``torch.Generator`` seeded with the given seed on the device
the tensors are drawn on.  CPU and CUDA generators give different streams, so a
workload is identified by (seed, device); every check compares the two
implementations on the very same tensors.
"""
import math

import torch

E4M3_MAX = 448.0
KBLOCK = 128  # scale granularity along k
NBLOCK = 128  # scale granularity along n

# The five synthetic workloads, by name.
CONFIGS = {
    "dense_128x256x256": dict(kind="dense", m=128, n=256, k=256, dist="uniform4",
                              scale_exp=(-4.0, 2.0), out_dtype="bf16", seed=1001),
    # run once with K-major and once with MN-major scales
    "dense_4096x7168x2048": dict(kind="dense", m=4096, n=7168, k=2048, dist="normal",
                                 scale_exp=(-6.0, 0.0), out_dtype="bf16", seed=1002,
                                 scale_layouts=("K", "MN")),
    # the same GEMM with FP8 (E4M3) output and a per-tensor output scale; with
    # these inputs R has an RMS near 5.4, so R / s (RMS ~87) spans the E4M3
    # range and under 0.1% of the outputs saturate
    "dense_4096x7168x2048_e4m3out": dict(kind="dense", m=4096, n=7168, k=2048, dist="normal",
                                         scale_exp=(-6.0, 0.0), out_dtype="e4m3",
                                         output_scale=0.0625, seed=1007),
    "grouped_4096tok_top8_e64_n4096_k7168": dict(
        kind="grouped", num_tokens=4096, top_k=8, num_experts=64, n=4096, k=7168,
        scale_exp=(-6.0, 0.0), seed=1003),
    "masked_g32_maxm256_n4096_k7168": dict(
        kind="masked", num_groups=32, max_m=256, n=4096, k=7168, expected_m=128,
        scale_exp=(-6.0, 0.0), seed=1004),
    # the masked form at decode: a few tokens per expert (masked_m ~ U{0..16},
    # expected_m 8) in buffers of 256 rows; bound by streaming the weights
    "masked_g32_maxm256_n4096_k7168_decode": dict(
        kind="masked", num_groups=32, max_m=256, n=4096, k=7168, expected_m=8, masked_hi=16,
        scale_exp=(-6.0, 0.0), seed=1010),
    "dense_16384x18432x7168": dict(kind="dense", m=16384, n=18432, k=7168, dist="normal",
                                   scale_exp=(-6.0, 0.0), out_dtype="f16", seed=1005),
    # the producer of the GEMM's activations: 4096 tokens of hidden size 7168
    # (the k of the MoE workloads above)
    "norm_quant_4096x7168": dict(kind="norm", rows=4096, hidden=7168, eps=1e-6, seed=1006),
    # bmm_fp8: 4 batches of 4096 x 4096 x 7168, E4M3, tensorwise scales
    "bmm_fp8_b4_4096x4096x7168": dict(kind="bmm", batch=4, m=4096, n=4096, k=7168, seed=1009),
    # the DeepSeek FP8 block-scale MoE layer around the grouped GEMM: fc1 is the
    # grouped workload above (n = 2 * inter = 4096, k = hidden = 7168), fc2 has
    # n = 7168, k = 2048
    "moe_4096tok_top8_e64_h7168_i2048": dict(kind="moe", tokens=4096, top_k=8, num_experts=64,
                                             hidden=7168, inter=2048, scale_exp=(-7.0, -5.0),
                                             seed=1008),
}


def generator(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def to_e4m3_codes(x):
    """E4M3 codes (uint8) of float values: clip to +-448, cast RNE."""
    x = x.float().clamp_(-E4M3_MAX, E4M3_MAX)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def _draw(shape, dist, gen, device, chunk_rows=None):
    """E4M3 codes of `shape`, drawn row-chunk by row-chunk to bound memory."""
    out = torch.empty(shape, dtype=torch.uint8, device=device)
    flat = out.view(-1, shape[-1])
    rows = flat.shape[0]
    step = chunk_rows or max(1, (1 << 24) // max(1, shape[-1]))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        v = torch.empty((r1 - r0, shape[-1]), dtype=torch.float32, device=device)
        if dist == "normal":
            v.normal_(0.0, 1.0, generator=gen)
        elif dist == "uniform4":
            v.uniform_(-1.0, 1.0, generator=gen).mul_(4.0)
        else:
            raise ValueError(dist)
        flat[r0:r1] = to_e4m3_codes(v)
    return out


def log_uniform(shape, lo, hi, gen, device="cpu"):
    """FP32 values 2**U(lo, hi)."""
    u = torch.empty(shape, dtype=torch.float32, device=device)
    u.uniform_(lo, hi, generator=gen)
    return torch.exp2(u)


def dense(m, n, k, seed, dist="normal", scale_exp=(-6.0, 0.0), scale_major="K",
          device="cpu", output_scale=None, **_):
    """a (m,k), b (n,k) E4M3 codes; scales in the requested layout; with
    `output_scale`, also the one-element FP32 scale of an E4M3 output."""
    gen = generator(seed, device)
    kb, nb = k // KBLOCK, n // NBLOCK
    a = _draw((m, k), dist, gen, device)
    b = _draw((n, k), dist, gen, device)
    sa = log_uniform((m, kb), scale_exp[0], scale_exp[1], gen, device)
    sb = log_uniform((nb, kb), scale_exp[0], scale_exp[1], gen, device)
    if scale_major == "MN":
        sa, sb = sa.t().contiguous(), sb.t().contiguous()
    elif scale_major != "K":
        raise ValueError(scale_major)
    d = dict(a=a, b=b, a_scale=sa, b_scale=sb, m=m, n=n, k=k, scale_major=scale_major)
    if output_scale is not None:
        d["output_scale"] = torch.tensor([output_scale], dtype=torch.float32, device=device)
    return d


def routing_m_indices(num_tokens, top_k, num_experts, gen, align=128):
    """m_indices of the contiguous grouped layout for a top-k routing.

    Each token picks `top_k` distinct experts uniformly at random (multinomial
    without replacement).  Rows are grouped by expert in ascending order and
    each expert's segment is padded with -1 up to a multiple of `align` rows.
    """
    w = torch.ones((num_tokens, num_experts), dtype=torch.float32)
    choice = torch.multinomial(w, top_k, replacement=False, generator=gen)
    counts = torch.bincount(choice.flatten(), minlength=num_experts).tolist()
    parts = []
    for e, c in enumerate(counts):
        if c == 0:
            continue
        padded = int(math.ceil(c / align) * align)
        seg = torch.full((padded,), -1, dtype=torch.int32)
        seg[:c] = e
        parts.append(seg)
    if not parts:
        return torch.empty(0, dtype=torch.int32)
    return torch.cat(parts)


def grouped(num_tokens, top_k, num_experts, n, k, seed, scale_exp=(-6.0, 0.0),
            device="cpu", m_indices=None, **_):
    """Contiguous grouped MoE operands; padding rows of a hold random data too."""
    cpu_gen = generator(seed, "cpu")
    mi = m_indices if m_indices is not None else routing_m_indices(
        num_tokens, top_k, num_experts, cpu_gen)
    mi = mi.to(torch.int32)
    gen = generator(seed + 7919, device)
    m = mi.numel()
    kb, nb = k // KBLOCK, n // NBLOCK
    a = _draw((m, k), "normal", gen, device)
    b = _draw((num_experts, n, k), "normal", gen, device)
    sa = log_uniform((m, kb), scale_exp[0], scale_exp[1], gen, device)
    sb = log_uniform((num_experts, nb, kb), scale_exp[0], scale_exp[1], gen, device)
    return dict(a=a, b=b, a_scale=sa, b_scale=sb, m_indices=mi.to(device), m=m, n=n,
                k=k, num_groups=num_experts)


def masked(num_groups, max_m, n, k, seed, scale_exp=(-6.0, 0.0), expected_m=None,
           device="cpu", masked_m=None, masked_hi=None, **_):
    """Masked batched MoE operands; masked_m ~ U{0..masked_hi} (masked_hi =
    max_m unless given) unless masked_m is given."""
    cpu_gen = generator(seed, "cpu")
    hi = max_m if masked_hi is None else masked_hi
    mm = masked_m if masked_m is not None else torch.randint(
        0, hi + 1, (num_groups,), generator=cpu_gen, dtype=torch.int64)
    mm = mm.to(torch.int32)
    gen = generator(seed + 7919, device)
    kb, nb = k // KBLOCK, n // NBLOCK
    a = _draw((num_groups, max_m, k), "normal", gen, device)
    b = _draw((num_groups, n, k), "normal", gen, device)
    sa = log_uniform((num_groups, max_m, kb), scale_exp[0], scale_exp[1], gen, device)
    sb = log_uniform((num_groups, nb, kb), scale_exp[0], scale_exp[1], gen, device)
    return dict(a=a, b=b, a_scale=sa, b_scale=sb, masked_m=mm.to(device),
                num_groups=num_groups, max_m=max_m, n=n, k=k,
                expected_m=expected_m if expected_m is not None else max_m // 2)


def norm(rows, hidden, seed, eps=1e-6, device="cpu", **_):
    """Operands of fused_add_rmsnorm_fp8_block_quant: BF16 input and residual
    ~ N(0, 1), BF16 weight ~ 1 + N(0, 0.2^2) (RMSNorm gains near one)."""
    gen = generator(seed, device)
    x = torch.empty((rows, hidden), dtype=torch.float32, device=device)
    x.normal_(0.0, 1.0, generator=gen)
    inp = x.to(torch.bfloat16)
    x.normal_(0.0, 1.0, generator=gen)
    res = x.to(torch.bfloat16)
    w = torch.empty((hidden,), dtype=torch.float32, device=device)
    w.normal_(0.0, 0.2, generator=gen)
    return dict(input=inp, residual=res, weight=(w + 1.0).to(torch.bfloat16), rows=rows,
                hidden=hidden, eps=eps)


def moe(tokens, top_k, num_experts, hidden, inter, seed, scale_exp=(-7.0, -5.0), device="cpu",
        **_):
    """Operands of the DeepSeek FP8 block-scale MoE layer: BF16 input ~ N(0, 1);
    token_selected (tokens, top_k) int32, each token's distinct experts drawn
    uniformly without replacement; E4M3 fc1 (E, 2 inter, hidden) and fc2 (E,
    hidden, inter) ~ N(0, 1); 128 x 128 block scales 2**U(lo, hi)."""
    cpu_gen = generator(seed, "cpu")
    w = torch.ones((tokens, num_experts), dtype=torch.float32)
    ts = torch.multinomial(w, top_k, replacement=False, generator=cpu_gen).to(torch.int32)
    gen = generator(seed + 7919, device)
    x = torch.empty((tokens, hidden), dtype=torch.float32, device=device)
    x.normal_(0.0, 1.0, generator=gen)
    fc1 = _draw((num_experts, 2 * inter, hidden), "normal", gen, device)
    fc2 = _draw((num_experts, hidden, inter), "normal", gen, device)
    s1 = log_uniform((num_experts, 2 * inter // KBLOCK, hidden // KBLOCK), scale_exp[0],
                     scale_exp[1], gen, device)
    s2 = log_uniform((num_experts, hidden // KBLOCK, inter // KBLOCK), scale_exp[0],
                     scale_exp[1], gen, device)
    return dict(input=x.to(torch.bfloat16), token_selected=ts.to(device), fc1=fc1, fc2=fc2,
                fc1_scale=s1, fc2_scale=s2, tokens=tokens, top_k=top_k,
                num_experts=num_experts, hidden=hidden, inter=inter)


def bmm(batch, m, n, k, seed, a_fmt="e4m3", b_fmt="e4m3", device="cpu", **_):
    """Operands of bmm_fp8: A (batch, m, k) and B (batch, k, n) FP8 codes of
    N(0, 1) values (E4M3 or E5M2, as torch float8 tensors), one tensorwise FP32
    scale each (2**U(-6, 0))."""
    gen = generator(seed, device)
    dts = {"e4m3": (torch.float8_e4m3fn, 448.0), "e5m2": (torch.float8_e5m2, 57344.0)}
    out = {}
    for name, shape, fmt in (("A", (batch, m, k), a_fmt), ("B", (batch, k, n), b_fmt)):
        x = torch.empty(shape, dtype=torch.float32, device=device)
        x.normal_(0.0, 1.0, generator=gen)
        dt, lim = dts[fmt]
        out[name] = x.clamp_(-lim, lim).to(dt)
    out["A_scale"] = log_uniform((1,), -6.0, 0.0, gen, device)
    out["B_scale"] = log_uniform((1,), -6.0, 0.0, gen, device)
    out.update(batch=batch, m=m, n=n, k=k)
    return out


def make(name, device="cpu", **overrides):
    """Operands of one of the named workloads."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    kind = cfg.pop("kind")
    if kind == "dense":
        return dense(device=device, **cfg)
    if kind == "grouped":
        return grouped(device=device, **cfg)
    if kind == "masked":
        return masked(device=device, **cfg)
    if kind == "norm":
        return norm(device=device, **cfg)
    if kind == "moe":
        return moe(device=device, **cfg)
    if kind == "bmm":
        return bmm(device=device, **cfg)
    raise ValueError(kind)


def sample_positions(rows, cols, count, seed, extra_rows=()):
    """`count` seeded (row, col) positions plus every column of `extra_rows`."""
    gen = generator(seed, "cpu")
    r = torch.randint(0, rows, (count,), generator=gen, dtype=torch.int64)
    c = torch.randint(0, cols, (count,), generator=gen, dtype=torch.int64)
    for er in extra_rows:
        r = torch.cat([r, torch.full((cols,), int(er), dtype=torch.int64)])
        c = torch.cat([c, torch.arange(cols, dtype=torch.int64)])
    return r, c
