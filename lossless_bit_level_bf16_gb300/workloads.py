"""Seeded synthetic inputs shaped like the codecs' target workloads.

This module only draws random numbers and lays them out; it holds none of the
codecs' arithmetic, so the CUDA path and the CPU oracle can both be fed from
it.  The real tensors the page summaries measured on (LLM weights, gradients
and activations; GNN / DLRM embedding tables) are not available, so these
draws stand in for them:

* ``zc_gaussian``   bf16 N(0, sigma) vector (ZipCCL: activations, gradients and
  weights are near-Gaussian).
* ``zc_gradient``   bf16 gradient-like buffer: per-layer-block sigma log-uniform
  in [1e-4, 1e-2], 1 % exact zeros, 0.1 % outliers scaled x100.
* ``zc_moe``        bf16 [tokens x hidden] N(0, 1) rows routed to experts with
  seeded truncated-Zipf(s) counts; rows grouped by expert, one segment each.
* ``ibp_table``     fp32 embedding table N(0, std) clipped to +-clip, plus the
  seeded sample rows used to build the IBP metadata.
* ``ibp_gaussian``  fp32 N(0, std) weight tensor.

Values are drawn in fp32 with torch's seeded generator on the requested device
and rounded to bf16 by torch's round-to-nearest-even cast.  CPU and CUDA
generators give different draws for the same seed; a test always hands both
the CUDA path and the oracle the same bytes.
"""
from __future__ import annotations

import math

import torch


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def zc_gaussian(n, sigma=0.02, seed=0, device="cpu", mean=0.0):
    """bf16 [n] drawn from N(mean, sigma)."""
    g = _gen(device, seed)
    x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    return (x * sigma + mean).to(torch.bfloat16)


def zc_gradient(n_blocks=256, block=262144, seed=0, device="cpu",
                log_sigma=(-4.0, -2.0), p_zero=0.01, p_outlier=0.001, scale=100.0):
    """bf16 [n_blocks*block] plus segment offsets (one segment per block)."""
    g = _gen(device, seed)
    u = torch.rand(n_blocks, generator=g, device=device, dtype=torch.float64)
    sig = torch.pow(10.0, log_sigma[0] + (log_sigma[1] - log_sigma[0]) * u).to(torch.float32)
    x = torch.randn(n_blocks, block, generator=g, device=device, dtype=torch.float32)
    x.mul_(sig[:, None])
    zero = torch.rand(n_blocks, block, generator=g, device=device) < p_zero
    out = torch.rand(n_blocks, block, generator=g, device=device) < p_outlier
    x = torch.where(out & ~zero, x * scale, x)
    x = torch.where(zero, torch.zeros_like(x), x)
    seg = [i * block for i in range(n_blocks + 1)]
    return x.reshape(-1).to(torch.bfloat16), seg


def zipf_counts(n_tokens=8192, n_experts=64, s=1.1, seed=0):
    """Token counts per expert from a truncated Zipf(s) law over ranks 1..E
    (expert r has rank r); they sum to n_tokens and may be zero."""
    g = _gen("cpu", seed)
    r = torch.arange(1, n_experts + 1, dtype=torch.float64)
    p = r.pow(-s)
    p = p / p.sum()
    draws = torch.multinomial(p, n_tokens, replacement=True, generator=g)
    return torch.bincount(draws, minlength=n_experts).tolist()


def zc_moe(n_tokens=8192, hidden=8192, n_experts=64, s=1.1, seed=0, device="cpu"):
    """bf16 [n_tokens*hidden] (rows grouped by expert) plus segment offsets
    (one segment per expert, in elements) and the per-expert counts."""
    counts = zipf_counts(n_tokens, n_experts, s, seed)
    g = _gen(device, seed)
    x = torch.randn(n_tokens * hidden, generator=g, device=device, dtype=torch.float32)
    seg = [0]
    for c in counts:
        seg.append(seg[-1] + c * hidden)
    return x.to(torch.bfloat16), seg, counts


def ibp_table(rows=1_000_000, cols=128, std=0.1, clip=1.0, seed=0, device="cpu",
              n_samples=10_000, sample_seed=1):
    """fp32 [rows, cols] N(0, std) clipped to +-clip, and the indices of the
    seeded sample rows (min(n_samples, rows) of them, drawn without
    replacement with their own seed)."""
    g = _gen(device, seed)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    x.mul_(std).clamp_(-clip, clip)
    idx = sample_rows(rows, n_samples, sample_seed, device)
    return x, idx


def sample_rows(rows, n_samples=10_000, seed=1, device="cpu"):
    g = _gen("cpu", seed)
    k = min(int(n_samples), int(rows))
    return torch.randperm(rows, generator=g)[:k].to(device)


def ibp_gaussian(n_elems, std=0.02, seed=0, device="cpu"):
    g = _gen(device, seed)
    return torch.randn(n_elems, generator=g, device=device, dtype=torch.float32) * std


SWEEP_BYTES = [1 << (20 + 2 * i) for i in range(7)]  # 1 MiB .. 4 GiB, x4 steps


def describe():
    """The workloads by name, with their sizes (used by the benchmark)."""
    return {
        "zc_gaussian_1m": dict(n=1 << 20, sigma=0.02, chunk=4096),
        "zc_gradient_64m": dict(n=256 * 262144, blocks=256, chunk=4096),
        "zc_moe_8192x8192": dict(n=8192 * 8192, experts=64, zipf_s=1.1, chunk=4096),
        "ibp_table_1m_x128": dict(rows=1_000_000, cols=128, std=0.1, T=0.9, samples=10_000),
        "sweep_bytes": SWEEP_BYTES,
    }


def bf16_bits(t):
    """The uint16 bit patterns of a bf16 tensor, as a CPU numpy array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def f32_bytes(t):
    return t.detach().contiguous().cpu().numpy().view("uint8").reshape(-1)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("math", "torch")]
