"""The seeded synthetic inputs match the recipes they stand for (CPU, small
sizes): same seed, same bytes; the stated distributions, fractions, segment
layouts and sample draws."""
import math

import numpy as np
import torch

from lossless_bit_level_bf16_gb300 import workloads as W


def test_gaussian_is_seeded_and_has_its_sigma():
    a = W.zc_gaussian(1 << 18, sigma=0.02, seed=3)
    b = W.zc_gaussian(1 << 18, sigma=0.02, seed=3)
    c = W.zc_gaussian(1 << 18, sigma=0.02, seed=4)
    assert a.dtype == torch.bfloat16 and torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
    x = a.float()
    assert abs(x.mean().item()) < 2e-4
    assert abs(x.std().item() / 0.02 - 1) < 0.01


def test_gradient_blocks_follow_the_recipe():
    nb, blk = 64, 65536
    x, seg = W.zc_gradient(n_blocks=nb, block=blk, seed=0)
    assert x.dtype == torch.bfloat16 and x.numel() == nb * blk
    assert seg == [i * blk for i in range(nb + 1)]
    v = x.float().view(nb, blk)
    zero = (v == 0).double().mean().item()
    assert abs(zero - 0.01) < 0.001  # 1 % exact zeros (a N(0, s) draw is never 0 in bf16 here)
    # per block: the bulk's sigma lies in [1e-4, 1e-2]; outliers are 100x the block's values
    med = v.abs().median(dim=1).values  # median |x| of N(0, s) is 0.674 s
    s_est = med / 0.6745
    assert s_est.min().item() > 1e-4 * 0.9 and s_est.max().item() < 1e-2 * 1.1
    big = (v.abs() > 8 * s_est[:, None]).double().mean().item()
    assert 0.0005 < big < 0.0015  # about 0.1 % outliers (x100), N(0,1) tails beyond 8 are nil


def test_zipf_counts_and_moe_segments():
    counts = W.zipf_counts(n_tokens=8192, n_experts=64, s=1.1, seed=0)
    assert len(counts) == 64 and sum(counts) == 8192
    assert counts == W.zipf_counts(n_tokens=8192, n_experts=64, s=1.1, seed=0)
    # rank 1 takes the largest share: p1 = 1 / H(64, 1.1)
    h = sum(r ** -1.1 for r in range(1, 65))
    assert abs(counts[0] / 8192 - 1 / h) < 0.02
    assert counts[0] > counts[10] > counts[50]
    x, seg, c2 = W.zc_moe(n_tokens=512, hidden=64, n_experts=16, s=1.1, seed=0)
    assert x.numel() == 512 * 64 and seg[0] == 0 and seg[-1] == x.numel()
    assert [seg[i + 1] - seg[i] for i in range(16)] == [c * 64 for c in c2]


def test_table_is_clipped_and_its_samples_distinct():
    t, idx = W.ibp_table(rows=20_000, cols=128, std=0.1, clip=1.0, seed=0, n_samples=10_000)
    assert t.shape == (20_000, 128) and t.dtype == torch.float32
    assert t.abs().max().item() <= 1.0
    assert abs(t.std().item() / 0.1 - 1) < 0.01
    assert idx.numel() == 10_000 and torch.unique(idx).numel() == 10_000
    assert int(idx.min()) >= 0 and int(idx.max()) < 20_000
    t2, idx2 = W.ibp_table(rows=20_000, cols=128, seed=0, n_samples=10_000)
    assert torch.equal(t, t2) and torch.equal(idx, idx2)
    _, few = W.ibp_table(rows=100, cols=4, n_samples=10_000)
    assert few.numel() == 100  # never more samples than rows


def test_sweep_sizes_and_byte_views():
    assert W.SWEEP_BYTES == [1 << 20, 1 << 22, 1 << 24, 1 << 26, 1 << 28, 1 << 30, 1 << 32]
    x = W.zc_gaussian(8, seed=1)
    b = W.bf16_bits(x)
    assert b.dtype == np.uint16 and b.size == 8
    assert np.array_equal(b, x.view(torch.int16).numpy().view(np.uint16))
    f = W.ibp_gaussian(4, seed=2)
    assert W.f32_bytes(f).size == 16
    assert math.isclose(float(np.frombuffer(W.f32_bytes(f).tobytes(), np.float32)[0]), float(f[0]))
