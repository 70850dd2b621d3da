"""Helpers for the GPU-vs-oracle parity tests of the ZipCCL codec."""
from __future__ import annotations

import numpy as np

import oracle as O

U = 2.0 ** -24  # fp32 unit roundoff


def fields(u16):
    return (np.asarray(u16, np.uint16) >> 7) & 0xFF


def finite_values(u16):
    u16 = np.asarray(u16, np.uint16)
    fin = fields(u16) != 255
    return (u16[fin].astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _sum_abs(u16, step=1 << 24):
    """Sum of |x| over the finite values, in pieces (large inputs)."""
    tot = 0.0
    for i in range(0, len(u16), step):
        tot += float(np.abs(finite_values(u16[i:i + step])).sum())
    return tot


def check_plan(x_bits, seg_off, books_gpu, mu_gpu, sig_gpu, allow_near_ties=False, rel=8):
    """Codebook parity for a plan computed on the GPU.

    The GPU sums each thread's 16 values as an fp32 tree (error at most 4 ulp
    of the sum of magnitudes) before accumulating exactly, so its mean and
    sigma may differ from the oracle's fp64 sums by that much (rel = 8 units
    of fp32 rounding allowed; the encoder's fused sums of zc_compress_fit add
    eight values per fp32 chain and then two levels, rel = 12).  Given the
    GPU's own (mu, sigma), the oracle's predictor must give the GPU's book
    exactly.  The oracle's book from its own statistics must agree too.  Only
    where the caller builds near-ties on purpose (allow_near_ties) may it
    differ, and then only inside the band those statistics' error allows:
    every field that one book has and the other lacks must carry, at the
    oracle's (mu, sigma), a mass within 1e-5 (relative) of the masses the
    other book has in its place.  Returns the number of such segments.
    """
    nseg = len(books_gpu)
    seg = [0, len(x_bits)] if seg_off is None else list(seg_off)
    near_ties = 0
    for s in range(nseg):
        xs = x_bits[seg[s]:seg[s + 1]]
        cnt, s1, s2 = O.zc_stats(xs)
        mu_o, sg_o = O.zc_moments(cnt, s1, s2)
        if cnt:
            mean_abs = _sum_abs(xs) / cnt
            ex2 = s2 / cnt
        else:
            mean_abs = ex2 = 0.0
        tol_mu = rel * U * mean_abs + 1e-300
        assert abs(mu_gpu[s] - mu_o) <= tol_mu, (s, mu_gpu[s], mu_o)
        # groups whose squares could underflow fp32 are summed in fp64 on the
        # GPU, so the only absolute term left is the fp32 subnormal spacing of
        # the squares of a group kept in fp32 (2^-150 each)
        tol_var = rel * U * ex2 + 2 * abs(mu_o) * tol_mu + 2.0 ** -140
        assert abs(sig_gpu[s] ** 2 - sg_o ** 2) <= tol_var, (s, sig_gpu[s], sg_o)
        b_from_gpu_stats = O.zc_predict(float(mu_gpu[s]), float(sig_gpu[s]))
        assert np.array_equal(b_from_gpu_stats, books_gpu[s]), (s, b_from_gpu_stats, books_gpu[s])
        b_own = O.zc_predict(mu_o, sg_o)
        if not np.array_equal(b_own, books_gpu[s]):
            assert allow_near_ties, (s, b_own, books_gpu[s], mu_o, sg_o)
            only_gpu = sorted(set(int(f) for f in books_gpu[s]) - set(int(f) for f in b_own))
            only_own = sorted(set(int(f) for f in b_own) - set(int(f) for f in books_gpu[s]))
            for a in only_gpu:
                for b in only_own:
                    ma, mb = O.zc_mass(mu_o, sg_o, a), O.zc_mass(mu_o, sg_o, b)
                    assert abs(ma - mb) <= 1e-5 * max(ma, mb), (s, a, b, ma, mb)
            near_ties += 1
    return near_ties


def check_stream_equal(stream_gpu, x_bits, seg_off, chunk, books):
    """The GPU stream must equal, byte for byte, the oracle's stream for the
    same input and codebooks."""
    st, _, _, _ = O.zc_encode(x_bits, seg_off=seg_off, chunk_elems=chunk,
                              books=np.asarray(books, np.uint8).reshape(-1))
    assert stream_gpu.size == st.size, (stream_gpu.size, st.size)
    diff = np.nonzero(stream_gpu != st)[0]
    assert diff.size == 0, f"{diff.size} bytes differ, first at {diff[:10]} of {st.size}"
    return st
