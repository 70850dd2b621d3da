// zc_plan.cu -- ZipCCL codebook prediction on the GPU.
//
// [ZipCCL] = "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", 2. Metodologia A: the top-7
// bf16 exponents of a near-Gaussian tensor follow from its standard
// deviation, so the exponent lookup table is computed in closed form instead
// of from a histogram or a sort.
//
// Two kernels:
//   zc_stats_kernel    one warp per statistics unit (U elements inside one
//                      segment): count, sum and sum of squares of the finite
//                      values.  HBM-bound: 2 bytes read per element.
//   zc_predict_kernel  K blocks per segment add fixed ranges of the unit
//                      partials; the segment's last block adds their totals
//                      in a fixed order, forms mu and sigma, evaluates the Gaussian
//                      mass of the exponent fields and keeps the 7 largest.
//                      fp64 is slow on this part, so each field edge's erfc
//                      ranking is done in fp32 unless the 7th and 8th masses
//                      are too close for fp32 to tell apart; then each field
//                      edge's erfc pair is computed once in fp64, only around
//                      the distribution's scale when bounds show that no
//                      other field can be among the 7, and the masses are
//                      ranked as integers (their fp64 bit patterns).
//
// Arithmetic of the statistics pass: the 16 values a thread holds are summed
// (and their squares, exact in fp32 for bf16 inputs) with four fp32
// additions on every value's path, run as packed fp32x2 operations on the
// pairs of values that share a word (error at most 4 units in the last place
// of the sum of magnitudes, as for a 16-leaf tree), the group sums
// are accumulated as unevaluated fp32 pairs (error-free two-sum), the pairs
// of a unit's lanes are added as pairs too, and only the unit's total is
// formed in fp64 (an fp64 tree when a pair overflows fp32).  A
// group of 16 whose fp32 sums are not finite (an inf/NaN input or an fp32
// overflow), or whose squares may have underflowed (sum of squares below
// 2^-96 with a nonzero value), is redone element by element in fp64,
// skipping non-finite values.  The whole pass is deterministic for a given
// plan: the partition into units and every reduction order are fixed.
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace lbb {
namespace {

#ifndef LBB_STAT_BATCH
#define LBB_STAT_BATCH 2
#endif
constexpr int kStatBatch = LBB_STAT_BATCH;  // groups loaded before summing


__device__ __forceinline__ int find_unit_segment(const ZcSegDev* segs, uint32_t nseg,
                                                 unsigned long long unit) {
  // largest s with unit_start[s] <= unit
  int lo = 0, hi = (int)nseg - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (segs[mid].unit_start <= unit) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// One warp per statistics unit; warp w of the grid takes a contiguous range
// of units, the same number (to one) as every other warp, and follows the
// segments along it after one search.  A step is 512 values: lane l takes 8
// at base + 8l and 8 at base + 256 + 8l, so each 16-byte load instruction of
// the warp reads 512 contiguous bytes; kStatBatch steps are loaded before any
// is summed.  No block barriers: a warp's loads overlap other warps' sums.
// The lanes' sums are added as fp32 (sum, error) pairs in a fixed tree order
// and only the unit's total goes to fp64 (fp64 is slow on this part); a pair
// that overflows fp32, or values already summed in fp64, take an fp64 tree of
// the same shape.  A unit's sums do not depend on which warp computes them:
// the partition into units and every order of addition depend only on the
// plan.
constexpr int kStatWarps = kThreads / 32;


// The warp's loads run ahead of its sums through a ring of kStatRing batches
// in shared memory (cp.async: each lane copies the 16-byte pieces it will sum
// itself, so the warp needs no synchronization), over its whole range of
// units.  Batches of 2 KB (two steps) in a 3-slot ring: 6 KB per warp, three
// blocks per SM.  Units of a segment that does not start 16-byte aligned, and the
// pieces at a unit's ragged end, are read with per-element loads when summed.
constexpr int kStatRing = 3;
constexpr uint32_t kStatSlotVecs = kStatBatch * 2 * 32;  // 16-byte pieces per batch
constexpr size_t kStatSmem = (size_t)kStatWarps * kStatRing * kStatSlotVecs * 16;

// red_cnt (not null when the predictor takes several blocks per segment):
// the predictor's per-segment block counters, zeroed here by block 0 (the
// predictor reads them only once this kernel has finished).
__global__ void __launch_bounds__(kThreads, 3) zc_stats_kernel(
    const uint16_t* __restrict__ x, const ZcSegDev* __restrict__ segs, uint32_t nseg,
    uint32_t U, unsigned long long nunits, StatPartial* __restrict__ parts, int x_al16,
    uint32_t* red_cnt) {
  extern __shared__ uint4 s_ring[];
  const int lane = threadIdx.x & 31;
  if (red_cnt && blockIdx.x == 0)
    for (uint32_t i = threadIdx.x; i < nseg; i += blockDim.x) red_cnt[i] = 0;
  uint4* ring = s_ring + (size_t)(threadIdx.x >> 5) * kStatRing * kStatSlotVecs;
  grid_dep_launch();  // the predictor may be scheduled as blocks finish
  unsigned long long ub;
  uint32_t nu;  // this warp's units: ub .. ub + nu - 1
  {
    const unsigned long long nwarps = (unsigned long long)gridDim.x * kStatWarps;
    const unsigned long long gw = (unsigned long long)blockIdx.x * kStatWarps + (threadIdx.x >> 5);
    const unsigned long long q = nunits / nwarps, r = nunits % nwarps;
    ub = gw * q + (gw < r ? gw : r);
    nu = (uint32_t)(q + (gw < r ? 1 : 0));
  }
  // A position in the warp's sequence of (unit, batch): the unit's element
  // range, whether it is 16-byte aligned, and the batch's first element.
  struct Cursor {
    uint32_t k;
    int sc;  // lane 0: segment of unit k
    unsigned long long lo, hi, base;
    int al;
  };
  auto load_unit = [&](Cursor& c) {  // the whole warp
    const unsigned long long unit = ub + c.k;
    unsigned long long lo = 0, hi = 0;
    int al = 0;
    if (lane == 0) {
      if (c.sc < 0) c.sc = find_unit_segment(segs, nseg, unit);
      while (c.sc + 1 < (int)nseg && segs[c.sc + 1].unit_start <= unit) ++c.sc;
      const int sg = c.sc;
      lo = segs[sg].elem_start + (unit - segs[sg].unit_start) * U;
      const unsigned long long e = segs[sg].elem_start + segs[sg].nelem;
      hi = (lo + U < e) ? lo + U : e;
      al = x_al16 && ((segs[sg].elem_start & 7ull) == 0);
    }
    c.lo = __shfl_sync(kFull, lo, 0);
    c.hi = __shfl_sync(kFull, hi, 0);
    c.al = __shfl_sync(kFull, al, 0);
    c.base = c.lo;
  };
  auto advance = [&](Cursor& c) -> bool {  // to the next batch; false past the last
    c.base += kStatBatch * 512ull;
    if (c.base < c.hi) return true;
    if (++c.k >= nu) return false;
    load_unit(c);
    return true;
  };
  auto issue = [&](const Cursor& c, int slot) {
    if (!c.al) return;
    if (c.hi - c.base >= kStatBatch * 512ull) {  // the whole batch: no test per piece
      uint4* dst = ring + (size_t)slot * kStatSlotVecs + lane;
      const uint16_t* src = x + c.base + 8ull * lane;
#pragma unroll
      for (int p = 0; p < 2 * kStatBatch; ++p) cp_async16(dst + 32 * p, src + 256 * p);
      return;
    }
#pragma unroll
    for (int g = 0; g < kStatBatch; ++g)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const unsigned long long e0 = c.base + g * 512ull + 256ull * h + 8ull * lane;
        if (e0 + 8 <= c.hi)
          cp_async16(ring + (size_t)slot * kStatSlotVecs + (2 * g + h) * 32 + lane, x + e0);
      }
  };

  Cursor ci{0, -1, 0, 0, 0, 0};
  bool more = nu > 0;  // the issue cursor has a batch
  if (more) load_unit(ci);
  Cursor cc = ci;      // the sum cursor, kStatRing - 1 batches behind
  int islot = 0, cslot = 0;
#pragma unroll
  for (int p = 0; p < kStatRing - 1; ++p) {
    if (more) {
      issue(ci, islot);
      more = advance(ci);
    }
    cp_async_commit();
    islot = islot + 1 == kStatRing ? 0 : islot + 1;
  }
  float hx = 0.f, lx = 0.f, hq = 0.f, lq = 0.f;
  double dx = 0.0, dq = 0.0;
  unsigned long long cnt = 0;
  bool have = nu > 0;  // the sum cursor has a batch
  while (have) {
    if (more) {
      issue(ci, islot);
      more = advance(ci);
    }
    cp_async_commit();
    islot = islot + 1 == kStatRing ? 0 : islot + 1;
    cp_async_wait_group<kStatRing - 1>();  // this lane's pieces of the batch
    // The batch, compiled twice: FULL (the unit is 16-byte aligned and the
    // batch lies wholly inside it, every piece in the ring: no test per
    // piece) and the general form (pieces past the unit's end count 0
    // values, pieces of an unaligned unit are read one value at a time).
    auto batch = [&](auto full_tag) {
      constexpr bool FULL = decltype(full_tag)::value;
      uint32_t w[kStatBatch][8];
      int vh[kStatBatch][2];
#pragma unroll
      for (int g = 0; g < kStatBatch; ++g) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const unsigned long long e0 = cc.base + g * 512ull + 256ull * h + 8ull * lane;
          int v = 8;
          if (!FULL) {
            const unsigned long long rem = e0 < cc.hi ? cc.hi - e0 : 0ull;
            v = rem < 8 ? (int)rem : 8;
          }
          vh[g][h] = v;
          if (FULL || (v == 8 && cc.al)) {
            const uint4 a4 = ring[(size_t)cslot * kStatSlotVecs + (2 * g + h) * 32 + lane];
            w[g][4 * h] = a4.x; w[g][4 * h + 1] = a4.y; w[g][4 * h + 2] = a4.z; w[g][4 * h + 3] = a4.w;
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t l = (2 * j < v) ? (uint32_t)__ldg(x + e0 + 2 * j) : 0u;
              const uint32_t hh = (2 * j + 1 < v) ? (uint32_t)__ldg(x + e0 + 2 * j + 1) : 0u;
              w[g][4 * h + j] = l | (hh << 16);
            }
          }
        }
      }
#pragma unroll
      for (int g = 0; g < kStatBatch; ++g) {
        const int valid = FULL ? 16 : vh[g][0] + vh[g][1];
        if (!FULL && valid == 0) continue;
        // word j's two values as one fp32x2 pair; pairs j and j + 4 are added
        // first, then the four sums in a tree, then the pair's two halves:
        // every value goes through four additions, as in a 16-leaf tree
        unsigned long long p1[4], p2[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const unsigned long long a = f2_pack(bf16_lo(w[g][j]), bf16_hi(w[g][j]));
          const unsigned long long b = f2_pack(bf16_lo(w[g][j + 4]), bf16_hi(w[g][j + 4]));
          p1[j] = f2_add(a, b);
          p2[j] = f2_fma(b, b, f2_mul(a, a));  // squares exact (bf16), one rounding each add
        }
        p1[0] = f2_add(f2_add(p1[0], p1[1]), f2_add(p1[2], p1[3]));
        p2[0] = f2_add(f2_add(p2[0], p2[1]), f2_add(p2[2], p2[3]));
        const float2 h1 = f2_unpack(p1[0]), h2 = f2_unpack(p2[0]);
        const float sv = __fadd_rn(h1.x, h1.y), sq = __fadd_rn(h2.x, h2.y);
        // Squares below 2^-126 lose bits in fp32 (below 2^-149 they vanish):
        // when the group's sum of squares is under 2^-96 and a value is not
        // zero, the loss could exceed the fp32 rounding bound, so the group
        // goes to fp64 like a non-finite one.
        bool fast = isfinite(sv) && isfinite(sq);
        if (fast && sq < 0x1p-96f) {
          uint32_t nz = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) nz |= w[g][j] & 0x7FFF7FFFu;
          fast = nz == 0;
        }
        if (fast) {
          two_sum_acc(hx, lx, sv);
          two_sum_acc(hq, lq, sq);
          cnt += (unsigned long long)valid;
        } else {
          // an inf/NaN input, an fp32 overflow or underflow: redo these
          // values in fp64
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint32_t bits = (j & 1) ? (w[g][j >> 1] >> 16) : (w[g][j >> 1] & 0xFFFFu);
            if ((j & 7) < vh[g][j >> 3] && ((bits >> 7) & 0xFFu) != 0xFFu) {
              const double d = (double)__uint_as_float(bits << 16);
              dx = __dadd_rn(dx, d);
              dq = __dadd_rn(dq, __dmul_rn(d, d));
              cnt += 1;
            }
          }
        }
      }
    };
    if (cc.al && cc.hi - cc.base >= kStatBatch * 512ull) batch(std::true_type{});
    else batch(std::false_type{});
    cslot = cslot + 1 == kStatRing ? 0 : cslot + 1;
    if (cc.base + kStatBatch * 512ull >= cc.hi) {
      // the unit's last batch: lanes' fp32 pairs, fp64 if a pair overflows or
      // fp64 sums exist
      float ax = hx, bx = lx, aq = hq, bq = lq;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ax2 = __shfl_down_sync(kFull, ax, o), bx2 = __shfl_down_sync(kFull, bx, o);
        const float aq2 = __shfl_down_sync(kFull, aq, o), bq2 = __shfl_down_sync(kFull, bq, o);
        pair_add(ax, bx, ax2, bx2);
        pair_add(aq, bq, aq2, bq2);
        cnt += __shfl_down_sync(kFull, cnt, o);
      }
      const bool fin = __shfl_sync(kFull, isfinite(ax) && isfinite(bx) && isfinite(aq) && isfinite(bq), 0);
      double t1, t2;
      if (!fin || __any_sync(kFull, dx != 0.0 || dq != 0.0)) {
        t1 = __dadd_rn(__dadd_rn((double)hx, (double)lx), dx);
        t2 = __dadd_rn(__dadd_rn((double)hq, (double)lq), dq);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          t1 = __dadd_rn(t1, __shfl_down_sync(kFull, t1, o));
          t2 = __dadd_rn(t2, __shfl_down_sync(kFull, t2, o));
        }
      } else {
        t1 = __dadd_rn((double)ax, (double)bx);
        t2 = __dadd_rn((double)aq, (double)bq);
      }
      if (lane == 0) {
        const unsigned long long unit = ub + cc.k;
        parts[unit].cnt = cnt;
        parts[unit].s1 = t1;
        parts[unit].s2 = t2;
      }
      hx = lx = hq = lq = 0.f;
      dx = dq = 0.0;
      cnt = 0;
    }
    have = advance(cc);
  }
  cp_async_wait_all();
}

// Gaussian mass of exponent field f, P(2^(f-127) <= |X| < 2^(f-126)) for
// X ~ N(mu, sigma), is a difference of complementary error functions at the
// field's two edges, for both signs.  Field f's upper edge is field f+1's
// lower edge, so the erfc terms are evaluated once per edge e = 2^(k-127),
// k = 1..255:  em = erfc((e - mu)/s),  ep = erfc((e + mu)/s),  s = sigma*sqrt(2).
// fp64, every operation rounded on its own (no fused multiply-add), so the
// result does not depend on contraction.
__device__ void edge_erfc(double mu, double sigma, int k, double* em, double* ep) {
  const double e = ldexp(1.0, k - 127);
  const double s = __dmul_rn(sigma, 1.4142135623730951);  // sigma * sqrt(2)
  *em = erfc(__ddiv_rn(__dsub_rn(e, mu), s));
  *ep = erfc(__ddiv_rn(__dadd_rn(e, mu), s));
}

// mass(f) from the edge terms of edges f and f+1; masses below 1e-300 read as 0.
__device__ double field_mass(const double* em, const double* ep, int f) {
  const double pos = __dmul_rn(0.5, __dsub_rn(em[f], em[f + 1]));
  const double neg = __dmul_rn(0.5, __dsub_rn(ep[f], ep[f + 1]));
  double m = __dadd_rn(pos, neg);
  if (!(m >= 1e-300)) m = 0.0;
  return m;
}

__device__ int field_of(double v) {
  double a = fabs(v);
  if (a == 0.0 || a < 1.1754943508222875e-38 /* 2^-126 */) return 0;
  int ex;
  (void)frexp(a, &ex);
  int f = ex + 126;
  return f > 254 ? 254 : (f < 0 ? 0 : f);
}

// parts: one partial per statistics unit (by_chunk = 0, after zc_stats_kernel)
// or per chunk (by_chunk = 1, after the encoder that also sums).
// K blocks per segment (block k of segment s is block s * K + k): block k
// adds the fixed range k of the segment's partials; with K > 1 it files its
// totals and the segment's last block to finish (a counter per segment,
// zeroed by the kernel that wrote the partials) adds the K totals with the same fixed tree
// as a range of partials and goes on with the codebook.  The sums depend
// only on the plan, not on which block is last.
__global__ void __launch_bounds__(kThreads) zc_predict_kernel(
    ZcSegDev* __restrict__ segs, uint32_t nseg, unsigned long long nunits,
    const StatPartial* __restrict__ parts, int by_chunk, uint32_t K, StatPartial* red,
    uint32_t* cnt) {
  __shared__ double s_r1[kThreads / 32], s_r2[kThreads / 32];
  __shared__ unsigned long long s_rc[kThreads / 32];
  __shared__ double s_mu, s_sigma;
  __shared__ double s_em[256], s_ep[256];
  __shared__ unsigned long long s_key[256];
  __shared__ int s_take[256];
  __shared__ double s_m7, s_hb, s_is;
  __shared__ int s_ok;
  __shared__ float s_emf[256], s_epf[256], s_m7f, s_m8f;
  __shared__ uint32_t s_keyf[256];
  __shared__ int s_lastblk;
  __shared__ unsigned char s_book[8];
  const int t = threadIdx.x;
  const uint32_t sg = blockIdx.x / K, kb = blockIdx.x % K;
  // the segment's range of partials (fields fixed when the plan was made)
  const unsigned long long s0 = by_chunk ? segs[sg].chunk_start : segs[sg].unit_start;
  const unsigned long long s1e = by_chunk ? s0 + segs[sg].nchunks
                                          : ((sg + 1 < nseg) ? segs[sg + 1].unit_start : nunits);
  grid_dep_wait();  // the statistics partials
  const unsigned long long per = (s1e - s0 + K - 1) / K;
  const unsigned long long u0 = s0 + per * kb < s1e ? s0 + per * kb : s1e;
  const unsigned long long u1 = u0 + per < s1e ? u0 + per : s1e;
  // The block's sum of partials lo .. hi - 1: thread t adds lo + t,
  // lo + t + 256, ... in index order, then a fixed shuffle tree per warp and
  // the 8 warp sums in order; thread 0 gets the totals.
  auto block_sum = [&](const StatPartial* p, unsigned long long lo, unsigned long long hi,
                       double* r1, double* r2, unsigned long long* rc) {
    double a = 0.0, b = 0.0;
    unsigned long long c = 0;
#pragma unroll 4
    for (unsigned long long u = lo + t; u < hi; u += kThreads) {
      a = __dadd_rn(a, __ldcg(&p[u].s1));
      b = __dadd_rn(b, __ldcg(&p[u].s2));
      c += __ldcg(&p[u].cnt);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a = __dadd_rn(a, __shfl_down_sync(kFull, a, o));
      b = __dadd_rn(b, __shfl_down_sync(kFull, b, o));
      c += __shfl_down_sync(kFull, c, o);
    }
    if ((t & 31) == 0) {
      s_r1[t >> 5] = a;
      s_r2[t >> 5] = b;
      s_rc[t >> 5] = c;
    }
    __syncthreads();
    if (t == 0) {
      double s1 = 0.0, s2 = 0.0;
      unsigned long long n = 0;
      for (int w = 0; w < kThreads / 32; ++w) {
        s1 = __dadd_rn(s1, s_r1[w]);
        s2 = __dadd_rn(s2, s_r2[w]);
        n += s_rc[w];
      }
      *r1 = s1;
      *r2 = s2;
      *rc = n;
    }
  };
  double s1 = 0.0, s2 = 0.0;
  unsigned long long n = 0;
  block_sum(parts, u0, u1, &s1, &s2, &n);
  if (t == 0) {
    s_lastblk = 1;
    if (K > 1) {
      StatPartial& mine = red[(unsigned long long)sg * K + kb];
      mine.cnt = n;
      mine.s1 = s1;
      mine.s2 = s2;
      __threadfence();
      s_lastblk = atomicAdd(cnt + sg, 1u) == K - 1;
    }
  }
  __syncthreads();
  if (!s_lastblk) return;  // another block of the segment finishes it
  if (K > 1) {
    // the segment's K block totals, read from L2 by the whole block and
    // added in the same fixed order whichever block is last
    __threadfence();
    block_sum(red + (unsigned long long)sg * K, 0, K, &s1, &s2, &n);
  }
  if (t == 0) {
    double mu = 0.0, sigma = 0.0;
    if (n) {
      mu = __ddiv_rn(s1, (double)n);
      double var = __dsub_rn(__ddiv_rn(s2, (double)n), __dmul_rn(mu, mu));
      sigma = var > 0.0 ? __dsqrt_rn(var) : 0.0;
    }
    s_mu = mu;
    s_sigma = sigma;
    s_is = sigma > 0.0 ? __drcp_rn(__dmul_rn(sigma, 1.4142135623730951)) : 0.0;  // 1/(sigma sqrt 2)
  }
  __syncthreads();
  const double mu = s_mu, sigma = s_sigma;
  // the codebook is built in s_book, then written with the segment's
  // classification table (publish_book)
  static_assert(kThreads == 256, "one thread per table entry");
  auto publish_book = [&]() {
    __syncthreads();
    if (t < 8) segs[sg].book[t] = s_book[t];
    zc_seg_luts(segs, nseg)[256u * sg + (uint32_t)t] = zc_lut_entry(s_book, (uint32_t)t);
    if (t == 0) {
      segs[sg].mu = mu;
      segs[sg].sigma = sigma;
    }
  };
  if (!(sigma > 0.0)) {
    if (t == 0) {
      int lo = field_of(mu) - 3;
      lo = lo < 0 ? 0 : (lo > 248 ? 248 : lo);
      for (int j = 0; j < 7; ++j) s_book[j] = (unsigned char)(lo + j);
      s_book[7] = 0;
    }
    publish_book();
    return;
  }
  // Fast ranking in fp32.  Edge terms with erfcf of the fp64 argument rounded
  // to fp32: each term is within EPS_TERM = 1e-6 of the exact erfc (erfcf's
  // error of a few units of 2^-23 on values <= 2, plus the argument's
  // rounding, which moves erfc by at most 2^-24 max|x erfc'(x)| < 3e-8), so
  // every fp32 mass (half the sum of two differences, each rounded once) is
  // within 2.5e-6 of the exact mass.  Taking a margin of 1e-5 per mass: when
  // the 7th largest fp32 mass exceeds the 8th by more than 2e-5, the 7 fields
  // whose exact masses are largest are the fp32 top 7, whatever the rounding
  // of an fp64 evaluation; the book is their set, in ascending order.
  if (t >= 1 && t <= 255) {
    const double e = __longlong_as_double((long long)(t - 127 + 1023) << 52), is = s_is;  // 2^(t-127)
    s_emf[t] = erfcf((float)__dmul_rn(__dsub_rn(e, mu), is));
    s_epf[t] = erfcf((float)__dmul_rn(__dadd_rn(e, mu), is));
  }
  __syncthreads();
  {
    float mf = 0.f;
    if (t >= 1 && t <= 254) {
      mf = 0.5f * (s_emf[t] - s_emf[t + 1]) + 0.5f * (s_epf[t] - s_epf[t + 1]);
      if (!(mf > 0.f)) mf = 0.f;
    }
    s_keyf[t] = __float_as_uint(mf);  // non-negative floats order like their bits
  }
  __syncthreads();
  if (t < 32) {
    // The 8 largest masses of fields 1..254 (ties to the lower field) by
    // eight rounds of a warp argmax, lane l holding fields 8l .. 8l + 7: the
    // first 7 are taken, the 7th and 8th masses decide the margin.
    const int f0 = 8 * t;
    uint32_t taken = 0;
    for (int r = 0; r < 8; ++r) {
      unsigned long long best = 0;  // (mass bits << 32) | (255 - field); 0 = none
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int f = f0 + i;
        if (f >= 1 && f <= 254 && !((taken >> i) & 1u)) {
          const unsigned long long cand = ((unsigned long long)s_keyf[f] << 32) | (unsigned)(255 - f);
          best = cand > best ? cand : best;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long y = __shfl_xor_sync(kFull, best, o);
        best = y > best ? y : best;
      }
      const int fs = 255 - (int)(best & 0xFFFFFFFFull);
      if (r < 7 && fs >= f0 && fs < f0 + 8) taken |= 1u << (fs - f0);
      if (t == 0 && r == 6) s_m7f = __uint_as_float((uint32_t)(best >> 32));
      if (t == 0 && r == 7) s_m8f = __uint_as_float((uint32_t)(best >> 32));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) s_take[f0 + i] = (taken >> i) & 1u;
  }
  __syncthreads();
  if (!(s_m7f - s_m8f > 2e-5f)) {
    // A near-tie at the 7th place: rank the exact fp64 masses.
    // The 7 largest masses among fields lo..hi (edge terms of edges lo..hi+1,
    // one edge per thread); s_take marks them, s_m7 gets the 7th largest.
    // Masses are finite and >= 0 (+0 below the cut-off), so their fp64 bit
    // patterns order like the values: the ranking compares 64-bit integers.
    auto rank_fields = [&](int lo, int hi) {
      if (t >= lo && t <= hi + 1) edge_erfc(mu, sigma, t, &s_em[t], &s_ep[t]);
      __syncthreads();
      s_key[t] = (t >= lo && t <= hi)
                     ? (unsigned long long)__double_as_longlong(field_mass(s_em, s_ep, t))
                     : 0ull;
      __syncthreads();
      int rank = 256;
      if (t >= lo && t <= hi) {
        const unsigned long long m = s_key[t];
        rank = 0;
        for (int g = lo; g <= hi; ++g) {
          const unsigned long long mg = s_key[g];
          rank += (mg > m || (mg == m && g < t)) ? 1 : 0;
        }
      }
      s_take[t] = rank < 7;
      if (rank == 6) s_m7 = __longlong_as_double((long long)s_key[t]);
      __syncthreads();
    };
    // First only a window of fields around the field of max(sigma, |mu|),
    // where the largest masses lie.  Every field below the window has mass at
    // most its width times the largest density of |X|, 2^(lo-128) * 2/(sigma
    // sqrt(2 pi)); every field above it at most P(|X| >= 2^(hi-126)) <=
    // erfc((2^(hi-126) - |mu|)/s).  When both bounds (plus 1e-15 for the
    // rounding of a mass computed as a difference of erfc values near 1) are
    // under half the window's 7th largest mass, no field outside the window
    // can be among the 7 largest, whichever way the masses are rounded, and
    // the window's 7 are the answer; otherwise all 254 fields are ranked.
    const int fc = field_of(fmax(sigma, fabs(mu)));
    const int lo = fc - 24 < 1 ? 1 : fc - 24, hi = fc + 8 > 254 ? 254 : fc + 8;
    if (t == 255) {  // the upper bound, next to the window's edge terms
      double hb = 0.0;
      if (hi < 254) {
        const double a = ldexp(1.0, hi - 126), am = fabs(mu);
        hb = a > am ? erfc((a - am) / __dmul_rn(sigma, 1.4142135623730951)) : 2.0;
      }
      s_hb = hb;
    }
    rank_fields(lo, hi);
    if (t == 0) {
      const double lb = lo > 1 ? ldexp(1.0, lo - 128) * 2.0 / (sigma * 2.5066282746310002) : 0.0;
      const double lim = 0.5 * s_m7;
      s_ok = (lb + 1e-15 < lim) && (s_hb + 1e-15 < lim);
    }
    __syncthreads();
    if (!s_ok) rank_fields(1, 254);
  }
  const int take = s_take[t];
  if (take) {
    int pos = 0;
    for (int g = 1; g < t; ++g) pos += s_take[g];
    s_book[pos] = (unsigned char)t;
  }
  if (t == 0) s_book[7] = 0;
  publish_book();
}

}  // namespace

namespace {
// The predictor over L's segments, K blocks per segment.
cudaError_t launch_predict(const ZcLayout& L, ZcSegDev* d_segs, unsigned long long nparts,
                           const StatPartial* parts, int by_chunk, uint32_t K, void* d_ws,
                           cudaStream_t s) {
  StatPartial* red = reinterpret_cast<StatPartial*>(static_cast<char*>(d_ws) + zc_red_offset(L));
  uint32_t* cnt = reinterpret_cast<uint32_t*>(static_cast<char*>(d_ws) + zc_cnt_offset(L));
  return launch_dependent(zc_predict_kernel, L.nseg * K, kThreads, 0, s, d_segs, L.nseg, nparts,
                          parts, by_chunk, K, red, cnt);
}
}  // namespace

cudaError_t zc_launch_plan(const ZcLayout& L, const ZcSegDev* d_segs,
                           const uint16_t* d_x, void* d_ws, cudaStream_t s) {
  StatPartial* parts = reinterpret_cast<StatPartial*>(static_cast<char*>(d_ws) + kCtrlBytes);
  const int al = (reinterpret_cast<uintptr_t>(d_x) & 15u) == 0;
  uint32_t* red_cnt =
      L.kred_u > 1 ? reinterpret_cast<uint32_t*>(static_cast<char*>(d_ws) + zc_cnt_offset(L)) : nullptr;
  if (L.nunits) {
    cudaError_t e = cudaFuncSetAttribute(zc_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kStatSmem);
    if (e != cudaSuccess) return e;
    const int res = resident_blocks((const void*)zc_stats_kernel, kThreads, kStatSmem);
    const unsigned long long need = (L.nunits + kStatWarps - 1) / kStatWarps;
    const unsigned grid = (unsigned)(need < (unsigned long long)res ? need : (unsigned long long)res);
    zc_stats_kernel<<<grid, kThreads, kStatSmem, s>>>(d_x, d_segs, L.nseg, L.U, L.nunits, parts, al,
                                                      red_cnt);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_predict(L, const_cast<ZcSegDev*>(d_segs), L.nunits, parts, 0, L.kred_u, d_ws, s);
}

cudaError_t zc_launch_predict_chunks(const ZcLayout& L, ZcSegDev* d_segs,
                                     const StatPartial* d_parts, void* d_ws, cudaStream_t s) {
  return launch_predict(L, d_segs, L.nchunks, d_parts, 1, L.kred_c, d_ws, s);
}

}  // namespace lbb
