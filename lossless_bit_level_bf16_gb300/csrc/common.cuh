// common.cuh -- device helpers shared by the codec kernels: the workspace
// control block and status word, memory-order primitives, a bounded
// decoupled look-back scan across thread blocks, and block-wide scans.
//
// Nothing here traps: every wait is bounded and reports ZC_ERR_TIMEOUT through
// the status word instead.
#pragma once

#include <cstdint>

#include "zc.h"

namespace lbb {

constexpr int kWarp = 32;

__host__ __device__ __forceinline__ unsigned long long round_up_dev(unsigned long long v,
                                                                  unsigned long long a) {
  return (v + a - 1) / a * a;
}
constexpr unsigned kFull = 0xFFFFFFFFu;

// First 256 bytes of every workspace.
struct Ctrl {
  int status;          // first error of the call (0 = none)
  int pad0;
  unsigned long long ticket;  // dynamic tile counter (ordered tile start)
  unsigned long long done;    // blocks finished (last one finalises)
  // Wait-failure test switch (zero, i.e. off, unless zc_test_wait_fault armed
  // it for the call): tile + 1 of the tile whose scan state is never
  // published, and the number of polls each inter-block wait may take.
  unsigned long long fault_tile1;
  unsigned max_spins;
  unsigned pad1;
  unsigned long long spare[27];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");
constexpr size_t kCtrlBytes = 256;

__device__ __forceinline__ void set_status(Ctrl* c, int code) {
  atomicCAS(&c->status, 0, code);
}
__device__ __forceinline__ int get_status(const Ctrl* c) {
  return *reinterpret_cast<const volatile int*>(&c->status);
}

// ---------------------------------------------------------------- fp32 sums

// The two bf16 values of a 32-bit word as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values in one 64-bit register (x in the low half) for the packed
// fp32x2 arithmetic of sm_100 and later: each half is rounded exactly as the
// fp32 operation on it alone would be.
__device__ __forceinline__ unsigned long long f2_pack(float x, float y) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long v) {
  float x, y;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
  return make_float2(x, y);
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// a * b + c, each half fused
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// Error-free transformation: hi + lo accumulates v exactly up to the rounding
// of lo itself.
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float v) {
  float s = __fadd_rn(hi, v);
  float bb = __fsub_rn(s, hi);
  float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(v, bb));
  hi = s;
  lo = __fadd_rn(lo, err);
}

// (a, b) += (a2, b2) for fp32 (sum, error) pairs: a takes the rounded sum of
// the sums, b the error of that addition and the errors so far.
__device__ __forceinline__ void pair_add(float& a, float& b, float a2, float b2) {
  two_sum_acc(a, b, a2);
  b = __fadd_rn(b, b2);
}

// ---------------------------------------------------------------- memory ops

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(
    const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(
    const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// 16-byte read-only load (data not written by this kernel).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Asynchronous global -> shared copies (cp.async, no register staging).
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---------------------------------------------------------------- TMA bulk copies
//
// One thread copies a contiguous global range into shared memory with
// cp.async.bulk (16-byte aligned addresses, size a multiple of 16); an
// mbarrier with one arrival counts the bytes in and flips its phase when all
// have landed.  Waits are bounded: they report failure instead of spinning on.

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// True once the phase with the given parity has completed; false if the
// bounded wait ran out.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < (1u << 20); ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Barrier `id` (1..15) over `count` threads (a multiple of 32) of the block.
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Orders this thread's earlier shared-memory accesses before later
// asynchronous-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 eviction policy for data read again soon (the cache-hinted prefetch below).
__device__ __forceinline__ unsigned long long l2_policy_keep() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ unsigned long long l2_policy_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// bulk_g2s with an L2 eviction-priority policy for the lines it reads.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              unsigned long long* bar, unsigned long long pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// st_v4 with an L2 eviction-priority policy.
__device__ __forceinline__ void st_v4_hint(void* p, uint4 v, unsigned long long pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}
// Asks L2 to fetch a contiguous range (16-byte aligned, size a multiple of
// 16); nothing waits for it.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes,
                                                 unsigned long long pol) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src),
               "r"(bytes), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// 16-byte relaxed load of words other blocks publish while this one runs.
__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
  uint4 r;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}

// ---------------------------------------------------------------- dependent launches
//
// A kernel launched with programmatic stream serialization (launch_dependent
// in internal.h) may start while the kernel before it on the stream is still
// finishing: it does its set-up, then grid_dep_wait() returns once that kernel
// has completed and its writes are visible.  grid_dep_launch() lets the next
// such kernel start.  Both do nothing in a kernel launched the ordinary way.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
  return __byte_perm(a, b, s);
}
// prmt.b32 in its default mode, where bit 3 of a selector nibble replicates
// the selected byte's sign bit over the output byte.
__device__ __forceinline__ uint32_t prmt_sx(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(s));
  return r;
}

// ---------------------------------------------------------------- warp sums

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// ---------------------------------------------------------------- look-back
//
// Tile state word: bits 63..62 = flag (0 empty, 1 aggregate, 2 inclusive
// prefix), bits 61..0 = value.  Tiles are numbered in the order blocks took
// them from the ticket counter, so every predecessor of a waiting tile is
// already running: the wait ends unless something is broken, and is bounded
// anyway.
constexpr unsigned long long kFlagAgg = 1ull << 62;
constexpr unsigned long long kFlagInc = 2ull << 62;
constexpr unsigned long long kValMask = (1ull << 62) - 1;
constexpr unsigned kMaxSpins = 1u << 22;  // ~1 s with the back-off below

// The poll limit of this call's inter-block waits, and whether `tile` may
// publish its scan state (both read from the control block: see Ctrl).
__device__ __forceinline__ unsigned wait_limit(const Ctrl* c) {
  const unsigned v = c->max_spins;
  return v ? v : kMaxSpins;
}
__device__ __forceinline__ bool may_publish(const Ctrl* c, unsigned long long tile) {
  return c->fault_tile1 != tile + 1;
}

// Look-back with an adaptive window (states are published with relaxed
// stores: they carry counts only, nothing else is read through them): the nearest 32 predecessors are read
// first (one state per lane; usually one of them already holds an inclusive
// prefix); if all 32 hold only aggregates the walk continues kLbDepth*32
// states per L2 round trip.  Spinning on a predecessor that has not published
// yet re-reads only the current window.
constexpr int kLbDepth = 8;
enum { kLbEmpty = 0, kLbFound = 1, kLbAllAgg = 2 };

template <int D>
__device__ __forceinline__ int lb_window(const unsigned long long* states, long long end,
                                         unsigned long long* sum) {
  const int lane = threadIdx.x & (kWarp - 1);
  unsigned long long s[D];
#pragma unroll
  for (int j = 0; j < D; ++j) {
    const long long idx = end - (32 * j + lane);
    s[j] = idx >= 0 ? ld_relaxed_u64(states + idx) : kFlagInc;
  }
  int jinc = D, linc = 32;
  bool empty_before = false;
#pragma unroll
  for (int j = 0; j < D; ++j) {
    const unsigned f = (unsigned)(s[j] >> 62);
    const unsigned inc = __ballot_sync(kFull, f == 2);
    const unsigned emp = __ballot_sync(kFull, f == 0);
    if (jinc == D) {
      if (inc) {
        jinc = j;
        linc = __ffs(inc) - 1;
        if (emp & ((1u << linc) - 1u)) empty_before = true;
      } else if (emp) {
        empty_before = true;
      }
    }
  }
  if (empty_before) return kLbEmpty;
  unsigned long long part = 0;
#pragma unroll
  for (int j = 0; j < D; ++j)
    if (j < jinc || (j == jinc && lane <= linc)) part += s[j] & kValMask;
  *sum = warp_sum_u64(part);
  return jinc < D ? kLbFound : kLbAllAgg;
}

// D0 * 32 predecessors are read in the first round trip and D1 * 32 in each
// further one; after FREE spins on a predecessor that has not published, the
// warp sleeps between re-reads (doubling up to 512 ns) to spare L2 bandwidth.
// `limit` bounds the polls of a predecessor that has not published; a tile
// with `publish` false publishes nothing (the wait-failure test).
template <int D0 = 1, int D1 = kLbDepth, unsigned FREE = 64>
__device__ __forceinline__ unsigned long long lookback_warp_wide(
    unsigned long long* states, unsigned long long tile, unsigned long long aggregate,
    bool* timed_out, unsigned limit = kMaxSpins, bool publish = true) {
  const int lane = threadIdx.x & (kWarp - 1);
  if (tile == 0) {
    if (lane == 0 && publish) st_relaxed_u64(states, kFlagInc | aggregate);
    return 0;
  }
  if (lane == 0 && publish) st_relaxed_u64(states + tile, kFlagAgg | aggregate);
  unsigned long long excl = 0;
  long long end = (long long)tile - 1;
  unsigned spins = 0, ns = 32;
  bool deep = false, to = false;
  while (true) {
    unsigned long long sum = 0;
    const int r = deep ? lb_window<D1>(states, end, &sum) : lb_window<D0>(states, end, &sum);
    if (r == kLbEmpty) {
      if (++spins > limit) {
        to = true;
        break;
      }
      if (spins > FREE) {
        __nanosleep(ns);
        if (ns < 512) ns <<= 1;
      }
      continue;
    }
    excl += sum;
    if (r == kLbFound) break;
    end -= deep ? 32 * D1 : 32 * D0;
    deep = true;
  }
  if (to) {
    *timed_out = true;
    if (lane == 0 && publish) st_relaxed_u64(states + tile, kFlagInc | aggregate);
    return 0;
  }
  if (lane == 0 && publish) st_relaxed_u64(states + tile, kFlagInc | ((excl + aggregate) & kValMask));
  return excl;
}

// ---------------------------------------------------------------- two-level look-back
//
// For kernels with many tickets in flight (every warp holds one), where the
// plain look-back would read back over all of them.  Tickets are grouped in
// blocks of kLbBlock, and each block has one word that only atomics change:
// bit 63 is the inclusive flag (kFlagInc), bits 61:52 count the tickets whose
// aggregate is in, bits 51:0 hold the value.  Every ticket adds (1 << 52) +
// its aggregate; the block's first ticket, once it knows its exclusive
// prefix, adds the flag + that prefix.  A word is read only as a whole: while its
// count is short of kLbBlock the block is incomplete whatever else is in it;
// once full it holds the block's sum, or with the flag the inclusive prefix
// through the block.  So no ordering between locations is needed.
// A look-back reads the tickets of its own block (one window), then the
// words of the blocks before it (32 * D per window), and reads a block's
// tickets only while that block is incomplete.
constexpr unsigned kLbBlock = 128;  // equal to kZcLbBlock (internal.h)
constexpr unsigned long long kBlkOne = 1ull << 52;
constexpr unsigned long long kBlkValMask = kBlkOne - 1;
static_assert(kLbBlock < 1024, "the count field holds a block's tickets");

// Lane 0, once ticket t's aggregate is known (values below 2^52).
__device__ __forceinline__ void lb2_publish_agg(unsigned long long* states,
                                                unsigned long long* bwords,
                                                unsigned long long t, unsigned long long agg) {
  atomicAdd(bwords + t / kLbBlock, kBlkOne + agg);
  st_relaxed_u64(states + t, (t == 0 ? kFlagInc : kFlagAgg) | agg);
}

// Lane 0, once ticket t's exclusive prefix is known: the ticket's inclusive
// state, and for a block's first ticket the block's exclusive prefix.
__device__ __forceinline__ void lb2_publish_inc(unsigned long long* states,
                                                unsigned long long* bwords,
                                                unsigned long long t, unsigned long long excl,
                                                unsigned long long agg) {
  st_relaxed_u64(states + t, kFlagInc | ((excl + agg) & kValMask));
  if (t % kLbBlock == 0) atomicAdd(bwords + t / kLbBlock, kFlagInc + excl);
}

// A window of 32 * D entries below `end`, down to `lo` (indices below lo
// are outside the range, except that with lo == 0 those below 0 read as an
// inclusive zero); BLK selects block words over ticket states.  Returns
// kLbFound (an inclusive entry in range; *sum = the values from end down to
// it), kLbAllAgg (none; *sum = every value in range) or kLbEmpty (an empty
// entry before any inclusive one; *empty_at = the nearest such index, *sum =
// the values above it).
template <int D, bool BLK>
__device__ __forceinline__ int lb2_window(const unsigned long long* words, long long end,
                                          long long lo, unsigned long long* sum,
                                          long long* empty_at) {
  const int lane = threadIdx.x & (kWarp - 1);
  constexpr unsigned long long kZeroInc = BLK ? (kFlagInc | ((unsigned long long)kLbBlock << 52))
                                              : kFlagInc;
  unsigned long long s[D];
#pragma unroll
  for (int j = 0; j < D; ++j) {
    const long long idx = end - (32 * j + lane);
    s[j] = idx < lo ? (idx < 0 && lo == 0 ? kZeroInc : 0ull) : ld_relaxed_u64(words + idx);
  }
  // nearest first: values count up to the first empty entry (excluded) or
  // the first inclusive one (included)
  unsigned long long part = 0;
  int res = kLbAllAgg;
#pragma unroll
  for (int j = 0; j < D; ++j) {
    const long long idx = end - (32 * j + lane);
    const bool in = idx >= lo || (idx < 0 && lo == 0);
    unsigned f = (unsigned)(s[j] >> 62);  // 0 empty, 1 aggregate, 2 inclusive
    if (BLK) f = ((s[j] >> 52) & 1023u) == kLbBlock ? 1u + (unsigned)(s[j] >> 63) : 0u;
    if (res == kLbAllAgg) {
      const unsigned emp = __ballot_sync(kFull, in && f == 0);
      const unsigned cut = emp | __ballot_sync(kFull, in && f == 2);
      const int lc = cut ? __ffs(cut) - 1 : 32;
      const bool e = (emp >> (lc & 31)) & (cut != 0);
      if (in && (lane < lc || (lane == lc && !e))) part += s[j] & (BLK ? kBlkValMask : kValMask);
      if (cut) {
        res = e ? kLbEmpty : kLbFound;
        if (e) *empty_at = end - (32 * j + lc);
      }
    }
  }
  *sum = warp_sum_u64(part);
  return res;
}

// The exclusive prefix of ticket t (whose aggregate is published), with the
// two-level look-back; bounded like lookback_warp_wide.  The caller then
// publishes with lb2_publish_inc (after a timeout: the ticket's own count
// as its inclusive state and nothing for the block, so that no one waits).
template <int D>
__device__ __forceinline__ unsigned long long lb2_lookback(const unsigned long long* states,
                                                           const unsigned long long* bwords,
                                                           unsigned long long t,
                                                           bool* timed_out,
                                                           unsigned limit = kMaxSpins) {
  static_assert(32 * D >= (int)kLbBlock, "a window covers a block's tickets");
  if (t == 0) return 0;
  unsigned long long excl = 0, sum = 0;
  unsigned spins = 0;
  long long at = 0;
  // the tickets of t's own block below t, then of any incomplete block below
  long long blk = (long long)(t / kLbBlock);
  long long tend = (long long)t - 1;
  for (;;) {
    int r;
    while ((r = lb2_window<D, false>(states, tend, blk * (long long)kLbBlock, &sum, &at)) ==
           kLbEmpty) {
      if (++spins > limit) {
        *timed_out = true;
        return excl;
      }
      if (spins > 64) __nanosleep(256);
    }
    excl += sum;
    if (r == kLbFound) return excl;
    // block words below blk, until an inclusive one or an incomplete block
    long long bend = blk - 1;
    for (;;) {
      if (bend < 0) return excl;
      const int q = lb2_window<D, true>(bwords, bend, 0, &sum, &at);
      excl += sum;
      if (q == kLbFound) return excl;
      if (q == kLbEmpty) {
        // the blocks above `at` are complete and counted; read block `at`
        // ticket by ticket
        blk = at;
        tend = at * (long long)kLbBlock + kLbBlock - 1;
        break;
      }
      bend -= 32 * D;
    }
  }
}

// ---------------------------------------------------------------- block scan
//
// Exclusive scan of one uint32 per thread over a block of NT threads
// (multiple of 32).  `warp_tot` is NT/32 words of shared memory.  Returns the
// thread's exclusive prefix; *total receives the block total.  Contains one
// __syncthreads (callers must not have warp_tot in use).
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_tot,
                                                    uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  uint32_t base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    uint32_t t = warp_tot[w];
    if (w < warp) base += t;
    tot += t;
  }
  *total = tot;
  return base + inc - v;
}

}  // namespace lbb
