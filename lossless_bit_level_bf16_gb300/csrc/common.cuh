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
  unsigned long long spare[29];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");
constexpr size_t kCtrlBytes = 256;

__device__ __forceinline__ void set_status(Ctrl* c, int code) {
  atomicCAS(&c->status, 0, code);
}
__device__ __forceinline__ int get_status(const Ctrl* c) {
  return *reinterpret_cast<const volatile int*>(&c->status);
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
template <int D0 = 1, int D1 = kLbDepth, unsigned FREE = 64>
__device__ __forceinline__ unsigned long long lookback_warp_wide(
    unsigned long long* states, unsigned long long tile, unsigned long long aggregate,
    bool* timed_out) {
  const int lane = threadIdx.x & (kWarp - 1);
  if (tile == 0) {
    if (lane == 0) st_relaxed_u64(states, kFlagInc | aggregate);
    return 0;
  }
  if (lane == 0) st_relaxed_u64(states + tile, kFlagAgg | aggregate);
  unsigned long long excl = 0;
  long long end = (long long)tile - 1;
  unsigned spins = 0, ns = 32;
  bool deep = false, to = false;
  while (true) {
    unsigned long long sum = 0;
    const int r = deep ? lb_window<D1>(states, end, &sum) : lb_window<D0>(states, end, &sum);
    if (r == kLbEmpty) {
      if (++spins > kMaxSpins) {
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
    if (lane == 0) st_relaxed_u64(states + tile, kFlagInc | aggregate);
    return 0;
  }
  if (lane == 0) st_relaxed_u64(states + tile, kFlagInc | ((excl + aggregate) & kValMask));
  return excl;
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
