// ibp_meta.cu -- IBP metadata: Mask and Bitval from sampled chunks.
//
// [IBP] = "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria
// GPU con la Compressione Lossless per il ML", Metodologia: Invariant Bit
// Packing (IBP), Algoritmo Core, step 1 (Preprocessing): bit positions that
// hold the same value across a high fraction T of the sampled tensors are
// invariant; Mask marks them and Bitval keeps their values; the result is a
// fixed-size blob kept in GPU memory and reused for the whole dataset.
//
// Kernels:
//   ibp_columns_kernel  a warp per 8 words of the chunk and 4 blocks of 32
//                       samples: a shuffle butterfly transposes each 32x32
//                       bit block, so lane b holds the column of position
//                       32w+b over those samples; its popcounts are summed
//                       and added to the ones count of that position.  The
//                       columns are kept for the joint reading.
//   ibp_meta_kernel     one block: threshold k = ceil(T*N) on each position's
//                       agreement max(ones, N-ones); per-position (mode 0) or
//                       joint greedy selection (mode 1: positions sorted by
//                       agreement, then index, with a block-wide bitonic
//                       sort; one warp then keeps a position while at least
//                       k samples still match every kept position);
//                       writes the IBPM blob with its FNV-1a-64 hash.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace lbb {
namespace {

constexpr int kMetaThreads = 1024;
constexpr uint32_t kWordsPerWarp = 8;
constexpr uint32_t kBlocksPerWarp = 4;  // blocks of 32 samples a warp takes

// 32x32 bit transpose across a warp: lane i holds row i on entry; lane b
// returns column b (bit i = bit b of row i).  Five butterfly levels, each
// swapping the off-diagonal j x j sub-blocks of lane pairs (i, i ^ j).
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
  uint32_t m = 0x0000FFFFu;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint32_t other = __shfl_xor_sync(kFull, x, j);
    const bool up = (lane & j) != 0;
    const uint32_t lo = up ? other : x, hi = up ? x : other;
    const uint32_t t = ((lo >> j) ^ hi) & m;
    x = up ? (hi ^ t) : (lo ^ (t << j));
    m ^= m << (j >> 1);
  }
  return x;
}

// A warp takes 8 words of the chunk for kBlocksPerWarp blocks of 32 samples:
// lane l loads words w0..w0+7 of sample 32*sb + l (two 16-byte loads, all
// blocks' loads issued before any is used), each word's 32x32 bit block is
// transposed so that lane b holds the column of position 32w+b over the 32
// samples, and the columns' popcounts are summed in registers; one atomic
// per position and warp adds them to the ones counts.  The columns are kept
// for the joint reading.
__global__ void __launch_bounds__(256) ibp_columns_kernel(
    const uint32_t* __restrict__ samples, unsigned long long N, uint32_t W,
    uint32_t* __restrict__ ones, uint32_t* __restrict__ cols, uint32_t Wn, int keep_cols) {
  const int lane = threadIdx.x & 31;
  grid_dep_launch();  // the metadata kernel may be scheduled as blocks finish
  const unsigned long long warp = (blockIdx.x * 256ull + threadIdx.x) >> 5;
  const uint32_t wgroups = (W + kWordsPerWarp - 1) / kWordsPerWarp;
  const unsigned long long sbq = warp / wgroups;  // group of kBlocksPerWarp sample blocks
  const uint32_t w0 = (uint32_t)(warp % wgroups) * kWordsPerWarp;
  if (sbq * kBlocksPerWarp >= Wn) return;
  const uint32_t nw = (W - w0) < kWordsPerWarp ? (W - w0) : kWordsPerWarp;
  uint32_t v[kBlocksPerWarp][kWordsPerWarp];
#pragma unroll
  for (uint32_t bi = 0; bi < kBlocksPerWarp; ++bi) {
    const unsigned long long sb = sbq * kBlocksPerWarp + bi;
    const unsigned long long s = sb * 32ull + lane;
    const bool have = sb < Wn && s < N;
    if (have && nw == kWordsPerWarp && (W & 3u) == 0) {  // 16-byte aligned: W and w0 multiples of 4
      const uint4 a = ld_nc_v4(samples + s * W + w0), b = ld_nc_v4(samples + s * W + w0 + 4);
      v[bi][0] = a.x; v[bi][1] = a.y; v[bi][2] = a.z; v[bi][3] = a.w;
      v[bi][4] = b.x; v[bi][5] = b.y; v[bi][6] = b.z; v[bi][7] = b.w;
    } else {
#pragma unroll
      for (uint32_t k = 0; k < kWordsPerWarp; ++k)
        v[bi][k] = (have && k < nw) ? __ldg(samples + s * W + w0 + k) : 0u;
    }
  }
  uint32_t cnt[kWordsPerWarp];
#pragma unroll
  for (uint32_t k = 0; k < kWordsPerWarp; ++k) cnt[k] = 0;
#pragma unroll
  for (uint32_t bi = 0; bi < kBlocksPerWarp; ++bi) {
    const unsigned long long sb = sbq * kBlocksPerWarp + bi;
    if (sb >= Wn) break;  // warp-uniform
#pragma unroll
    for (uint32_t k = 0; k < kWordsPerWarp; ++k) {
      const uint32_t col = warp_transpose32(v[bi][k], lane);
      cnt[k] += (uint32_t)__popc(col);
      if (keep_cols && k < nw) cols[(32ull * (w0 + k) + lane) * Wn + sb] = col;
    }
  }
#pragma unroll
  for (uint32_t k = 0; k < kWordsPerWarp; ++k)
    if (k < nw && cnt[k]) atomicAdd(ones + 32u * (w0 + k) + lane, cnt[k]);
}

__device__ __forceinline__ uint32_t block_sum_1024(uint32_t v, uint32_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  __syncthreads();  // red reuse
  if (lane == 0) red[warp] = v;
  __syncthreads();
  uint32_t t = 0;
#pragma unroll
  for (int w = 0; w < kMetaThreads / 32; ++w) t += red[w];
  return t;
}

// Joint reading, greedy pass over the sorted candidates (one warp): a
// candidate is kept when at least k samples still match every kept position
// and it.
constexpr int kGreedyRegs = 12;
constexpr uint32_t kRing = 8;  // candidate columns in flight

__device__ __forceinline__ void greedy_warp(const unsigned long long* keys, uint32_t Bp,
                                            const uint32_t* __restrict__ ones,
                                            const uint32_t* __restrict__ cols, uint32_t Wn,
                                            unsigned long long k, uint32_t* alive,
                                            uint32_t* smask, uint32_t* sbitv, uint32_t* ring) {
  const int lane = threadIdx.x & 31;
  if (Wn <= 32u * kGreedyRegs) {
    // columns of the next kRing candidates in flight (cp.async into a ring in
    // shared memory; each lane copies and reads only its own words)
    uint32_t al[kGreedyRegs];
#pragma unroll
    for (int r = 0; r < kGreedyRegs; ++r) {
      const uint32_t w = lane + 32u * r;
      al[r] = w < Wn ? alive[w] : 0u;
    }
    auto fetch = [&](uint32_t c) {
      const unsigned long long key = c < Bp ? keys[c] : ~0ull;
      if (key != ~0ull) {
        const uint32_t* col = cols + (unsigned long long)((uint32_t)key >> 1) * Wn;
        uint32_t* slot = ring + (c % kRing) * (32u * kGreedyRegs);
#pragma unroll
        for (int r = 0; r < kGreedyRegs; ++r) {
          const uint32_t w = lane + 32u * r;
          if (w < Wn) cp_async4(slot + w, col + w);
        }
      }
      cp_async_commit();  // (possibly empty) group per candidate
    };
#pragma unroll 1
    for (uint32_t d = 0; d < kRing; ++d) fetch(d);
    for (uint32_t c = 0; c < Bp; ++c) {
      const unsigned long long key = keys[c];
      if (key == ~0ull) break;
      const uint32_t j = (uint32_t)(key & 0xFFFFFFFFu) >> 1;
      cp_async_wait_group<kRing - 1>();  // this candidate's column has landed
      const uint32_t* slot = ring + (c % kRing) * (32u * kGreedyRegs);
      const bool v = (key & 1u) != 0;
      uint32_t keep[kGreedyRegs], cnt = 0;
#pragma unroll
      for (int r = 0; r < kGreedyRegs; ++r) {
        const uint32_t w = lane + 32u * r;
        const uint32_t cw = w < Wn ? slot[w] : 0u;
        keep[r] = al[r] & (v ? cw : ~cw);
        cnt += __popc(keep[r]);
      }
      fetch(c + kRing);  // the slot just read is refilled
      cnt = __reduce_add_sync(kFull, cnt);
      if (cnt >= k) {
#pragma unroll
        for (int r = 0; r < kGreedyRegs; ++r) al[r] = keep[r];
        if (lane == 0) {
          smask[j >> 5] |= 1u << (j & 31);
          if (v) sbitv[j >> 5] |= 1u << (j & 31);
        }
      }
    }
    cp_async_wait_all();
    return;
  }
  // many samples: the mask stays in shared memory, two passes per candidate
  for (uint32_t c = 0; c < Bp; ++c) {
    const unsigned long long key = keys[c];
    if (key == ~0ull) break;
    const uint32_t j = (uint32_t)(key & 0xFFFFFFFFu) >> 1;
    const bool v = (key & 1u) != 0;
    const uint32_t* col = cols + (unsigned long long)j * Wn;
    uint32_t cnt = 0;
    for (uint32_t w = lane; w < Wn; w += 32) {
      const uint32_t cw = __ldg(col + w);
      cnt += __popc(alive[w] & (v ? cw : ~cw));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
    if (cnt >= k) {
      for (uint32_t w = lane; w < Wn; w += 32) {
        const uint32_t cw = __ldg(col + w);
        alive[w] &= v ? cw : ~cw;
      }
      if (lane == 0) {
        smask[j >> 5] |= 1u << (j & 31);
        if (v) sbitv[j >> 5] |= 1u << (j & 31);
      }
    }
    __syncwarp();
  }
}

// Dynamic shared memory: keys (8*Bp bytes, mode 1), alive (4*Wn), mask and
// bitval words (4*W each), the greedy pass's column ring (mode 1).
__global__ void __launch_bounds__(kMetaThreads) ibp_meta_kernel(
    const uint32_t* __restrict__ ones, const uint32_t* __restrict__ cols, uint32_t Wn,
    unsigned long long N, uint32_t chunk_bytes, unsigned long long k, double T, int mode,
    uint32_t Bp, uint8_t* __restrict__ meta) {
  extern __shared__ __align__(16) unsigned char dyn[];
  __shared__ uint32_t red[kMetaThreads / 32];
  const uint32_t B = chunk_bytes * 8u, W = chunk_bytes / 4u;
  const int t = threadIdx.x;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(dyn);
  uint32_t* alive = reinterpret_cast<uint32_t*>(dyn + (mode == 1 ? 8ull * Bp : 0ull));
  uint32_t* smask = alive + (mode == 1 ? Wn : 0u);
  uint32_t* sbitv = smask + W;
  grid_dep_wait();  // the ones counts and bit columns

  for (uint32_t w = t; w < W; w += kMetaThreads) {
    smask[w] = 0;
    sbitv[w] = 0;
  }
  if (mode == 0) {
    __syncthreads();
    // lane b of a warp decides position 32 w + b of word w; the warp's two
    // votes are the word's Mask and Bitval
    for (uint32_t j0 = (uint32_t)t & ~31u; j0 < B; j0 += kMetaThreads) {
      const unsigned long long o = ones[j0 + (t & 31)];
      const unsigned long long agree = o > N - o ? o : N - o;
      const uint32_t mk = __ballot_sync(kFull, agree >= k);
      const uint32_t bv = __ballot_sync(kFull, agree >= k && o >= k);
      if ((t & 31) == 0) {
        smask[j0 >> 5] = mk;
        sbitv[j0 >> 5] = bv;
      }
    }
  } else {
    // candidates sorted by (agreement descending, position ascending)
    for (uint32_t j = t; j < Bp; j += kMetaThreads) {
      unsigned long long key = ~0ull;
      if (j < B) {
        const unsigned long long o = ones[j];
        const unsigned long long agree = o > N - o ? o : N - o;
        // low word: position, then its majority value (ties stay by position)
        if (agree >= k) key = ((N - agree) << 32) | ((unsigned long long)j << 1) | (o >= k ? 1u : 0u);
      }
      keys[j] = key;
    }
    for (uint32_t w = t; w < Wn; w += kMetaThreads) {
      const unsigned long long rem = N - 32ull * w;
      alive[w] = rem >= 32 ? 0xFFFFFFFFu : ((1u << rem) - 1u);
    }
    __syncthreads();
    for (uint32_t size = 2; size <= Bp; size <<= 1) {
      for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
        for (uint32_t i = t; i < Bp / 2; i += kMetaThreads) {
          const uint32_t lo = 2 * i - (i & (stride - 1));
          const uint32_t hi = lo + stride;
          const bool up = (lo & size) == 0;
          const unsigned long long a = keys[lo], b = keys[hi];
          if ((a > b) == up) {
            keys[lo] = b;
            keys[hi] = a;
          }
        }
        __syncthreads();
      }
    }
    // The greedy pass is sequential over candidates: one warp runs it, with
    // no block barrier per candidate.  Lane l owns words l, l + 32, ... of the
    // surviving-sample mask; for up to 32 * kGreedyRegs words those stay in
    // registers and the next candidate's column is loaded while the current
    // one is decided.
    if (t < 32) greedy_warp(keys, Bp, ones, cols, Wn, k, alive, smask, sbitv, sbitv + W);
  }
  __syncthreads();
  // write Mask, Bitval and the header
  uint32_t* om = reinterpret_cast<uint32_t*>(meta + kIbpmHeader);
  uint32_t* ob = reinterpret_cast<uint32_t*>(meta + kIbpmHeader + chunk_bytes);
  uint32_t pc = 0;
  for (uint32_t w = t; w < W; w += kMetaThreads) {
    om[w] = smask[w];
    ob[w] = sbitv[w];
    pc += __popc(smask[w]);
  }
  const uint32_t m = block_sum_1024(pc, red);
  if (t == 0) {
    // FNV-1a-64 over the chunk size (4 bytes, little-endian), Mask and
    // Bitval.  The prime is 2^40 + 435, so h * prime = h * 435 + (h << 40):
    // in 32-bit halves the low half's chain per byte is one XOR and one
    // widening multiply, and the high half follows beside it.
    uint32_t lo = 0x84222325u, hi = 0xcbf29ce4u;  // the offset basis
    auto step = [&](uint32_t byte) {
      lo ^= byte;
      const unsigned long long p = (unsigned long long)lo * 435ull;
      hi = hi * 435u + (uint32_t)(p >> 32) + (lo << 8);
      lo = (uint32_t)p;
    };
    auto word = [&](uint32_t v) {
      step(v & 0xFFu);
      step((v >> 8) & 0xFFu);
      step((v >> 16) & 0xFFu);
      step(v >> 24);
    };
    word(chunk_bytes);
    for (uint32_t w = 0; w < W; ++w) word(smask[w]);
    for (uint32_t w = 0; w < W; ++w) word(sbitv[w]);
    const unsigned long long h = ((unsigned long long)hi << 32) | lo;
    unsigned long long* hd = reinterpret_cast<unsigned long long*>(meta);
    hd[0] = (unsigned long long)kIbpmMagic | (1ull << 32) | ((unsigned long long)kIbpmHeader << 48);
    hd[1] = (unsigned long long)chunk_bytes | ((unsigned long long)B << 32);
    hd[2] = (unsigned long long)m | ((unsigned long long)(uint32_t)mode << 32);
    hd[3] = N;
    hd[4] = k;
    hd[5] = (unsigned long long)__double_as_longlong(T);
    hd[6] = h;
    hd[7] = 0;
  }
}

}  // namespace

cudaError_t ibp_launch_build_meta(const void* d_samples, unsigned long long N,
                                  uint32_t chunk_bytes, unsigned long long k, double T, int mode,
                                  void* d_meta, void* d_ws, cudaStream_t s) {
  const uint32_t W = chunk_bytes / 4, B = chunk_bytes * 8;
  const uint32_t Wn = (uint32_t)((N + 31) / 32);
  uint32_t* ones = reinterpret_cast<uint32_t*>(static_cast<char*>(d_ws) + kCtrlBytes);
  uint32_t* cols = ones + B;
  cudaError_t e = cudaMemsetAsync(d_ws, 0, kCtrlBytes + 4ull * B, s);
  if (e != cudaSuccess) return e;
  const uint32_t wgroups = (W + kWordsPerWarp - 1) / kWordsPerWarp;
  const unsigned long long warps =
      (unsigned long long)((Wn + kBlocksPerWarp - 1) / kBlocksPerWarp) * wgroups;
  const unsigned long long blocks = (warps + 7) / 8;
  if (blocks > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  ibp_columns_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint32_t*>(d_samples), N,
                                                      W, ones, cols, Wn, mode == 1);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  uint32_t Bp = 1;
  while (Bp < B) Bp <<= 1;
  const size_t smem = (mode == 1 ? 8ull * Bp + 4ull * Wn + 4ull * kRing * 32 * kGreedyRegs : 0ull) +
                      8ull * W;
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(ibp_meta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_dependent(ibp_meta_kernel, 1u, (unsigned)kMetaThreads, smem, s,
                          static_cast<const uint32_t*>(ones), static_cast<const uint32_t*>(cols),
                          Wn, N, chunk_bytes, k, T, mode, Bp, static_cast<uint8_t*>(d_meta));
}

}  // namespace lbb
