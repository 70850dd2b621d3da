// ibp_slots.cu -- IBP chunks kept in place in fixed-size slots, and the
// gather that reads selected slots back.
//
// [IBP] = "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria
// GPU con la Compressione Lossless per il ML":
//   Integrazione del Sistema (PCIe transfer compression): tensors are
//     compressed in CPU memory before they are transferred; compressed
//     tensors of varying size live in place in fixed-size buffers, of which
//     only the compressed part is read, and a bitmask in GPU memory records
//     which tensors are compressed;
//   Algoritmo Core, step 2: the GPU compresses through zero-copy access to
//     CPU memory; step 3: warps read a contiguous compressed segment from CPU
//     memory into shared memory and re-insert the Bitval bits.
//
// Layout (one "tensor" is one chunk): chunk s owns the slot of chunk_bytes at
// slots + s * chunk_bytes (the last slot is as long as the last chunk).  A
// compressed slot (the chunk's participation bit, as in the IBP1 stream, is
// set) starts with the chunk's body -- its B - m kept bits in ascending
// position order, zero bits up to a whole word -- and its later bytes are not
// written; any other slot holds the raw chunk.  Bit s % 32 of bitmask word
// s / 32 is the participation bit of slot s.
//
// Both kernels give each warp whole chunks: the chunk (or the slot's stored
// part) is staged in the warp's shared-memory buffer with coalesced 4-byte
// accesses -- the slots are normally pinned host memory, read and written in
// place over the host link -- and the words are closed up (or re-expanded)
// with the per-word tables of ibp_common.cuh.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ibp_common.cuh"
#include "internal.h"

namespace lbb {
namespace {

constexpr int kSlotThreads = 256;  // ibp_load_tables wants >= 256 threads for 4096-byte chunks
constexpr int kSlotWarps = kSlotThreads / 32;

struct SlotArgs {
  const uint8_t* meta;
  const uint32_t* x;      // compress: input chunks (may be the slots themselves)
  uint32_t* slots;        // compress: written; gather: read (as const)
  uint32_t* bitmask;
  const unsigned long long* idx;
  unsigned long long n_idx;
  uint32_t* y;            // gather: one row of chunk_bytes per index
  unsigned long long* read_bytes;
  unsigned long long n_bytes, nchunks, ngroups;
  uint32_t cb;
  int in_place;
  Ctrl* ctrl;
};

// Shared memory: the block's tables, then per warp a chunk buffer and a body
// buffer of W + 1 words each (the extra word is read by get_bits).
__host__ __device__ inline size_t slot_smem_bytes(uint32_t cb) {
  const uint32_t W = cb / 4;
  return 4ull * ibp_table_words(W) + 4ull * kSlotWarps * 2ull * (W + 1);
}

__global__ void __launch_bounds__(kSlotThreads) ibp_slots_encode_kernel(SlotArgs A) {
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ uint32_t s_scr[kSlotWarps + 4];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t cb = A.cb, W = cb / 4, B = 8 * cb;
  IbpTables T;
  if (!ibp_load_tables<kSlotThreads>(A.meta, cb, dyn, T, s_scr)) {
    if (t == 0) set_status(A.ctrl, ZC_ERR_META_MISMATCH);
    return;
  }
  const uint32_t m = T.m;
  const uint32_t body_words = (B - m + 31) / 32;
  uint32_t* buf = dyn + ibp_table_words(W) + (size_t)warp * 2 * (W + 1);
  uint32_t* body = buf + (W + 1);
  const unsigned long long gw = (unsigned long long)blockIdx.x * kSlotWarps + warp;
  const unsigned long long nw = (unsigned long long)gridDim.x * kSlotWarps;
  for (unsigned long long g = gw; g < A.ngroups; g += nw) {
    uint32_t pword = 0;
    const uint32_t nin = (uint32_t)((A.nchunks - 32 * g) < 32 ? (A.nchunks - 32 * g) : 32);
    for (uint32_t i = 0; i < nin; ++i) {
      const unsigned long long s = 32 * g + i;
      const unsigned long long first = s * cb;
      const uint32_t len = (uint32_t)((A.n_bytes - first) < cb ? (A.n_bytes - first) : cb);
      const uint32_t wl = len / 4;
      const uint32_t* src = A.x + s * W;
      // the whole chunk is read before any of its slot is written (in place)
      uint32_t bad = 0;
      for (uint32_t w = lane; w < wl; w += 32) {
        const uint32_t v = src[w];
        buf[w] = v;
        bad |= (v ^ T.V[w]) & ~T.K[w];
      }
      const bool p = len == cb && m > 0 && !__any_sync(kFull, bad != 0);
      uint32_t* dst = A.slots + s * W;
      if (p) {
        for (uint32_t w = lane; w <= body_words; w += 32) body[w] = 0;
        __syncwarp();
        for (uint32_t w = lane; w < W; w += 32) {
          const uint32_t K = T.K[w];
          const uint32_t k = __popc(K);
          if (k) put_bits(body, T.P[w], hd_compress(buf[w], K, T.MV + w, W), k);
        }
        __syncwarp();
        for (uint32_t w = lane; w < body_words; w += 32) dst[w] = body[w];
      } else if (!A.in_place) {
        __syncwarp();
        for (uint32_t w = lane; w < wl; w += 32) dst[w] = buf[w];
      }
      pword |= (p ? 1u : 0u) << i;
      __syncwarp();  // the buffers are reused by the next chunk
    }
    if (lane == 0) A.bitmask[g] = pword;
  }
}

__global__ void __launch_bounds__(kSlotThreads) ibp_slots_gather_kernel(SlotArgs A) {
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ uint32_t s_scr[kSlotWarps + 4];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t cb = A.cb, W = cb / 4, B = 8 * cb;
  IbpTables T;
  if (!ibp_load_tables<kSlotThreads>(A.meta, cb, dyn, T, s_scr)) {
    if (t == 0) set_status(A.ctrl, ZC_ERR_META_MISMATCH);
    return;
  }
  const uint32_t m = T.m;
  const uint32_t body_words = (B - m + 31) / 32;
  uint32_t* buf = dyn + ibp_table_words(W) + (size_t)warp * 2 * (W + 1);
  const uint32_t* slots = A.slots;
  const unsigned long long gw = (unsigned long long)blockIdx.x * kSlotWarps + warp;
  const unsigned long long nw = (unsigned long long)gridDim.x * kSlotWarps;
  unsigned long long read = 0;
  for (unsigned long long i = gw; i < A.n_idx; i += nw) {
    const unsigned long long s = A.idx[i];
    if (s >= A.nchunks) {
      if (lane == 0) set_status(A.ctrl, ZC_ERR_ARG);
      continue;  // warp-uniform
    }
    const unsigned long long first = s * cb;
    const uint32_t len = (uint32_t)((A.n_bytes - first) < cb ? (A.n_bytes - first) : cb);
    const bool p = (A.bitmask[s >> 5] >> (s & 31)) & 1u;
    if (p && (len != cb || m == 0)) {  // no body could be stored there
      if (lane == 0) set_status(A.ctrl, ZC_ERR_FORMAT);
      continue;
    }
    // only the stored part of the slot is read
    const uint32_t rw = p ? body_words : len / 4;
    const uint32_t* src = slots + s * W;
    for (uint32_t w = lane; w < rw; w += 32) buf[w] = src[w];
    if (lane == 0) buf[rw] = 0;
    __syncwarp();
    uint32_t* dst = A.y + i * W;
    if (p) {
      for (uint32_t w = lane; w < W; w += 32) {
        const uint32_t K = T.K[w];
        const uint32_t k = __popc(K);
        const uint32_t f = k ? get_bits(buf, T.P[w], k) : 0u;
        dst[w] = hd_expand(f, K, T.MV + w, W) | T.V[w];
      }
    } else {
      for (uint32_t w = lane; w < rw; w += 32) dst[w] = buf[w];
    }
    read += 4ull * rw;
    __syncwarp();  // the buffer is reused by the next index
  }
  if (A.read_bytes && lane == 0 && read) atomicAdd(A.read_bytes, read);
}

template <typename K>
cudaError_t launch_slots(K k, const SlotArgs& A, unsigned long long work, cudaStream_t s) {
  const size_t smem = slot_smem_bytes(A.cb);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned long long res = (unsigned long long)resident_blocks((const void*)k, kSlotThreads, smem);
  unsigned long long grid = (work + kSlotWarps - 1) / kSlotWarps;
  if (grid > res) grid = res;
  if (grid == 0) grid = 1;
  k<<<(unsigned)grid, kSlotThreads, smem, s>>>(A);
  return cudaGetLastError();
}

}  // namespace

cudaError_t ibp_launch_slots_compress(const void* d_meta, uint32_t cb, const void* d_x,
                                      unsigned long long n_bytes, void* d_slots,
                                      uint32_t* d_bitmask, void* d_ws, cudaStream_t s) {
  SlotArgs A{};
  A.meta = static_cast<const uint8_t*>(d_meta);
  A.x = static_cast<const uint32_t*>(d_x);
  A.slots = static_cast<uint32_t*>(d_slots);
  A.bitmask = d_bitmask;
  A.n_bytes = n_bytes;
  A.nchunks = (n_bytes + cb - 1) / cb;
  A.ngroups = (A.nchunks + 31) / 32;
  A.cb = cb;
  A.in_place = d_x == d_slots;
  A.ctrl = static_cast<Ctrl*>(d_ws);
  cudaError_t e = cudaMemsetAsync(d_ws, 0, kCtrlBytes, s);
  if (e != cudaSuccess || A.ngroups == 0) return e;
  return launch_slots(ibp_slots_encode_kernel, A, A.ngroups, s);
}

cudaError_t ibp_launch_slots_gather(const void* d_meta, uint32_t cb, const void* d_slots,
                                    unsigned long long n_bytes, const uint32_t* d_bitmask,
                                    const unsigned long long* d_idx, unsigned long long n_idx,
                                    void* d_y, unsigned long long* d_read_bytes, void* d_ws,
                                    cudaStream_t s) {
  SlotArgs A{};
  A.meta = static_cast<const uint8_t*>(d_meta);
  A.slots = static_cast<uint32_t*>(const_cast<void*>(d_slots));
  A.bitmask = const_cast<uint32_t*>(d_bitmask);
  A.idx = d_idx;
  A.n_idx = n_idx;
  A.y = static_cast<uint32_t*>(d_y);
  A.read_bytes = d_read_bytes;
  A.n_bytes = n_bytes;
  A.nchunks = (n_bytes + cb - 1) / cb;
  A.ngroups = (A.nchunks + 31) / 32;
  A.cb = cb;
  A.ctrl = static_cast<Ctrl*>(d_ws);
  cudaError_t e = cudaMemsetAsync(d_ws, 0, kCtrlBytes, s);
  if (e == cudaSuccess && d_read_bytes) e = cudaMemsetAsync(d_read_bytes, 0, 8, s);
  if (e != cudaSuccess || n_idx == 0) return e;
  return launch_slots(ibp_slots_gather_kernel, A, n_idx, s);
}

}  // namespace lbb
