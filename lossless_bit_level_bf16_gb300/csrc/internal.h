// internal.h -- structures and launchers shared between the C-ABI layer
// (api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "zc.h"

namespace lbb {

// ---------------------------------------------------------------- ZipCCL

constexpr uint32_t kZcMagic = 0x3143435Au;  // "ZCC1"
constexpr uint32_t kZcHeader = 128;
constexpr uint32_t kZcSegRec = 64;
constexpr uint32_t kZcAlign = 128;
constexpr uint32_t kTileLanes = 8192;   // lanes (element slots) per encoder tile
constexpr unsigned long long kZcLbBlock = 128;  // tiles per look-back block

// Slots of one encoder tile (ticket) for chunks of C slots (a multiple of
// 1024): whole chunks only, as many as fit in kTileLanes (one chunk when C is
// larger), so that every chunk's escape count -- and with it the choice of
// the raw form for an incompressible chunk -- is known inside one tile.
// Powers of two up to kTileLanes give kTileLanes.
__host__ __device__ constexpr uint32_t zc_tile_slots(uint32_t C) {
  return C >= kTileLanes ? C : C * (kTileLanes / C);
}
__host__ __device__ constexpr uint32_t zc_chunks_per_tile(uint32_t C) {
  return zc_tile_slots(C) / C;
}

// Bit 63 of a chunk's escape-offset table entry: the chunk is stored raw.
constexpr unsigned long long kZcRawFlag = 1ull << 63;

// ZipCCL encoder scratch after the control block: one look-back state per
// tile, then one look-back word per block of kZcLbBlock tiles.
constexpr unsigned long long zc_enc_blocks(unsigned long long ntiles) {
  return (ntiles + kZcLbBlock - 1) / kZcLbBlock;
}
constexpr unsigned long long zc_enc_scratch_bytes(unsigned long long ntiles) {
  return (8 * ntiles + 15) / 16 * 16 + (8 * zc_enc_blocks(ntiles) + 15) / 16 * 16;
}
constexpr int kThreads = 256;           // 16 lanes per thread

// Per-segment record of a plan, in device memory (64 bytes).
struct ZcSegDev {
  unsigned long long elem_start, nelem, chunk_start, nchunks;
  unsigned long long unit_start;  // first statistics unit of the segment
  unsigned char book[8];          // 7 ascending exponent fields + 0
  double mu, sigma;
};
static_assert(sizeof(ZcSegDev) == 64, "segment record is 64 bytes");

// The encoder's 256-entry classification table of a segment (entry e for
// exponent field e): the 3-bit code's bits at bits 0, 8 and 16, or bit 24
// for an escape.  Shifting an entry left by the element's index (0..7) drops
// its bits into four per-plane bytes.  A plan keeps each segment's table
// after its segment records, in the same device allocation (zc_seg_luts),
// written wherever the codebook is set.
__host__ __device__ inline uint32_t zc_lut_entry(const unsigned char* book, uint32_t e) {
  uint32_t code = 0;
  for (int j = 0; j < 7; ++j)
    if (book[j] == e) code = (uint32_t)j + 1;
  if (code == 0) return 1u << 24;
  return (code & 1u) | (((code >> 1) & 1u) << 8) | (((code >> 2) & 1u) << 16);
}
__host__ __device__ inline uint32_t* zc_seg_luts(ZcSegDev* segs, uint32_t nseg) {
  return reinterpret_cast<uint32_t*>(segs + nseg);
}
__host__ __device__ inline const uint32_t* zc_seg_luts(const ZcSegDev* segs, uint32_t nseg) {
  return reinterpret_cast<const uint32_t*>(segs + nseg);
}
// After the tables: the segment of every chunk (one word per chunk).
__host__ __device__ inline uint32_t* zc_chunk_seg(ZcSegDev* segs, uint32_t nseg) {
  return zc_seg_luts(segs, nseg) + 256ull * nseg;
}
__host__ __device__ inline const uint32_t* zc_chunk_seg(const ZcSegDev* segs, uint32_t nseg) {
  return zc_seg_luts(segs, nseg) + 256ull * nseg;
}

struct ZcLayout {
  unsigned long long n, nchunks, ntiles, nunits;
  uint32_t nseg, C, log2C, U;  // U: elements per statistics unit
  unsigned long long off_seg, off_escoff, off_static, off_esc;
  unsigned long long slot_bytes;
  // predictor blocks per segment over unit partials (plan) and over chunk
  // partials (fit): each block adds a fixed range of at most 1024 partials
  uint32_t kred_u, kred_c;
};

// Predictor blocks per segment for `maxparts` partials in the largest segment.
inline uint32_t zc_red_blocks(unsigned long long maxparts) {
  const unsigned long long k = (maxparts + 1023) / 1024;
  return k < 1 ? 1u : (k > 128 ? 128u : (uint32_t)k);
}

// One partial of the statistics pass (one unit of U elements).
struct StatPartial {
  unsigned long long cnt;
  double s1, s2;
};

inline unsigned long long round_up(unsigned long long v, unsigned long long a) {
  return (v + a - 1) / a * a;
}

cudaError_t zc_launch_plan(const ZcLayout& L, const ZcSegDev* d_segs,
                           const uint16_t* d_x, void* d_ws, cudaStream_t s);
// fit: the encoder also sums each chunk's finite values (count, sum, sum of
// squares) into partials after its scratch, and the predictor then replaces
// the plan's statistics and codebooks from them (zc_compress_fit).
cudaError_t zc_launch_compress(const ZcLayout& L, const ZcSegDev* d_segs,
                               const uint16_t* d_x, void* d_out,
                               unsigned long long out_cap,
                               unsigned long long* d_out_bytes, void* d_ws,
                               cudaStream_t s, bool fit = false);
// The predictor over per-chunk partials (the second launch of a fit).
cudaError_t zc_launch_predict_chunks(const ZcLayout& L, ZcSegDev* d_segs,
                                     const StatPartial* d_parts, void* d_ws, cudaStream_t s);
// Offset of the per-chunk statistics partials in an encoder workspace.
constexpr unsigned long long zc_fit_parts_offset(unsigned long long ntiles) {
  return 256 + (zc_enc_scratch_bytes(ntiles) + 15) / 16 * 16;
}
// The predictor's per-block totals (nseg * max(kred_u, kred_c) partials) and
// one block counter per segment follow the partials of the plan or the fit.
inline unsigned long long zc_red_offset(const ZcLayout& L) {
  const unsigned long long a = 256 + L.nunits * sizeof(StatPartial);
  const unsigned long long b = zc_fit_parts_offset(L.ntiles) + L.nchunks * sizeof(StatPartial);
  return round_up(a > b ? a : b, 256);
}
inline unsigned long long zc_cnt_offset(const ZcLayout& L) {
  const unsigned long long k = L.kred_u > L.kred_c ? L.kred_u : L.kred_c;
  return round_up(zc_red_offset(L) + (unsigned long long)L.nseg * k * sizeof(StatPartial), 256);
}
cudaError_t zc_launch_decompress(const void* d_in, unsigned long long in_bytes,
                                 uint16_t* d_y, unsigned long long y_cap,
                                 void* d_ws, cudaStream_t s);

// ---------------------------------------------------------------- IBP

constexpr uint32_t kIbpmMagic = 0x4D504249u;  // "IBPM"
constexpr uint32_t kIbp1Magic = 0x31504249u;  // "IBP1"
constexpr uint32_t kIbpmHeader = 64;
constexpr uint32_t kIbp1Header = 128;

cudaError_t ibp_launch_build_meta(const void* d_samples, unsigned long long N,
                                  uint32_t chunk_bytes, unsigned long long k,
                                  double T, int mode, void* d_meta, void* d_ws,
                                  cudaStream_t s);
// x_host: d_x is pinned host memory, read with plain loads by the
// single-kernel encoder (no bulk copies from system memory).
cudaError_t ibp_launch_compress(const void* d_meta, uint32_t chunk_bytes,
                                const void* d_x, unsigned long long n_bytes,
                                void* d_out, unsigned long long out_cap,
                                unsigned long long* d_out_bytes, void* d_ws,
                                cudaStream_t s, bool x_host);
// in_host: d_in is pinned host memory, read in place over the host link by
// the plain-load decoder (no bulk copies from system memory).
cudaError_t ibp_launch_decompress(const void* d_meta, uint32_t chunk_bytes,
                                  const void* d_in, unsigned long long in_bytes,
                                  void* d_y, unsigned long long y_cap,
                                  void* d_ws, cudaStream_t s, bool in_host);

// IBP in-place slots (ibp_slots.cu): the slot form of every chunk of d_x
// (which may be d_slots itself) and the bitmask of compressed slots; the
// gather of the chunks d_idx[0..n_idx) from their slots into rows of d_y.
cudaError_t ibp_launch_slots_compress(const void* d_meta, uint32_t chunk_bytes, const void* d_x,
                                      unsigned long long n_bytes, void* d_slots,
                                      uint32_t* d_bitmask, void* d_ws, cudaStream_t s);
cudaError_t ibp_launch_slots_gather(const void* d_meta, uint32_t chunk_bytes, const void* d_slots,
                                    unsigned long long n_bytes, const uint32_t* d_bitmask,
                                    const unsigned long long* d_idx, unsigned long long n_idx,
                                    void* d_y, unsigned long long* d_read_bytes, void* d_ws,
                                    cudaStream_t s);

// TMA-pipelined IBP kernels (ibp_pipe.cu) for chunks of up to 2048 bytes;
// the launchers above use them whenever ibp_pipe_supported says so.
bool ibp_pipe_supported(uint32_t chunk_bytes, bool encode);
// Test switch (zc_test_ibp_single_pass): 0 sends chunks of up to 512 bytes to
// the three-launch encode, the path taken when the single-pass encoder's grid
// cannot be resident at once.
void ibp_set_single_pass(int on);
// Waves between a group's match and its packing in the single-pass encoder
// for 1024- and 2048-byte chunks (1..3; tests and measurements).
void ibp_set_wsp_lag(int lag);
cudaError_t ibp_pipe_compress(const void* d_meta, uint32_t chunk_bytes, const void* d_x,
                              unsigned long long n_bytes, void* d_out,
                              unsigned long long out_cap, unsigned long long* d_out_bytes,
                              void* d_ws, cudaStream_t s);
cudaError_t ibp_pipe_decompress(const void* d_meta, uint32_t chunk_bytes, const void* d_in,
                                unsigned long long in_bytes, void* d_y,
                                unsigned long long y_cap, void* d_ws, cudaStream_t s);

// Wait-failure test switch (zc_test_wait_fault): when armed, writes the
// fault tile and the poll limit into the control block of the workspace at
// d_ws, after the launcher has cleared it; otherwise does nothing.
cudaError_t arm_wait_fault(void* d_ws, cudaStream_t s);

// Blocks of `kernel` resident per SM times SMs on the current device.
int resident_blocks(const void* kernel, int threads, size_t smem);

// Launches a kernel that depends on the kernel launched just before it on the
// same stream with programmatic stream serialization: its blocks may start
// while that kernel finishes, and must call grid_dep_wait() (common.cuh)
// before reading what it wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*k)(KArgs...), unsigned grid, unsigned threads, size_t smem,
                             cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace lbb

// A ZipCCL plan (the opaque zc_plan_t of zc.h): layout, the device segment
// table the kernels read, and its host copy.
struct zc_plan_s {
  int device;
  lbb::ZcLayout L;
  lbb::ZcSegDev* d_segs;
  std::vector<lbb::ZcSegDev> h_segs;
};
