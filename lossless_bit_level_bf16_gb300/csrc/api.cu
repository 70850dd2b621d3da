// api.cu -- the C ABI declared in include/zc.h: argument checks, plan objects,
// workspace sizing and kernel launches.  No arithmetic of the codecs lives
// here; see zc_plan.cu, zc_codec.cu, ibp_meta.cu and ibp_codec.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstddef>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "zc.h"

namespace lbb {

int resident_blocks(const void* kernel, int threads, size_t smem) {
  struct Entry {
    const void* k;
    int dev, threads;
    size_t smem;
    int blocks;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> g(mu);
    for (const Entry& e : cache)
      if (e.k == kernel && e.dev == dev && e.threads == threads && e.smem == smem) return e.blocks;
  }
  int sms = 1, per = 1;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, threads, smem) != cudaSuccess ||
      per < 1)
    per = 1;
  const int blocks = per * sms;
  std::lock_guard<std::mutex> g(mu);
  cache.push_back(Entry{kernel, dev, threads, smem, blocks});
  return blocks;
}

namespace {
std::atomic<unsigned long long> g_fault_tile1{0};
std::atomic<unsigned> g_fault_spins{0};
}  // namespace

cudaError_t arm_wait_fault(void* d_ws, cudaStream_t s) {
  const unsigned long long f = g_fault_tile1.load();
  const unsigned sp = g_fault_spins.load();
  if (!f && !sp) return cudaSuccess;
  struct {
    unsigned long long fault_tile1;
    unsigned max_spins, pad1;
  } v{f, sp, 0};
  static_assert(sizeof(v) == 16, "two fields of Ctrl");
  return cudaMemcpyAsync(static_cast<char*>(d_ws) + offsetof(Ctrl, fault_tile1), &v, sizeof(v),
                         cudaMemcpyHostToDevice, s);
}

}  // namespace lbb

namespace {

using lbb::kCtrlBytes;

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? ZC_OK : ZC_ERR_CUDA; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Whether the GPU can reach *p: device memory, or pinned host memory (then
// *host is set and *p becomes its device-side address).  Unregistered host
// memory is not reachable.
bool reachable(const void** p, bool* host) {
  *host = false;
  if (!*p) return true;
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, *p) != cudaSuccess) {
    cudaGetLastError();  // clear the lookup's error; treat as device memory
    return true;
  }
  if (pa.type == cudaMemoryTypeUnregistered) return false;
  if (pa.type == cudaMemoryTypeHost) {
    *host = true;
    if (pa.devicePointer) *p = pa.devicePointer;
  }
  return true;
}

// The classification tables of the codebooks in p->h_segs, after the segment
// records on the device.
int upload_luts(zc_plan_s* p) {
  std::vector<uint32_t> luts(256ull * p->L.nseg);
  for (uint32_t s = 0; s < p->L.nseg; ++s)
    for (uint32_t e = 0; e < 256; ++e) luts[256ull * s + e] = lbb::zc_lut_entry(p->h_segs[s].book, e);
  return cudaMemcpy(lbb::zc_seg_luts(p->d_segs, p->L.nseg), luts.data(), 4ull * luts.size(),
                    cudaMemcpyHostToDevice) == cudaSuccess
             ? ZC_OK
             : ZC_ERR_CUDA;
}

// Workspace of a plan: the control block, then the statistics partials (one
// per unit) or the encoder's look-back words followed by one statistics
// partial per chunk (zc_compress_fit), whichever is larger; then the
// predictor's per-block totals and one block counter per segment.
size_t zc_ws_bytes(const lbb::ZcLayout& L) {
  return (size_t)lbb::round_up_dev(lbb::zc_cnt_offset(L) + 4ull * L.nseg, 256);
}

}  // namespace

extern "C" {

const char* zc_strerror(int code) {
  switch (code) {
    case ZC_OK: return "ok";
    case ZC_ERR_ARG: return "invalid argument";
    case ZC_ERR_CAPACITY: return "output or workspace buffer too small";
    case ZC_ERR_FORMAT: return "stream is corrupt or inconsistent";
    case ZC_ERR_META_MISMATCH: return "stream was made with other IBP metadata";
    case ZC_ERR_TIMEOUT: return "a bounded wait between thread blocks ran out";
    case ZC_ERR_CUDA: return "CUDA runtime error";
    case ZC_ERR_UNSUPPORTED: return "parameter legal in the format but not supported by the GPU path";
    case ZC_ERR_NOMEM: return "allocation failed";
    default: return "unknown error";
  }
}

int zc_version(void) { return 100; }

int zc_test_ibp_single_pass(int enable) {
  lbb::ibp_set_single_pass(enable);
  return ZC_OK;
}

int zc_test_wait_fault(uint64_t tile, uint32_t max_spins) {
  lbb::g_fault_tile1.store(tile == UINT64_MAX ? 0ull : tile + 1);
  lbb::g_fault_spins.store(max_spins);
  return ZC_OK;
}

int zc_status(const void* d_ws, zc_stream_t stream, int* h_status) {
  if (!d_ws || !h_status) return ZC_ERR_ARG;
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, d_ws, sizeof(int), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return ZC_ERR_CUDA;
  *h_status = v;
  return ZC_OK;
}

// ------------------------------------------------------------------ ZipCCL

int zc_plan_create(uint64_t n, const uint64_t* h_seg_off, uint32_t nseg, uint32_t C,
                   zc_plan_t* out_plan) {
  if (!out_plan) return ZC_ERR_ARG;
  *out_plan = nullptr;
  if (nseg == 0 || (!h_seg_off && nseg != 1)) return ZC_ERR_ARG;
  if (C < 1024u || C > 65536u || (C % 1024u) != 0) return ZC_ERR_ARG;
  if (n > (1ull << 46)) return ZC_ERR_ARG;
  if (h_seg_off) {
    if (h_seg_off[0] != 0 || h_seg_off[nseg] != n) return ZC_ERR_ARG;
    for (uint32_t s = 0; s < nseg; ++s)
      if (h_seg_off[s + 1] < h_seg_off[s]) return ZC_ERR_ARG;
  }
  zc_plan_s* p = new (std::nothrow) zc_plan_s();
  if (!p) return ZC_ERR_NOMEM;
  lbb::ZcLayout& L = p->L;
  L.n = n;
  L.nseg = nseg;
  L.C = C;
  L.log2C = 0;
  while ((1u << L.log2C) < C) ++L.log2C;
  // statistics unit: a power of two between 4096 and 16384 elements, fixed by
  // n (one warp of the statistics kernel; small units keep its tail short:
  // 16384 units or more once they are 16384 elements)
  unsigned long long U = 4096;
  while (U < 16384 && U * 2 <= n / 16384) U *= 2;
  L.U = (uint32_t)U;
  try {
    p->h_segs.resize(nseg);
  } catch (...) {
    delete p;
    return ZC_ERR_NOMEM;
  }
  unsigned long long chunks = 0, units = 0, max_units = 0, max_chunks = 0;
  for (uint32_t s = 0; s < nseg; ++s) {
    const unsigned long long b = h_seg_off ? h_seg_off[s] : 0;
    const unsigned long long e = h_seg_off ? h_seg_off[s + 1] : n;
    lbb::ZcSegDev& r = p->h_segs[s];
    std::memset(&r, 0, sizeof r);
    r.elem_start = b;
    r.nelem = e - b;
    r.chunk_start = chunks;
    r.nchunks = (r.nelem + C - 1) / C;
    r.unit_start = units;
    chunks += r.nchunks;
    units += (r.nelem + U - 1) / U;
    max_units = std::max(max_units, (r.nelem + U - 1) / U);
    max_chunks = std::max(max_chunks, r.nchunks);
  }
  L.nchunks = chunks;
  L.nunits = units;
  L.kred_u = lbb::zc_red_blocks(max_units);
  L.kred_c = lbb::zc_red_blocks(max_chunks);
  const unsigned long long tl = lbb::zc_tile_slots(C);
  L.ntiles = (chunks * C + tl - 1) / tl;
  L.slot_bytes = (unsigned long long)C * 11ull / 8ull;
  L.off_seg = lbb::kZcHeader;
  L.off_escoff = L.off_seg + lbb::round_up_dev((unsigned long long)lbb::kZcSegRec * nseg, lbb::kZcAlign);
  L.off_static = L.off_escoff + lbb::round_up_dev(8ull * (chunks + 1), lbb::kZcAlign);
  L.off_esc = L.off_static + chunks * L.slot_bytes;
  if (units > 0x7FFFFFFFull) {
    delete p;
    return ZC_ERR_ARG;
  }
  cudaGetDevice(&p->device);
  // segment records, each segment's classification table, the segment of
  // every chunk
  if (cudaMalloc(&p->d_segs, (sizeof(lbb::ZcSegDev) + 1024) * nseg + 4ull * chunks) != cudaSuccess) {
    delete p;
    return ZC_ERR_NOMEM;
  }
  std::vector<uint32_t> cseg;
  try {
    cseg.resize(chunks);
  } catch (...) {
    cudaFree(p->d_segs);
    delete p;
    return ZC_ERR_NOMEM;
  }
  for (uint32_t s = 0; s < nseg; ++s)
    for (unsigned long long c = 0; c < p->h_segs[s].nchunks; ++c) cseg[p->h_segs[s].chunk_start + c] = s;
  if (cudaMemcpy(p->d_segs, p->h_segs.data(), sizeof(lbb::ZcSegDev) * nseg,
                 cudaMemcpyHostToDevice) != cudaSuccess ||
      upload_luts(p) != ZC_OK ||
      (chunks && cudaMemcpy(lbb::zc_chunk_seg(p->d_segs, nseg), cseg.data(), 4ull * chunks,
                            cudaMemcpyHostToDevice) != cudaSuccess)) {
    cudaFree(p->d_segs);
    delete p;
    return ZC_ERR_CUDA;
  }
  *out_plan = p;
  return ZC_OK;
}

void zc_plan_destroy(zc_plan_t p) {
  if (!p) return;
  cudaFree(p->d_segs);
  delete p;
}

size_t zc_workspace_bytes(zc_plan_t p) { return p ? zc_ws_bytes(p->L) : 0; }

uint64_t zc_max_compressed_bytes(zc_plan_t p) {
  if (!p) return 0;
  // dynamic bytes: a full chunk at most 5C/8 (beyond that it is stored raw),
  // a segment's short last chunk one escape per element
  const unsigned long long C = p->L.C;
  unsigned long long dyn = 0;
  for (const lbb::ZcSegDev& r : p->h_segs) dyn += (r.nelem / C) * (5 * C / 8) + r.nelem % C;
  return p->L.off_esc + lbb::round_up_dev(dyn, lbb::kZcAlign);
}

int zc_plan(zc_plan_t p, const uint16_t* d_x, void* d_ws, size_t ws_bytes, zc_stream_t stream) {
  if (!p || !d_ws || (!d_x && p->L.n) || !aligned(d_ws, 256) || !aligned(d_x, 2)) return ZC_ERR_ARG;
  if (ws_bytes < zc_ws_bytes(p->L)) return ZC_ERR_CAPACITY;
  cudaError_t e = cudaMemsetAsync(d_ws, 0, kCtrlBytes, (cudaStream_t)stream);
  if (e == cudaSuccess) e = lbb::zc_launch_plan(p->L, p->d_segs, d_x, d_ws, (cudaStream_t)stream);
  return cuda_rc(e);
}

int zc_plan_set_books(zc_plan_t p, const uint8_t* h_books) {
  if (!p || !h_books) return ZC_ERR_ARG;
  for (uint32_t s = 0; s < p->L.nseg; ++s)
    for (int j = 1; j < 7; ++j)
      if (h_books[7 * s + j] <= h_books[7 * s + j - 1]) return ZC_ERR_ARG;
  std::vector<lbb::ZcSegDev> segs(p->L.nseg);
  if (cudaMemcpy(segs.data(), p->d_segs, sizeof(lbb::ZcSegDev) * p->L.nseg,
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return ZC_ERR_CUDA;
  for (uint32_t s = 0; s < p->L.nseg; ++s) {
    std::memcpy(segs[s].book, h_books + 7 * s, 7);
    segs[s].book[7] = 0;
    std::memcpy(p->h_segs[s].book, segs[s].book, 8);
  }
  if (cudaMemcpy(p->d_segs, segs.data(), sizeof(lbb::ZcSegDev) * p->L.nseg,
                 cudaMemcpyHostToDevice) != cudaSuccess)
    return ZC_ERR_CUDA;
  return upload_luts(p);
}

int zc_plan_info(zc_plan_t p, zc_stream_t stream, uint8_t* h_books, double* h_mu_sigma) {
  if (!p) return ZC_ERR_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return ZC_ERR_CUDA;
  std::vector<lbb::ZcSegDev> segs(p->L.nseg);
  if (cudaMemcpy(segs.data(), p->d_segs, sizeof(lbb::ZcSegDev) * p->L.nseg,
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return ZC_ERR_CUDA;
  for (uint32_t s = 0; s < p->L.nseg; ++s) {
    if (h_books) std::memcpy(h_books + 7 * s, segs[s].book, 7);
    if (h_mu_sigma) {
      h_mu_sigma[2 * s] = segs[s].mu;
      h_mu_sigma[2 * s + 1] = segs[s].sigma;
    }
  }
  return ZC_OK;
}

int zc_compress(zc_plan_t p, const uint16_t* d_x, void* d_out, uint64_t out_cap,
                uint64_t* d_out_bytes, void* d_ws, size_t ws_bytes, zc_stream_t stream) {
  if (!p || !d_out || !d_ws || (!d_x && p->L.n)) return ZC_ERR_ARG;
  if (!aligned(d_out, 16) || !aligned(d_ws, 256) || !aligned(d_x, 2) || !aligned(d_out_bytes, 8))
    return ZC_ERR_ARG;
  if (ws_bytes < zc_ws_bytes(p->L)) return ZC_ERR_CAPACITY;
  if (out_cap < p->L.off_esc) return ZC_ERR_CAPACITY;
  return cuda_rc(lbb::zc_launch_compress(p->L, p->d_segs, d_x, d_out, out_cap,
                                         reinterpret_cast<unsigned long long*>(d_out_bytes), d_ws,
                                         (cudaStream_t)stream));
}

int zc_compress_fit(zc_plan_t p, const uint16_t* d_x, void* d_out, uint64_t out_cap,
                    uint64_t* d_out_bytes, void* d_ws, size_t ws_bytes, zc_stream_t stream) {
  if (!p || !d_out || !d_ws || (!d_x && p->L.n)) return ZC_ERR_ARG;
  if (!aligned(d_out, 16) || !aligned(d_ws, 256) || !aligned(d_x, 2) || !aligned(d_out_bytes, 8))
    return ZC_ERR_ARG;
  if (ws_bytes < zc_ws_bytes(p->L)) return ZC_ERR_CAPACITY;
  if (out_cap < p->L.off_esc) return ZC_ERR_CAPACITY;
  return cuda_rc(lbb::zc_launch_compress(p->L, p->d_segs, d_x, d_out, out_cap,
                                         reinterpret_cast<unsigned long long*>(d_out_bytes), d_ws,
                                         (cudaStream_t)stream, true));
}

size_t zc_decompress_workspace_bytes(void) { return kCtrlBytes; }

int zc_decompress(const void* d_in, uint64_t in_bytes, uint16_t* d_y, uint64_t y_cap_elems,
                  void* d_ws, size_t ws_bytes, zc_stream_t stream) {
  if (!d_in || !d_ws || (!d_y && y_cap_elems)) return ZC_ERR_ARG;
  if (!aligned(d_in, 16) || !aligned(d_ws, 256) || !aligned(d_y, 2)) return ZC_ERR_ARG;
  if (ws_bytes < kCtrlBytes) return ZC_ERR_CAPACITY;
  return cuda_rc(lbb::zc_launch_decompress(d_in, in_bytes, d_y, y_cap_elems, d_ws,
                                           (cudaStream_t)stream));
}

// ------------------------------------------------------------------ IBP

uint64_t ibp_meta_bytes(uint32_t chunk_bytes) {
  return lbb::kIbpmHeader + 2ull * chunk_bytes;
}

// Any multiple of 4 bytes up to 4096: multiples of 16 up to 2048 take the
// TMA-pipelined kernels, the others the word-granular ones.
static bool ibp_chunk_ok(uint32_t cb) { return cb >= 4 && cb <= 4096 && (cb % 4) == 0; }

size_t ibp_workspace_bytes(uint32_t cb, uint64_t n_bytes, uint64_t n_samples) {
  if (!ibp_chunk_ok(cb)) return 0;
  const unsigned long long nch = (n_bytes + cb - 1) / cb;
  const unsigned long long ng = (nch + 31) / 32;
  // look-back states per group (chunks above 2048 bytes), or the encode's
  // offsets-pass states and one participation word per group
  const unsigned long long codec = 8ull * ng + 512;
  const unsigned long long B = 8ull * cb;
  const unsigned long long words = (n_samples + 31) / 32;
  const unsigned long long meta = 8ull * B + 4ull * B * words;      // counts + columns
  return (size_t)lbb::round_up_dev(kCtrlBytes + std::max(codec, meta), 256);
}

uint64_t ibp_max_compressed_bytes(uint32_t cb, uint64_t n_bytes) {
  if (!ibp_chunk_ok(cb)) return 0;
  const unsigned long long nch = (n_bytes + cb - 1) / cb;
  const unsigned long long ng = (nch + 31) / 32;
  // every chunk raw, 4 bytes of participation bits and up to 15 bytes of
  // padding per group
  return lbb::kIbp1Header + lbb::round_up_dev(8ull * (ng + 1), 128) + n_bytes + 20ull * ng + 16;
}

int ibp_build_meta(const void* d_samples, uint64_t n_samples, uint32_t cb, double T, int mode,
                   void* d_meta, void* d_ws, size_t ws_bytes, zc_stream_t stream) {
  if (!d_samples || !d_meta || !d_ws || n_samples == 0) return ZC_ERR_ARG;
  if (!ibp_chunk_ok(cb) || !(T > 0.5 && T <= 1.0) || (mode != 0 && mode != 1)) return ZC_ERR_ARG;
  if (mode == 1 && (cb > 2048 || n_samples > 262144)) return ZC_ERR_UNSUPPORTED;
  if (n_samples >= (1ull << 32)) return ZC_ERR_UNSUPPORTED;
  if (!aligned(d_samples, 16) || !aligned(d_meta, 16) || !aligned(d_ws, 256)) return ZC_ERR_ARG;
  if (ws_bytes < ibp_workspace_bytes(cb, 0, n_samples)) return ZC_ERR_CAPACITY;
  const unsigned long long k = (unsigned long long)std::ceil(T * (double)n_samples);
  return cuda_rc(lbb::ibp_launch_build_meta(d_samples, n_samples, cb, k, T, mode, d_meta, d_ws,
                                            (cudaStream_t)stream));
}

int ibp_compress(const void* d_meta, uint32_t cb, const void* d_x, uint64_t n_bytes, void* d_out,
                 uint64_t out_cap, uint64_t* d_out_bytes, void* d_ws, size_t ws_bytes,
                 zc_stream_t stream) {
  if (!d_meta || !d_out || !d_ws || (!d_x && n_bytes) || !ibp_chunk_ok(cb) || (n_bytes % 4) != 0)
    return ZC_ERR_ARG;
  if (!aligned(d_meta, 16) || !aligned(d_x, 16) || !aligned(d_out, 16) || !aligned(d_ws, 256) ||
      !aligned(d_out_bytes, 8))
    return ZC_ERR_ARG;
  if (ws_bytes < ibp_workspace_bytes(cb, n_bytes, 0)) return ZC_ERR_CAPACITY;
  const unsigned long long nch = (n_bytes + cb - 1) / cb, ng = (nch + 31) / 32;
  if (out_cap < lbb::kIbp1Header + lbb::round_up_dev(8ull * (ng + 1), 128)) return ZC_ERR_CAPACITY;
  // input and stream may be pinned host memory (zero-copy)
  bool x_host = false, out_host = false;
  const void* o = d_out;
  if (!reachable(&d_x, &x_host) || !reachable(&o, &out_host)) return ZC_ERR_ARG;
  d_out = const_cast<void*>(o);
  return cuda_rc(lbb::ibp_launch_compress(d_meta, cb, d_x, n_bytes, d_out, out_cap,
                                          reinterpret_cast<unsigned long long*>(d_out_bytes),
                                          d_ws, (cudaStream_t)stream, x_host));
}

int ibp_decompress(const void* d_meta, uint32_t cb, const void* d_in, uint64_t in_bytes,
                   void* d_y, uint64_t y_cap, void* d_ws, size_t ws_bytes, zc_stream_t stream) {
  if (!d_meta || !d_in || !d_ws || (!d_y && y_cap) || !ibp_chunk_ok(cb)) return ZC_ERR_ARG;
  if (!aligned(d_meta, 16) || !aligned(d_in, 16) || !aligned(d_y, 16) || !aligned(d_ws, 256))
    return ZC_ERR_ARG;
  if (ws_bytes < kCtrlBytes) return ZC_ERR_CAPACITY;
  // the stream may stay in pinned host memory: it is then read in place
  bool in_host = false, out_host = false;
  const void* yo = d_y;
  if (!reachable(&d_in, &in_host) || !reachable(&yo, &out_host)) return ZC_ERR_ARG;
  d_y = const_cast<void*>(yo);
  return cuda_rc(lbb::ibp_launch_decompress(d_meta, cb, d_in, in_bytes, d_y, y_cap, d_ws,
                                            (cudaStream_t)stream, in_host));
}

int ibp_slots_compress(const void* d_meta, uint32_t cb, const void* d_x, uint64_t n_bytes,
                       void* d_slots, uint32_t* d_bitmask, void* d_ws, size_t ws_bytes,
                       zc_stream_t stream) {
  if (!d_meta || !d_slots || !d_bitmask || !d_ws || (!d_x && n_bytes) || !ibp_chunk_ok(cb) ||
      (n_bytes % 4) != 0)
    return ZC_ERR_ARG;
  if (!aligned(d_meta, 16) || !aligned(d_x, 4) || !aligned(d_slots, 4) || !aligned(d_bitmask, 4) ||
      !aligned(d_ws, 256))
    return ZC_ERR_ARG;
  if (ws_bytes < kCtrlBytes) return ZC_ERR_CAPACITY;
  // the input is the slots themselves (compression in place) or apart from them
  const char* xb = static_cast<const char*>(d_x);
  const char* sb = static_cast<const char*>(d_slots);
  if (xb != sb && xb < sb + n_bytes && sb < xb + n_bytes) return ZC_ERR_ARG;
  bool x_host = false, s_host = false;
  const void* sl = d_slots;
  if (!reachable(&d_x, &x_host) || !reachable(&sl, &s_host)) return ZC_ERR_ARG;
  if (xb == sb) d_x = sl;  // the same memory, by its device-side address
  return cuda_rc(lbb::ibp_launch_slots_compress(d_meta, cb, d_x, n_bytes, const_cast<void*>(sl),
                                                d_bitmask, d_ws, (cudaStream_t)stream));
}

int ibp_slots_gather(const void* d_meta, uint32_t cb, const void* d_slots, uint64_t n_bytes,
                     const uint32_t* d_bitmask, const uint64_t* d_idx, uint64_t n_idx, void* d_y,
                     uint64_t* d_read_bytes, void* d_ws, size_t ws_bytes, zc_stream_t stream) {
  if (!d_meta || !d_slots || !d_bitmask || !d_ws || (!d_idx && n_idx) || (!d_y && n_idx) ||
      !ibp_chunk_ok(cb) || (n_bytes % 4) != 0)
    return ZC_ERR_ARG;
  if (!aligned(d_meta, 16) || !aligned(d_slots, 4) || !aligned(d_bitmask, 4) ||
      !aligned(d_idx, 8) || !aligned(d_y, 4) || !aligned(d_read_bytes, 8) || !aligned(d_ws, 256))
    return ZC_ERR_ARG;
  if (ws_bytes < kCtrlBytes) return ZC_ERR_CAPACITY;
  bool s_host = false, y_host = false;
  const void* yo = d_y;
  if (!reachable(&d_slots, &s_host) || !reachable(&yo, &y_host)) return ZC_ERR_ARG;
  return cuda_rc(lbb::ibp_launch_slots_gather(
      d_meta, cb, d_slots, n_bytes, d_bitmask, reinterpret_cast<const unsigned long long*>(d_idx),
      n_idx, const_cast<void*>(yo), reinterpret_cast<unsigned long long*>(d_read_bytes), d_ws,
      (cudaStream_t)stream));
}

}  // extern "C"
