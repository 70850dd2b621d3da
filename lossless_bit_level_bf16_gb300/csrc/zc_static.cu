// zc_static.cu -- zc_compress_static: ZipCCL encoding without a caller
// workspace.  The encoder's scratch (its status/ticket block and one
// look-back word per 8192-slot tile and per block of 128 tiles) lives in a
// fixed array in device memory
// that belongs to the library, so this entry point allocates nothing and
// needs no workspace from the caller.  The encoding itself is the one
// zc_compress runs (same launcher, same kernel, same stream bytes).
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "zc.h"

namespace {

// 1 MiB: the 256-byte control block, then the encoder's look-back states,
// enough for plans of up to 130,024 tiles of 8192 slots (1,065,156,608 slots).
constexpr size_t kStaticScratchBytes = 1u << 20;
constexpr unsigned long long kStaticMaxTiles = 130024;
static_assert(lbb::kCtrlBytes + lbb::zc_enc_scratch_bytes(kStaticMaxTiles) <= kStaticScratchBytes &&
                  lbb::kCtrlBytes + lbb::zc_enc_scratch_bytes(kStaticMaxTiles + 1) > kStaticScratchBytes,
              "the largest plan the fixed scratch holds");
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_zc_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// The array's device address on the current device.  Outside a stream
// capture it is looked up on every call (with that device current): a device
// reset reloads the library's module, and the array may then sit elsewhere.
// During a capture the address the last such lookup found is used.
int scratch_for_current_device(cudaStream_t s, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ZC_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();  // e.g. the legacy stream while another stream captures
    cs = cudaStreamCaptureStatusActive;
  }
  std::lock_guard<std::mutex> g(g_mu);
  if (cs == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_zc_scratch) != cudaSuccess || !p) return ZC_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ZC_OK;
}

}  // namespace

extern "C" int zc_compress_static(zc_plan_t p, const uint16_t* d_x, void* d_out,
                                  uint64_t out_cap, uint64_t* d_out_bytes, int* d_status,
                                  zc_stream_t stream) {
  if (!p || !d_out || (!d_x && p->L.n)) return ZC_ERR_ARG;
  const auto al = [](const void* q, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0;
  };
  if (!al(d_out, 16) || !al(d_x, 2) || !al(d_out_bytes, 8) || !al(d_status, 4)) return ZC_ERR_ARG;
  if (p->L.ntiles > kStaticMaxTiles) return ZC_ERR_CAPACITY;
  if (out_cap < p->L.off_esc) return ZC_ERR_CAPACITY;
  const cudaStream_t s = (cudaStream_t)stream;
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(s, &scratch);
  if (rc != ZC_OK) return rc;
  // the launcher clears the control block and the look-back words it uses
  cudaError_t e = lbb::zc_launch_compress(p->L, p->d_segs, d_x, d_out, out_cap,
                                          reinterpret_cast<unsigned long long*>(d_out_bytes),
                                          scratch, s);
  if (e == cudaSuccess && d_status)
    e = cudaMemcpyAsync(d_status, scratch, sizeof(int), cudaMemcpyDeviceToDevice, s);
  return e == cudaSuccess ? ZC_OK : ZC_ERR_CUDA;
}
