// ibp_codec.cu -- IBP invariant bit packing: encode and decode kernels.
//
// [IBP] = "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria
// GPU con la Compressione Lossless per il ML", Metodologia: Invariant Bit
// Packing (IBP), Algoritmo Core:
//   2 (Compressione)  per chunk, compare the invariant positions with Bitval;
//     on a match drop those bits and close the gap; a participation bit tells
//     whether the chunk was compressed (raw when compression saves nothing);
//   3 (Decompressione) a warp reads a contiguous compressed segment into
//     shared memory, a warp prefix scan of the chunk bit lengths gives each
//     chunk's start bit, and the Bitval bits are re-inserted.
//
// Stream "IBP1": header (128 B) | group bit offsets (u64, ngroups+1) |
// payload.  A group is 32 chunks: 32 participation bits, then the bodies, then
// zero bits up to a multiple of 128, so every group starts 16-byte aligned.
//
// GPU mapping: one block per group at a time (persistent blocks).  Each warp
// owns CPW chunks of the group; a lane owns WPL words of a chunk (VEC=4: four
// consecutive words per 16-byte access, VEC=1: one word, for chunk sizes that
// are not a multiple of 512 bytes).
//   encode: match test -> participation word -> group length -> aggregate
//     published for the decoupled look-back -> kept bits closed up
//     (compress) and OR-ed into the group image in shared memory -> look-back
//     resolves the group's bit offset -> 16-byte copy-out.
//   decode: group bytes staged into shared memory with 16-byte loads -> warp
//     prefix scan of the 32 chunk lengths -> every word re-expanded from its
//     bit offset with Bitval OR-ed in -> 16-byte stores.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ibp_common.cuh"
#include "internal.h"

namespace lbb {
namespace {

struct IbpEncArgs {
  const uint8_t* meta;
  const uint32_t* x;
  unsigned long long n_bytes, nchunks, ngroups;
  uint32_t cb;
  uint8_t* out;
  unsigned long long out_cap, off_payload;
  unsigned long long* out_bytes;
  Ctrl* ctrl;
  unsigned long long* states;
};

__host__ __device__ constexpr uint32_t ibp_group_words(uint32_t cb) {
  // 32 p-bits + 32 raw chunks, rounded up to 128 bits, plus one spare word
  return (uint32_t)(((32ull + 32ull * 8ull * cb + 127ull) / 128ull) * 4ull + 4ull);
}

// Word index of lane `lane`'s slot j within a chunk.
template <int VEC>
__device__ __forceinline__ uint32_t owned_word(int lane, int j) {
  if (VEC == 4) return (uint32_t)(128 * (j >> 2) + 4 * lane + (j & 3));
  return (uint32_t)(32 * j + lane);
}

template <int VEC, int WPL, int CPW>
__global__ void __launch_bounds__(32 * (32 / CPW)) ibp_encode_kernel(IbpEncArgs A) {
  constexpr int NT = 32 * (32 / CPW);
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ uint32_t s_scr[NT / 32 + 4];
  __shared__ uint32_t s_pword;
  __shared__ unsigned long long s_g, s_excl;
  __shared__ int s_last;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t cb = A.cb, W = cb / 4, B = cb * 8;

  IbpTables T;
  const bool ok = ibp_load_tables<NT>(A.meta, cb, dyn, T, s_scr);
  if (!ok) {
    if (t == 0) set_status(A.ctrl, ZC_ERR_META_MISMATCH);
  }
  uint32_t* gbuf = dyn + ibp_table_words(W);
  const uint32_t m = T.m;
  const unsigned long long tail_bytes = A.n_bytes - (A.nchunks ? (A.nchunks - 1) * cb : 0ull);
  for (uint32_t w = t; w < ibp_group_words(cb); w += NT) gbuf[w] = 0;
  __syncthreads();

  for (;;) {
    if (t == 0) {
      // the ticket is taken when the group starts (see the look-back notes)
      s_g = ok ? atomicAdd(&A.ctrl->ticket, 1ull) : A.ngroups;
      s_pword = 0;
    }
    __syncthreads();
    const unsigned long long g = s_g;
    if (g >= A.ngroups) break;
    const unsigned long long c0 = g * 32ull;
    const uint32_t nch = (uint32_t)(A.nchunks - c0 < 32 ? A.nchunks - c0 : 32);

    // ---- phase 1: load my chunks, participation bits
    uint32_t d[CPW][WPL];
#pragma unroll
    for (int r = 0; r < CPW; ++r) {
      const uint32_t i = (uint32_t)warp * CPW + r;
      const unsigned long long c = c0 + i;
      const bool present = i < nch;
      const bool full = present && (c + 1 < A.nchunks || tail_bytes == cb);
      const uint32_t wv = present ? (full ? W : (uint32_t)(tail_bytes / 4)) : 0u;
      const uint32_t* src = A.x + c * (unsigned long long)W;
      uint32_t bad = 0;
#pragma unroll
      for (int j = 0; j < WPL; j += VEC) {
        const uint32_t w = owned_word<VEC>(lane, j);
        if (VEC == 4 && w + 3 < wv) {
          const uint4 q = ld_nc_v4(src + w);
          d[r][j] = q.x;
          d[r][j + 1] = q.y;
          d[r][j + 2] = q.z;
          d[r][j + 3] = q.w;
        } else {
#pragma unroll
          for (int q = 0; q < VEC; ++q) d[r][j + q] = (w + q < wv) ? __ldg(src + w + q) : 0u;
        }
#pragma unroll
        for (int q = 0; q < VEC; ++q) {
          const uint32_t ww = w + q;
          if (ww < wv) bad |= (d[r][j + q] ^ T.V[ww]) & ~T.K[ww];
        }
      }
      const bool match = !__any_sync(kFull, bad != 0);
      if (lane == 0 && full && m > 0 && match) atomicOr(&s_pword, 1u << i);
    }
    __syncthreads();
    const uint32_t pword = s_pword;
    // group length: 32 + sum of body lengths (the short last chunk, if any,
    // is always raw and is the last chunk of the last group)
    const uint32_t np = __popc(pword);
    unsigned long long bits = 32ull + (unsigned long long)nch * B - (unsigned long long)np * m;
    if (c0 + nch == A.nchunks && tail_bytes != cb) bits -= 8ull * (cb - tail_bytes);
    const unsigned long long padded = round_up_dev(bits, 128);
    // publish the aggregate now; the look-back below resolves it later
    if (t == 0 && g > 0 && may_publish(A.ctrl, g)) st_relaxed_u64(A.states + g, kFlagAgg | padded);
    if (t == 0) gbuf[0] = pword;  // the image is all zeros here (cleared at copy-out)

    // ---- phase 2: close up kept bits into the group image
#pragma unroll
    for (int r = 0; r < CPW; ++r) {
      const uint32_t i = (uint32_t)warp * CPW + r;
      if (i >= nch) continue;
      const unsigned long long c = c0 + i;
      const bool full = c + 1 < A.nchunks || tail_bytes == cb;
      const uint32_t wv = full ? W : (uint32_t)(tail_bytes / 4);
      const bool p = (pword >> i) & 1u;
      const unsigned long long off =
          32ull + (unsigned long long)i * B - (unsigned long long)__popc(pword & ((1u << i) - 1u)) * m;
#pragma unroll
      for (int j = 0; j < WPL; ++j) {
        const uint32_t w = owned_word<VEC>(lane, j);
        if (w >= wv) continue;
        if (p) {
          const uint32_t K = T.K[w];
          const uint32_t k = __popc(K);
          if (k) put_bits(gbuf, off + T.P[w], hd_compress(d[r][j], K, T.MV + w, W), k);
        } else {
          put_bits(gbuf, off + 32ull * w, d[r][j], 32);
        }
      }
    }
    // ---- look-back for the group's bit offset
    if (warp == 0) {
      bool to = false;
      const unsigned long long e = lookback_warp_wide(A.states, g, padded, &to, wait_limit(A.ctrl),
                                                      may_publish(A.ctrl, g));
      if (lane == 0) {
        s_excl = e;
        if (to) set_status(A.ctrl, ZC_ERR_TIMEOUT);
      }
    }
    __syncthreads();
    const unsigned long long gpos = s_excl;  // bits, multiple of 128
    const unsigned long long dst = A.off_payload + (gpos >> 3);
    const unsigned long long nbytes = padded >> 3;
    {
      // copy the image out and clear it for the next group in the same pass
      uint4* s4 = reinterpret_cast<uint4*>(gbuf);
      const bool fits = dst + nbytes <= A.out_cap;
      for (uint32_t v = t; v < (uint32_t)(nbytes >> 4); v += NT) {
        if (fits) st_v4(A.out + dst + 16ull * v, s4[v]);
        s4[v] = make_uint4(0, 0, 0, 0);
      }
      if (!fits && t == 0) set_status(A.ctrl, ZC_ERR_CAPACITY);
    }
    if (t == 0) reinterpret_cast<unsigned long long*>(A.out + kIbp1Header)[g] = gpos;
    __syncthreads();
  }

  // ---- last block: header and table end
  __syncthreads();
  if (t == 0) {
    __threadfence();
    const unsigned long long dn = atomicAdd(&A.ctrl->done, 1ull);
    s_last = (dn == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  unsigned long long pay = 0;
  if (A.ngroups) pay = ld_acquire_u64(A.states + A.ngroups - 1) & kValMask;
  ibp_write_tail(A.meta, cb, m, A.n_bytes, A.nchunks, A.ngroups, A.out, A.out_cap,
                 A.off_payload, A.out_bytes, A.ctrl, pay, t, NT);
}

// ------------------------------------------------------------------ decode

struct IbpDecArgs {
  const uint8_t* meta;
  const uint8_t* in;
  unsigned long long in_bytes;
  uint32_t* y;
  unsigned long long y_cap;
  uint32_t cb;
  Ctrl* ctrl;
};

template <int VEC, int WPL, int CPW>
__global__ void __launch_bounds__(32 * (32 / CPW)) ibp_decode_kernel(IbpDecArgs A) {
  constexpr int NT = 32 * (32 / CPW);
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ uint32_t s_scr[NT / 32 + 4];
  __shared__ unsigned long long s_h[10];
  __shared__ int s_ok, s_bad;
  __shared__ unsigned long long s_off[33];
  __shared__ uint32_t s_pword;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t cb = A.cb, W = cb / 4, B = cb * 8;

  IbpTables T;
  const bool meta_ok = ibp_load_tables<NT>(A.meta, cb, dyn, T, s_scr);
  uint32_t* gbuf = dyn + ibp_table_words(W);
  const uint32_t m = T.m;
  if (t == 0) {
    const int err = ibp_check_stream(A.meta, meta_ok, cb, m, A.in, A.in_bytes, A.y_cap,
                                     blockIdx.x == 0, s_h);
    if (err) set_status(A.ctrl, err);
    s_ok = err == 0;
    s_bad = 0;
  }
  __syncthreads();
  if (!s_ok) return;
  const unsigned long long n_bytes = s_h[2], nchunks = s_h[3], ngroups = s_h[4];
  const unsigned long long off_payload = s_h[7], pay_bits = s_h[8];
  const unsigned long long* grp = reinterpret_cast<const unsigned long long*>(A.in + kIbp1Header);
  const unsigned long long tail_bytes = n_bytes - (nchunks ? (nchunks - 1) * cb : 0ull);
  const uint32_t max_words = ibp_group_words(cb);
  // small chunks: keep this lane's per-word tables in registers
  constexpr bool kRegTab = false;  // registers per lane outweigh the saved loads at 4 blocks/SM
  uint32_t rK[kRegTab ? WPL : 1], rV[kRegTab ? WPL : 1], rP[kRegTab ? WPL : 1];
  uint32_t rMV[kRegTab ? WPL : 1][5];
  if (kRegTab) {
#pragma unroll
    for (int j = 0; j < WPL; ++j) {
      const uint32_t w = owned_word<VEC>(lane, j);
      const bool in = w < W;
      rK[j] = in ? T.K[w] : 0u;
      rV[j] = in ? T.V[w] : 0u;
      rP[j] = in ? T.P[w] : 0u;
#pragma unroll
      for (int i = 0; i < 5; ++i) rMV[j][i] = in ? T.MV[i * W + w] : 0u;
    }
  }

  for (unsigned long long g = blockIdx.x; g < ngroups; g += gridDim.x) {
    const unsigned long long g0 = grp[g], g1 = grp[g + 1];
    const unsigned long long c0 = g * 32ull;
    const uint32_t nch = (uint32_t)(nchunks - c0 < 32 ? nchunks - c0 : 32);
    const bool span_ok = g0 <= g1 && g1 <= pay_bits && (g0 & 127) == 0 && (g1 & 127) == 0 &&
                         ((g1 - g0) >> 5) + 1 <= max_words && g1 > g0;
    if (span_ok) {
      const uint4* src = reinterpret_cast<const uint4*>(A.in + off_payload + (g0 >> 3));
      uint4* dst4 = reinterpret_cast<uint4*>(gbuf);
      const uint32_t nv = (uint32_t)((g1 - g0) >> 7);
      for (uint32_t v = t; v < nv; v += NT) dst4[v] = ld_nc_v4(src + v);
      if (t == 0) gbuf[nv * 4] = 0;  // spare word read by the last fragment
    }
    __syncthreads();
    if (warp == 0) {
      // warp prefix scan of the chunk bit lengths (one lane per chunk)
      const uint32_t pw = span_ok ? gbuf[0] : 0u;
      const unsigned long long c = c0 + lane;
      const bool present = (uint32_t)lane < nch;
      const bool full = present && (c + 1 < nchunks || tail_bytes == cb);
      const bool p = (pw >> lane) & 1u;
      bool bad = !span_ok || (p && (!full || m == 0));
      unsigned long long len = !present ? 0ull : (p ? (unsigned long long)(B - m) : (full ? (unsigned long long)B : 8ull * tail_bytes));
      unsigned long long inc = len;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long v = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += v;
      }
      s_off[lane] = 32ull + inc - len;
      const unsigned long long tot = __shfl_sync(kFull, inc, 31);
      if (lane == 0) {
        s_pword = pw;
        if (round_up_dev(32ull + tot, 128) != g1 - g0) bad = true;
      }
      if (__any_sync(kFull, bad) && lane == 0) s_bad = 1;
    }
    __syncthreads();
    if (!s_bad) {
      const uint32_t pword = s_pword;
#pragma unroll
      for (int r = 0; r < CPW; ++r) {
        const uint32_t i = (uint32_t)warp * CPW + r;
        if (i >= nch) continue;
        const unsigned long long c = c0 + i;
        const bool full = c + 1 < nchunks || tail_bytes == cb;
        const uint32_t wv = full ? W : (uint32_t)(tail_bytes / 4);
        const bool p = (pword >> i) & 1u;
        const unsigned long long off = s_off[i];
        uint32_t* dst = A.y + c * (unsigned long long)W;
#pragma unroll
        for (int j = 0; j < WPL; j += VEC) {
          const uint32_t w = owned_word<VEC>(lane, j);
          uint32_t o[VEC];
#pragma unroll
          for (int q = 0; q < VEC; ++q) {
            const uint32_t ww = w + q;
            o[q] = 0;
            if (ww < wv) {
              if (p) {
                if (kRegTab) {  // this lane's words are the same in every chunk
                  const uint32_t K = rK[j + q];
                  const uint32_t k = __popc(K);
                  const uint32_t f = k ? get_bits(gbuf, off + rP[j + q], k) : 0u;
                  o[q] = hd_expand(f, K, rMV[j + q], 1) | rV[j + q];
                } else {
                  const uint32_t K = T.K[ww];
                  const uint32_t k = __popc(K);
                  const uint32_t f = k ? get_bits(gbuf, off + T.P[ww], k) : 0u;
                  o[q] = hd_expand(f, K, T.MV + ww, W) | T.V[ww];
                }
              } else {
                o[q] = get_bits(gbuf, off + 32ull * ww, 32);
              }
            }
          }
          if (VEC == 4 && w + 3 < wv) {
            st_v4(dst + w, make_uint4(o[0], o[1], o[2], o[3]));
          } else {
#pragma unroll
            for (int q = 0; q < VEC; ++q)
              if (w + q < wv) dst[w + q] = o[q];
          }
        }
      }
    }
    __syncthreads();
    if (t == 0) {
      if (s_bad) set_status(A.ctrl, ZC_ERR_FORMAT);
      s_bad = 0;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ launch

template <int VEC, int WPL>
struct Cfg {
  static constexpr int CPW = (16 / WPL) >= 4 ? 4 : ((16 / WPL) < 1 ? 1 : 16 / WPL);
  static constexpr int NT = 32 * (32 / CPW);
};

size_t smem_bytes(uint32_t cb) {
  return 4ull * (ibp_table_words(cb / 4) + ibp_group_words(cb));
}

template <int VEC, int WPL>
cudaError_t launch_enc(const IbpEncArgs& A, cudaStream_t s) {
  using C = Cfg<VEC, WPL>;
  auto k = ibp_encode_kernel<VEC, WPL, C::CPW>;
  const size_t smem = smem_bytes(A.cb);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int res = resident_blocks((const void*)k, C::NT, smem);
  unsigned long long grid = A.ngroups < (unsigned long long)res ? A.ngroups : (unsigned long long)res;
  if (grid == 0) grid = 1;
  k<<<(unsigned)grid, C::NT, smem, s>>>(A);
  return cudaGetLastError();
}

template <int VEC, int WPL>
cudaError_t launch_dec(const IbpDecArgs& A, cudaStream_t s) {
  using C = Cfg<VEC, WPL>;
  auto k = ibp_decode_kernel<VEC, WPL, C::CPW>;
  const size_t smem = smem_bytes(A.cb);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int res = resident_blocks((const void*)k, C::NT, smem);
  k<<<res, C::NT, smem, s>>>(A);
  return cudaGetLastError();
}

// words per lane needed for chunk_bytes (a lane covers 32 words per unit)
int wpl_for(uint32_t cb) {
  const uint32_t W = cb / 4;
  const uint32_t need = (W + 31) / 32;
  if (need <= 4) return 4;
  if (need <= 8) return 8;
  if (need <= 16) return 16;
  return 32;
}

}  // namespace

cudaError_t ibp_launch_compress(const void* d_meta, uint32_t cb, const void* d_x,
                                unsigned long long n_bytes, void* d_out,
                                unsigned long long out_cap, unsigned long long* d_out_bytes,
                                void* d_ws, cudaStream_t s, bool x_host) {
  IbpEncArgs A;
  A.meta = static_cast<const uint8_t*>(d_meta);
  A.x = static_cast<const uint32_t*>(d_x);
  A.n_bytes = n_bytes;
  A.nchunks = (n_bytes + cb - 1) / cb;
  A.ngroups = (A.nchunks + 31) / 32;
  A.cb = cb;
  A.out = static_cast<uint8_t*>(d_out);
  A.out_cap = out_cap;
  A.off_payload = kIbp1Header + round_up_dev(8ull * (A.ngroups + 1), 128);
  A.out_bytes = d_out_bytes;
  A.ctrl = static_cast<Ctrl*>(d_ws);
  A.states = reinterpret_cast<unsigned long long*>(static_cast<char*>(d_ws) + kCtrlBytes);
  cudaError_t e = cudaMemsetAsync(d_ws, 0, kCtrlBytes + 8ull * A.ngroups, s);
  if (e != cudaSuccess) return e;
  e = arm_wait_fault(d_ws, s);
  if (e != cudaSuccess) return e;
  if (!x_host && ibp_pipe_supported(cb, true))
    return ibp_pipe_compress(d_meta, cb, d_x, n_bytes, d_out, out_cap, d_out_bytes, d_ws, s);
  const bool vec = (cb % 512) == 0;
  switch (wpl_for(cb)) {
    case 4: return vec ? launch_enc<4, 4>(A, s) : launch_enc<1, 4>(A, s);
    case 8: return vec ? launch_enc<4, 8>(A, s) : launch_enc<1, 8>(A, s);
    case 16: return vec ? launch_enc<4, 16>(A, s) : launch_enc<1, 16>(A, s);
    default: return vec ? launch_enc<4, 32>(A, s) : launch_enc<1, 32>(A, s);
  }
}

cudaError_t ibp_launch_decompress(const void* d_meta, uint32_t cb, const void* d_in,
                                  unsigned long long in_bytes, void* d_y,
                                  unsigned long long y_cap, void* d_ws, cudaStream_t s,
                                  bool in_host) {
  IbpDecArgs A;
  A.meta = static_cast<const uint8_t*>(d_meta);
  A.in = static_cast<const uint8_t*>(d_in);
  A.in_bytes = in_bytes;
  A.y = static_cast<uint32_t*>(d_y);
  A.y_cap = y_cap;
  A.cb = cb;
  A.ctrl = static_cast<Ctrl*>(d_ws);
  cudaError_t e = cudaMemsetAsync(d_ws, 0, kCtrlBytes, s);
  if (e != cudaSuccess) return e;
  if (!in_host && ibp_pipe_supported(cb, false))
    return ibp_pipe_decompress(d_meta, cb, d_in, in_bytes, d_y, y_cap, d_ws, s);
  const bool vec = (cb % 512) == 0;
  switch (wpl_for(cb)) {
    case 4: return vec ? launch_dec<4, 4>(A, s) : launch_dec<1, 4>(A, s);
    case 8: return vec ? launch_dec<4, 8>(A, s) : launch_dec<1, 8>(A, s);
    case 16: return vec ? launch_dec<4, 16>(A, s) : launch_dec<1, 16>(A, s);
    default: return vec ? launch_dec<4, 32>(A, s) : launch_dec<1, 32>(A, s);
  }
}

}  // namespace lbb
