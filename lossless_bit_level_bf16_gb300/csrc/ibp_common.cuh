// ibp_common.cuh -- helpers shared by the IBP kernels: the per-word tables a
// block derives from the metadata, and bit gather/scatter under a mask.
//
// [IBP] = "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria
// GPU con la Compressione Lossless per il ML", Metodologia: Invariant Bit
// Packing (IBP), Algoritmo Core, steps 2-3: the bits of a chunk at invariant
// positions (Mask) are dropped when they equal Bitval and the rest is closed
// up; decoding puts the Bitval bits back.
//
// Closing up the kept bits of a 32-bit word (and the inverse) uses the
// parallel-suffix "compress" and "expand" method of H. S. Warren, Hacker's
// Delight (2nd ed.), sections 7-4 and 7-5: five rounds, each moving the bits
// whose count of dropped positions to their right has bit i set by 2^i places.
// The five move masks depend only on the mask word, so a block computes them
// once per word of the chunk and keeps them in shared memory; a data word then
// costs 3 logic operations per round.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace lbb {

// Move masks of the compress/expand rounds for keep-mask `k`.
__device__ __forceinline__ void hd_move_masks(uint32_t k, uint32_t mv[5]) {
  uint32_t mk = ~k << 1;  // count the dropped positions to the right
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    uint32_t mp = mk ^ (mk << 1);  // parallel suffix (prefix XOR)
    mp ^= mp << 2;
    mp ^= mp << 4;
    mp ^= mp << 8;
    mp ^= mp << 16;
    const uint32_t v = mp & k;
    mv[i] = v;
    k = (k ^ v) | (v >> (1u << i));
    mk &= ~mp;
  }
}

// Kept bits of x (positions set in k), closed up toward bit 0.
__device__ __forceinline__ uint32_t hd_compress(uint32_t x, uint32_t k, const uint32_t* mv,
                                                int stride) {
  x &= k;
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    const uint32_t t = x & mv[i * stride];
    x = (x ^ t) | (t >> (1u << i));
  }
  return x;
}

// Inverse: the low popc(k) bits of x spread out to the positions set in k.
__device__ __forceinline__ uint32_t hd_expand(uint32_t x, uint32_t k, const uint32_t* mv,
                                              int stride) {
#pragma unroll
  for (int i = 4; i >= 0; --i) {
    const uint32_t t = x << (1u << i);
    const uint32_t v = mv[i * stride];
    x = (x & ~v) | (t & v);
  }
  return x & k;
}

// OR k (1..32) bits of v into the shared-memory bit string at bit position
// pos (words the fragment shares with others take an atomic OR).
__device__ __forceinline__ void put_bits(uint32_t* buf, unsigned long long pos, uint32_t v,
                                         uint32_t k) {
  const uint32_t wi = (uint32_t)(pos >> 5), sh = (uint32_t)(pos & 31);
  if (sh == 0 && k == 32) {
    buf[wi] = v;  // the whole word belongs to this fragment
    return;
  }
  atomicOr(buf + wi, v << sh);
  if (sh + k > 32) atomicOr(buf + wi + 1, v >> (32 - sh));
}

// k (1..32) bits of a bit string from bit position pos (the word after the
// one holding pos must be readable).
__device__ __forceinline__ uint32_t get_bits(const uint32_t* buf, unsigned long long pos,
                                             uint32_t k) {
  const uint32_t wi = (uint32_t)(pos >> 5), sh = (uint32_t)(pos & 31);
  const uint32_t v = __funnelshift_r(buf[wi], buf[wi + 1], sh);
  return k >= 32 ? v : (v & ((1u << k) - 1u));
}

// Per-word tables of one chunk layout, in shared memory:
//   K[w]  keep mask (~Mask word)      V[w]  Bitval word (zero outside Mask)
//   P[w]  kept bits in words < w      MV[i*W + w]  move masks of round i
struct IbpTables {
  uint32_t* K;
  uint32_t* V;
  uint32_t* P;
  uint32_t* MV;
  uint32_t W;
  uint32_t m;  // invariant positions in a chunk
};

__host__ __device__ constexpr size_t ibp_table_words(uint32_t W) { return 8ull * W; }

// Fill the tables from the IBPM blob (all NT threads of the block; ends with
// a barrier).  Returns false in every thread if the blob's header is not a
// version-1 IBPM for chunk_bytes or its m disagrees with its Mask.
template <int NT>
__device__ bool ibp_load_tables(const uint8_t* meta, uint32_t chunk_bytes, uint32_t* smem,
                                IbpTables& T, uint32_t* s_scratch /* NT/32 + 4 words */) {
  const uint32_t W = chunk_bytes / 4;
  T.W = W;
  T.K = smem;
  T.V = smem + W;
  T.P = smem + 2 * W;
  T.MV = smem + 3 * W;
  const uint32_t* hdr = reinterpret_cast<const uint32_t*>(meta);
  // the header is checked before any Mask/Bitval word is read, so a blob made
  // for another chunk size is never read past its end
  const bool hdr_ok = hdr[0] == kIbpmMagic && (hdr[1] & 0xFFFFu) == 1u &&
                      (hdr[1] >> 16) == kIbpmHeader && hdr[2] == chunk_bytes &&
                      hdr[3] == chunk_bytes * 8u;
  const uint32_t* mask = reinterpret_cast<const uint32_t*>(meta + kIbpmHeader);
  const uint32_t* bitv = reinterpret_cast<const uint32_t*>(meta + kIbpmHeader + chunk_bytes);
  // each thread takes a run of consecutive words
  constexpr int kMaxPer = 4;  // W <= 1024 words, NT >= 256
  const uint32_t per = (W + NT - 1) / NT;
  const uint32_t w0 = threadIdx.x * per;
  uint32_t kc[kMaxPer];
  uint32_t local = 0;
#pragma unroll
  for (int j = 0; j < kMaxPer; ++j) {
    const uint32_t w = w0 + j;
    kc[j] = 0;
    if (j < (int)per && w < W) {
      const uint32_t M = hdr_ok ? mask[w] : 0u;
      const uint32_t K = ~M;
      T.K[w] = K;
      T.V[w] = hdr_ok ? (bitv[w] & M) : 0u;
      uint32_t mv[5];
      hd_move_masks(K, mv);
#pragma unroll
      for (int i = 0; i < 5; ++i) T.MV[i * W + w] = mv[i];
      kc[j] = __popc(K);
      local += kc[j];
    }
  }
  uint32_t total;
  uint32_t excl = block_excl_scan<NT>(local, s_scratch, &total);
#pragma unroll
  for (int j = 0; j < kMaxPer; ++j) {
    const uint32_t w = w0 + j;
    if (j < (int)per && w < W) {
      T.P[w] = excl;
      excl += kc[j];
    }
  }
  T.m = 8u * chunk_bytes - total;
  __syncthreads();
  return hdr_ok && T.m == hdr[4];
}

// Closing step of an IBP encode, run by every thread of the last block to
// finish once `pay` (payload bits, the scan total) is known: the end of the
// group-offset table, the output size, zero padding and the 128-byte header.
__device__ __forceinline__ void ibp_write_tail(const uint8_t* meta, uint32_t cb, uint32_t m,
                                               unsigned long long n_bytes,
                                               unsigned long long nchunks,
                                               unsigned long long ngroups, uint8_t* out,
                                               unsigned long long out_cap,
                                               unsigned long long off_payload,
                                               unsigned long long* out_bytes, Ctrl* ctrl,
                                               unsigned long long pay, int t, int nt) {
  const unsigned long long total = off_payload + (pay >> 3);
  unsigned long long* grp = reinterpret_cast<unsigned long long*>(out + kIbp1Header);
  if (t == 0) {
    grp[ngroups] = pay;
    if (out_bytes) *out_bytes = total;
    if (total > out_cap) set_status(ctrl, ZC_ERR_CAPACITY);
  }
  for (unsigned long long p = kIbp1Header + 8ull * (ngroups + 1) + t; p < off_payload; p += nt)
    out[p] = 0;
  if (t < 16) {
    const unsigned long long* mh = reinterpret_cast<const unsigned long long*>(meta);
    unsigned long long h = 0;
    switch (t) {
      case 0: h = (unsigned long long)kIbp1Magic | (1ull << 32) | ((unsigned long long)kIbp1Header << 48); break;
      case 1: h = (unsigned long long)cb | ((unsigned long long)m << 32); break;
      case 2: h = n_bytes; break;
      case 3: h = nchunks; break;
      case 4: h = ngroups; break;
      case 5: h = mh[6]; break;  // metadata hash
      case 6: h = kIbp1Header; break;
      case 7: h = off_payload; break;
      case 8: h = pay; break;
      case 9: h = total; break;
      default: h = 0; break;
    }
    reinterpret_cast<unsigned long long*>(out)[t] = h;
  }
}

// Checks an IBP1 stream header against the metadata (its chunk size, m and
// hash), the stream length and the output capacity; copies the first ten
// header words to h.  With check_table the group-offset table's two ends are
// checked too.  Returns 0 or the error code.  One thread.
__device__ __forceinline__ int ibp_check_stream(const uint8_t* meta, bool meta_ok, uint32_t cb,
                                                uint32_t m, const uint8_t* in,
                                                unsigned long long in_bytes,
                                                unsigned long long y_cap, bool check_table,
                                                unsigned long long* h) {
  if (!meta_ok) return ZC_ERR_META_MISMATCH;
  if (in_bytes < kIbp1Header) return ZC_ERR_FORMAT;
  const unsigned long long* hd = reinterpret_cast<const unsigned long long*>(in);
  for (int i = 0; i < 10; ++i) h[i] = hd[i];
  const unsigned long long h0 = h[0], h1 = h[1];
  const unsigned long long n_bytes = h[2], nch = h[3], ng = h[4];
  const unsigned long long mh = reinterpret_cast<const unsigned long long*>(meta)[6];
  if ((uint32_t)h0 != kIbp1Magic || ((h0 >> 32) & 0xFFFF) != 1 || (h0 >> 48) != kIbp1Header)
    return ZC_ERR_FORMAT;
  if ((uint32_t)h1 != cb || (uint32_t)(h1 >> 32) != m || h[5] != mh) return ZC_ERR_META_MISMATCH;
  if ((n_bytes & 3) || nch != (n_bytes + cb - 1) / cb || ng != (nch + 31) / 32 ||
      h[6] != kIbp1Header || ng > in_bytes / 8 ||
      h[7] != kIbp1Header + round_up_dev(8ull * (ng + 1), 128) || h[9] > in_bytes ||
      h[7] > h[9] || (h[8] & 127) || (h[8] >> 3) != h[9] - h[7])
    return ZC_ERR_FORMAT;
  if (n_bytes > y_cap) return ZC_ERR_CAPACITY;
  if (check_table) {
    const unsigned long long* grp = reinterpret_cast<const unsigned long long*>(in + kIbp1Header);
    if (grp[0] != 0 || grp[ng] != h[8]) return ZC_ERR_FORMAT;
  }
  return 0;
}

}  // namespace lbb
