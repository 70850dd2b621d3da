// ibp_pipe.cu -- IBP encode and decode for chunks of up to 2048 bytes, with
// tiles of the input staged into shared memory by TMA bulk copies several
// tiles ahead of the threads that work on them.
//
// [IBP] = "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria
// GPU con la Compressione Lossless per il ML", Metodologia: Invariant Bit
// Packing (IBP), Algoritmo Core, steps 2 (Compressione) and 3
// (Decompressione).  The stream is the same "IBP1" stream ibp_codec.cu writes
// and reads (groups of 32 chunks: 32 participation bits, the bodies, zero bits
// up to a multiple of 128).
//
// Tile = Q consecutive groups (Q = 512 / chunk_bytes below 512-byte chunks,
// else 1), so a tile is about 16 KB of input or more.  A block owns a ring of
// S shared-memory stages; one thread keeps up to S tiles in flight with
// cp.async.bulk, each completing on its stage's mbarrier.
//
// A thread owns 16-byte vectors of the tile: 4 consecutive words, which never
// straddle a chunk because chunk_bytes is a multiple of 16.  When the number
// of vectors per chunk is a power of two dividing the block size, a thread's
// vectors all sit at the same position r in their chunks, so the Mask tables
// of its 4 words (keep masks, Bitval, compress/expand move masks) live in
// registers for the whole kernel (REG); otherwise they are read from shared
// memory per vector.
//
// Encode: for chunks of up to 512 bytes, and of 1024 and 2048 bytes, one
// launch (a control warp matches and resolves offsets, four pack warps pack;
// described at ibp_encode_ws_kernel and ibp_encode_wsp_kernel); for other
// chunk sizes, and when a single-pass grid cannot be resident at once, three
// launches (match -> offsets -> pack, described at the encode kernels below),
// which read the input twice.  Packing closes up the kept bits of a vector's 4 words into
// one run of at most 128 bits and ORs it into a shared-memory image of the
// tile's stream (a shared atomicOr per word, with no choice between words a
// run owns alone and words it shares), which is then copied out with 16-byte
// stores and cleared; a tile in which no chunk participates is copied
// straight from the stage.  The image holds stream word j at image word j.
//
// Decode, per tile: the tile's compressed bytes (its span taken from the
// stream's group-offset table, checked first) are staged; one warp per group
// scans the 32 chunk lengths; every thread then reads the <= 128 bits of each
// of its vectors with two 16-byte shared loads, splits them into the 4 words'
// fields, expands them, ORs in Bitval and stores 16 bytes.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "ibp_common.cuh"
#include "internal.h"

namespace lbb {
namespace {

constexpr uint32_t kMaxStages = 6;
constexpr uint32_t kMaxQ = 32;
constexpr uint32_t kStageSlack = 128;  // bytes readable past a stage's data

struct PipeArgs {
  const uint8_t* meta;
  const uint32_t* pw;             // encode: participation word of every group
  const uint8_t* src;             // encode: raw input; decode: the stream
  unsigned long long src_bytes;   // decode: stream bytes
  uint8_t* dst;                   // encode: the stream; decode: the output
  unsigned long long dst_cap;
  unsigned long long n_bytes, nchunks, ngroups, ntiles, off_payload;
  unsigned long long* out_bytes;
  Ctrl* ctrl;
  unsigned long long* states;
  uint32_t cb, vpc, lvpc;  // chunk bytes, 16-byte vectors per chunk, log2 (REG)
  uint32_t Q, S, stage_bytes, img_words;
  uint32_t* lens;  // single-pass encode: every tile's published stream length
  uint32_t lag;    // single-pass encode in pieces: waves between a group's match and its packing
};

// Mask tables of the 4 words at vector position r of a chunk.  When every
// keep mask of the 4 words is at most two runs of ones (fast), MV holds the
// runs instead of the move masks: MV[0] = first run's start a0, MV[1] = its
// mask m0, MV[2] = second run's start a1, MV[3] = its mask m1, MV[4] = the
// first run's length l0 (0 when there is no second run).
struct VecTab {
  uint32_t K[4], V[4], MV[5][4];
  uint32_t R3[3][4];  // three-run form (decoder): third run's start a2, mask m2, field offset l01
  uint32_t Pr;        // kept bits of the chunk before this vector
  bool fast, fast3;
};

// Switch vt to the two-run form if every word allows it (called once, on
// the tables in registers).
__device__ __forceinline__ void make_runs(VecTab& v) {
  bool ok = true;
#pragma unroll
  for (int j = 0; j < 4; ++j) ok = ok && __popc(v.K[j] & ~(v.K[j] << 1)) <= 2;
  v.fast = ok;
  if (!ok) return;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t k = v.K[j];
    uint32_t a0 = 0, m0 = 0, a1 = 0, m1 = 0, l0 = 0;
    if (k) {
      a0 = __ffs(k) - 1;
      const uint32_t y = k >> a0;
      const uint32_t len0 = (y == 0xFFFFFFFFu) ? 32u : (uint32_t)(__ffs(~y) - 1);
      m0 = len0 >= 32 ? 0xFFFFFFFFu : ((1u << len0) - 1u);
      const uint32_t k1 = k & ~(m0 << a0);
      if (k1) {
        a1 = __ffs(k1) - 1;
        m1 = (1u << __popc(k1)) - 1u;  // the second run is shorter than 32
        l0 = len0;
      }
    }
    v.MV[0][j] = a0;
    v.MV[1][j] = m0;
    v.MV[2][j] = a1;
    v.MV[3][j] = m1;
    v.MV[4][j] = l0;
  }
}

// The decoder's three-run form, for tables whose keep masks are three runs
// of ones in some word (16-bit values: a sign run and a low run per half) and
// at most three in every word: MV[0..4] as in the two-run form, R3 the third
// run.  fast3 is set only when the two-run form does not apply.
__device__ __forceinline__ void make_runs3(VecTab& v) {
  v.fast3 = false;
  if (v.fast) {  // no third run: the three-run form reduces to the two-run one
#pragma unroll
    for (int j = 0; j < 4; ++j) v.R3[0][j] = v.R3[1][j] = v.R3[2][j] = 0;
    return;
  }
  bool ok = true;
#pragma unroll
  for (int j = 0; j < 4; ++j) ok = ok && __popc(v.K[j] & ~(v.K[j] << 1)) <= 3;
  if (!ok) return;
  v.fast3 = true;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t k = v.K[j];
    uint32_t a[3] = {0, 0, 0}, mk[3] = {0, 0, 0}, len[3] = {0, 0, 0};
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      if (k) {
        a[i] = __ffs(k) - 1;
        const uint32_t y = k >> a[i];
        len[i] = (y == 0xFFFFFFFFu) ? 32u : (uint32_t)(__ffs(~y) - 1);
        mk[i] = len[i] >= 32 ? 0xFFFFFFFFu : ((1u << len[i]) - 1u);
        k &= ~(mk[i] << a[i]);
      }
    }
    v.MV[0][j] = a[0];
    v.MV[1][j] = mk[0];
    v.MV[2][j] = a[1];
    v.MV[3][j] = mk[1];
    v.MV[4][j] = mk[1] ? len[0] : 0u;
    v.R3[0][j] = a[2];
    v.R3[1][j] = mk[2];
    v.R3[2][j] = mk[2] ? len[0] + len[1] : 0u;
  }
}

// Kept bits of word w of x closed up toward bit 0 (the keep mask's runs, or
// the general method).
__device__ __forceinline__ uint32_t vt_compress(const VecTab& v, uint32_t x, int w) {
  if (v.fast)
    return ((x >> v.MV[0][w]) & v.MV[1][w]) | (((x >> v.MV[2][w]) & v.MV[3][w]) << v.MV[4][w]);
  return hd_compress(x, v.K[w], &v.MV[0][w], 4);
}
// Kept bits per word of the vector (recomputed: cheaper than registers).
__device__ __forceinline__ void kept_bits(const VecTab& v, uint32_t k[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) k[j] = __popc(v.K[j]);
}

__device__ __forceinline__ void load_vectab(const IbpTables& T, uint32_t r, VecTab& v) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = 4 * r + j;
    v.K[j] = T.K[w];
    v.V[j] = T.V[w];
#pragma unroll
    for (int i = 0; i < 5; ++i) v.MV[i][j] = T.MV[i * T.W + w];
  }
  v.Pr = T.P[4 * r];
  v.fast = false;
  v.fast3 = false;
}

// Fields f[0..3] (f[j] has k[j] <= 32 bits) laid end to end, LSB first.
__device__ __forceinline__ void cat4(const uint32_t f[4], const uint32_t k[4], uint32_t o[4]) {
  const unsigned long long a = (unsigned long long)f[0] | ((unsigned long long)f[1] << k[0]);
  const unsigned long long b = (unsigned long long)f[2] | ((unsigned long long)f[3] << k[2]);
  const uint32_t s = k[0] + k[1];
  unsigned long long lo, hi;
  if (s == 0) {
    lo = b;
    hi = 0;
  } else if (s >= 64) {
    lo = a;
    hi = b;
  } else {
    lo = a | (b << s);
    hi = b >> (64 - s);
  }
  o[0] = (uint32_t)lo;
  o[1] = (uint32_t)(lo >> 32);
  o[2] = (uint32_t)hi;
  o[3] = (uint32_t)(hi >> 32);
}

// Inverse of cat4: the fields of lengths k[0..3] from the 128 bits u.
__device__ __forceinline__ void split4(const uint32_t u[4], const uint32_t k[4], uint32_t f[4]) {
  const unsigned long long lo = (unsigned long long)u[0] | ((unsigned long long)u[1] << 32);
  const unsigned long long hi = (unsigned long long)u[2] | ((unsigned long long)u[3] << 32);
  const uint32_t s = k[0] + k[1];
  f[0] = (uint32_t)(lo & ((1ull << k[0]) - 1ull));
  f[1] = (uint32_t)((lo >> k[0]) & ((1ull << k[1]) - 1ull));
  unsigned long long b;
  if (s == 0) b = lo;
  else if (s >= 64) b = hi;
  else b = (lo >> s) | (hi << (64 - s));
  f[2] = (uint32_t)(b & ((1ull << k[2]) - 1ull));
  f[3] = (uint32_t)((b >> k[2]) & ((1ull << k[3]) - 1ull));
}

// OR the run o[0..3] (n <= 128 bits, LSB first, zero above n) into the image
// at bit pos: one shared atomicOr for each of the 5 words from pos / 32 on,
// with no choice per word (the image is zero before the tile; words past
// the run take an OR of zero, and the image has slack for them past the
// tile's last vector).
__device__ __forceinline__ void img_or(uint32_t* img, uint32_t pos, const uint32_t o[4]) {
  const uint32_t sh = pos & 31;
  uint32_t* p = img + (pos >> 5);
  atomicOr(p, o[0] << sh);
  atomicOr(p + 1, __funnelshift_l(o[0], o[1], sh));
  atomicOr(p + 2, __funnelshift_l(o[1], o[2], sh));
  atomicOr(p + 3, __funnelshift_l(o[2], o[3], sh));
  atomicOr(p + 4, __funnelshift_l(o[3], 0u, sh));
}

// Per-thread constants of the packing fast path, for the thread's vector
// position when every keep mask of its 4 words has at most three runs of
// ones.  Word j's field is ((x >> a0) & m0) | ((x >> d1) & M1) |
// ((x >> d2) & M2): each later run is shifted straight to its place in the
// field (d = the run's start minus the kept bits before it, M = its mask at
// that place).  k0..k2: kept bits of words 0..2; n: of all four; Pr: kept
// bits of the chunk before the vector.
struct PackTab {
  uint32_t a0[4], m0[4], d1[4], M1[4], d2[4], M2[4];
  uint32_t k0, k1, k2, n, Pr;
  bool ok, three, low;  // low: every word's first run starts at bit 0
};

// From a VecTab on which make_runs (and, for three runs, make_runs3) ran.
__device__ __forceinline__ void make_packtab(const VecTab& v, PackTab& p) {
  p.ok = v.fast || v.fast3;
  p.three = !v.fast && v.fast3;
  p.low = v.MV[0][0] == 0 && v.MV[0][1] == 0 && v.MV[0][2] == 0 && v.MV[0][3] == 0;
  uint32_t k[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    k[j] = __popc(v.K[j]);
    p.a0[j] = v.MV[0][j];
    p.m0[j] = v.MV[1][j];
    const uint32_t m1 = v.MV[3][j], l0 = v.MV[4][j];  // l0 < 32 when there is a second run
    p.d1[j] = m1 ? v.MV[2][j] - l0 : 0u;
    p.M1[j] = m1 << l0;
    const uint32_t m2 = p.three ? v.R3[1][j] : 0u, l01 = p.three ? v.R3[2][j] : 0u;
    p.d2[j] = m2 ? v.R3[0][j] - l01 : 0u;
    p.M2[j] = m2 << l01;
  }
  p.k0 = k[0];
  p.k1 = k[1];
  p.k2 = k[2];
  p.n = k[0] + k[1] + k[2] + k[3];
  p.Pr = v.Pr;
}

// Bits below bit n (n <= 32).
__device__ __forceinline__ uint32_t lowmask(uint32_t n) { return n >= 32 ? 0xFFFFFFFFu : (1u << n) - 1u; }

// A group's chunk table for the packing: entry c is chunk c's first bit in
// the group's stream, from the group's first bit g (g + 32 + c * B minus the
// kept-bit savings of the participating chunks before it), shifted left by
// one, with the chunk's participation bit below.  Filled by threads 0..31.
__device__ __forceinline__ void fill_chunk_table(uint32_t* coff, uint32_t t, uint32_t pw, uint32_t g,
                                                 uint32_t B, uint32_t m) {
  if (t < 32)
    coff[t] = ((g + 32u + t * B - (uint32_t)__popc(pw & lowmask(t)) * m) << 1) | ((pw >> t) & 1u);
}

// Per-thread constants of the decoder's fast path, for the thread's vector
// position when every keep mask of its 4 words has at most three runs of
// ones: word w's field is the km[w] low bits read c_w bits into the vector's
// run (c_0 = 0, then c1, c2, c3), and expands to ((f << a0) & M0) |
// ((f << e1) & M1) | ((f << e2) & M2) (each run's mask already at its place
// in the word), ORed with Bitval V.
struct UnpackTab {
  uint32_t km[4], c1, c2, c3;
  uint32_t a0[4], M0[4], e1[4], M1[4], e2[4], M2[4], V[4];
  uint32_t Pr;
  bool ok, three;
};

// From a VecTab on which make_runs and make_runs3 ran.
__device__ __forceinline__ void make_unpacktab(const VecTab& v, UnpackTab& u) {
  u.ok = v.fast || v.fast3;
  u.three = !v.fast && v.fast3;
  uint32_t k[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    k[j] = __popc(v.K[j]);
    u.km[j] = lowmask(k[j]);
    u.a0[j] = v.MV[0][j];
    u.M0[j] = v.MV[1][j] << v.MV[0][j];
    const uint32_t m1 = v.MV[3][j], l0 = v.MV[4][j];
    u.e1[j] = m1 ? v.MV[2][j] - l0 : 0u;
    u.M1[j] = m1 << v.MV[2][j];
    const uint32_t m2 = u.three ? v.R3[1][j] : 0u, l01 = u.three ? v.R3[2][j] : 0u;
    u.e2[j] = m2 ? v.R3[0][j] - l01 : 0u;
    u.M2[j] = m2 ? m2 << v.R3[0][j] : 0u;
    u.V[j] = v.V[j];
  }
  u.c1 = k[0];
  u.c2 = k[0] + k[1];
  u.c3 = k[0] + k[1] + k[2];
  u.Pr = v.Pr;
}

// x << s for s in 0..32 (0 at 32).
__device__ __forceinline__ uint32_t shl32(uint32_t x, uint32_t s) { return __funnelshift_lc(0u, x, s); }

// The kept bits of the 4 words x as one run o[0..3] (LSB first, zero above
// p.n): fields concatenated from the last one down, each step a 128-bit
// shift by the next field's length (clamped funnel shifts: no branches).
template <bool THREE, bool LOW>
__device__ __forceinline__ void pack_run(const PackTab& p, const uint4& d, uint32_t o[4]) {
  const uint32_t x[4] = {d.x, d.y, d.z, d.w};
  uint32_t f[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[j] = ((LOW ? x[j] : x[j] >> p.a0[j]) & p.m0[j]) | ((x[j] >> p.d1[j]) & p.M1[j]);
    if (THREE) f[j] |= (x[j] >> p.d2[j]) & p.M2[j];
  }
  uint32_t o0 = f[3], o1, o2, o3;
  o1 = __funnelshift_lc(o0, 0u, p.k2);
  o0 = shl32(o0, p.k2) | f[2];
  o2 = __funnelshift_lc(o1, 0u, p.k1);
  o1 = __funnelshift_lc(o0, o1, p.k1);
  o0 = shl32(o0, p.k1) | f[1];
  o3 = __funnelshift_lc(o2, 0u, p.k0);
  o2 = __funnelshift_lc(o1, o2, p.k0);
  o1 = __funnelshift_lc(o0, o1, p.k0);
  o0 = shl32(o0, p.k0) | f[0];
  o[0] = o0;
  o[1] = o1;
  o[2] = o2;
  o[3] = o3;
}

// Packs the staged tile's vectors v = t, t + NT, ... (< nvec) into the image
// (fast path: REG positions, run-form keep masks).  E vectors per step: the
// words and chunk offsets of all E are read before any is placed, so their
// chains interleave (a placement's shared atomics would otherwise keep the
// next vector's loads behind them).  MODE 0 (several groups): spw / sgex
// hold the groups' participation words and bit offsets.  MODE 1 (one
// group): pw1 is its participation word, the staged vectors belong to its
// chunks cbase, cbase + 1, ..., and chunk c's body starts at image bit
// g1 + c * B - (kept-bit savings of the chunks before it), g1 folding in
// the group's first image bit and its 32 participation bits.  MODE 2 (one
// group, table): chunk c's entry in coff (fill_chunk_table) gives its first
// bit, plus g1.  r: the thread's vector position.
template <bool THREE, bool LOW, int MODE, int E, int NT>
__device__ __forceinline__ void pack_fast(const PackTab& p, const uint32_t* sd, uint32_t nvec,
                                          uint32_t twords, const uint32_t* spw,
                                          const uint32_t* sgex, const uint32_t* coff, uint32_t pw1,
                                          uint32_t g1, uint32_t cbase, uint32_t lvpc, uint32_t r,
                                          uint32_t B, uint32_t m, uint32_t* img, uint32_t t) {
  const uint32_t rawpos = 128u * r;
  for (uint32_t v0 = t; v0 < nvec; v0 += E * NT) {
    uint4 d[E];
    uint32_t off[E], in[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint32_t v = v0 + e * NT;
      const uint32_t vv = v < nvec ? v : v0;  // a vector of the tile
      const uint32_t c = (MODE ? cbase : 0u) + (vv >> lvpc), i5 = c & 31;
      d[e] = *reinterpret_cast<const uint4*>(sd + 4 * vv);
      if (MODE == 2) {
        const uint32_t ce = coff[c];
        off[e] = (ce >> 1) + g1;
        in[e] = ce & 1u;
      } else {
        const uint32_t pw = MODE ? pw1 : spw[c >> 5];
        const uint32_t g = MODE ? g1 : sgex[c >> 5] + 32u;
        off[e] = g + i5 * B - (uint32_t)__popc(pw & ((1u << i5) - 1u)) * m;
        in[e] = (pw >> i5) & 1u;
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint32_t v = v0 + e * NT;
      if (v >= nvec) continue;
      uint32_t o[4];
      if (in[e]) {
        pack_run<THREE, LOW>(p, d[e], o);
        off[e] += p.Pr;
      } else {
        const uint32_t wv = twords - 4 * v;  // >= 1; < 4 only for a short last vector
        o[0] = d[e].x;
        o[1] = wv > 1 ? d[e].y : 0u;
        o[2] = wv > 2 ? d[e].z : 0u;
        o[3] = wv > 3 ? d[e].w : 0u;
        off[e] += rawpos;
      }
      img_or(img, off[e], o);
    }
  }
}

// pack_fast in the form the thread's run constants allow.
template <int MODE, int E, int NT>
__device__ __forceinline__ void pack_any(const PackTab& p, const uint32_t* sd, uint32_t nvec,
                                         uint32_t twords, const uint32_t* spw, const uint32_t* sgex,
                                         const uint32_t* coff, uint32_t pw1, uint32_t g1,
                                         uint32_t cbase, uint32_t lvpc, uint32_t r, uint32_t B,
                                         uint32_t m, uint32_t* img, uint32_t t) {
  if (p.three) {
    if (p.low)
      pack_fast<true, true, MODE, E, NT>(p, sd, nvec, twords, spw, sgex, coff, pw1, g1, cbase, lvpc,
                                         r, B, m, img, t);
    else
      pack_fast<true, false, MODE, E, NT>(p, sd, nvec, twords, spw, sgex, coff, pw1, g1, cbase,
                                          lvpc, r, B, m, img, t);
  } else {
    if (p.low)
      pack_fast<false, true, MODE, E, NT>(p, sd, nvec, twords, spw, sgex, coff, pw1, g1, cbase,
                                          lvpc, r, B, m, img, t);
    else
      pack_fast<false, false, MODE, E, NT>(p, sd, nvec, twords, spw, sgex, coff, pw1, g1, cbase,
                                           lvpc, r, B, m, img, t);
  }
}

// The 128 bits at bit position pos of a shared-memory bit string, read with
// two 16-byte loads (the string must be readable 32 bytes past pos / 8).
__device__ __forceinline__ void win128(const uint32_t* buf, uint32_t pos, uint32_t u[4]) {
  const uint32_t a = pos >> 5, a4 = a & ~3u, d = a - a4, sh = pos & 31;
  const uint4 x = *reinterpret_cast<const uint4*>(buf + a4);
  const uint4 y = *reinterpret_cast<const uint4*>(buf + a4 + 4);
  const uint32_t q[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
  uint32_t s[5];
#pragma unroll
  for (int j = 0; j < 5; ++j) s[j] = d == 0 ? q[j] : (d == 1 ? q[j + 1] : (d == 2 ? q[j + 2] : q[j + 3]));
#pragma unroll
  for (int j = 0; j < 4; ++j) u[j] = __funnelshift_r(s[j], s[j + 1], sh);
}

__host__ __device__ __forceinline__ bool pow2_dev(uint32_t v) { return v && !(v & (v - 1)); }
inline bool pow2(uint32_t v) { return pow2_dev(v); }

// Tile-local chunk and vector position of vector v.
template <bool REG>
__device__ __forceinline__ void vec_pos(const PipeArgs& A, uint32_t v, uint32_t& c, uint32_t& r) {
  if (REG) {
    c = v >> A.lvpc;
    r = v & (A.vpc - 1);
  } else {
    c = v / A.vpc;
    r = v - c * A.vpc;
  }
}

// ------------------------------------------------------------------ encode
//
// Three launches, none of which waits on another block's progress:
//   match    reads the input once and writes each group's participation
//            word (its full chunks whose Mask bits all equal Bitval);
//   offsets  scans the groups' padded bit lengths into the stream's
//            group-offset table (tiles of 4096 groups chained by decoupled
//            look-back: a handful of tiles, so the chain is short);
//   pack     stages tiles of the input with TMA bulk copies, packs each group
//            at its now-known offset and writes the header.
// The match pass costs one extra read of the input; in exchange no tile ever
// holds its data while it waits for its predecessors' lengths.

struct MatchArgs {
  const uint8_t* meta;
  const uint32_t* x;
  unsigned long long n_bytes, nchunks, ngroups;
  uint32_t cb, vpc, lvpc;
  uint32_t* pw;  // out: one participation word per group
  Ctrl* ctrl;
};

// MODE 0: vpc <= 32, a power of two: a lane's vectors all sit at position
//         lane % vpc of their chunks.
// MODE 1, 2, 4: vpc = 32 * MODE: row i of a step of 8 rows is at positions
//         lane + 32 * (i % MODE).
// MODE 3: any other vpc: the tables are read per vector.
template <int MODE>
__global__ void __launch_bounds__(256) ibp_match_kernel(MatchArgs A) {
  extern __shared__ __align__(128) uint8_t dyn[];
  __shared__ uint32_t s_scr[256 / 32 + 4];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  grid_dep_launch();  // the offsets kernel may be scheduled as blocks finish
  IbpTables T;
  const bool ok = ibp_load_tables<256>(A.meta, A.cb, reinterpret_cast<uint32_t*>(dyn), T, s_scr);
  if (!ok) {
    if (t == 0) set_status(A.ctrl, ZC_ERR_META_MISMATCH);
    return;
  }
  const uint32_t cb = A.cb, W = cb / 4, vpc = A.vpc, m = T.m;
  constexpr int NR = (MODE == 1 || MODE == 2 || MODE == 4) ? MODE : 1;
  uint32_t rK[NR][4], rV[NR][4];
  if (MODE != 3) {
#pragma unroll
    for (int k = 0; k < NR; ++k) {
      const uint32_t r0 = MODE == 0 ? ((uint32_t)lane & (vpc - 1)) : (uint32_t)lane + 32u * k;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        rK[k][j] = T.K[4 * r0 + j];
        rV[k][j] = T.V[4 * r0 + j];
      }
    }
  }
  const unsigned long long total_words = A.n_bytes / 4;
  const unsigned long long tail_bytes = A.n_bytes - (A.nchunks ? (A.nchunks - 1) * cb : 0ull);
  const bool short_tail = A.nchunks && tail_bytes != cb;
  const unsigned long long nwarps = (unsigned long long)gridDim.x * 8;
  for (unsigned long long g = (unsigned long long)blockIdx.x * 8 + warp; g < A.ngroups; g += nwarps) {
    const unsigned long long c0 = 32ull * g;
    const uint32_t nch = (uint32_t)((A.nchunks - c0) < 32 ? (A.nchunks - c0) : 32);
    const uint32_t* xg = A.x + c0 * W;
    const uint32_t gwords =
        (uint32_t)((total_words - c0 * W) < 32ull * W ? (total_words - c0 * W) : 32ull * W);
    const uint32_t nvec = (gwords + 3) / 4;
    uint32_t lw = 0;  // bad bits of this lane's vectors, per chunk of the group
    for (uint32_t v0 = 0; v0 < nvec; v0 += 256) {
      uint4 d[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t v = v0 + 32 * i + lane;
        if (4 * v + 3 < gwords) {
          d[i] = ld_nc_v4(xg + 4 * v);
        } else {
          uint32_t w[4];
#pragma unroll
          for (uint32_t k = 0; k < 4; ++k) w[k] = 4 * v + k < gwords ? __ldg(xg + 4 * v + k) : 0u;
          d[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t v = v0 + 32 * i + lane;
        if (v >= nvec) continue;
        uint32_t K[4], V[4];
        if (MODE == 3) {
          const uint32_t r = v % vpc;
          const uint4 k4 = *reinterpret_cast<const uint4*>(T.K + 4 * r);
          const uint4 v4 = *reinterpret_cast<const uint4*>(T.V + 4 * r);
          K[0] = k4.x; K[1] = k4.y; K[2] = k4.z; K[3] = k4.w;
          V[0] = v4.x; V[1] = v4.y; V[2] = v4.z; V[3] = v4.w;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            K[q] = rK[i % NR][q];
            V[q] = rV[i % NR][q];
          }
        }
        const uint32_t dw[4] = {d[i].x, d[i].y, d[i].z, d[i].w};
        const uint32_t wv = (gwords - 4 * v) < 4u ? (gwords - 4 * v) : 4u;
        uint32_t x = 0;
#pragma unroll
        for (uint32_t q = 0; q < 4; ++q)
          if (q < wv) x |= (dw[q] ^ V[q]) & ~K[q];
        const uint32_t c = MODE == 3 ? v / vpc : v >> A.lvpc;
        if (x) lw |= 1u << (c & 31);
      }
    }
    const uint32_t bad = __reduce_or_sync(kFull, lw);
    if (lane == 0) {
      uint32_t valid = nch >= 32 ? kFull : ((1u << nch) - 1u);
      if (short_tail && c0 + nch == A.nchunks) valid &= ~(1u << (nch - 1));
      A.pw[g] = m ? (~bad & valid) : 0u;
    }
  }
}

// Padded bit length of group g with participation word pw.
__device__ __forceinline__ unsigned long long ibp_group_bits(unsigned long long g, uint32_t pw,
                                                             unsigned long long nchunks,
                                                             unsigned long long tail_bytes,
                                                             uint32_t cb, uint32_t m) {
  const unsigned long long c0 = 32ull * g;
  const uint32_t nch = (uint32_t)((nchunks - c0) < 32 ? (nchunks - c0) : 32);
  unsigned long long bits = 32ull + (unsigned long long)nch * 8ull * cb - (unsigned long long)__popc(pw) * m;
  if (c0 + nch == nchunks && tail_bytes != cb) bits -= 8ull * (cb - tail_bytes);
  return round_up_dev(bits, 128);
}

constexpr int kOffNT = 512, kOffIPT = 8;  // 4096 groups per offsets tile

struct OffArgs {
  const uint32_t* pw;
  const uint8_t* meta;
  unsigned long long n_bytes, nchunks, ngroups, ntiles;
  uint32_t cb;
  unsigned long long* grp;  // the stream's group-offset table (ngroups + 1 entries)
  Ctrl* ctrl;
  unsigned long long* states;
};

__global__ void __launch_bounds__(kOffNT) ibp_offsets_kernel(OffArgs A) {
  __shared__ uint32_t s_wt[kOffNT / 32];
  __shared__ unsigned long long s_tile, s_excl;
  const int t = threadIdx.x, warp = t >> 5;
  const uint32_t m = reinterpret_cast<const uint32_t*>(A.meta)[4];
  const unsigned long long tail_bytes = A.n_bytes - (A.nchunks ? (A.nchunks - 1) * A.cb : 0ull);
  grid_dep_wait();    // the match kernel's participation words
  grid_dep_launch();  // the pack kernel may start its set-up
  if (t == 0) s_tile = atomicAdd(&A.ctrl->ticket, 1ull);
  __syncthreads();
  const unsigned long long tile = s_tile;
  if (tile >= A.ntiles) return;
  const unsigned long long g0 = tile * (kOffNT * kOffIPT) + (unsigned long long)t * kOffIPT;
  uint32_t len[kOffIPT];  // group lengths fit 32 bits (chunks of at most 2048 bytes)
  uint32_t local = 0;
#pragma unroll
  for (int i = 0; i < kOffIPT; ++i) {
    const unsigned long long g = g0 + i;
    len[i] = g < A.ngroups ? (uint32_t)ibp_group_bits(g, A.pw[g], A.nchunks, tail_bytes, A.cb, m) : 0u;
    local += len[i];
  }
  uint32_t total;
  const uint32_t excl_local = block_excl_scan<kOffNT>(local, s_wt, &total);
  if (warp == 0) {
    bool to = false;
    const unsigned long long ex = lookback_warp_wide(A.states, tile, total, &to, wait_limit(A.ctrl),
                                                     may_publish(A.ctrl, tile));
    if (t == 0) {
      s_excl = ex;
      if (to) set_status(A.ctrl, ZC_ERR_TIMEOUT);
    }
  }
  __syncthreads();
  unsigned long long run = s_excl + excl_local;
#pragma unroll
  for (int i = 0; i < kOffIPT; ++i) {
    const unsigned long long g = g0 + i;
    if (g < A.ngroups) A.grp[g] = run;
    run += len[i];
    if (g + 1 == A.ngroups) A.grp[A.ngroups] = run;
  }
}

template <int NT, bool REG>
__global__ void __launch_bounds__(NT, 512 / NT) ibp_pack_kernel(PipeArgs A) {
  constexpr int NW = NT / 32;
  extern __shared__ __align__(128) uint8_t dyn[];
  __shared__ uint32_t s_scr[NW + 4];
  __shared__ unsigned long long s_tile[kMaxStages];
  // per stage, read when its copy is issued: participation words, group bit
  // offsets in the tile's stream, the tile's stream offset and bits
  __shared__ uint32_t s_pw[kMaxStages][kMaxQ], s_gex[kMaxStages][kMaxQ];
  __shared__ unsigned long long s_base[kMaxStages];
  __shared__ uint32_t s_agg[kMaxStages];
  __shared__ int s_raw[kMaxStages], s_last;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t cb = A.cb, W = cb / 4, B = 8 * cb, Q = A.Q, S = A.S;

  uint32_t* tab = reinterpret_cast<uint32_t*>(dyn);
  uint8_t* stages = dyn + 4 * ibp_table_words(W);
  uint32_t* img = reinterpret_cast<uint32_t*>(stages + (size_t)S * A.stage_bytes);
  uint4* img4 = reinterpret_cast<uint4*>(img);
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(img + A.img_words);
  const unsigned long long* grp = reinterpret_cast<const unsigned long long*>(A.dst + kIbp1Header);

  IbpTables T;
  const bool ok = ibp_load_tables<NT>(A.meta, cb, tab, T, s_scr);
  const uint32_t m = T.m;
  const unsigned long long tile_raw = 32ull * Q * cb;
  const uint32_t gvec = 8 * W + 1;  // 16-byte vectors of a full group stored raw

  const uint32_t r_own = (uint32_t)t & (A.vpc - 1);  // REG: every vector's position
  PackTab pt{};
  if (REG) {
    VecTab v0;
    load_vectab(T, r_own, v0);
    make_runs(v0);
    make_runs3(v0);
    make_packtab(v0, pt);
  }
  for (uint32_t i = t; i < A.img_words / 4; i += NT) img4[i] = make_uint4(0, 0, 0, 0);

  // warp 0: prefetch() loads the participation words and group offsets of
  // this block's kk-th tile into registers (their latency overlaps the
  // current tile's work); issue() files them per stage and starts the copy of
  // the tile's input into stage s.
  uint32_t pf_pw = 0;
  unsigned long long pf_go = 0, pf_gend = 0;
  bool run = ok;  // false: nothing to pack (bad metadata, or the call failed before)
  // the largest legal stream of a group (every chunk raw), in bits
  const unsigned long long max_group_bits = (32ull + 32ull * B + 127ull) / 128ull * 128ull;
  auto prefetch = [&](unsigned long long kk) {
    const unsigned long long tile = run ? blockIdx.x + kk * gridDim.x : A.ntiles;
    if (tile >= A.ntiles) return;
    const unsigned long long g0 = tile * Q;
    const uint32_t nq = (uint32_t)((A.ngroups - g0) < Q ? (A.ngroups - g0) : Q);
    pf_pw = (uint32_t)lane < nq ? A.pw[g0 + lane] : 0u;
    pf_go = (uint32_t)lane < nq ? grp[g0 + lane] : 0ull;
    pf_gend = grp[g0 + nq];
  };
  auto issue = [&](unsigned long long kk, uint32_t s) {
    const unsigned long long tile = run ? blockIdx.x + kk * gridDim.x : A.ntiles;
    if (lane == 0) s_tile[s] = tile;
    if (tile >= A.ntiles) return;
    const unsigned long long g0 = tile * Q;
    const uint32_t nq = (uint32_t)((A.ngroups - g0) < Q ? (A.ngroups - g0) : Q);
    const uint32_t pw = pf_pw;
    const unsigned long long go = pf_go;
    const unsigned long long base = __shfl_sync(kFull, go, 0);
    const bool raw = __ballot_sync(kFull, pw != 0) == 0;
    // The offsets come from the scan pass through global memory: a tile whose
    // span could not be its stream (offsets out of order, or longer than its
    // groups stored raw) is not packed -- its sizes would index the image out
    // of bounds -- and the call reports the inconsistency.
    const unsigned long long span = pf_gend - base;
    const bool bad = __any_sync(kFull, pf_gend < base || span > nq * max_group_bits ||
                                           ((uint32_t)lane < nq && (go < base || go - base > span)));
    if ((uint32_t)lane < nq) {
      s_pw[s][lane] = pw;
      s_gex[s][lane] = bad ? 0u : (uint32_t)(go - base);
    }
    if (lane == 0) {
      if (bad) set_status(A.ctrl, ZC_ERR_FORMAT);
      s_base[s] = bad ? 0ull : base;
      s_agg[s] = bad ? 0u : (uint32_t)span;  // nothing to write for a bad tile
      s_raw[s] = bad ? 1 : raw;
      const unsigned long long b0 = tile * tile_raw;
      const unsigned long long tb = (A.n_bytes - b0) < tile_raw ? (A.n_bytes - b0) : tile_raw;
      const uint32_t b16 = (uint32_t)(tb & ~15ull);
      uint8_t* st = stages + (size_t)s * A.stage_bytes;
      for (uint32_t w = b16 / 4; w < (uint32_t)(tb / 4); ++w)  // the last 4..12 bytes
        reinterpret_cast<uint32_t*>(st)[w] = __ldg(reinterpret_cast<const uint32_t*>(A.src + b0) + w);
      // Only the last tile has words written through the generic proxy; the
      // stage's earlier reads are ordered by the barrier, as with any TMA ring.
      if (b16 != tb) fence_proxy_async_smem();
      mbar_arrive_expect_tx(bars + s, b16);
      if (b16) bulk_g2s(st, A.src + b0, b16, bars + s);
    }
  };
  if (t == 0)
    for (uint32_t s = 0; s < S; ++s) mbar_init(bars + s, 1);
  grid_dep_wait();  // the participation words and the group-offset table
  // a call whose match or scan pass failed (a wait that ran out) packs
  // nothing: its offsets cannot be trusted (one read, the same for the block)
  if (t == 0) s_last = ok && get_status(A.ctrl) == 0;
  __syncthreads();
  run = s_last != 0;
  __syncthreads();
  if (warp == 0)
    for (uint32_t s = 0; s < S; ++s) {
      prefetch(s);
      issue(s, s);
    }
  __syncthreads();

  for (uint32_t k = 0;; ++k) {
    const uint32_t s = k % S;
    const unsigned long long tile = s_tile[s];
    if (tile >= A.ntiles) break;
    if (warp == 0) prefetch(k + S);
    if (!mbar_wait(bars + s, (k / S) & 1)) set_status(A.ctrl, ZC_ERR_TIMEOUT);
    const uint32_t* sd = reinterpret_cast<const uint32_t*>(stages + (size_t)s * A.stage_bytes);
    const unsigned long long g0 = tile * Q, b0 = tile * tile_raw;
    const uint32_t nq = (uint32_t)((A.ngroups - g0) < Q ? (A.ngroups - g0) : Q);
    const uint32_t tb = (uint32_t)((A.n_bytes - b0) < tile_raw ? (A.n_bytes - b0) : tile_raw);
    const uint32_t twords = tb / 4, nvec = (tb + 15) / 16;
    const bool raw = s_raw[s] != 0;
    const unsigned long long dst = A.off_payload + (s_base[s] >> 3);
    const uint32_t nv = s_agg[s] >> 7;  // 16-byte vectors of the tile's stream
    const bool fits = dst + 16ull * nv <= A.dst_cap;
    if (!fits && t == 0) set_status(A.ctrl, ZC_ERR_CAPACITY);
    if (raw) {
      // [0][input words][zero padding] per group, straight from the stage
      for (uint32_t u0 = t; u0 < nv; u0 += 4 * NT) {
        uint4 o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t u = u0 + e * NT;
          if (u >= nv) continue;
          const uint32_t q = Q == 1 ? 0u : u / gvec, lu = u - q * gvec;
          const uint32_t ib = q * 32u * W;  // group's first input word in the stage
          const uint32_t bw = (q + 1 == nq) ? twords - ib : 32u * W;
          if (lu > 0 && 4 * lu + 3 <= bw) {
            const uint4 x = *reinterpret_cast<const uint4*>(sd + ib + 4 * lu);
            o[e] = make_uint4(sd[ib + 4 * lu - 1], x.x, x.y, x.z);
          } else {
            uint32_t w[4];
#pragma unroll
            for (uint32_t kk = 0; kk < 4; ++kk) {
              const uint32_t ow = 4 * lu + kk;  // word of the group's stream
              w[kk] = (ow >= 1 && ow - 1 < bw) ? sd[ib + ow - 1] : 0u;
            }
            o[e] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        if (fits) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t u = u0 + e * NT;
            if (u < nv) st_v4(A.dst + dst + 16ull * u, o[e]);
          }
        }
      }
    } else {
      // the group's participation word (atomic: a neighbouring run may OR a
      // zero into the same word)
      if ((uint32_t)t < nq) atomicOr(img + (s_gex[s][t] >> 5), s_pw[s][t]);
      // run-form keep masks: constants in registers; otherwise the position's
      // tables are read per vector
      if (REG && pt.ok) {
        const uint32_t* pw_ = s_pw[s];
        const uint32_t* gx_ = s_gex[s];
        const uint32_t pw1 = pw_[0], g1 = gx_[0] + 32u;
        if (Q == 1)
          pack_any<1, 2, NT>(pt, sd, nvec, twords, pw_, gx_, nullptr, pw1, g1, 0u, A.lvpc, r_own, B, m, img, t);
        else
          pack_any<0, 2, NT>(pt, sd, nvec, twords, pw_, gx_, nullptr, pw1, g1, 0u, A.lvpc, r_own, B, m, img, t);
      } else {
        for (uint32_t v = t; v < nvec; v += NT) {
          uint32_t c, r;
          vec_pos<REG>(A, v, c, r);
          const uint32_t q = c >> 5, i = c & 31;
          const uint32_t pwq = s_pw[s][q];
          VecTab vt;
          load_vectab(T, r, vt);
          const uint4 d = *reinterpret_cast<const uint4*>(sd + 4 * v);
          const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
          const uint32_t off =
              s_gex[s][q] + 32u + i * B - (uint32_t)__popc(pwq & ((1u << i) - 1u)) * m;
          uint32_t o[4], pos;
          if ((pwq >> i) & 1u) {
            uint32_t f[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) f[w] = vt_compress(vt, dw[w], w);
            uint32_t kk[4];
            kept_bits(vt, kk);
            cat4(f, kk, o);
            pos = off + vt.Pr;
          } else {
            const uint32_t wv = (twords - 4 * v) < 4u ? (twords - 4 * v) : 4u;
#pragma unroll
            for (uint32_t w = 0; w < 4; ++w) o[w] = w < wv ? dw[w] : 0u;
            pos = off + 128u * r;
          }
          img_or(img, pos, o);
        }
      }
      __syncthreads();
      // stream vector u is image vector u: copied out, and cleared for the
      // next tile by the thread that read it
      for (uint32_t u0 = t; u0 < nv; u0 += 4 * NT) {
        uint4 o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t u = u0 + e * NT;
          if (u < nv) {
            o[e] = img4[u];
            img4[u] = make_uint4(0, 0, 0, 0);
          }
        }
        if (fits) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t u = u0 + e * NT;
            if (u < nv) st_v4(A.dst + dst + 16ull * u, o[e]);
          }
        }
      }
    }
    __syncthreads();  // the stage has been read, the image cleared
    if (warp == 0) issue(k + S, s);
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
  const unsigned long long pay = A.ngroups ? grp[A.ngroups] : 0ull;
  ibp_write_tail(A.meta, cb, m, A.n_bytes, A.nchunks, A.ngroups, A.dst, A.dst_cap, A.off_payload,
                 A.out_bytes, A.ctrl, pay, t, NT);
}

// -------------------------------------------------------- single-pass encode
//
// For chunks of up to 512 bytes (tiles of at most 16 KB) the input is read
// from DRAM once.  A block has four pack warps and one control warp; block b
// owns tiles b, b + G, b + 2G, ... (G = the grid; wave i = tiles iG .. iG+G-1).
//   The control warp, in its iteration i, asks L2 to prefetch its tile of
//   wave i + 2, matches its tile of wave i from its own TMA stage (the first
//   read of that tile) and publishes the tile's stream length in lens[tile]
//   (bit 31 | length in 128-bit units).  It then resolves its tile of wave
//   i - D: the tile's stream offset is the length of the waves before it,
//   which the warp carries from wave to wave, plus the lengths of the tiles
//   before it in its wave, copied into shared memory one iteration earlier.
//   It writes the tile's entries of the group-offset table and hands the
//   participation words and offsets to the pack warps through a two-entry
//   ring of mbarrier-guarded slots.
//   The pack warps run the pack kernel's pipeline: two TMA stages of input,
//   read again right after the match read, while it is still in L2.
// The pack warps wait only for their staged input and the handed-over slot.
// The control warp waits for other blocks only in the resolve, D waves after
// they published: a block that is behind never waits for one that is ahead
// (every wave it needs was matched before the others went on), and the grid
// is no larger than the blocks resident at once, so the waits end; each is
// bounded all the same.
constexpr int kWsPack = 128, kWsThreads = kWsPack + 32;
constexpr uint32_t kWsLag = 3, kWsInfo = 2, kWsStages = 2;  // D = 3 waves (measured best)
constexpr uint32_t kWsLensBytes = 2048;                  // a wave's lengths, padded
constexpr unsigned kWsMaxGrid = kWsLensBytes / 4 - 8;    // 504 tiles per wave
std::atomic<int> g_wsp_lag{2};  // waves between a group's match and its packing (pieces; 2 measured best)

struct WsInfo {
  unsigned long long base;  // the tile's first stream bit, from the payload start
  uint32_t pw[kMaxQ], gex[kMaxQ];
  uint32_t agg;             // the tile's stream bits
  int raw;
};

// Dynamic shared memory of the single-pass encoder.
__host__ __device__ inline size_t ws_smem_bytes(uint32_t cb, uint32_t stage_bytes,
                                                uint32_t img_words) {
  return 4 * ibp_table_words(cb / 4) + (size_t)(kWsStages + 1) * stage_bytes +
         4ull * img_words + 2ull * kWsLensBytes + 8ull * (kWsStages + 1 + 2 * kWsInfo);
}

template <bool REG>
__global__ void __launch_bounds__(kWsThreads, 3) ibp_encode_ws_kernel(PipeArgs A) {
  extern __shared__ __align__(128) uint8_t dyn[];
  __shared__ uint32_t s_scr[kWsThreads / 32 + 4];
  __shared__ WsInfo s_info[kWsInfo];
  __shared__ uint32_t s_cpw[kWsLag + 1][kMaxQ];  // control warp: matched tiles' words
  __shared__ uint32_t s_coff[32];                 // pack warps: a one-group tile's chunk table
  __shared__ int s_last;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t cb = A.cb, W = cb / 4, B = 8 * cb, Q = A.Q;
  const unsigned long long G = gridDim.x, bid = blockIdx.x;

  uint32_t* tab = reinterpret_cast<uint32_t*>(dyn);
  uint8_t* stages = dyn + 4 * ibp_table_words(W);
  uint8_t* mstage = stages + (size_t)kWsStages * A.stage_bytes;
  uint32_t* img = reinterpret_cast<uint32_t*>(mstage + A.stage_bytes);
  uint4* img4 = reinterpret_cast<uint4*>(img);
  uint8_t* lensbuf = reinterpret_cast<uint8_t*>(img + A.img_words);
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(lensbuf + 2 * kWsLensBytes);
  unsigned long long* b_sfull = bars;                    // pack stages landed
  unsigned long long* b_mfull = bars + kWsStages;        // match stage landed
  unsigned long long* b_ifull = b_mfull + 1;             // slot handed over
  unsigned long long* b_iempty = b_ifull + kWsInfo;      // slot read
  unsigned long long* grp = reinterpret_cast<unsigned long long*>(A.dst + kIbp1Header);

  IbpTables T;
  if (!ibp_load_tables<kWsThreads>(A.meta, cb, tab, T, s_scr)) {  // the same in every block
    if (t == 0) set_status(A.ctrl, ZC_ERR_META_MISMATCH);
    return;
  }
  const uint32_t m = T.m;
  const unsigned long long tile_raw = 32ull * Q * cb;
  const unsigned long long tail_bytes = A.n_bytes - (A.nchunks ? (A.nchunks - 1) * cb : 0ull);
  const bool short_tail = A.nchunks && tail_bytes != cb;
  const uint32_t mine = bid < A.ntiles ? (uint32_t)((A.ntiles - bid + G - 1) / G) : 0u;
  auto tile_bytes = [&](unsigned long long tile) -> uint32_t {
    const unsigned long long b0 = tile * tile_raw;
    return (uint32_t)((A.n_bytes - b0) < tile_raw ? (A.n_bytes - b0) : tile_raw);
  };
  // one thread: copy a tile's input into a stage (its last 4..12 bytes with
  // plain loads), completing on the stage's mbarrier
  auto stage_in = [&](unsigned long long tile, uint8_t* st, unsigned long long* bar) {
    const unsigned long long b0 = tile * tile_raw;
    const uint32_t tb = tile_bytes(tile), b16 = tb & ~15u;
    for (uint32_t w = b16 / 4; w < tb / 4; ++w)
      reinterpret_cast<uint32_t*>(st)[w] = __ldg(reinterpret_cast<const uint32_t*>(A.src + b0) + w);
    // Only the last tile has words written through the generic proxy (a fence
    // here would also wait for the thread's outstanding global stores); the
    // stage's earlier reads are ordered by the barrier, as with any TMA ring.
    if (b16 != tb) fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, b16);
    if (b16) bulk_g2s(st, A.src + b0, b16, bar);
  };
  if (t == 0) {
    for (uint32_t s = 0; s < kWsStages; ++s) mbar_init(b_sfull + s, 1);
    mbar_init(b_mfull, 1);
    for (uint32_t k = 0; k < kWsInfo; ++k) {
      mbar_init(b_ifull + k, 1);
      mbar_init(b_iempty + k, 1);
    }
  }
  for (uint32_t i = t; i < A.img_words / 4; i += kWsThreads) img4[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();

  if (warp == kWsPack / 32) {
    // ================================================= control warp
    uint32_t cK[4] = {0, 0, 0, 0}, cV[4] = {0, 0, 0, 0};
    if (REG) {
      const uint32_t r = (uint32_t)lane & (A.vpc - 1);  // every vector of this lane
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        cK[q] = T.K[4 * r + q];
        cV[q] = T.V[4 * r + q];
      }
    }
    auto prefetch_l2 = [&](uint32_t k) {
      if (k >= mine) return;
      const unsigned long long tile = bid + k * G;
      const uint32_t b16 = tile_bytes(tile) & ~15u;
      if (b16) bulk_prefetch_l2(A.src + tile * tile_raw, b16, l2_policy_keep());
    };
    // lengths of the tiles of wave w (as 16-byte vectors from the tile index
    // rounded down to 4) into lens buffer w & 1
    auto lens_fetch = [&](uint32_t w) {
      if (w < mine) {
        const unsigned long long wf = (unsigned long long)w * G, la0 = wf & ~3ull;
        const uint32_t nw = (uint32_t)((A.ntiles - wf) < G ? (A.ntiles - wf) : G);
        const uint32_t nv4 = (uint32_t)((wf + nw - la0 + 3) / 4);
        uint8_t* lb = lensbuf + (w & 1u) * kWsLensBytes;
        for (uint32_t vi = lane; vi < nv4; vi += 32) cp_async16(lb + 16u * vi, A.lens + la0 + 4ull * vi);
      }
      cp_async_commit();
    };
    if (lane == 0) {
      prefetch_l2(0);
      prefetch_l2(1);
      if (mine) stage_in(bid, mstage, b_mfull);
    }
    const unsigned lim = wait_limit(A.ctrl);
    const unsigned long long fault1 = A.ctrl->fault_tile1;  // 0 unless a wait-failure test
    unsigned long long wave_base = 0;  // 128-bit units of the waves resolved so far
    for (uint32_t i = 0; i < mine + kWsLag; ++i) {
      if (i < mine) {
        // ---- match the tile of wave i
        const unsigned long long tile = bid + (unsigned long long)i * G, g0 = tile * Q;
        if (lane == 0) prefetch_l2(i + 2);
        if (!mbar_wait(b_mfull, i & 1u)) set_status(A.ctrl, ZC_ERR_TIMEOUT);
        const uint32_t tb = tile_bytes(tile), twords = tb / 4, nvec = (tb + 15) / 16;
        const uint32_t* sd = reinterpret_cast<const uint32_t*>(mstage);
        uint32_t bad = 0;  // lane q: chunks of the tile's group q that differ
        if (REG && A.vpc == 32) {
          // a 512-byte chunk per step of 32 vectors: one vote per chunk, four
          // chunks at a time (lane l's vector sits at position l of its chunk)
          const uint32_t nfull = twords / 128;  // chunks wholly in the tile
          uint32_t c0 = 0;
          for (; c0 + 4 <= nfull; c0 += 4) {
            uint32_t any4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint4 d = *reinterpret_cast<const uint4*>(sd + 128 * (c0 + u) + 4 * lane);
              const uint32_t x = ((d.x ^ cV[0]) & ~cK[0]) | ((d.y ^ cV[1]) & ~cK[1]) |
                                 ((d.z ^ cV[2]) & ~cK[2]) | ((d.w ^ cV[3]) & ~cK[3]);
              any4[u] = __any_sync(kFull, x != 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t c = c0 + u;
              if (any4[u] && (uint32_t)lane == (c >> 5)) bad |= 1u << (c & 31);
            }
          }
          for (; c0 < nfull; ++c0) {
            const uint4 d = *reinterpret_cast<const uint4*>(sd + 128 * c0 + 4 * lane);
            const uint32_t x = ((d.x ^ cV[0]) & ~cK[0]) | ((d.y ^ cV[1]) & ~cK[1]) |
                               ((d.z ^ cV[2]) & ~cK[2]) | ((d.w ^ cV[3]) & ~cK[3]);
            if (__any_sync(kFull, x != 0) && (uint32_t)lane == (c0 >> 5)) bad |= 1u << (c0 & 31);
          }
          // a short last chunk never participates: its bits are not needed
        } else
        for (uint32_t v0 = 0; v0 < nvec; v0 += 32) {
          const uint32_t v = v0 + lane;
          uint32_t bits = 0, qq = 0xFFFFFFFFu;
          if (v < nvec) {
            uint32_t c, r;
            vec_pos<REG>(A, v, c, r);
            uint32_t K[4], V[4];
            if (REG) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                K[q] = cK[q];
                V[q] = cV[q];
              }
            } else {
              const uint4 k4 = *reinterpret_cast<const uint4*>(T.K + 4 * r);
              const uint4 v4 = *reinterpret_cast<const uint4*>(T.V + 4 * r);
              K[0] = k4.x; K[1] = k4.y; K[2] = k4.z; K[3] = k4.w;
              V[0] = v4.x; V[1] = v4.y; V[2] = v4.z; V[3] = v4.w;
            }
            const uint4 d = *reinterpret_cast<const uint4*>(sd + 4 * v);
            const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
            const uint32_t wv = (twords - 4 * v) < 4u ? (twords - 4 * v) : 4u;
            uint32_t x = 0;
#pragma unroll
            for (uint32_t q = 0; q < 4; ++q)
              if (q < wv) x |= (dw[q] ^ V[q]) & ~K[q];
            qq = c >> 5;
            bits = x ? 1u << (c & 31) : 0u;
          }
          // the warp's 32 consecutive vectors touch at most two groups
          const uint32_t q0 = __shfl_sync(kFull, qq, 0);
          const uint32_t r0 = __reduce_or_sync(kFull, qq == q0 ? bits : 0u);
          const uint32_t r1 = __reduce_or_sync(kFull, qq != q0 ? bits : 0u);
          if ((uint32_t)lane == q0) bad |= r0;
          if ((uint32_t)lane == q0 + 1) bad |= r1;
        }
        __syncwarp();  // the match stage has been read
        if (lane == 0 && i + 1 < mine) stage_in(tile + G, mstage, b_mfull);
        const uint32_t nq = (uint32_t)((A.ngroups - g0) < Q ? (A.ngroups - g0) : Q);
        uint32_t pw = 0, units = 0;
        if ((uint32_t)lane < nq) {
          const unsigned long long g = g0 + lane, c0 = 32ull * g;
          const uint32_t nch = (uint32_t)((A.nchunks - c0) < 32 ? (A.nchunks - c0) : 32);
          uint32_t valid = nch >= 32 ? kFull : ((1u << nch) - 1u);
          if (short_tail && c0 + nch == A.nchunks) valid &= ~(1u << (nch - 1));
          pw = m ? (~bad & valid) : 0u;
          units = (uint32_t)(ibp_group_bits(g, pw, A.nchunks, tail_bytes, cb, m) >> 7);
        }
        s_cpw[i % (kWsLag + 1)][lane] = pw;
        units = __reduce_add_sync(kFull, units);
        if (lane == 0 && tile + 1 != fault1) st_relaxed_u32(A.lens + tile, 0x80000000u | units);
      }
      if (i + 1 == kWsLag) lens_fetch(0);
      if (i >= kWsLag) {
        // ---- resolve the tile of wave j = i - D and hand it over
        const uint32_t j = i - kWsLag;
        const unsigned long long wf = (unsigned long long)j * G, la0 = wf & ~3ull;
        const uint32_t nw = (uint32_t)((A.ntiles - wf) < G ? (A.ntiles - wf) : G);
        const uint32_t nv4 = (uint32_t)((wf + nw - la0 + 3) / 4);
        uint4* lb = reinterpret_cast<uint4*>(lensbuf + (j & 1u) * kWsLensBytes);
        cp_async_wait_all();
        __syncwarp();
        uint32_t pre = 0, tot = 0;
        for (unsigned spins = 0;; ++spins) {
          bool all = true;
          pre = 0;
          tot = 0;
          for (uint32_t vi = lane; vi < nv4; vi += 32) {
            const uint4 e4 = lb[vi];
            const uint32_t e[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
            for (uint32_t q = 0; q < 4; ++q) {
              const unsigned long long idx = la0 + 4ull * vi + q;  // tile index
              if (idx >= wf && idx < wf + nw) {
                if (!(e[q] >> 31)) all = false;
                const uint32_t u = e[q] & 0x7FFFFFFFu;
                tot += u;
                if (idx < wf + bid) pre += u;
              }
            }
          }
          if (__all_sync(kFull, all)) break;
          if (spins >= lim) {
            if (lane == 0) set_status(A.ctrl, ZC_ERR_TIMEOUT);
            break;
          }
          // the call has failed: no more waiting (one vote, so that the
          // whole warp leaves the loop together)
          if (__any_sync(kFull, get_status(A.ctrl) != 0)) break;
          __nanosleep(spins < 64 ? 32 : 256);
          for (uint32_t vi = lane; vi < nv4; vi += 32) lb[vi] = ld_relaxed_v4(A.lens + la0 + 4ull * vi);
          __syncwarp();
        }
        __syncwarp();  // lens buffer j & 1 has been read
        lens_fetch(j + 1);
        pre = __reduce_add_sync(kFull, pre);
        tot = __reduce_add_sync(kFull, tot);
        const unsigned long long base = (wave_base + pre) * 128ull;
        wave_base += tot;
        const unsigned long long tile = bid + wf, g0 = tile * Q;
        const uint32_t nq = (uint32_t)((A.ngroups - g0) < Q ? (A.ngroups - g0) : Q);
        const uint32_t pw = (uint32_t)lane < nq ? s_cpw[j % (kWsLag + 1)][lane] : 0u;
        const uint32_t gb =
            (uint32_t)lane < nq ? (uint32_t)ibp_group_bits(g0 + lane, pw, A.nchunks, tail_bytes, cb, m)
                                : 0u;
        uint32_t inc = gb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(kFull, inc, o);
          if (lane >= o) inc += y;
        }
        const uint32_t agg = __shfl_sync(kFull, inc, 31);
        const bool raw = __ballot_sync(kFull, pw != 0) == 0;
        if ((uint32_t)lane < nq) grp[g0 + lane] = base + (inc - gb);
        if (lane == 0 && tile + 1 == A.ntiles) grp[A.ngroups] = base + agg;
        // slot j % R, once the pack warps have read its previous contents
        const uint32_t k = j % kWsInfo, f = j / kWsInfo;
        if (f > 0 && !mbar_wait(b_iempty + k, (f - 1) & 1u)) set_status(A.ctrl, ZC_ERR_TIMEOUT);
        WsInfo& si = s_info[k];
        si.pw[lane] = pw;
        si.gex[lane] = inc - gb;
        if (lane == 0) {
          si.base = base;
          si.agg = agg;
          si.raw = raw;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(b_ifull + k);
      }
    }
    cp_async_wait_all();
  } else {
    // ================================================= pack warps
    const uint32_t gvec = 8 * W + 1;  // 16-byte vectors of a full group stored raw
    const uint32_t r_own = (uint32_t)t & (A.vpc - 1);  // REG: every vector's position
    PackTab pt{};
    if (REG) {
      VecTab v0;
      load_vectab(T, r_own, v0);
      make_runs(v0);
      make_runs3(v0);
      make_packtab(v0, pt);
    }
    if (t == 0)
      for (uint32_t s = 0; s < kWsStages && s < mine; ++s)
        stage_in(bid + s * G, stages + (size_t)s * A.stage_bytes, b_sfull + s);
    for (uint32_t j = 0; j < mine; ++j) {
      const uint32_t s = j % kWsStages, k = j % kWsInfo;
      bool ok = mbar_wait(b_sfull + s, (j / kWsStages) & 1u);
      ok = mbar_wait(b_ifull + k, (j / kWsInfo) & 1u) && ok;
      if (!ok) set_status(A.ctrl, ZC_ERR_TIMEOUT);
      if (Q == 1 && !s_info[k].raw)  // one group: its chunk table (the previous tile is done with it)
        fill_chunk_table(s_coff, (uint32_t)t, s_info[k].pw[0], s_info[k].gex[0], B, m);
      named_bar(1, kWsPack);  // the previous tile's image is cleared, the chunk table filled
      const WsInfo& si = s_info[k];
      const uint32_t* sd = reinterpret_cast<const uint32_t*>(stages + (size_t)s * A.stage_bytes);
      const unsigned long long tile = bid + (unsigned long long)j * G, g0 = tile * Q;
      const uint32_t nq = (uint32_t)((A.ngroups - g0) < Q ? (A.ngroups - g0) : Q);
      const uint32_t tb = tile_bytes(tile);
      const uint32_t twords = tb / 4, nvec = (tb + 15) / 16;
      const bool raw = si.raw != 0;
      const unsigned long long dst = A.off_payload + (si.base >> 3);
      const uint32_t nv = si.agg >> 7;  // 16-byte vectors of the tile's stream
      const bool fits = dst + 16ull * nv <= A.dst_cap;
      if (!fits && t == 0) set_status(A.ctrl, ZC_ERR_CAPACITY);
      if (raw) {
        // [0][input words][zero padding] per group, straight from the stage:
        // stream vector lu of group q is input words 4 lu - 1 .. 4 lu + 2; a
        // lane loads words 4 lu .. 4 lu + 3 and takes word 4 lu - 1 from the
        // lane before it (lane 0 reads it), which keeps the loads 16-byte;
        // the loop runs while the warp's first vector is in (the shuffles
        // take every lane)
        for (uint32_t u0 = t; u0 - lane < nv; u0 += 4 * kWsPack) {
          uint4 o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t u = u0 + e * kWsPack;
            const uint32_t q = Q == 1 ? 0u : u / gvec, lu = u - q * gvec;
            const uint32_t ib = q * 32u * W;  // group's first input word in the stage
            const uint32_t bw = (q + 1 == nq) ? twords - ib : 32u * W;
            uint4 x = make_uint4(0, 0, 0, 0);
            if (u < nv) {
              if (4 * lu + 3 < bw) {
                x = *reinterpret_cast<const uint4*>(sd + ib + 4 * lu);
              } else {
                x.x = 4 * lu < bw ? sd[ib + 4 * lu] : 0u;
                x.y = 4 * lu + 1 < bw ? sd[ib + 4 * lu + 1] : 0u;
                x.z = 4 * lu + 2 < bw ? sd[ib + 4 * lu + 2] : 0u;
              }
            }
            uint32_t prev = __shfl_up_sync(kFull, x.w, 1);
            if (lu == 0) prev = 0u;  // the group's participation word: none
            else if (lane == 0) prev = (u < nv && 4 * lu - 1 < bw) ? sd[ib + 4 * lu - 1] : 0u;
            o[e] = make_uint4(prev, x.x, x.y, x.z);
          }
          if (fits) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t u = u0 + e * kWsPack;
              if (u < nv) st_v4(A.dst + dst + 16ull * u, o[e]);
            }
          }
        }
      } else {
        if ((uint32_t)t < nq) atomicOr(img + (si.gex[t] >> 5), si.pw[t]);
        // A thread whose vector position has run-form keep masks packs with
        // its constants in registers; any other reads its position's tables
        // per vector (the loops have no warp-wide operation).
        if (REG && pt.ok) {
          // one group: chunk offsets from the table filled at the tile's start
          if (Q == 1)
            pack_any<2, 4, kWsPack>(pt, sd, nvec, twords, si.pw, si.gex, s_coff, 0u, 0u, 0u, A.lvpc,
                                    r_own, B, m, img, t);
          else
            pack_any<0, 4, kWsPack>(pt, sd, nvec, twords, si.pw, si.gex, nullptr, 0u, 0u, 0u, A.lvpc,
                                    r_own, B, m, img, t);
        } else {
          for (uint32_t v = t; v < nvec; v += kWsPack) {
            uint32_t c, r;
            vec_pos<REG>(A, v, c, r);
            const uint32_t q = c >> 5, i5 = c & 31;
            const uint32_t pwq = si.pw[q];
            VecTab vt;
            load_vectab(T, r, vt);
            const uint4 d = *reinterpret_cast<const uint4*>(sd + 4 * v);
            const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
            const uint32_t off =
                si.gex[q] + 32u + i5 * B - (uint32_t)__popc(pwq & ((1u << i5) - 1u)) * m;
            uint32_t o[4], pos;
            if ((pwq >> i5) & 1u) {
              uint32_t f[4];
#pragma unroll
              for (int w = 0; w < 4; ++w) f[w] = vt_compress(vt, dw[w], w);
              uint32_t kk[4];
              kept_bits(vt, kk);
              cat4(f, kk, o);
              pos = off + vt.Pr;
            } else {
              const uint32_t wv = (twords - 4 * v) < 4u ? (twords - 4 * v) : 4u;
#pragma unroll
              for (uint32_t w = 0; w < 4; ++w) o[w] = w < wv ? dw[w] : 0u;
              pos = off + 128u * r;
            }
            img_or(img, pos, o);
          }
        }
        named_bar(1, kWsPack);
        // stream vector u is image vector u: copied out, and cleared for the
        // next tile (the barrier at its top) by the thread that read it
        for (uint32_t u0 = t; u0 < nv; u0 += 4 * kWsPack) {
          uint4 o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t u = u0 + e * kWsPack;
            if (u < nv) {
              o[e] = img4[u];
              img4[u] = make_uint4(0, 0, 0, 0);
            }
          }
          if (fits) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t u = u0 + e * kWsPack;
              if (u < nv) st_v4(A.dst + dst + 16ull * u, o[e]);
            }
          }
        }
      }
      named_bar(1, kWsPack);  // the stage, the image and the slot have been read
      if (t == 0) {
        mbar_arrive(b_iempty + k);
        if (j + kWsStages < mine)
          stage_in(tile + kWsStages * G, stages + (size_t)s * A.stage_bytes, b_sfull + s);
      }
    }
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
  const unsigned long long pay = A.ngroups ? grp[A.ngroups] : 0ull;
  ibp_write_tail(A.meta, cb, m, A.n_bytes, A.nchunks, A.ngroups, A.dst, A.dst_cap, A.off_payload,
                 A.out_bytes, A.ctrl, pay, t, kWsThreads);
}

// ------------------------------------------ single-pass encode in pieces
//
// For chunks of 1024 and 2048 bytes a group is 32 or 64 KB of input, too
// large to stage whole beside a match stage.  Here a block takes whole
// groups (tile = group; block b owns groups b, b + G, ...) and moves each
// through shared memory in pieces of 16 KB (cpp = 16 or 8 chunks, np = 2 or
// 4 pieces per group).
//   The control warp matches a group piece by piece from two stages (the
//   next piece's copy in flight while it matches one), publishes the group's
//   stream length after its last piece, and resolves the group of wave
//   i - D (D = A.lag, 1..3) as the single-pass encoder above does.
//   The pack warps take the pieces through two stages of their own.  A piece
//   is packed into an image of its part of the group's stream, starting at
//   the 16-byte vector that holds the piece's first bit; that vector already
//   holds the previous piece's bits in it.  The full vectors are written
//   out and the partial last one is moved to the front for the next piece.
//   A group's stream is thus written by one block, in order, 16 bytes at a
//   time: no block waits for another's output.
constexpr int kWspPack = 128, kWspThreads = kWspPack + 32;
constexpr uint32_t kWspPiece = 16384;  // input bytes per piece
constexpr uint32_t kWspMS = 2, kWspPS = 2;  // match stages, pack stages

__host__ __device__ inline size_t wsp_smem_bytes(uint32_t cb, uint32_t stage_bytes,
                                                 uint32_t img_words) {
  return 4 * ibp_table_words(cb / 4) + (size_t)(kWspMS + kWspPS) * stage_bytes +
         4ull * img_words + 2ull * kWsLensBytes + 8ull * (kWspMS + kWspPS + 2 * kWsInfo);
}

template <int VPW>  // 16-byte vectors of a chunk per lane of a warp (vpc / 32)
__global__ void __launch_bounds__(kWspThreads, 2) ibp_encode_wsp_kernel(PipeArgs A) {
  extern __shared__ __align__(128) uint8_t dyn[];
  __shared__ uint32_t s_scr[kWspThreads / 32 + 4];
  __shared__ WsInfo s_info[kWsInfo];
  __shared__ uint32_t s_cpw[4];  // control warp: matched groups' participation words
  __shared__ uint32_t s_coff[32];  // pack warps: the group's chunk table
  __shared__ int s_last;
  constexpr uint32_t vpc = 32 * VPW;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t cb = A.cb, W = cb / 4, B = 8 * cb;
  const uint32_t cpp = kWspPiece / cb, np = 32 / cpp;  // chunks per piece, pieces per group
  const uint32_t lag = A.lag;
  const unsigned long long G = gridDim.x, bid = blockIdx.x;

  uint32_t* tab = reinterpret_cast<uint32_t*>(dyn);
  uint8_t* pstages = dyn + 4 * ibp_table_words(W);
  uint8_t* mstages = pstages + (size_t)kWspPS * A.stage_bytes;
  uint32_t* img = reinterpret_cast<uint32_t*>(mstages + (size_t)kWspMS * A.stage_bytes);
  uint4* img4 = reinterpret_cast<uint4*>(img);
  uint8_t* lensbuf = reinterpret_cast<uint8_t*>(img + A.img_words);
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(lensbuf + 2 * kWsLensBytes);
  unsigned long long* b_sfull = bars;                    // pack stages landed
  unsigned long long* b_mfull = bars + kWspPS;           // match stages landed
  unsigned long long* b_ifull = b_mfull + kWspMS;        // slot handed over
  unsigned long long* b_iempty = b_ifull + kWsInfo;  // slot read
  unsigned long long* grp = reinterpret_cast<unsigned long long*>(A.dst + kIbp1Header);

  IbpTables T;
  if (!ibp_load_tables<kWspThreads>(A.meta, cb, tab, T, s_scr)) {  // the same in every block
    if (t == 0) set_status(A.ctrl, ZC_ERR_META_MISMATCH);
    return;
  }
  const uint32_t m = T.m;
  const unsigned long long group_raw = 32ull * cb;
  const unsigned long long tail_bytes = A.n_bytes - (A.nchunks ? (A.nchunks - 1) * cb : 0ull);
  const bool short_tail = A.nchunks && tail_bytes != cb;
  const uint32_t mine = bid < A.ntiles ? (uint32_t)((A.ntiles - bid + G - 1) / G) : 0u;
  // input bytes of piece p of group g (0: no such piece)
  auto piece_bytes = [&](unsigned long long g, uint32_t p) -> uint32_t {
    const unsigned long long b0 = g * group_raw + (unsigned long long)p * kWspPiece;
    if (b0 >= A.n_bytes) return 0u;
    return (uint32_t)((A.n_bytes - b0) < kWspPiece ? (A.n_bytes - b0) : kWspPiece);
  };
  // one thread: copy this block's piece number seq (its group seq / np, piece
  // seq % np) into a stage (its last 4..12 bytes with plain loads), with an
  // L2 policy for the lines read: the match keeps them for the pack warps'
  // second read, which lets them go
  auto stage_piece = [&](uint32_t seq, uint8_t* st, unsigned long long* bar,
                         unsigned long long pol) {
    const uint32_t k = seq / np, p = seq % np;
    if (k >= mine) return;
    const unsigned long long g = bid + (unsigned long long)k * G;
    const uint32_t tb = piece_bytes(g, p), b16 = tb & ~15u;
    if (tb == 0) return;
    const unsigned long long b0 = g * group_raw + (unsigned long long)p * kWspPiece;
    for (uint32_t w = b16 / 4; w < tb / 4; ++w)
      reinterpret_cast<uint32_t*>(st)[w] = __ldg(reinterpret_cast<const uint32_t*>(A.src + b0) + w);
    if (b16 != tb) fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, b16);
    if (b16) bulk_g2s_hint(st, A.src + b0, b16, bar, pol);
  };
  if (t == 0) {
    for (uint32_t s = 0; s < kWspPS; ++s) mbar_init(b_sfull + s, 1);
    for (uint32_t s = 0; s < kWspMS; ++s) mbar_init(b_mfull + s, 1);
    for (uint32_t k = 0; k < kWsInfo; ++k) {
      mbar_init(b_ifull + k, 1);
      mbar_init(b_iempty + k, 1);
    }
  }
  for (uint32_t i = t; i < A.img_words / 4; i += kWspThreads) img4[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();

  if (warp == kWspPack / 32) {
    // ================================================= control warp
    // lane l matches vector positions l, l + 32, ... of every chunk
    uint32_t cK[VPW][4], cV[VPW][4];
#pragma unroll
    for (int k = 0; k < VPW; ++k)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        cK[k][q] = T.K[4 * (lane + 32 * k) + q];
        cV[k][q] = T.V[4 * (lane + 32 * k) + q];
      }
    auto differs = [&](const uint32_t* sd, uint32_t c) -> uint32_t {
      uint32_t x = 0;
#pragma unroll
      for (int k = 0; k < VPW; ++k) {
        const uint4 d = *reinterpret_cast<const uint4*>(sd + 4 * (c * vpc + 32 * k + lane));
        x |= ((d.x ^ cV[k][0]) & ~cK[k][0]) | ((d.y ^ cV[k][1]) & ~cK[k][1]) |
             ((d.z ^ cV[k][2]) & ~cK[k][2]) | ((d.w ^ cV[k][3]) & ~cK[k][3]);
      }
      return x;
    };
    // lengths of the groups of wave w into lens buffer w & 1 (as in the
    // single-pass encoder)
    auto lens_fetch = [&](uint32_t w) {
      if (w < mine) {
        const unsigned long long wf = (unsigned long long)w * G, la0 = wf & ~3ull;
        const uint32_t nw = (uint32_t)((A.ntiles - wf) < G ? (A.ntiles - wf) : G);
        const uint32_t nv4 = (uint32_t)((wf + nw - la0 + 3) / 4);
        uint8_t* lb = lensbuf + (w & 1u) * kWsLensBytes;
        for (uint32_t vi = lane; vi < nv4; vi += 32) cp_async16(lb + 16u * vi, A.lens + la0 + 4ull * vi);
      }
      cp_async_commit();
    };
    const unsigned long long keep = l2_policy_keep();
    if (lane == 0)
      for (uint32_t s = 0; s < kWspMS; ++s)
        stage_piece(s, mstages + (size_t)s * A.stage_bytes, b_mfull + s, keep);
    const unsigned lim = wait_limit(A.ctrl);
    const unsigned long long fault1 = A.ctrl->fault_tile1;  // 0 unless a wait-failure test
    unsigned long long wave_base = 0;  // 128-bit units of the waves resolved so far
    for (uint32_t i = 0; i < mine + lag; ++i) {
      if (i < mine) {
        // ---- match the group of wave i, piece by piece
        const unsigned long long g = bid + (unsigned long long)i * G;
        uint32_t bad = 0;  // the same in every lane
        for (uint32_t p = 0; p < np; ++p) {
          const uint32_t tb = piece_bytes(g, p);
          if (tb == 0) break;
          const uint32_t seq = i * np + p, ms = seq % kWspMS;
          if (!mbar_wait(b_mfull + ms, (seq / kWspMS) & 1u)) set_status(A.ctrl, ZC_ERR_TIMEOUT);
          const uint32_t* sd = reinterpret_cast<const uint32_t*>(mstages + (size_t)ms * A.stage_bytes);
          const uint32_t nfull = tb / cb;  // a short last chunk never participates
          uint32_t c = 0;
          for (; c + 2 <= nfull; c += 2) {
            const uint32_t x0 = differs(sd, c), x1 = differs(sd, c + 1);
            if (__any_sync(kFull, x0 != 0)) bad |= 1u << (p * cpp + c);
            if (__any_sync(kFull, x1 != 0)) bad |= 1u << (p * cpp + c + 1);
          }
          if (c < nfull && __any_sync(kFull, differs(sd, c) != 0)) bad |= 1u << (p * cpp + c);
          __syncwarp();  // the match stage has been read
          if (lane == 0)
            stage_piece(seq + kWspMS, mstages + (size_t)ms * A.stage_bytes, b_mfull + ms, keep);
        }
        const unsigned long long c0 = 32ull * g;
        const uint32_t nch = (uint32_t)((A.nchunks - c0) < 32 ? (A.nchunks - c0) : 32);
        uint32_t valid = nch >= 32 ? kFull : ((1u << nch) - 1u);
        if (short_tail && c0 + nch == A.nchunks) valid &= ~(1u << (nch - 1));
        const uint32_t pw = m ? (~bad & valid) : 0u;
        const uint32_t units = (uint32_t)(ibp_group_bits(g, pw, A.nchunks, tail_bytes, cb, m) >> 7);
        if (lane == 0) {
          s_cpw[i % (lag + 1)] = pw;
          if (g + 1 != fault1) st_relaxed_u32(A.lens + g, 0x80000000u | units);
        }
      }
      if (i + 1 == lag) lens_fetch(0);
      if (i >= lag) {
        // ---- resolve the group of wave j = i - D and hand it over
        const uint32_t j = i - lag;
        const unsigned long long wf = (unsigned long long)j * G, la0 = wf & ~3ull;
        const uint32_t nw = (uint32_t)((A.ntiles - wf) < G ? (A.ntiles - wf) : G);
        const uint32_t nv4 = (uint32_t)((wf + nw - la0 + 3) / 4);
        uint4* lb = reinterpret_cast<uint4*>(lensbuf + (j & 1u) * kWsLensBytes);
        cp_async_wait_all();
        __syncwarp();
        uint32_t pre = 0, tot = 0;
        for (unsigned spins = 0;; ++spins) {
          bool all = true;
          pre = 0;
          tot = 0;
          for (uint32_t vi = lane; vi < nv4; vi += 32) {
            const uint4 e4 = lb[vi];
            const uint32_t e[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
            for (uint32_t q = 0; q < 4; ++q) {
              const unsigned long long idx = la0 + 4ull * vi + q;  // group index
              if (idx >= wf && idx < wf + nw) {
                if (!(e[q] >> 31)) all = false;
                const uint32_t u = e[q] & 0x7FFFFFFFu;
                tot += u;
                if (idx < wf + bid) pre += u;
              }
            }
          }
          if (__all_sync(kFull, all)) break;
          if (spins >= lim) {
            if (lane == 0) set_status(A.ctrl, ZC_ERR_TIMEOUT);
            break;
          }
          // the call has failed: no more waiting (one vote for the warp)
          if (__any_sync(kFull, get_status(A.ctrl) != 0)) break;
          __nanosleep(spins < 64 ? 32 : 256);
          for (uint32_t vi = lane; vi < nv4; vi += 32) lb[vi] = ld_relaxed_v4(A.lens + la0 + 4ull * vi);
          __syncwarp();
        }
        __syncwarp();  // lens buffer j & 1 has been read
        lens_fetch(j + 1);
        pre = __reduce_add_sync(kFull, pre);
        tot = __reduce_add_sync(kFull, tot);
        const unsigned long long base = (wave_base + pre) * 128ull;
        wave_base += tot;
        const unsigned long long g = bid + wf;
        const uint32_t pw = s_cpw[j % (lag + 1)];
        const uint32_t gb = (uint32_t)ibp_group_bits(g, pw, A.nchunks, tail_bytes, cb, m);
        if (lane == 0) {
          grp[g] = base;
          if (g + 1 == A.ntiles) grp[A.ngroups] = base + gb;
        }
        // slot j % R, once the pack warps have read its previous contents
        const uint32_t k = j % kWsInfo, f = j / kWsInfo;
        if (f > 0 && !mbar_wait(b_iempty + k, (f - 1) & 1u)) set_status(A.ctrl, ZC_ERR_TIMEOUT);
        if (lane == 0) {
          WsInfo& si = s_info[k];
          si.base = base;
          si.pw[0] = pw;
          si.gex[0] = 0;
          si.agg = gb;
          si.raw = pw == 0;
          mbar_arrive(b_ifull + k);
        }
        __syncwarp();
      }
    }
    cp_async_wait_all();
  } else {
    // ================================================= pack warps
    const uint32_t r_own = (uint32_t)t & (vpc - 1);  // every vector's position
    PackTab pt{};
    {
      VecTab v0;
      load_vectab(T, r_own, v0);
      make_runs(v0);
      make_runs3(v0);
      make_packtab(v0, pt);
    }
    const unsigned long long drop = l2_policy_first();
    if (t == 0)
      for (uint32_t s = 0; s < kWspPS; ++s)
        stage_piece(s, pstages + (size_t)s * A.stage_bytes, b_sfull + s, drop);
    uint32_t carry = 0;  // thread 0, raw groups: the previous piece's last input word
    for (uint32_t j = 0; j < mine; ++j) {
      const uint32_t k = j % kWsInfo;
      if (!mbar_wait(b_ifull + k, (j / kWsInfo) & 1u)) set_status(A.ctrl, ZC_ERR_TIMEOUT);
      const unsigned long long base = s_info[k].base;
      const uint32_t pw = s_info[k].pw[0], agg = s_info[k].agg;
      const bool raw = s_info[k].raw != 0;
      // the group's chunk table (every pack thread is past the previous group)
      if (!raw) fill_chunk_table(s_coff, (uint32_t)t, pw, 0u, B, m);
      named_bar(1, kWspPack);  // every pack thread has read the slot; the table is filled
      if (t == 0) mbar_arrive(b_iempty + k);
      const unsigned long long g = bid + (unsigned long long)j * G;
      const unsigned long long dst0 = A.off_payload + (base >> 3);
      const bool fits = dst0 + (agg >> 3) <= A.dst_cap;
      if (!fits && t == 0) set_status(A.ctrl, ZC_ERR_CAPACITY);
      carry = 0;  // a raw group's participation word
      for (uint32_t p = 0; p < np; ++p) {
        const uint32_t tb = piece_bytes(g, p);
        if (tb == 0) break;
        const bool last = p + 1 == np || piece_bytes(g, p + 1) == 0;
        const uint32_t seq = j * np + p, s = seq % kWspPS;
        if (!mbar_wait(b_sfull + s, (seq / kWspPS) & 1u)) set_status(A.ctrl, ZC_ERR_TIMEOUT);
        const uint32_t* sd = reinterpret_cast<const uint32_t*>(pstages + (size_t)s * A.stage_bytes);
        const uint32_t twords = tb / 4, nvec = (tb + 15) / 16;
        const uint32_t c0 = p * cpp;  // the piece's first chunk in the group
        if (raw) {
          // [0][input words][zero padding]: output vector u of piece p is
          // stream words 4096 p + 4 u .. + 3, i.e. the piece's input words
          // 4 u - 1 .. 4 u + 2 (word -1: the previous piece's last word)
          const uint32_t ibase = c0 * B;  // the piece's first 128-bit boundary
          const uint32_t nfull = last ? (agg - ibase) >> 7 : kWspPiece / 16;
          const unsigned long long dst = dst0 + (ibase >> 3);
          for (uint32_t u0 = t; u0 - lane < nfull; u0 += 4 * kWspPack) {
            uint4 o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t u = u0 + e * kWspPack;
              uint4 x = make_uint4(0, 0, 0, 0);
              if (u < nfull) {
                if (4 * u + 3 < twords) {
                  x = *reinterpret_cast<const uint4*>(sd + 4 * u);
                } else {
                  x.x = 4 * u < twords ? sd[4 * u] : 0u;
                  x.y = 4 * u + 1 < twords ? sd[4 * u + 1] : 0u;
                  x.z = 4 * u + 2 < twords ? sd[4 * u + 2] : 0u;
                }
              }
              uint32_t prev = __shfl_up_sync(kFull, x.w, 1);
              if (lane == 0)
                prev = u == 0 ? carry : ((u < nfull && 4 * u - 1 < twords) ? sd[4 * u - 1] : 0u);
              o[e] = make_uint4(prev, x.x, x.y, x.z);
            }
            if (fits) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const uint32_t u = u0 + e * kWspPack;
                if (u < nfull) st_v4_hint(A.dst + dst + 16ull * u, o[e], drop);
              }
            }
          }
          if (t == 0) carry = sd[twords - 1];
          named_bar(1, kWspPack);  // the stage has been read
          if (t == 0) stage_piece(seq + kWspPS, pstages + (size_t)s * A.stage_bytes, b_sfull + s, drop);
        } else {
          // bit P of the group's stream starts the piece; the image holds the
          // stream from ibase = P rounded down to 128 bits
          const uint32_t P = 32u + c0 * B - (uint32_t)__popc(pw & lowmask(c0)) * m;
          const uint32_t ibase = P & ~127u;
          const uint32_t Pn = last ? agg : 32u + (c0 + cpp) * B - (uint32_t)__popc(pw & lowmask(c0 + cpp)) * m;
          const uint32_t nfull = (Pn - ibase) >> 7;  // vectors complete after this piece
          if (p == 0 && t == 0) atomicOr(img, pw);  // the participation word
          const uint32_t g1 = 32u - ibase;  // modulo 2^32: chunk starts relative to the image
          if (pt.ok) {
            // chunk c's first bit relative to the image: its table entry - ibase
            pack_any<2, 2, kWspPack>(pt, sd, nvec, twords, nullptr, nullptr, s_coff, pw, 0u - ibase,
                                     c0, A.lvpc, r_own, B, m, img, t);
          } else {
            for (uint32_t v = t; v < nvec; v += kWspPack) {
              const uint32_t c = c0 + (v >> A.lvpc);
              VecTab vt;
              load_vectab(T, r_own, vt);
              const uint4 d = *reinterpret_cast<const uint4*>(sd + 4 * v);
              const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
              const uint32_t off = g1 + c * B - (uint32_t)__popc(pw & lowmask(c)) * m;
              uint32_t o[4], pos;
              if ((pw >> c) & 1u) {
                uint32_t f[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) f[w] = vt_compress(vt, dw[w], w);
                uint32_t kk[4];
                kept_bits(vt, kk);
                cat4(f, kk, o);
                pos = off + vt.Pr;
              } else {
                const uint32_t wv = (twords - 4 * v) < 4u ? (twords - 4 * v) : 4u;
#pragma unroll
                for (uint32_t w = 0; w < 4; ++w) o[w] = w < wv ? dw[w] : 0u;
                pos = off + 128u * r_own;
              }
              img_or(img, pos, o);
            }
          }
          named_bar(1, kWspPack);  // the piece is in the image; the stage has been read
          if (t == 0) stage_piece(seq + kWspPS, pstages + (size_t)s * A.stage_bytes, b_sfull + s, drop);
          const unsigned long long dst = dst0 + (ibase >> 3);
          for (uint32_t u0 = t; u0 < nfull; u0 += 4 * kWspPack) {
            uint4 o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const uint32_t u = u0 + e * kWspPack;
              if (u < nfull) {
                o[e] = img4[u];
                img4[u] = make_uint4(0, 0, 0, 0);
              }
            }
            if (fits) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const uint32_t u = u0 + e * kWspPack;
                if (u < nfull) st_v4_hint(A.dst + dst + 16ull * u, o[e], drop);
              }
            }
          }
          // the partial vector (the next piece's first) to the front: thread 0
          // copied out vector 0 above, and no thread copies vector nfull
          if (t == 0 && !last && nfull > 0) {
            img4[0] = img4[nfull];
            img4[nfull] = make_uint4(0, 0, 0, 0);
          }
          named_bar(1, kWspPack);  // the image is ready for the next piece
        }
      }
    }
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
  const unsigned long long pay = A.ngroups ? grp[A.ngroups] : 0ull;
  ibp_write_tail(A.meta, cb, m, A.n_bytes, A.nchunks, A.ngroups, A.dst, A.dst_cap, A.off_payload,
                 A.out_bytes, A.ctrl, pay, t, kWspThreads);
}

template <int NT, bool REG>
__global__ void __launch_bounds__(NT, 512 / NT) ibp_decode_pipe_kernel(PipeArgs A) {
  constexpr int NW = NT / 32;
  extern __shared__ __align__(128) uint8_t dyn[];
  __shared__ uint32_t s_scr[NW + 4];
  __shared__ unsigned long long s_h[10];
  __shared__ int s_ok;
  __shared__ unsigned long long s_tile[kMaxStages];
  __shared__ unsigned long long s_goff[kMaxStages][kMaxQ + 1];
  __shared__ int s_sbad[kMaxStages];
  __shared__ uint32_t s_pw[2][kMaxQ];
  __shared__ int s_gbad[2][kMaxQ];
  __shared__ uint32_t s_off[2][kMaxQ][32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t cb = A.cb, W = cb / 4, B = 8 * cb, Q = A.Q, S = A.S;

  uint32_t* tab = reinterpret_cast<uint32_t*>(dyn);
  uint8_t* stages = dyn + 4 * ibp_table_words(W);
  unsigned long long* bars =
      reinterpret_cast<unsigned long long*>(stages + (size_t)S * A.stage_bytes);

  IbpTables T;
  const bool meta_ok = ibp_load_tables<NT>(A.meta, cb, tab, T, s_scr);
  const uint32_t m = T.m;
  if (t == 0) {
    const int err = ibp_check_stream(A.meta, meta_ok, cb, m, A.src, A.src_bytes, A.dst_cap,
                                     blockIdx.x == 0, s_h);
    if (err) set_status(A.ctrl, err);
    s_ok = err == 0;
    for (uint32_t s = 0; s < S; ++s) mbar_init(bars + s, 1);
  }
  __syncthreads();
  if (!s_ok) return;
  const unsigned long long n_bytes = s_h[2], nchunks = s_h[3], ngroups = s_h[4];
  const unsigned long long off_payload = s_h[7], pay_bits = s_h[8];
  const unsigned long long ntiles = (ngroups + Q - 1) / Q;
  const unsigned long long tail_bytes = n_bytes - (nchunks ? (nchunks - 1) * cb : 0ull);
  const unsigned long long tile_raw = 32ull * Q * cb;
  const unsigned long long* grp = reinterpret_cast<const unsigned long long*>(A.src + kIbp1Header);
  const uint32_t cap = A.stage_bytes - kStageSlack;

  UnpackTab ut{};
  if (REG) {
    VecTab v0;
    load_vectab(T, (uint32_t)t & (A.vpc - 1), v0);
    make_runs(v0);
    make_runs3(v0);
    make_unpacktab(v0, ut);
  }

  // warp 0: the span of this block's kk-th tile.  prefetch() loads its
  // group-table entries into registers (their latency overlaps the current
  // tile's work); issue() checks them and starts the copy into stage s.
  unsigned long long pf_go = 0, pf_gend = 0;
  auto prefetch = [&](unsigned long long kk) {
    const unsigned long long tile = blockIdx.x + kk * gridDim.x;
    if (tile >= ntiles) return;
    const unsigned long long g0 = tile * Q;
    const uint32_t nq = (uint32_t)((ngroups - g0) < Q ? (ngroups - g0) : Q);
    pf_gend = grp[g0 + nq];
    pf_go = (uint32_t)lane < nq ? grp[g0 + lane] : 0ull;
  };
  auto issue = [&](unsigned long long kk, uint32_t s) {
    const unsigned long long tile = blockIdx.x + kk * gridDim.x;
    if (tile >= ntiles) {
      if (lane == 0) s_tile[s] = tile;
      return;
    }
    const unsigned long long g0 = tile * Q;
    const uint32_t nq = (uint32_t)((ngroups - g0) < Q ? (ngroups - g0) : Q);
    const unsigned long long gend = pf_gend;
    const unsigned long long go = (uint32_t)lane < nq ? pf_go : gend;
    const unsigned long long nx0 = __shfl_down_sync(kFull, go, 1);
    const unsigned long long nx = (uint32_t)lane + 1 < nq ? nx0 : gend;
    bool bad = false;
    if ((uint32_t)lane < nq) bad = (go & 127) != 0 || nx < go + 128 || nx > pay_bits;
    const unsigned long long first = __shfl_sync(kFull, go, 0);
    bad = __any_sync(kFull, bad) || ((gend - first) >> 3) > cap;
    if ((uint32_t)lane < nq) s_goff[s][lane] = go;
    if (lane == 0) {
      s_goff[s][nq] = gend;
      s_tile[s] = tile;
      s_sbad[s] = bad;
      if (bad) {
        mbar_arrive_expect_tx(bars + s, 0);  // nothing to copy: the phase completes now
      } else {
        const uint32_t bytes = (uint32_t)((gend - first) >> 3);
        mbar_arrive_expect_tx(bars + s, bytes);
        bulk_g2s(stages + (size_t)s * A.stage_bytes, A.src + off_payload + (first >> 3), bytes,
                 bars + s);
      }
    }
  };
  // The scan of the kk-th tile (in stage s) into buffer bf: the chunk bit
  // offsets of its groups (one warp per group, from the last warp down).
  auto scan = [&](uint32_t kk, uint32_t s, uint32_t bf) {
    const unsigned long long tile = s_tile[s];
    if (tile >= ntiles) return;
    const unsigned long long g0 = tile * Q;
    const uint32_t nq = (uint32_t)((ngroups - g0) < Q ? (ngroups - g0) : Q);
    const uint32_t qw = (uint32_t)(NW - 1 - warp);  // the last warp takes group 0
    if (qw >= nq) return;
    const bool waited = mbar_wait(bars + s, (kk / S) & 1);
    if (!waited) set_status(A.ctrl, ZC_ERR_TIMEOUT);
    const uint32_t* sd = reinterpret_cast<const uint32_t*>(stages + (size_t)s * A.stage_bytes);
    const bool sbad = s_sbad[s] != 0 || !waited;
    const unsigned long long base = s_goff[s][0];
    for (uint32_t q = qw; q < nq; q += NW) {
      const uint32_t gs = (uint32_t)(s_goff[s][q] - base), ge = (uint32_t)(s_goff[s][q + 1] - base);
      const uint32_t pw = sbad ? 0u : sd[gs >> 5];
      const unsigned long long c = (g0 + q) * 32ull + lane;
      const bool present = c < nchunks;
      const bool full = present && (c + 1 < nchunks || tail_bytes == cb);
      const bool p = (pw >> lane) & 1u;
      bool bad = sbad || (p && (!full || m == 0));
      const uint32_t len = !present ? 0u : (p ? B - m : (full ? B : 8u * (uint32_t)tail_bytes));
      uint32_t inc = len;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += u;
      }
      s_off[bf][q][lane] = gs + 32u + inc - len;
      const uint32_t tot = __shfl_sync(kFull, inc, 31);
      if (round_up_dev(32ull + tot, 128) != (unsigned long long)(ge - gs)) bad = true;
      bad = __any_sync(kFull, bad);
      if (lane == 0) {
        s_pw[bf][q] = pw;
        s_gbad[bf][q] = bad;
      }
    }
  };
  if (warp == 0)
    for (uint32_t s = 0; s < S; ++s) {
      prefetch(s);
      issue(s, s);
    }
  __syncthreads();
  scan(0, 0, 0);
  __syncthreads();

  // Tile k is expanded, then tile k + 1 scanned; one barrier per tile.  The
  // loop is compiled for two-run and for three-run tables; a block whose
  // threads all have two-run tables takes the first (the choice is the same
  // for every thread of the block, so all take the same barriers).
  auto tiles = [&](auto three_runs) {
  constexpr bool THREE = decltype(three_runs)::value;
  for (uint32_t k = 0;; ++k) {
    const uint32_t s = k % S, bf = k & 1;
    const unsigned long long tile = s_tile[s];
    if (tile >= ntiles) break;
    if (warp == 0) prefetch(k + S);
    const bool waited = mbar_wait(bars + s, (k / S) & 1);
    if (!waited) set_status(A.ctrl, ZC_ERR_TIMEOUT);
    const uint32_t* sd = reinterpret_cast<const uint32_t*>(stages + (size_t)s * A.stage_bytes);
    const unsigned long long b0 = tile * tile_raw, g0 = tile * Q;
    const uint32_t nq = (uint32_t)((ngroups - g0) < Q ? (ngroups - g0) : Q);
    const uint32_t tb = (uint32_t)((n_bytes - b0) < tile_raw ? (n_bytes - b0) : tile_raw);
    const uint32_t twords = tb / 4, nvec = (tb + 15) / 16;
    uint32_t* yt = reinterpret_cast<uint32_t*>(A.dst + b0);
    if (Q == 1 && s_pw[bf][0] == 0 && !s_gbad[bf][0]) {
      // A tile of one group in which no chunk participates: output word j is
      // stream word 1 + j.  A lane loads stage vector v (words 4v .. 4v + 3)
      // and takes word 4v + 4 from the lane above (lane 31 reads it), so the
      // lane just past the last vector loads too (inside the stage: a stage
      // holds 16 bytes more than a tile's vectors); the loop runs while the
      // warp's first vector is in (the shuffle takes every lane).  The same
      // for every thread of the block.
      const uint4* sd4 = reinterpret_cast<const uint4*>(sd);
      for (uint32_t v = t; v - lane < nvec; v += NT) {
        const uint4 x = v <= nvec ? sd4[v] : make_uint4(0, 0, 0, 0);
        uint32_t nx = __shfl_down_sync(kFull, x.x, 1);
        if (lane == 31) nx = v < nvec ? sd[4 * v + 4] : 0u;
        if (v < nvec) {
          const uint32_t wv = (twords - 4 * v) < 4u ? (twords - 4 * v) : 4u;
          if (wv == 4) {
            st_v4(yt + 4 * v, make_uint4(x.y, x.z, x.w, nx));
          } else {
            const uint32_t o[3] = {x.y, x.z, x.w};
#pragma unroll
            for (uint32_t w = 0; w < 3; ++w)
              if (w < wv) yt[4 * v + w] = o[w];
          }
        }
      }
    } else
    // two vectors per thread per step (same chunk position, so the same
    // register tables): two independent dependency chains to interleave
    for (uint32_t v0 = t; v0 < nvec; v0 += 2 * NT) {
      uint32_t o[2][4];
      bool live[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t v = v0 + e * NT;
        live[e] = false;
        if (v >= nvec) continue;
        uint32_t c, r;
        vec_pos<REG>(A, v, c, r);
        const uint32_t q = c >> 5, i = c & 31;
        if (s_gbad[bf][q]) continue;
        live[e] = true;
        const uint32_t off = s_off[bf][q][i];
        uint32_t u[4];
        if ((s_pw[bf][q] >> i) & 1u) {
          if (REG && ut.ok) {
            // each word's field read at its own bit offset, expanded from runs
            const uint32_t p0 = off + ut.Pr;
            const uint32_t cw[4] = {0u, ut.c1, ut.c2, ut.c3};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const uint32_t pos = p0 + cw[w], a = pos >> 5, sh = pos & 31;
              const uint32_t f = __funnelshift_r(sd[a], sd[a + 1], sh) & ut.km[w];
              uint32_t x = ((f << ut.a0[w]) & ut.M0[w]) | ((f << ut.e1[w]) & ut.M1[w]);
              if (THREE) x |= (f << ut.e2[w]) & ut.M2[w];
              o[e][w] = x | ut.V[w];
            }
          } else {
            VecTab vt;
            load_vectab(T, r, vt);
            win128(sd, off + vt.Pr, u);
            uint32_t f[4];
            uint32_t kk[4];
            kept_bits(vt, kk);
            split4(u, kk, f);
#pragma unroll
            for (int w = 0; w < 4; ++w) o[e][w] = hd_expand(f[w], vt.K[w], &vt.MV[0][w], 4) | vt.V[w];
          }
        } else {
          win128(sd, off + 128u * r, u);
#pragma unroll
          for (int w = 0; w < 4; ++w) o[e][w] = u[w];
        }
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t v = v0 + e * NT;
        if (!live[e]) continue;
        const uint32_t wv = (twords - 4 * v) < 4u ? (twords - 4 * v) : 4u;
        if (wv == 4) {
          st_v4(yt + 4 * v, make_uint4(o[e][0], o[e][1], o[e][2], o[e][3]));
        } else {
#pragma unroll
          for (uint32_t w = 0; w < 4; ++w)
            if (w < wv) yt[4 * v + w] = o[e][w];
        }
      }
    }
    if ((uint32_t)t < nq && s_gbad[bf][t]) set_status(A.ctrl, ZC_ERR_FORMAT);
    // after this warp's share, so that waiting for the next tile to land
    // overlaps the expansion
    scan(k + 1, (k + 1) % S, bf ^ 1);
    __syncthreads();  // stage s read; the next tile's scan written
    if (warp == 0) issue(k + S, s);
  }
  };
  if (__syncthreads_or(REG && ut.three ? 1 : 0)) tiles(std::true_type{});
  else tiles(std::false_type{});
}

// ------------------------------------------------------------------ launch

struct Geo {
  bool ok;
  int nt;   // decode: threads per block; encode: packer warps
  bool reg;
  uint32_t Q, S, stage_bytes, img_words;
  size_t smem;
};

constexpr size_t kSmemPerSm = 233472;     // shared memory per SM
constexpr size_t kSmemPerBlock = 232448;  // most one block may use
constexpr size_t kSmemReserved = 1024;    // the system's share per resident block

template <typename K>
void attrs(K k, size_t* stat, int* regs) {
  cudaFuncAttributes a{};
  cudaFuncGetAttributes(&a, k);
  *stat = a.sharedSizeBytes;
  *regs = a.numRegs;
}

void tile_shape(uint32_t cb, bool enc, Geo& g) {
  g.Q = cb >= 512 ? 1u : std::min<uint32_t>(kMaxQ, 512u / cb);
  const uint64_t raw = 32ull * g.Q * cb;
  const uint64_t maxc = (uint64_t)g.Q * (32ull * cb + 16ull);  // largest compressed tile
  g.stage_bytes = (uint32_t)(round_up(enc ? raw : maxc, 128) + kStageSlack);
  g.img_words = enc ? (uint32_t)round_up(raw / 4 + 4ull * g.Q + 16, 4) : 0u;
}

// Stages that fit `blocks` resident blocks per SM (0 if fewer than 2).
uint32_t stages_for(int blocks, size_t stat, size_t fixed, uint32_t stage_bytes) {
  const size_t per = std::min(kSmemPerSm / blocks - kSmemReserved, kSmemPerBlock);
  if (per <= stat + fixed) return 0;
  const size_t st = std::min<size_t>((per - stat - fixed) / stage_bytes, kMaxStages);
  return st >= 2 ? (uint32_t)st : 0u;
}

// Encode (the pack kernel): the smallest block (most blocks per SM, each with
// its own pipeline) whose shared memory holds the image and at least 2 stages.
Geo pick_enc(uint32_t cb) {
  Geo g{};
  tile_shape(cb, true, g);
  const uint32_t vpc = cb / 16;
  const size_t fixed = 4 * ibp_table_words(cb / 4) + 4ull * g.img_words + 8 * kMaxStages;
  for (int nt : {128, 256, 512}) {
    size_t stat = 0, s2 = 0;
    int regs = 0, r2 = 0;
    if (nt == 128) {
      attrs(ibp_pack_kernel<128, true>, &stat, &regs);
      attrs(ibp_pack_kernel<128, false>, &s2, &r2);
    } else if (nt == 256) {
      attrs(ibp_pack_kernel<256, true>, &stat, &regs);
      attrs(ibp_pack_kernel<256, false>, &s2, &r2);
    } else {
      attrs(ibp_pack_kernel<512, true>, &stat, &regs);
      attrs(ibp_pack_kernel<512, false>, &s2, &r2);
    }
    const uint32_t st = stages_for(512 / nt, std::max(stat, s2), fixed, g.stage_bytes);
    if (st) {
      g.ok = true;
      g.nt = nt;
      g.reg = pow2(vpc) && (uint32_t)nt % vpc == 0;
      g.S = st;
      g.smem = fixed + st * g.stage_bytes;
      return g;
    }
  }
  return g;
}

// Decode: the smallest block (most blocks per SM, each with its own
// pipeline) whose shared memory holds at least 2 stages.
Geo pick_dec(uint32_t cb) {
  Geo g{};
  tile_shape(cb, false, g);
  const uint32_t vpc = cb / 16;
  const size_t fixed = 4 * ibp_table_words(cb / 4) + 8 * kMaxStages;
  for (int nt : {128, 256, 512}) {
    size_t stat = 0, s2 = 0;
    int regs = 0, r2 = 0;
    if (nt == 128) {
      attrs(ibp_decode_pipe_kernel<128, true>, &stat, &regs);
      attrs(ibp_decode_pipe_kernel<128, false>, &s2, &r2);
    } else if (nt == 256) {
      attrs(ibp_decode_pipe_kernel<256, true>, &stat, &regs);
      attrs(ibp_decode_pipe_kernel<256, false>, &s2, &r2);
    } else {
      attrs(ibp_decode_pipe_kernel<512, true>, &stat, &regs);
      attrs(ibp_decode_pipe_kernel<512, false>, &s2, &r2);
    }
    const uint32_t st = stages_for(512 / nt, std::max(stat, s2), fixed, g.stage_bytes);
    if (st) {
      g.ok = true;
      g.nt = nt;
      g.reg = pow2(vpc) && (uint32_t)nt % vpc == 0;
      g.S = st;
      g.smem = fixed + st * g.stage_bytes;
      return g;
    }
  }
  return g;
}

Geo pick(uint32_t cb, bool enc) {
  static std::mutex mu;
  static Geo cache[2][2048 / 16 + 1];
  static bool have[2][2048 / 16 + 1];
  if (cb == 0 || cb > 2048 || cb % 16) return Geo{};
  std::lock_guard<std::mutex> lk(mu);
  const int e = enc ? 1 : 0, i = (int)(cb / 16);
  if (!have[e][i]) {
    cache[e][i] = enc ? pick_enc(cb) : pick_dec(cb);
    have[e][i] = true;
  }
  return cache[e][i];
}

template <typename K, typename Args>
cudaError_t launch(K k, int nt, const Args& A, size_t smem, unsigned long long work,
                   cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int res = resident_blocks((const void*)k, nt, smem);
  unsigned long long grid = work < (unsigned long long)res ? work : (unsigned long long)res;
  if (grid == 0) grid = 1;
  k<<<(unsigned)grid, nt, smem, s>>>(A);
  return cudaGetLastError();
}

// dep: launched with launch_dependent (the kernel calls grid_dep_wait()).
template <typename K>
cudaError_t launch(K k, int nt, const PipeArgs& A, const Geo& g, unsigned long long work,
                   cudaStream_t s, bool dep = false) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem);
  if (e != cudaSuccess) return e;
  const int res = resident_blocks((const void*)k, nt, g.smem);
  unsigned long long grid = work < (unsigned long long)res ? work : (unsigned long long)res;
  if (grid == 0) grid = 1;
  if (dep) return launch_dependent(k, (unsigned)grid, (unsigned)nt, g.smem, s, A);
  k<<<(unsigned)grid, nt, g.smem, s>>>(A);
  return cudaGetLastError();
}

void fill_shape(PipeArgs& A, const Geo& g) {
  A.vpc = A.cb / 16;
  A.lvpc = 0;
  while ((1u << A.lvpc) < A.vpc) ++A.lvpc;
  A.Q = g.Q;
  A.S = g.S;
  A.stage_bytes = g.stage_bytes;
  A.img_words = g.img_words;
}

// The single-pass encoder for chunks of up to 512 bytes (one group of 16 KB
// per tile, or several groups of smaller chunks).
cudaError_t ibp_ws_compress(const void* d_meta, uint32_t cb, const void* d_x,
                            unsigned long long n_bytes, void* d_out, unsigned long long out_cap,
                            unsigned long long* d_out_bytes, void* d_ws, cudaStream_t s) {
  Geo g{};
  tile_shape(cb, true, g);
  const unsigned long long nchunks = (n_bytes + cb - 1) / cb, ngroups = (nchunks + 31) / 32;
  PipeArgs A{};
  A.meta = static_cast<const uint8_t*>(d_meta);
  A.src = static_cast<const uint8_t*>(d_x);
  A.dst = static_cast<uint8_t*>(d_out);
  A.dst_cap = out_cap;
  A.n_bytes = n_bytes;
  A.cb = cb;
  A.nchunks = nchunks;
  A.ngroups = ngroups;
  A.ntiles = (ngroups + g.Q - 1) / g.Q;
  A.off_payload = kIbp1Header + round_up(8ull * (ngroups + 1), 128);
  A.out_bytes = d_out_bytes;
  A.ctrl = static_cast<Ctrl*>(d_ws);
  A.lens = reinterpret_cast<uint32_t*>(static_cast<char*>(d_ws) + kCtrlBytes);
  g.S = kWsStages;
  fill_shape(A, g);
  const bool reg = pow2(A.vpc) && A.vpc <= 32;
  const size_t smem = ws_smem_bytes(cb, g.stage_bytes, g.img_words);
  auto k = reg ? ibp_encode_ws_kernel<true> : ibp_encode_ws_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  unsigned long long grid = (unsigned long long)resident_blocks((const void*)k, kWsThreads, smem);
  if (grid > kWsMaxGrid) grid = kWsMaxGrid;
  if (grid > A.ntiles) grid = A.ntiles;
  if (grid == 0) grid = 1;
  // workspace: control block | one length word per tile (+ one vector of slack)
  e = cudaMemsetAsync(d_ws, 0, kCtrlBytes + 4ull * A.ntiles + 16, s);
  if (e != cudaSuccess) return e;
  e = arm_wait_fault(d_ws, s);
  if (e != cudaSuccess) return e;
  // The blocks wait for lengths that every other block of the launch
  // publishes: a cooperative launch makes the whole grid resident at once (or
  // is refused, cudaErrorCooperativeLaunchTooLarge, e.g. on a GPU whose SMs
  // are shared out), so no block ever waits for one that cannot start.
  void* kargs[] = {&A};
  return cudaLaunchCooperativeKernel((const void*)k, dim3((unsigned)grid), dim3(kWsThreads), kargs,
                                     smem, s);
}

// The single-pass encoder in pieces, for chunks of 1024 and 2048 bytes (a
// group per tile, moved through shared memory 16 KB at a time).
cudaError_t ibp_wsp_compress(const void* d_meta, uint32_t cb, const void* d_x,
                             unsigned long long n_bytes, void* d_out, unsigned long long out_cap,
                             unsigned long long* d_out_bytes, void* d_ws, cudaStream_t s) {
  const unsigned long long nchunks = (n_bytes + cb - 1) / cb, ngroups = (nchunks + 31) / 32;
  PipeArgs A{};
  A.meta = static_cast<const uint8_t*>(d_meta);
  A.src = static_cast<const uint8_t*>(d_x);
  A.dst = static_cast<uint8_t*>(d_out);
  A.dst_cap = out_cap;
  A.n_bytes = n_bytes;
  A.cb = cb;
  A.nchunks = nchunks;
  A.ngroups = ngroups;
  A.ntiles = ngroups;
  A.off_payload = kIbp1Header + round_up(8ull * (ngroups + 1), 128);
  A.out_bytes = d_out_bytes;
  A.ctrl = static_cast<Ctrl*>(d_ws);
  A.lens = reinterpret_cast<uint32_t*>(static_cast<char*>(d_ws) + kCtrlBytes);
  A.vpc = cb / 16;
  A.lvpc = 0;
  while ((1u << A.lvpc) < A.vpc) ++A.lvpc;
  A.Q = 1;
  A.S = 2;
  A.stage_bytes = (uint32_t)(round_up(kWspPiece, 128) + kStageSlack);
  A.img_words = kWspPiece / 4 + 16;
  A.lag = g_wsp_lag.load();
  const size_t smem = wsp_smem_bytes(cb, A.stage_bytes, A.img_words);
  auto k = cb == 2048 ? ibp_encode_wsp_kernel<4> : ibp_encode_wsp_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  unsigned long long grid = (unsigned long long)resident_blocks((const void*)k, kWspThreads, smem);
  if (grid > kWsMaxGrid) grid = kWsMaxGrid;
  if (grid > A.ntiles) grid = A.ntiles;
  if (grid == 0) grid = 1;
  // workspace: control block | one length word per group (+ one vector of slack)
  e = cudaMemsetAsync(d_ws, 0, kCtrlBytes + 4ull * A.ntiles + 16, s);
  if (e != cudaSuccess) return e;
  e = arm_wait_fault(d_ws, s);
  if (e != cudaSuccess) return e;
  // blocks wait for every other block's group lengths: the whole grid must
  // be resident at once (see ibp_ws_compress)
  void* kargs[] = {&A};
  return cudaLaunchCooperativeKernel((const void*)k, dim3((unsigned)grid), dim3(kWspThreads), kargs,
                                     smem, s);
}

std::atomic<int> g_single_pass{1};  // 0: the three-launch encode for every chunk size (tests)

}  // namespace

void ibp_set_single_pass(int on) { g_single_pass.store(on ? 1 : 0); }

void ibp_set_wsp_lag(int lag) { g_wsp_lag.store(lag < 1 ? 1 : (lag > 3 ? 3 : lag)); }

bool ibp_pipe_supported(uint32_t cb, bool encode) { return cb <= 2048 && pick(cb, encode).ok; }

cudaError_t ibp_pipe_compress(const void* d_meta, uint32_t cb, const void* d_x,
                              unsigned long long n_bytes, void* d_out, unsigned long long out_cap,
                              unsigned long long* d_out_bytes, void* d_ws, cudaStream_t s) {
  if ((cb <= 512 || cb == 1024 || cb == 2048) && g_single_pass.load()) {
    const cudaError_t e =
        cb <= 512 ? ibp_ws_compress(d_meta, cb, d_x, n_bytes, d_out, out_cap, d_out_bytes, d_ws, s)
                  : ibp_wsp_compress(d_meta, cb, d_x, n_bytes, d_out, out_cap, d_out_bytes, d_ws, s);
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    cudaGetLastError();  // the grid cannot be resident at once here: three launches instead
  }
  const Geo g = pick(cb, true);
  const unsigned long long nchunks = (n_bytes + cb - 1) / cb, ngroups = (nchunks + 31) / 32;
  const unsigned long long ntiles2 = (ngroups + kOffNT * kOffIPT - 1) / (kOffNT * kOffIPT);
  // workspace: control block | offsets-pass look-back states | participation words
  char* ws = static_cast<char*>(d_ws);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws);
  unsigned long long* states = reinterpret_cast<unsigned long long*>(ws + kCtrlBytes);
  uint32_t* pw = reinterpret_cast<uint32_t*>(ws + kCtrlBytes + round_up(8ull * ntiles2, 256));
  cudaError_t e = cudaMemsetAsync(d_ws, 0, kCtrlBytes + 8ull * ntiles2, s);
  if (e != cudaSuccess) return e;
  e = arm_wait_fault(d_ws, s);
  if (e != cudaSuccess) return e;
  unsigned long long* grp =
      reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(d_out) + kIbp1Header);
  if (ngroups) {
    MatchArgs M{};
    M.meta = static_cast<const uint8_t*>(d_meta);
    M.x = static_cast<const uint32_t*>(d_x);
    M.n_bytes = n_bytes;
    M.nchunks = nchunks;
    M.ngroups = ngroups;
    M.cb = cb;
    M.vpc = cb / 16;
    M.lvpc = 0;
    while ((1u << M.lvpc) < M.vpc) ++M.lvpc;
    M.pw = pw;
    M.ctrl = ctrl;
    const size_t msmem = 4 * ibp_table_words(cb / 4);
    const unsigned long long mwork = (ngroups + 7) / 8;
    const int mode = !pow2(M.vpc) ? 3 : (M.vpc <= 32 ? 0 : (int)(M.vpc / 32));
    switch (mode) {
      case 0: e = launch(ibp_match_kernel<0>, 256, M, msmem, mwork, s); break;
      case 2: e = launch(ibp_match_kernel<2>, 256, M, msmem, mwork, s); break;
      case 4: e = launch(ibp_match_kernel<4>, 256, M, msmem, mwork, s); break;
      default: e = launch(ibp_match_kernel<3>, 256, M, msmem, mwork, s); break;
    }
    if (e != cudaSuccess) return e;
    OffArgs O{};
    O.pw = pw;
    O.meta = static_cast<const uint8_t*>(d_meta);
    O.n_bytes = n_bytes;
    O.nchunks = nchunks;
    O.ngroups = ngroups;
    O.ntiles = ntiles2;
    O.cb = cb;
    O.grp = grp;
    O.ctrl = ctrl;
    O.states = states;
    e = launch_dependent(ibp_offsets_kernel, (unsigned)ntiles2, kOffNT, 0, s, O);
    if (e != cudaSuccess) return e;
  }
  PipeArgs A{};
  A.meta = static_cast<const uint8_t*>(d_meta);
  A.pw = pw;
  A.src = static_cast<const uint8_t*>(d_x);
  A.dst = static_cast<uint8_t*>(d_out);
  A.dst_cap = out_cap;
  A.n_bytes = n_bytes;
  A.cb = cb;
  A.nchunks = nchunks;
  A.ngroups = ngroups;
  A.ntiles = (ngroups + g.Q - 1) / g.Q;
  A.off_payload = kIbp1Header + round_up(8ull * (ngroups + 1), 128);
  A.out_bytes = d_out_bytes;
  A.ctrl = ctrl;
  fill_shape(A, g);
  const unsigned long long w = A.ntiles;
  const bool dep = ngroups != 0;  // after the offsets kernel
  if (g.nt == 128)
    return g.reg ? launch(ibp_pack_kernel<128, true>, 128, A, g, w, s, dep)
                 : launch(ibp_pack_kernel<128, false>, 128, A, g, w, s, dep);
  if (g.nt == 256)
    return g.reg ? launch(ibp_pack_kernel<256, true>, 256, A, g, w, s, dep)
                 : launch(ibp_pack_kernel<256, false>, 256, A, g, w, s, dep);
  return g.reg ? launch(ibp_pack_kernel<512, true>, 512, A, g, w, s, dep)
               : launch(ibp_pack_kernel<512, false>, 512, A, g, w, s, dep);
}

cudaError_t ibp_pipe_decompress(const void* d_meta, uint32_t cb, const void* d_in,
                                unsigned long long in_bytes, void* d_y, unsigned long long y_cap,
                                void* d_ws, cudaStream_t s) {
  const Geo g = pick(cb, false);
  PipeArgs A{};
  A.meta = static_cast<const uint8_t*>(d_meta);
  A.src = static_cast<const uint8_t*>(d_in);
  A.src_bytes = in_bytes;
  A.dst = static_cast<uint8_t*>(d_y);
  A.dst_cap = y_cap;
  A.cb = cb;
  A.ctrl = static_cast<Ctrl*>(d_ws);
  // the tile count is only known once the header is read on the device: the
  // grid is sized for the largest stream that fits y_cap
  const unsigned long long nch = (y_cap + cb - 1) / cb, ng = (nch + 31) / 32;
  const unsigned long long w = (ng + g.Q - 1) / g.Q;
  fill_shape(A, g);
  if (g.nt == 128)
    return g.reg ? launch(ibp_decode_pipe_kernel<128, true>, 128, A, g, w, s)
                 : launch(ibp_decode_pipe_kernel<128, false>, 128, A, g, w, s);
  if (g.nt == 256)
    return g.reg ? launch(ibp_decode_pipe_kernel<256, true>, 256, A, g, w, s)
                 : launch(ibp_decode_pipe_kernel<256, false>, 256, A, g, w, s);
  return g.reg ? launch(ibp_decode_pipe_kernel<512, true>, 512, A, g, w, s)
               : launch(ibp_decode_pipe_kernel<512, false>, 512, A, g, w, s);
}

}  // namespace lbb
