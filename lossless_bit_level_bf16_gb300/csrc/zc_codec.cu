// zc_codec.cu -- ZipCCL exponent coding of bf16: encode and decode kernels.
//
// [ZipCCL] = "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", 2. Metodologia:
//   B  each bf16 splits into sign+mantissa (kept as one byte) and an 8-bit
//      exponent; an exponent in the segment's 7-entry codebook becomes a 3-bit
//      code 001..111, any other gets 000 and goes, whole, to a separate escape
//      array;
//   C  blocks padded to 128 bytes for full 128-bit coalesced accesses; the
//      3-bit codes kept as three 1-bit planes;
//   D  fixed-size parts first, variable-size parts after.
//
// Stream "ZCC1": header (128 B) | segment table (64 B per segment) |
// per-chunk escape offsets (u64) | static region: one slot of 11*C/8 bytes
// per chunk = [C sign+mantissa bytes][plane 0][plane 1][plane 2] | escape
// bytes.  Every region starts on a 128-byte boundary.
//
// Encode: every warp takes 8192-slot tickets of the chunked slot space from a
// ticket counter and classifies a ticket 1024 slots at a time, 32 consecutive
// slots per lane (so a lane builds whole 32-bit words of each bit plane); it
// writes the slot bytes and plane words with plain stores and stages its
// escape bytes in shared memory.  One decoupled look-back per ticket, resolved
// after the warp's next ticket, gives the ticket's escape offset, and the
// staged bytes are copied out compacted.  The last warp to finish writes the
// header, the segment table and the padding.  Bytes per element: 2 read,
// 11/8 + escapes written.
//
// Decode: every warp decodes whole chunks on its own (512 slots per step, 16
// per lane); the escape offsets come from the stream's table, so warps are
// independent.  Every offset read from the stream is checked before it is
// used as an address; a bad stream sets ZC_ERR_FORMAT and is not written past.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace lbb {
namespace {

struct EncArgs {
  const uint16_t* x;
  uint8_t* out;
  unsigned long long out_cap;
  unsigned long long* out_bytes;
  const ZcSegDev* segs;
  ZcLayout L;
  Ctrl* ctrl;
  unsigned long long* states;  // look-back state per tile
  unsigned long long* bwords;  // look-back word per block of kLbBlock tiles
  StatPartial* parts;          // zc_compress_fit: one statistics partial per chunk
  uint32_t* red_cnt;           // zc_compress_fit: the predictor's block counters, zeroed here
  int x_al16;
};

__device__ __forceinline__ uint32_t sm4(uint32_t w0, uint32_t w1) {
  // sign+mantissa bytes of 4 consecutive bf16 held in w0, w1
  return (prmt(w0, w1, 0x7531) & 0x80808080u) | (prmt(w0, w1, 0x6420) & 0x7F7F7F7Fu);
}

constexpr uint32_t kWTile = kTileLanes;             // slots per warp ticket
constexpr int kEncWarps = kThreads / 32;
constexpr int kMaxLutSlots = kWTile / 1024;          // chunks per ticket at C = 1024
constexpr uint32_t kStages = 2, kAhead = 1;          // input ring: 2 KB steps, copied 1 ahead
constexpr uint32_t kEscCap = 1024;                   // escape bytes a warp stages per ticket

// Warp-level encoder.  A ticket is 8192 slots and belongs to one warp: it
// classifies them 1024 at a time (32 per lane), writes the slot bytes and plane
// words, stages its escape bytes in its own shared-memory window, then runs
// the decoupled look-back for its ticket and copies the escapes to their place.
// Warps never wait for each other inside a block, so one warp's look-back is
// covered by the other warps' loads.
// Dynamic shared memory per warp: the input ring (kStages x 2 KB), one
// 256-word lookup table per chunk of a ticket, kEscCap staged escape bytes.
static_assert(kLbBlock == kZcLbBlock, "the scratch layout and the look-back agree");

// STATS (zc_compress_fit): each lane also sums its finite values and their
// squares per step (four fp32 chains of eight values, in packed fp32x2
// operations, then fp32 (sum, error)
// pairs across steps; a step whose fp32 sums are not finite, or whose squares
// may have underflowed, is summed in fp64), and the warp writes each chunk's
// count and fp64 sums to A.parts when the chunk's last step is done.  The
// lane's rare fp64 sums live in shared memory (s_stdx, s_stdq) and its count
// in 32 bits (a chunk has at most 65536 values), so that both forms of the
// kernel run at three blocks per SM.
template <bool STATS>
__global__ void __launch_bounds__(kThreads, 3) zc_encode_kernel(EncArgs A) {
  extern __shared__ __align__(16) unsigned char dyn[];
  __shared__ int s_lseg[kEncWarps][kMaxLutSlots];
  __shared__ double s_stdx[STATS ? kEncWarps : 1][32], s_stdq[STATS ? kEncWarps : 1][32];
  __shared__ uint32_t s_cs[kEncWarps][kMaxLutSlots];  // escape position where a chunk starts
  // the pending (previous) ticket of each warp: its index, first chunk, escape
  // count, staging window, and its chunks' escape starts (lanes < chunks per ticket)
  __shared__ unsigned long long s_ptile[kEncWarps], s_pcfirst[kEncWarps];
  __shared__ uint32_t s_prun[kEncWarps], s_pbuf[kEncWarps], s_pcs[kEncWarps][kMaxLutSlots];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const ZcLayout& L = A.L;
  const uint32_t C = L.C, log2C = L.log2C;
  // the predictor that follows a fit reads these only once this kernel is done
  if (STATS && A.red_cnt && blockIdx.x == 0)
    for (uint32_t i = (uint32_t)t; i < L.nseg; i += kThreads) A.red_cnt[i] = 0;
  // chunk sizes that are powers of two divide by shifts; the others (any
  // multiple of 1024) by division, once per ticket and per 1024-slot step
  const bool p2 = (C & (C - 1)) == 0;
  const unsigned long long S = L.slot_bytes;
  const unsigned long long lanes_total = L.nchunks * (unsigned long long)C;
  const uint32_t TL = zc_tile_slots(C);        // slots per ticket: whole chunks
  const unsigned long long ntiles = (lanes_total + TL - 1) / TL;
  const uint32_t nct = zc_chunks_per_tile(C);  // chunks per ticket
  const uint32_t raw_dyn = 5u * C / 8u;        // dynamic bytes of a chunk stored raw
  uint8_t* wring = dyn + (size_t)warp * (kStages * 2048u + nct * 1024u + 2 * kEscCap);  // input steps
  uint32_t* wlut = reinterpret_cast<uint32_t*>(wring + kStages * 2048u);
  uint8_t* const wst_base = wring + kStages * 2048u + nct * 1024u;  // two escape staging windows
  uint32_t buf = 0;                 // the window the current ticket stages into
  uint8_t* wst = wst_base;
  // The previous ticket: its escape count is published, its offset is
  // resolved after the next ticket is classified (by then its predecessors
  // have published), so the warp never waits on the look-back with its
  // slots still to write.
  bool p_has = false;
  // a ticket's inclusive prefix (after a timeout: its own count, and nothing
  // for its block, so that no one waits)
  const unsigned lim = wait_limit(A.ctrl);
  const unsigned long long fault1 = A.ctrl->fault_tile1;  // 0 unless a wait-failure test
  auto publish_inc = [&](unsigned long long tl, unsigned long long excl, unsigned long long agg,
                         bool to) {
    if (lane == 0 && tl + 1 != fault1) {
      if (to) {
        set_status(A.ctrl, ZC_ERR_TIMEOUT);
        st_relaxed_u64(A.states + tl, kFlagInc | agg);
      } else {
        lb2_publish_inc(A.states, A.bwords, tl, excl, agg);
      }
    }
  };
  auto resolve = [&]() {
    const unsigned long long p_tile = s_ptile[warp], p_cfirst = s_pcfirst[warp];
    const uint32_t p_run = s_prun[warp], p_buf = s_pbuf[warp];
    bool to = false;
    const unsigned long long excl = lb2_lookback<4>(A.states, A.bwords, p_tile, &to, lim);
    publish_inc(p_tile, excl, p_run, to);
    const unsigned long long dst = L.off_esc + excl;
    const uint8_t* pst = wst_base + p_buf * kEscCap;
    if (dst + p_run > A.out_cap) {
      if (lane == 0) set_status(A.ctrl, ZC_ERR_CAPACITY);
    } else {
      for (uint32_t i = lane; i < p_run; i += 32) A.out[dst + i] = pst[i];
    }
    if (lane < (int)nct) {
      const unsigned long long c = p_cfirst + lane;
      if (c < L.nchunks) reinterpret_cast<unsigned long long*>(A.out + L.off_escoff)[c] = excl + s_pcs[warp][lane];
    }
    __syncwarp();
    p_has = false;
  };
  if (lane < kMaxLutSlots) s_lseg[warp][lane] = -1;
  // ring offsets of this lane: it copies pieces lane + 32j, reads pieces 4*lane + k
  uint32_t cp_dst[4], rd_src[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t q = (uint32_t)lane + 32u * j, r = 4u * lane + j;
    cp_dst[j] = 16u * (q ^ ((q >> 3) & 3u));
    rd_src[j] = 16u * (r ^ ((r >> 3) & 3u));
  }
  __syncwarp();
  int my_seg = -1;  // segment cache of lanes < nct
  unsigned long long my_c0 = 0, my_c1 = 0;
  // statistics of the chunk being classified (STATS only)
  float st_hx = 0.f, st_lx = 0.f, st_hq = 0.f, st_lq = 0.f;
  uint32_t st_cnt = 0;  // values of the chunk summed so far (a chunk has at most 65536)
  if constexpr (STATS) {
    s_stdx[warp][lane] = 0.0;
    s_stdq[warp][lane] = 0.0;
  }

  // A ticket is taken only when the warp is ready to work on it: taking the
  // next one early delays its published escape count, which other warps'
  // look-backs wait for (measured slower).
  for (;;) {
    unsigned long long tile = 0;
    if (lane == 0) tile = atomicAdd(&A.ctrl->ticket, 1ull);
    tile = __shfl_sync(kFull, tile, 0);
    if (tile >= ntiles) {
      if (p_has) resolve();
      break;
    }
    const unsigned long long tlane0 = tile * TL;
    const unsigned long long cfirst = tile * nct;  // tickets start at chunk starts
    // chunk information, held by lane k for the ticket's chunk k
    unsigned long long ce0 = 0;
    uint32_t cval = 0;
    int cal = 0, cseg = -1;
    if (lane < (int)nct) {
      const unsigned long long c = cfirst + lane;
      if (c < L.nchunks) {
        if (my_seg < 0 || c < my_c0 || c >= my_c1) {
          my_seg = (int)__ldg(zc_chunk_seg(A.segs, L.nseg) + c);  // the plan's chunk index
          my_c0 = A.segs[my_seg].chunk_start;
          my_c1 = my_c0 + A.segs[my_seg].nchunks;
        }
        const ZcSegDev& r = A.segs[my_seg];
        ce0 = r.elem_start + (c - r.chunk_start) * (unsigned long long)C;
        const unsigned long long end = r.elem_start + r.nelem;
        cval = (uint32_t)((end - ce0) < C ? (end - ce0) : C);
        cal = A.x_al16 && ((r.elem_start & 7ull) == 0);
        cseg = my_seg;
      }
    }
    const unsigned long long t_e0 = __shfl_sync(kFull, ce0, 0);
    const uint32_t t_val = __shfl_sync(kFull, cval, 0);
    const bool t_al = __shfl_sync(kFull, cal, 0) != 0;

    // ---- steps of 1024 slots, 32 consecutive slots per lane: a lane builds whole
    // 32-bit plane words; a step lies inside one chunk (C is a multiple of 1024)
    uint32_t run = 0, cs_pos = 0;  // escapes staged so far; chunk-start position (lane k)
    const uint32_t steps =
        (uint32_t)((lanes_total - tlane0) < TL ? (lanes_total - tlane0) : TL) / 1024u;
    // Step input: a full, 16-byte aligned step is copied into the warp's ring
    // with coalesced cp.async pieces (lane l copies 16-byte pieces l, l+32,
    // l+64, l+96), kAhead steps before it is used; each lane then reads its own
    // 64 contiguous bytes.  Piece q sits at q ^ ((q >> 3) & 3) so those reads
    // are free of bank conflicts.  Other steps use plain per-lane loads.
    // With C >= 4096 the whole ticket lies in one chunk and the step's chunk
    // data need no shuffles.
    const bool one = nct == 1;
    // chunk (within the ticket) and slot (within the chunk) of step st's first slot
    auto where = [&](uint32_t st, uint32_t& s0) -> int {
      const uint32_t q = st * 1024u;
      const uint32_t k = p2 ? (q >> log2C) : q / C;
      s0 = q - k * C;
      return (int)k;
    };
    auto info = [&](uint32_t st, int& lct, unsigned long long& e0, uint32_t& vch, bool& al) {
      if (one) {
        lct = 0;
        e0 = t_e0;
        vch = t_val;
        al = t_al;
      } else {
        uint32_t s0_;
        lct = where(st, s0_);
        e0 = __shfl_sync(kFull, ce0, lct);
        vch = __shfl_sync(kFull, cval, lct);
        al = __shfl_sync(kFull, cal, lct) != 0;
      }
    };
    auto issue = [&](uint32_t st) {
      if (st < steps) {
        int l_;
        unsigned long long e_;
        uint32_t v_;
        bool a_;
        info(st, l_, e_, v_, a_);
        uint32_t s0;
        where(st, s0);
        if (a_ && v_ >= s0 + 1024u) {
          uint8_t* slotbuf = wring + (st % kStages) * 2048u;
          const uint16_t* src = A.x + e_ + s0;
#pragma unroll
          for (int j = 0; j < 4; ++j) cp_async16(slotbuf + cp_dst[j], src + 8u * lane + 256u * j);
        }
      }
      cp_async_commit();
    };
    auto lane_load = [&](const uint16_t* src, int valid, uint32_t(&w)[16]) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t lo = (2 * j < valid) ? (uint32_t)__ldg(src + 2 * j) : 0u;
        const uint32_t hi = (2 * j + 1 < valid) ? (uint32_t)__ldg(src + 2 * j + 1) : 0u;
        w[j] = lo | (hi << 16);
      }
    };
    // byte k of acc[q] = plane k bits of slots 8q..8q+7 (k = 3: escapes); the
    // entries' bits never overlap, so shifting and adding (one LEA) is an OR
    auto classify = [&](const uint32_t(&w)[16], const uint32_t* Lt, int valid, uint32_t(&acc)[4]) {
      const char* Lb = reinterpret_cast<const char*>(Lt);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t a = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t x = w[4 * q + j];
          a += *reinterpret_cast<const uint32_t*>(Lb + ((x >> 5) & 0x3FCu)) << (2 * j);
          a += *reinterpret_cast<const uint32_t*>(Lb + ((x >> 21) & 0x3FCu)) << (2 * j + 1);
        }
        if (valid < 32) {  // slots past the segment end: code 0, no escape
          const int vq = valid - 8 * q;
          const uint32_t m = vq >= 8 ? 0xFFu : (vq <= 0 ? 0u : ((1u << vq) - 1u));
          a &= m * 0x01010101u;
        }
        acc[q] = a;
      }
    };
    auto warp_excl = [&](uint32_t ne, uint32_t& total) {
      uint32_t inc = ne;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += v;
      }
      total = __shfl_sync(kFull, inc, 31);
      return inc - ne;
    };
    // escaped exponent fields, in slot order, from the lane's 16 words
    // (the stash is the step's ring slot, free once every lane has read it)
    // (each lane's 64 bytes go to the slot as four 16-byte pieces, piece j at
    // 4 * lane + (j ^ ((lane >> 1) & 3)), so each store instruction of the warp
    // spreads over all eight 16-byte bank groups)
    auto put_escapes = [&](const uint32_t(&w)[16], uint32_t esc, uint32_t pos, uint8_t* dst,
                           uint32_t cap, uint8_t* slotbuf) {
      __syncwarp();
      uint4* st4 = reinterpret_cast<uint4*>(slotbuf);
      const uint32_t sw = ((uint32_t)lane >> 1) & 3u, b4 = 4u * lane;
      st4[b4 + (0u ^ sw)] = make_uint4(w[0], w[1], w[2], w[3]);
      st4[b4 + (1u ^ sw)] = make_uint4(w[4], w[5], w[6], w[7]);
      st4[b4 + (2u ^ sw)] = make_uint4(w[8], w[9], w[10], w[11]);
      st4[b4 + (3u ^ sw)] = make_uint4(w[12], w[13], w[14], w[15]);
      // value i of the lane sits at half-word 32 * lane + (i ^ 8 * sw): its
      // 16-byte piece i >> 3 was stored at piece (i >> 3) ^ sw
      const uint16_t* h = reinterpret_cast<const uint16_t*>(slotbuf) + 32u * lane;
      const uint32_t sw8 = sw << 3;
      while (esc) {
        const uint32_t i = (uint32_t)__ffs(esc) - 1u;
        esc &= esc - 1;
        const uint32_t hv = h[i ^ sw8];
        if (pos < cap) dst[pos] = (uint8_t)((hv >> 7) & 0xFFu);
        ++pos;
      }
    };

#pragma unroll
    for (uint32_t k = 0; k < kAhead; ++k) issue(k);
    // lookup tables of the ticket's chunks (rebuilt only when the segment
    // changes), copied while the first step's input is on its way
    for (uint32_t k = 0; k < nct; ++k) {
      const int sg = __shfl_sync(kFull, cseg, (int)k);
      if (sg >= 0 && s_lseg[warp][k] != sg) {
        // the segment's table, kept by the plan
        const uint32_t* src = zc_seg_luts(A.segs, L.nseg) + 256u * (uint32_t)sg;
        for (uint32_t e = lane; e < 256u; e += 32u) wlut[k * 256u + e] = __ldg(src + e);
        __syncwarp();
        if (lane == 0) s_lseg[warp][k] = sg;
      }
    }
    __syncwarp();
    for (uint32_t st = 0; st < steps; ++st) {
      issue(st + kAhead);
      int lct;
      unsigned long long e0;
      uint32_t vch;
      bool al;
      info(st, lct, e0, vch, al);
      uint32_t s0;
      where(st, s0);
      const uint32_t i0 = s0 + 32u * lane;
      const int valid = vch > i0 ? ((vch - i0) < 32u ? (int)(vch - i0) : 32) : 0;
      uint32_t w[16];
      if (al && vch >= s0 + 1024u) {  // the ring holds this step
        cp_async_wait_group<kAhead>();
        __syncwarp();
        const uint8_t* slotbuf = wring + (st % kStages) * 2048u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = *reinterpret_cast<const uint4*>(slotbuf + rd_src[k]);
          w[4 * k] = v.x;
          w[4 * k + 1] = v.y;
          w[4 * k + 2] = v.z;
          w[4 * k + 3] = v.w;
        }
        __syncwarp();  // every lane has its bytes before the slot is refilled
      } else {  // unaligned segment or a ragged end; padding slots read as 0
        lane_load(A.x + e0 + i0, valid, w);
      }
      const unsigned long long c = cfirst + lct;
      if constexpr (STATS) {
        // four fp32 chains of eight values: the low and the high value of the
        // even and of the odd words, two chains per packed fp32x2 operation
        unsigned long long s1[2] = {0ull, 0ull}, s2[2] = {0ull, 0ull};
#pragma unroll
        for (int j = 0; j < 16; ++j) {  // padding slots hold 0
          const unsigned long long v = f2_pack(bf16_lo(w[j]), bf16_hi(w[j]));
          s1[j & 1] = f2_add(s1[j & 1], v);
          s2[j & 1] = f2_fma(v, v, s2[j & 1]);
        }
        const float2 a0 = f2_unpack(s1[0]), a1 = f2_unpack(s1[1]);
        const float2 q0 = f2_unpack(s2[0]), q1 = f2_unpack(s2[1]);
        const float t1 = __fadd_rn(__fadd_rn(a0.x, a0.y), __fadd_rn(a1.x, a1.y));
        const float t2 = __fadd_rn(__fadd_rn(q0.x, q0.y), __fadd_rn(q1.x, q1.y));
        bool fast = isfinite(t1) && isfinite(t2);
        if (fast && t2 < 0x1p-96f) {  // squares may have lost bits: only if a value is not 0
          uint32_t nz = 0;
#pragma unroll
          for (int j = 0; j < 16; ++j) nz |= w[j] & 0x7FFF7FFFu;
          fast = nz == 0;
        }
        if (fast) {
          two_sum_acc(st_hx, st_lx, t1);
          two_sum_acc(st_hq, st_lq, t2);
          st_cnt += (uint32_t)valid;
        } else {  // an inf/NaN value, an fp32 overflow or underflow: fp64, finite values only
          // (rare: the lane's values are read again, one at a time)
          const uint16_t* xs = A.x + e0 + s0 + 32u * lane;
#pragma unroll 1
          for (int j = 0; j < valid; ++j) {
            const uint32_t bits = xs[j];
            if (((bits >> 7) & 0xFFu) != 0xFFu) {
              const double d = (double)__uint_as_float(bits << 16);
              s_stdx[warp][lane] = __dadd_rn(s_stdx[warp][lane], d);
              s_stdq[warp][lane] = __dadd_rn(s_stdq[warp][lane], __dmul_rn(d, d));
              st_cnt += 1;
            }
          }
        }
        if (s0 + 1024u == C || st + 1 == steps) {  // the chunk's last step (warp-uniform)
          float ax = st_hx, bx = st_lx, aq = st_hq, bq = st_lq;
          unsigned long long n = st_cnt;
          const double st_dx = s_stdx[warp][lane], st_dq = s_stdq[warp][lane];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ax2 = __shfl_down_sync(kFull, ax, o), bx2 = __shfl_down_sync(kFull, bx, o);
            const float aq2 = __shfl_down_sync(kFull, aq, o), bq2 = __shfl_down_sync(kFull, bq, o);
            pair_add(ax, bx, ax2, bx2);
            pair_add(aq, bq, aq2, bq2);
            n += __shfl_down_sync(kFull, n, o);
          }
          const bool fin =
              __shfl_sync(kFull, isfinite(ax) && isfinite(bx) && isfinite(aq) && isfinite(bq), 0);
          double r1, r2;
          if (!fin || __any_sync(kFull, st_dx != 0.0 || st_dq != 0.0)) {
            r1 = __dadd_rn(__dadd_rn((double)st_hx, (double)st_lx), st_dx);
            r2 = __dadd_rn(__dadd_rn((double)st_hq, (double)st_lq), st_dq);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              r1 = __dadd_rn(r1, __shfl_down_sync(kFull, r1, o));
              r2 = __dadd_rn(r2, __shfl_down_sync(kFull, r2, o));
            }
          } else {
            r1 = __dadd_rn((double)ax, (double)bx);
            r2 = __dadd_rn((double)aq, (double)bq);
          }
          if (lane == 0) A.parts[c] = StatPartial{n, r1, r2};
          st_hx = st_lx = st_hq = st_lq = 0.f;
          s_stdx[warp][lane] = 0.0;
          s_stdq[warp][lane] = 0.0;
          st_cnt = 0;
        }
      }
      uint32_t acc[4];
      classify(w, wlut + (uint32_t)lct * 256u, valid, acc);
      uint8_t* slot = A.out + L.off_static + c * S;
      uint4 s0v, s1v;
      s0v.x = sm4(w[0], w[1]);
      s0v.y = sm4(w[2], w[3]);
      s0v.z = sm4(w[4], w[5]);
      s0v.w = sm4(w[6], w[7]);
      s1v.x = sm4(w[8], w[9]);
      s1v.y = sm4(w[10], w[11]);
      s1v.z = sm4(w[12], w[13]);
      s1v.w = sm4(w[14], w[15]);
      st_v4(slot + i0, s0v);
      st_v4(slot + i0 + 16, s1v);
      const uint32_t tA = prmt(acc[0], acc[1], 0x5140), tB = prmt(acc[2], acc[3], 0x5140);
      const uint32_t tC = prmt(acc[0], acc[1], 0x7362), tD = prmt(acc[2], acc[3], 0x7362);
      uint32_t* pw = reinterpret_cast<uint32_t*>(slot + C + (i0 >> 3));
      const uint32_t pwords = C >> 5;
      pw[0] = prmt(tA, tB, 0x5410);
      pw[pwords] = prmt(tA, tB, 0x7632);
      pw[2 * pwords] = prmt(tC, tD, 0x5410);
      const uint32_t esc = prmt(tC, tD, 0x7632);
      uint32_t tot;
      const uint32_t pos0 = run + warp_excl((uint32_t)__popc(esc), tot);
      if (s0 == 0 && lane == 0) s_cs[warp][lct] = pos0;  // a chunk starts at this step
      if (__any_sync(kFull, esc != 0 && pos0 < kEscCap))
      {
        put_escapes(w, (esc != 0 && pos0 < kEscCap) ? esc : 0u, pos0, wst, kEscCap,
                    wring + (st % kStages) * 2048u);
        __syncwarp();  // the stash is read before the next copy lands in the ring
      }
      run += tot;
    }
    __syncwarp();
    // Chunk `lane` of the ticket: its escapes (to the next chunk's start or
    // the ticket's end), whether it is stored raw (a full chunk with more
    // escapes than the 5C/8 bytes its raw form puts past the slot), its
    // dynamic bytes and their place within the ticket's.
    if (lane < (int)nct) cs_pos = s_cs[warp][lane];
    const uint32_t nxt = __shfl_down_sync(kFull, cs_pos, 1);
    const bool have_c = lane < (int)nct && cfirst + lane < L.nchunks;
    const bool have_n = lane + 1 < (int)nct && cfirst + lane + 1 < L.nchunks;
    const uint32_t cesc = have_c ? (have_n ? nxt : run) - cs_pos : 0u;
    const bool craw = have_c && cval == C && cesc > raw_dyn;
    uint32_t dtot;
    const uint32_t dpos = warp_excl(craw ? raw_dyn : cesc, dtot);
    const bool any_raw = __any_sync(kFull, craw);

    if (!any_raw && run <= kEscCap) {
      // publish this ticket's escape count now, resolve the previous ticket,
      // and keep this one pending in its window
      if (lane == 0 && tile + 1 != fault1) lb2_publish_agg(A.states, A.bwords, tile, run);
      if (p_has) resolve();
      p_has = true;
      if (lane == 0) {
        s_ptile[warp] = tile;
        s_pcfirst[warp] = cfirst;
        s_prun[warp] = run;
        s_pbuf[warp] = buf;
      }
      if (lane < kMaxLutSlots) s_pcs[warp][lane] = cs_pos;
      __syncwarp();
      buf ^= 1u;
      wst = wst_base + buf * kEscCap;
      continue;
    }
    if (p_has) resolve();
    // ---- more escapes than a window holds, or a chunk stored raw: the
    // look-back now, then the ticket is read again and its dynamic bytes
    // (escapes, or a raw chunk's last 5C/8 bytes) written straight out
    bool to = false;
    if (lane == 0 && tile + 1 != fault1) lb2_publish_agg(A.states, A.bwords, tile, dtot);
    __syncwarp();  // also orders the slot stores above before the raw chunks' below
    const unsigned long long excl = lb2_lookback<4>(A.states, A.bwords, tile, &to, lim);
    publish_inc(tile, excl, dtot, to);
    const unsigned long long dst = L.off_esc + excl;
    if (dst + dtot > A.out_cap) {
      if (lane == 0) set_status(A.ctrl, ZC_ERR_CAPACITY);
    } else {
      uint32_t r2 = 0;  // dynamic position within the ticket
      for (uint32_t st = 0; st < steps; ++st) {
        int lct;
        unsigned long long e0;
        uint32_t vch;
        bool al;
        info(st, lct, e0, vch, al);
        uint32_t s0;
        where(st, s0);
        const bool raw_c = __shfl_sync(kFull, craw, lct);
        const uint32_t pos_c = __shfl_sync(kFull, dpos, lct);
        if (s0 == 0) r2 = pos_c;
        const uint32_t i0 = s0 + 32u * lane;
        const int valid = vch > i0 ? ((vch - i0) < 32u ? (int)(vch - i0) : 32) : 0;
        uint32_t w[16];
        lane_load(A.x + e0 + i0, valid, w);
        if (raw_c) {
          // the lane's 32 values are raw bytes 2*i0 .. 2*i0+63 of the chunk,
          // wholly in the slot or wholly past it (S is a multiple of 64)
          const uint32_t b = 2u * i0;
          if (b < S) {
            uint8_t* sp = A.out + L.off_static + (cfirst + lct) * S + b;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              st_v4(sp + 16 * k, make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]));
          } else {
            uint8_t* dp = A.out + dst + pos_c + (b - (uint32_t)S);
#pragma unroll
            for (int k = 0; k < 64; ++k) dp[k] = (uint8_t)(w[k >> 2] >> (8 * (k & 3)));
          }
          continue;  // warp-uniform
        }
        uint32_t acc[4];
        classify(w, wlut + (uint32_t)lct * 256u, valid, acc);
        const uint32_t esc = prmt(prmt(acc[0], acc[1], 0x7362), prmt(acc[2], acc[3], 0x7362), 0x7632);
        uint32_t tot;
        const uint32_t pos = r2 + warp_excl((uint32_t)__popc(esc), tot);
        put_escapes(w, esc, pos, A.out + dst, 0xFFFFFFFFu, wring);
        __syncwarp();
        r2 += tot;
      }
    }
    if (have_c)
      reinterpret_cast<unsigned long long*>(A.out + L.off_escoff)[cfirst + lane] =
          (excl + dpos) | (craw ? kZcRawFlag : 0ull);
    __syncwarp();  // the window is reused by the next ticket
  }

  // ---- the last warp to finish writes the header, tables and padding
  unsigned last = 0;
  if (lane == 0) {
    __threadfence();
    const unsigned long long d = atomicAdd(&A.ctrl->done, 1ull);
    last = (d == (unsigned long long)gridDim.x * kEncWarps - 1) ? 1u : 0u;
  }
  if (!__shfl_sync(kFull, last, 0)) return;
  __threadfence();
  unsigned long long esc_total = 0;
  if (ntiles) esc_total = ld_acquire_u64(A.states + ntiles - 1) & kValMask;
  const unsigned long long total = L.off_esc + round_up_dev(esc_total, kZcAlign);
  unsigned long long* escoff = reinterpret_cast<unsigned long long*>(A.out + L.off_escoff);
  if (lane == 0) {
    escoff[L.nchunks] = esc_total;
    if (total > A.out_cap) set_status(A.ctrl, ZC_ERR_CAPACITY);
    if (A.out_bytes) *A.out_bytes = total;
  }
  // zero padding: escape tail, segment-table tail, offset-table tail
  const unsigned long long pad_end = total < A.out_cap ? total : A.out_cap;
  for (unsigned long long p = L.off_esc + esc_total + lane; p < pad_end; p += 32) A.out[p] = 0;
  for (unsigned long long p = L.off_seg + (unsigned long long)kZcSegRec * L.nseg + lane;
       p < L.off_escoff; p += 32)
    A.out[p] = 0;
  for (unsigned long long p = L.off_escoff + 8ull * (L.nchunks + 1) + lane; p < L.off_static;
       p += 32)
    A.out[p] = 0;
  __syncwarp();
  for (uint32_t s = lane; s < L.nseg; s += 32) {
    const ZcSegDev& r = A.segs[s];
    const volatile unsigned long long* ve = escoff;
    const unsigned long long es = ve[r.chunk_start] & ~kZcRawFlag;
    const unsigned long long ee = ve[r.chunk_start + r.nchunks] & ~kZcRawFlag;
    unsigned long long* rec =
        reinterpret_cast<unsigned long long*>(A.out + L.off_seg + (unsigned long long)kZcSegRec * s);
    unsigned long long bk = 0;
#pragma unroll
    for (int j = 0; j < 7; ++j) bk |= (unsigned long long)r.book[j] << (8 * j);
    rec[0] = r.elem_start;
    rec[1] = r.nelem;
    rec[2] = r.chunk_start;
    rec[3] = r.nchunks;
    rec[4] = es;
    rec[5] = ee - es;
    rec[6] = bk;
    rec[7] = 0;
  }
  if (lane < 16) {
    unsigned long long h = 0;
    switch (lane) {
      case 0: h = (unsigned long long)kZcMagic | (1ull << 32) | ((unsigned long long)kZcHeader << 48); break;
      case 1: h = (unsigned long long)C | ((unsigned long long)L.nseg << 32); break;
      case 2: h = L.n; break;
      case 3: h = L.nchunks; break;
      case 4: h = esc_total; break;
      case 5: h = L.off_seg; break;
      case 6: h = L.off_escoff; break;
      case 7: h = L.off_static; break;
      case 8: h = L.off_esc; break;
      case 9: h = total; break;
      default: h = 0; break;
    }
    reinterpret_cast<unsigned long long*>(A.out)[lane] = h;
  }
}

// ------------------------------------------------------------------ decode

struct DecHdr {
  unsigned long long n, nchunks, esc_total, off_seg, off_escoff, off_static, off_esc, total;
  uint32_t C, log2C, nseg;
};

__device__ __forceinline__ unsigned long long rd_u64(const uint8_t* p) {
  return *reinterpret_cast<const unsigned long long*>(p);
}

// Validates the header against in_bytes and y_cap; false on any mismatch.
__device__ bool parse_header(const uint8_t* in, unsigned long long in_bytes,
                             unsigned long long y_cap, DecHdr& h, int& err) {
  err = ZC_ERR_FORMAT;
  if (in_bytes < kZcHeader) return false;
  const unsigned long long w0 = rd_u64(in), w1 = rd_u64(in + 8);
  if ((uint32_t)w0 != kZcMagic || ((w0 >> 32) & 0xFFFFu) != 1u || (w0 >> 48) != kZcHeader)
    return false;
  h.C = (uint32_t)w1;
  h.nseg = (uint32_t)(w1 >> 32);
  h.n = rd_u64(in + 16);
  h.nchunks = rd_u64(in + 24);
  h.esc_total = rd_u64(in + 32);
  h.off_seg = rd_u64(in + 40);
  h.off_escoff = rd_u64(in + 48);
  h.off_static = rd_u64(in + 56);
  h.off_esc = rd_u64(in + 64);
  h.total = rd_u64(in + 72);
  if (h.C < 1024u || h.C > 65536u || (h.C % 1024u) != 0 || h.nseg == 0) return false;
  h.log2C = 31 - __clz(h.C);  // used only when C is a power of two
  if (h.total > in_bytes) return false;
  const unsigned long long S = (unsigned long long)h.C * 11ull / 8ull;
  if (h.off_seg != kZcHeader) return false;
  if (h.nseg > h.total / kZcSegRec) return false;
  if (h.off_escoff != h.off_seg + round_up_dev((unsigned long long)kZcSegRec * h.nseg, kZcAlign))
    return false;
  if (h.nchunks > h.total / 8ull) return false;
  if (h.off_static != h.off_escoff + round_up_dev(8ull * (h.nchunks + 1), kZcAlign)) return false;
  if (h.nchunks > h.total / S) return false;
  if (h.off_esc != h.off_static + h.nchunks * S) return false;
  if (h.off_esc > h.total || h.esc_total > h.total - h.off_esc) return false;
  if (h.total != h.off_esc + round_up_dev(h.esc_total, kZcAlign)) return false;
  if (h.n > h.nchunks * (unsigned long long)h.C) return false;
  if (h.n > y_cap) {
    err = ZC_ERR_CAPACITY;
    return false;
  }
  return true;
}

// Segment record s of the stream, checked for consistency with the header and
// with record s-1; false if anything is off.
struct SegRec {
  unsigned long long elem_start, nelem, chunk_start, nchunks;
  uint32_t R0, R1;  // book bytes for the byte-permute lookup (code 0 -> 0)
};

__device__ bool load_seg(const uint8_t* in, const DecHdr& h, uint32_t s, SegRec& r) {
  const uint8_t* p = in + h.off_seg + (unsigned long long)kZcSegRec * s;
  r.elem_start = rd_u64(p);
  r.nelem = rd_u64(p + 8);
  r.chunk_start = rd_u64(p + 16);
  r.nchunks = rd_u64(p + 24);
  const unsigned long long bk = rd_u64(p + 48);
  r.R0 = (uint32_t)(bk << 8);
  r.R1 = (uint32_t)(bk >> 24);
  if (r.nelem > h.n || r.elem_start > h.n - r.nelem) return false;
  if (r.nchunks > h.nchunks || r.chunk_start > h.nchunks - r.nchunks) return false;
  if (r.nchunks != (r.nelem + h.C - 1) / h.C) return false;
  if (s == 0) return r.elem_start == 0 && r.chunk_start == 0;
  const uint8_t* q = p - kZcSegRec;
  return rd_u64(q) + rd_u64(q + 8) == r.elem_start && rd_u64(q + 16) + rd_u64(q + 24) == r.chunk_start;
}

// Two bf16 from (sign+mantissa byte, exponent byte) pairs: selP takes each
// sign+mantissa byte twice, the second time with its sign replicated over
// the byte (selector bit 3), so that masking leaves the sign at bit 15 and
// the mantissa at bits 0..6; selQ puts each exponent byte at bits 8..15 of
// its half (zeros from the second operand elsewhere), one shift down.
__device__ __forceinline__ uint32_t out_word(uint32_t S, uint32_t E, uint32_t selP, uint32_t selQ) {
  return (prmt_sx(S, E, selP) & 0x807F807Fu) | (prmt(E, 0u, selQ) >> 1);
}

constexpr uint32_t kWarpEscBytes = 512;  // escape bytes a warp stages per chunk
constexpr int kDecWarps = kThreads / 32;

// Segment record of chunk c, found by interpolation (segments of equal size
// need no search) and checked against the header and the record before it.
__device__ bool find_seg_checked(const uint8_t* in, const DecHdr& h, unsigned long long c,
                                 SegRec& r) {
  uint32_t g = (uint32_t)(((double)c * (double)h.nseg) / (double)h.nchunks);
  if (g >= h.nseg) g = h.nseg - 1;
  const unsigned long long cs = rd_u64(in + h.off_seg + (unsigned long long)kZcSegRec * g + 16);
  const unsigned long long cn = rd_u64(in + h.off_seg + (unsigned long long)kZcSegRec * g + 24);
  if (!(c >= cs && c - cs < cn)) {
    int lo = 0, hi = (int)h.nseg - 1;  // largest s with chunk_start <= c
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rd_u64(in + h.off_seg + (unsigned long long)kZcSegRec * mid + 16) <= c) lo = mid;
      else hi = mid - 1;
    }
    g = (uint32_t)lo;
  }
  if (!load_seg(in, h, g, r)) return false;
  return c >= r.chunk_start && c < r.chunk_start + r.nchunks;
}

// Each warp decodes a contiguous range of whole chunks on its own, 512 slots
// (16 per lane) per step, carrying the chunk's escape count from step to
// step; no block
// barrier after the header is read.  The chunk's escape bytes are staged in
// the warp's shared-memory window when they fit (one 16-byte load per lane).
__global__ void __launch_bounds__(kThreads, 3) zc_decode_kernel(
    const uint8_t* __restrict__ in, unsigned long long in_bytes, uint16_t* __restrict__ y,
    unsigned long long y_cap, Ctrl* ctrl, int y_al16) {
  __shared__ uint32_t s_nib[256];
  __shared__ __align__(16) uint8_t s_esc[kDecWarps][kWarpEscBytes + 16];
  __shared__ __align__(16) uint8_t s_ex[kDecWarps][32 * 16];  // a lane's 16 exponent bytes
  __shared__ DecHdr s_h;
  __shared__ int s_ok;

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) {
    int err;
    s_ok = parse_header(in, in_bytes, y_cap, s_h, err);
    if (!s_ok) set_status(ctrl, err);
  }
  {
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) v |= ((t >> i) & 1u) << (4 * i);
    s_nib[t] = v;  // bit i of a plane byte -> nibble i
  }
  __syncthreads();
  if (!s_ok) return;
  const DecHdr h = s_h;
  const uint32_t C = h.C;
  const unsigned long long S = (unsigned long long)C * 11ull / 8ull;
  const uint8_t* escoff = in + h.off_escoff;
  const uint8_t* esc_base = in + h.off_esc;

  // whole-table checks, once (block 0): segment chain and offset-table ends
  if (blockIdx.x == 0) {
    for (uint32_t s = t; s < h.nseg; s += kThreads) {
      SegRec r;
      if (!load_seg(in, h, s, r)) set_status(ctrl, ZC_ERR_FORMAT);
      if (s + 1 == h.nseg && (r.elem_start + r.nelem != h.n || r.chunk_start + r.nchunks != h.nchunks))
        set_status(ctrl, ZC_ERR_FORMAT);
    }
    if (t == 0 && ((rd_u64(escoff) & ~kZcRawFlag) != 0 ||
                   rd_u64(escoff + 8 * h.nchunks) != h.esc_total))
      set_status(ctrl, ZC_ERR_FORMAT);
  }

  const unsigned long long nwarps = (unsigned long long)gridDim.x * kDecWarps;
  const uint32_t steps = C / 512u;
  uint8_t* wesc = s_esc[warp];
  // The checked record of the last segment used (chunks of one segment take
  // it without reading the table again) and the next chunk's escape offsets,
  // read one chunk ahead.
  // Warp w takes a contiguous range of chunks, as many (to one) as every
  // other warp, so consecutive chunks mostly share a segment.
  SegRec r;
  bool have_r = false;
  unsigned long long c, c_end;
  {
    const unsigned long long gw = (unsigned long long)blockIdx.x * kDecWarps + warp;
    const unsigned long long q = h.nchunks / nwarps, rem = h.nchunks % nwarps;
    c = gw * q + (gw < rem ? gw : rem);
    c_end = c + q + (gw < rem ? 1 : 0);
  }
  unsigned long long n_lo = 0, n_hi = 0;
  if (c < c_end) {
    n_lo = rd_u64(escoff + 8 * c);
    n_hi = rd_u64(escoff + 8 * (c + 1));
  }
  for (; c < c_end; ++c) {
    const uint8_t* slot = in + h.off_static + c * S;
    // step 0 data and the chunk's table entries in flight together
    uint4 smv = ld_nc_v4(slot + 16u * lane);
    const uint8_t* pb = slot + C + 2u * lane;
    uint32_t p0 = __ldg(reinterpret_cast<const unsigned short*>(pb));
    uint32_t p1 = __ldg(reinterpret_cast<const unsigned short*>(pb + (C >> 3)));
    uint32_t p2 = __ldg(reinterpret_cast<const unsigned short*>(pb + (C >> 2)));
    const bool craw = (n_lo & kZcRawFlag) != 0;  // the chunk is stored raw
    const unsigned long long elo = n_lo & ~kZcRawFlag, ehi = n_hi & ~kZcRawFlag;
    const unsigned long long cn = c + 1;
    if (cn < c_end) {
      n_lo = rd_u64(escoff + 8 * cn);
      n_hi = rd_u64(escoff + 8 * (cn + 1));
    }
    if (!(have_r && c >= r.chunk_start && c - r.chunk_start < r.nchunks))
      have_r = find_seg_checked(in, h, c, r);
    bool ok = have_r && elo <= ehi && ehi <= h.esc_total;
    if (!ok) {
      if (lane == 0) set_status(ctrl, ZC_ERR_FORMAT);
      continue;  // warp-uniform
    }
    const unsigned long long e0 = r.elem_start + (c - r.chunk_start) * (unsigned long long)h.C;
    const unsigned long long vch_ll = r.elem_start + r.nelem - e0;
    const uint32_t vch = (uint32_t)(vch_ll < C ? vch_ll : C);
    const bool al = y_al16 && ((r.elem_start & 7ull) == 0);
    if (craw) {
      // a full chunk's 2C raw bytes: the slot, then its 5C/8 dynamic bytes
      // (each 16-byte piece lies wholly in one: S is a multiple of 64)
      if (vch != C || ehi - elo != 5ull * C / 8ull) {
        if (lane == 0) set_status(ctrl, ZC_ERR_FORMAT);
        continue;  // warp-uniform
      }
      for (uint32_t b = 16u * lane; b < 2u * C; b += 512u) {
        uint4 v;
        if (b < S) {
          v = ld_nc_v4(slot + b);
        } else {
          const uint8_t* q = esc_base + elo + (b - S);
          uint32_t u[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            u[k] = (uint32_t)q[4 * k] | ((uint32_t)q[4 * k + 1] << 8) |
                   ((uint32_t)q[4 * k + 2] << 16) | ((uint32_t)q[4 * k + 3] << 24);
          v = make_uint4(u[0], u[1], u[2], u[3]);
        }
        const unsigned long long elem = e0 + b / 2;
        if (al) {
          st_v4(y + elem, v);
        } else {
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            y[elem + 2 * k] = (uint16_t)(u[k] & 0xFFFFu);
            y[elem + 2 * k + 1] = (uint16_t)(u[k] >> 16);
          }
        }
      }
      __syncwarp();
      continue;
    }
    const unsigned long long ea = elo & ~15ull;  // staged window starts 16-byte aligned
    const bool staged = ehi - ea <= kWarpEscBytes;
    if (staged && ea + 16ull * lane < ehi)
      *reinterpret_cast<uint4*>(wesc + 16 * lane) = ld_nc_v4(esc_base + ea + 16ull * lane);
    __syncwarp();
    unsigned long long carry = elo;
    for (uint32_t st = 0; st < steps; ++st) {
      const uint32_t i0 = st * 512u + 16u * lane;
      // next step's loads go out before this step is decoded
      uint4 smn = make_uint4(0, 0, 0, 0);
      uint32_t q0 = 0, q1 = 0, q2 = 0;
      if (st + 1 < steps) {
        smn = ld_nc_v4(slot + i0 + 512u);
        const uint8_t* qb = slot + C + ((i0 + 512u) >> 3);
        q0 = __ldg(reinterpret_cast<const unsigned short*>(qb));
        q1 = __ldg(reinterpret_cast<const unsigned short*>(qb + (C >> 3)));
        q2 = __ldg(reinterpret_cast<const unsigned short*>(qb + (C >> 2)));
      }
      const int valid = vch > i0 ? ((vch - i0) < 16u ? (int)(vch - i0) : 16) : 0;
      const uint32_t vmask = valid >= 16 ? 0xFFFFu : ((1u << valid) - 1u);
      const uint32_t esc = ~(p0 | p1 | p2) & vmask;
      const uint32_t ne = (uint32_t)__popc(esc);
      uint32_t inc = ne;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += v;
      }
      const unsigned long long base = carry + inc - ne;
      carry += __shfl_sync(kFull, inc, 31);
      const uint32_t cA = s_nib[p0 & 0xFFu] | (s_nib[p1 & 0xFFu] << 1) | (s_nib[p2 & 0xFFu] << 2);
      const uint32_t cB = s_nib[p0 >> 8] | (s_nib[p1 >> 8] << 1) | (s_nib[p2 >> 8] << 2);
      uint32_t E0 = prmt(r.R0, r.R1, cA), E1 = prmt(r.R0, r.R1, cA >> 16);
      uint32_t E2 = prmt(r.R0, r.R1, cB), E3 = prmt(r.R0, r.R1, cB >> 16);
      if (esc && base + ne <= ehi) {
        // the lane's exponent bytes go through its own 16 bytes of shared
        // memory: each escaped one is one byte store
        uint4* mine = reinterpret_cast<uint4*>(s_ex[warp] + 16 * lane);
        *mine = make_uint4(E0, E1, E2, E3);
        uint8_t* mb = reinterpret_cast<uint8_t*>(mine);
        uint32_t m = esc;
        unsigned long long pos = base;
        while (m) {
          const int i = __ffs(m) - 1;
          m &= m - 1;
          mb[i] = staged ? wesc[pos - ea] : esc_base[pos];
          ++pos;
        }
        const uint4 v = *mine;
        E0 = v.x;
        E1 = v.y;
        E2 = v.z;
        E3 = v.w;
      }
      if (valid) {
        uint32_t o[8];
        o[0] = out_word(smv.x, E0, 0x9180, 0x1404);
        o[1] = out_word(smv.x, E0, 0xB3A2, 0x3424);
        o[2] = out_word(smv.y, E1, 0x9180, 0x1404);
        o[3] = out_word(smv.y, E1, 0xB3A2, 0x3424);
        o[4] = out_word(smv.z, E2, 0x9180, 0x1404);
        o[5] = out_word(smv.z, E2, 0xB3A2, 0x3424);
        o[6] = out_word(smv.w, E3, 0x9180, 0x1404);
        o[7] = out_word(smv.w, E3, 0xB3A2, 0x3424);
        const unsigned long long elem = e0 + i0;
        if (valid == 16 && al) {
          st_v4(y + elem, make_uint4(o[0], o[1], o[2], o[3]));
          st_v4(y + elem + 8, make_uint4(o[4], o[5], o[6], o[7]));
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (2 * j < valid) y[elem + 2 * j] = (uint16_t)(o[j] & 0xFFFFu);
            if (2 * j + 1 < valid) y[elem + 2 * j + 1] = (uint16_t)(o[j] >> 16);
          }
        }
      }
      smv = smn;
      p0 = q0;
      p1 = q1;
      p2 = q2;
    }
    // the escapes counted in the planes must be exactly the table's
    if (lane == 0 && carry != ehi) set_status(ctrl, ZC_ERR_FORMAT);
    __syncwarp();  // window reuse
  }
}

}  // namespace

cudaError_t zc_launch_compress(const ZcLayout& L, const ZcSegDev* d_segs,
                               const uint16_t* d_x, void* d_out,
                               unsigned long long out_cap,
                               unsigned long long* d_out_bytes, void* d_ws,
                               cudaStream_t s, bool fit) {
  Ctrl* ctrl = static_cast<Ctrl*>(d_ws);
  unsigned long long* states =
      reinterpret_cast<unsigned long long*>(static_cast<char*>(d_ws) + kCtrlBytes);
  const unsigned long long tl = zc_tile_slots(L.C);
  const unsigned long long ntiles = (L.nchunks * (unsigned long long)L.C + tl - 1) / tl;
  char* lb = static_cast<char*>(d_ws) + kCtrlBytes;
  cudaError_t e = cudaMemsetAsync(d_ws, 0, kCtrlBytes + zc_enc_scratch_bytes(ntiles), s);
  if (e != cudaSuccess) return e;
  e = arm_wait_fault(d_ws, s);
  if (e != cudaSuccess) return e;
  EncArgs A;
  A.x = d_x;
  A.out = static_cast<uint8_t*>(d_out);
  A.out_cap = out_cap;
  A.out_bytes = d_out_bytes;
  A.segs = d_segs;
  A.L = L;
  A.ctrl = ctrl;
  A.states = states;
  A.bwords = reinterpret_cast<unsigned long long*>(lb + (8 * ntiles + 15) / 16 * 16);
  A.x_al16 = (reinterpret_cast<uintptr_t>(d_x) & 15u) == 0;
  A.parts = fit ? reinterpret_cast<StatPartial*>(static_cast<char*>(d_ws) + zc_fit_parts_offset(ntiles))
                : nullptr;
  A.red_cnt = fit && L.kred_c > 1
                  ? reinterpret_cast<uint32_t*>(static_cast<char*>(d_ws) + zc_cnt_offset(L))
                  : nullptr;
  const uint32_t nct = zc_chunks_per_tile(L.C);
  const size_t smem = (size_t)kEncWarps * (kStages * 2048u + nct * 1024u + 2 * kEscCap);
  auto k = fit ? zc_encode_kernel<true> : zc_encode_kernel<false>;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  const int res = resident_blocks((const void*)k, kThreads, smem);
  const unsigned long long need = (ntiles + kEncWarps - 1) / kEncWarps;
  unsigned long long grid = need < (unsigned long long)res ? need : (unsigned long long)res;
  if (grid == 0) grid = 1;
  k<<<(unsigned)grid, kThreads, smem, s>>>(A);
  e = cudaGetLastError();
  if (e != cudaSuccess || !fit) return e;
  // every chunk's partial is written before the predictor reads them
  return zc_launch_predict_chunks(L, const_cast<ZcSegDev*>(d_segs), A.parts, d_ws, s);
}

cudaError_t zc_launch_decompress(const void* d_in, unsigned long long in_bytes,
                                 uint16_t* d_y, unsigned long long y_cap,
                                 void* d_ws, cudaStream_t s) {
  Ctrl* ctrl = static_cast<Ctrl*>(d_ws);
  cudaError_t e = cudaMemsetAsync(d_ws, 0, kCtrlBytes, s);
  if (e != cudaSuccess) return e;
  const int res = resident_blocks((const void*)zc_decode_kernel, kThreads, 0);
  const int y_al = (reinterpret_cast<uintptr_t>(d_y) & 15u) == 0;
  zc_decode_kernel<<<res, kThreads, 0, s>>>(static_cast<const uint8_t*>(d_in), in_bytes, d_y,
                                            y_cap, ctrl, y_al);
  return cudaGetLastError();
}

}  // namespace lbb
