/*
 * oracle.c -- plain, slow, bit-serial CPU oracle for the ZipCCL exponent codec
 * and IBP invariant bit packing.
 *
 * TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
 * CPU-baseline leg call it; the product library never does.  It is written one
 * element and one bit at a time, in the order the page summaries describe the
 * steps, so that it can be checked against them by eye.  Citations use the page
 * titles and sections listed in oracle.h.
 *
 * Floating point: fp64 throughout; built with -ffp-contract=off so the same
 * source gives the same bits on x86-64 and aarch64 hosts.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- helpers */

static void wr16(uint8_t* p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xFF);
  p[1] = (uint8_t)(v >> 8);
}
static void wr32(uint8_t* p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = (uint8_t)((v >> (8 * i)) & 0xFF);
}
static void wr64(uint8_t* p, uint64_t v) {
  for (int i = 0; i < 8; ++i) p[i] = (uint8_t)((v >> (8 * i)) & 0xFF);
}
static uint16_t rd16(const uint8_t* p) {
  return (uint16_t)(p[0] | (p[1] << 8));
}
static uint32_t rd32(const uint8_t* p) {
  uint32_t v = 0;
  for (int i = 3; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}
static uint64_t rd64(const uint8_t* p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}
static uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

static int get_bit(const uint8_t* base, uint64_t pos) {
  return (base[pos >> 3] >> (pos & 7)) & 1;
}
static void set_bit(uint8_t* base, uint64_t pos, int b) {
  if (b)
    base[pos >> 3] = (uint8_t)(base[pos >> 3] | (1u << (pos & 7)));
  else
    base[pos >> 3] = (uint8_t)(base[pos >> 3] & ~(1u << (pos & 7)));
}

/* bf16 bit pattern -> its exact value as a double (a bf16 is the top half of
 * an IEEE binary32). */
static double bf16_value(uint16_t v) {
  uint32_t u = (uint32_t)v << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ============================================================ ZipCCL
 *
 * Stream "ZCC1" (this project's reading of [ZipCCL] 2.B-2.D):
 *   header, 128 bytes:
 *     0 u32 magic 0x3143435A ('Z','C','C','1')   4 u16 version 1
 *     6 u16 header bytes 128                     8 u32 chunk elements C
 *    12 u32 nseg   16 u64 n   24 u64 nchunks   32 u64 escape bytes total
 *    40 u64 off_seg  48 u64 off_escoff  56 u64 off_static  64 u64 off_esc
 *    72 u64 total bytes   80..127 zero
 *   segment table at off_seg (=128): nseg records of 64 bytes
 *     0 elem_start  8 nelem  16 chunk_start  24 nchunks  32 esc_start
 *    40 esc_bytes (all u64)  48 u8 book[7] ascending  55..63 zero
 *     region padded with zeros to a multiple of 128 bytes
 *   chunk escape-offset table at off_escoff: u64 x (nchunks+1), exclusive
 *     prefix of per-chunk dynamic byte counts (bits 62..0); bit 63 of entry c
 *     (c < nchunks) set when chunk c is stored raw; padded to 128 bytes
 *   static region at off_static: one slot of S = 11*C/8 bytes per chunk:
 *     [C sign+mantissa bytes][plane 0: C bits][plane 1][plane 2]
 *     bit i (LSB first within bytes) of plane k is bit k of element i's code
 *   escape (dynamic) region at off_esc: per chunk, in chunk order, the 8-bit
 *     exponent fields of its escaped elements (element order); zero padded to
 *     128 bytes at the end.
 *   Elements past the end of a segment's last chunk: byte 0, code 0, no escape.
 *   Raw fallback: a full chunk (L = C) with more escapes than the 5C/8 bytes
 *     its raw form puts past the slot is stored raw: its 2C bytes (the bf16
 *     values, little-endian) fill the slot first and their last 5C/8 bytes
 *     are the chunk's dynamic part, so no full chunk takes more than 2C
 *     bytes.  A segment's short last chunk is always coded.
 */

#define ZC_MAGIC 0x3143435Au
#define ZC_HDR 128u
#define ZC_SEGREC 64u
#define ZC_ALIGN 128u

void ora_zc_stats(const uint16_t* x, uint64_t n, uint64_t* cnt, double* sum,
                  double* sumsq) {
  uint64_t c = 0;
  double s1 = 0.0, s2 = 0.0;
  for (uint64_t i = 0; i < n; ++i) {
    uint16_t v = x[i];
    unsigned e = (v >> 7) & 0xFFu;
    if (e == 255u) continue; /* inf / NaN carry no statistics */
    double d = bf16_value(v);
    s1 = s1 + d;
    s2 = s2 + d * d;
    c = c + 1;
  }
  *cnt = c;
  *sum = s1;
  *sumsq = s2;
}

void ora_zc_moments(uint64_t cnt, double sum, double sumsq, double* mu,
                    double* sigma) {
  if (cnt == 0) {
    *mu = 0.0;
    *sigma = 0.0;
    return;
  }
  double m = sum / (double)cnt;
  double var = sumsq / (double)cnt - m * m;
  *mu = m;
  *sigma = var > 0.0 ? sqrt(var) : 0.0;
}

/* [ZipCCL] 2.A: the frequent exponents follow from the Gaussian law with the
 * layer's standard deviation.  Mass of field f = probability that |X| lies in
 * the binade [2^(f-127), 2^(f-126)), X ~ N(mu, sigma), both signs. */
double ora_zc_mass(double mu, double sigma, int f) {
  double a = ldexp(1.0, f - 127);
  double b = ldexp(1.0, f - 126);
  double s = sigma * 1.4142135623730951; /* sigma * sqrt(2) */
  double pos = 0.5 * (erfc((a - mu) / s) - erfc((b - mu) / s));
  double neg = 0.5 * (erfc((a + mu) / s) - erfc((b + mu) / s));
  double m = pos + neg;
  if (!(m >= 1e-300)) m = 0.0;
  return m;
}

/* Exponent field of a double's magnitude, clamped to the bf16 range 0..254. */
static int field_of(double v) {
  double a = fabs(v);
  if (a == 0.0 || a < ldexp(1.0, -126)) return 0;
  int ex;
  (void)frexp(a, &ex); /* a = fr * 2^ex, fr in [0.5, 1) */
  int f = ex + 126;
  if (f > 254) f = 254;
  if (f < 0) f = 0;
  return f;
}

void ora_zc_predict(double mu, double sigma, uint8_t book[7]) {
  if (!(sigma > 0.0)) {
    int lo = field_of(mu) - 3;
    if (lo < 0) lo = 0;
    if (lo > 248) lo = 248;
    for (int j = 0; j < 7; ++j) book[j] = (uint8_t)(lo + j);
    return;
  }
  double mass[256];
  int taken[256];
  for (int f = 0; f < 256; ++f) {
    mass[f] = (f >= 1 && f <= 254) ? ora_zc_mass(mu, sigma, f) : -1.0;
    taken[f] = 0;
  }
  int pick[7];
  for (int r = 0; r < 7; ++r) {
    int best = -1;
    for (int f = 1; f <= 254; ++f) { /* ascending: ties keep the smaller f */
      if (taken[f]) continue;
      if (best < 0 || mass[f] > mass[best]) best = f;
    }
    taken[best] = 1;
    pick[r] = best;
  }
  int k = 0;
  for (int f = 0; f < 256; ++f)
    if (taken[f]) book[k++] = (uint8_t)f;
  (void)pick;
}

static uint64_t zc_slot_bytes(uint32_t C) { return (uint64_t)C * 11u / 8u; }

static int zc_check_layout(uint64_t n, uint32_t nseg, const uint64_t* seg_off,
                           uint32_t C) {
  if (C < 1024u || C > 65536u || (C % 1024u) != 0) return ORA_E_ARG;
  if (nseg == 0) return ORA_E_ARG;
  if (seg_off) {
    if (seg_off[0] != 0 || seg_off[nseg] != n) return ORA_E_ARG;
    for (uint32_t s = 0; s < nseg; ++s)
      if (seg_off[s + 1] < seg_off[s]) return ORA_E_ARG;
  } else if (nseg != 1) {
    return ORA_E_ARG;
  }
  return ORA_OK;
}

static uint64_t seg_begin(const uint64_t* seg_off, uint32_t s) {
  return seg_off ? seg_off[s] : 0;
}
static uint64_t seg_end(const uint64_t* seg_off, uint32_t s, uint64_t n) {
  return seg_off ? seg_off[s + 1] : n;
}

uint64_t ora_zc_stream_bytes(uint64_t n, uint32_t nseg, const uint64_t* seg_off,
                             uint32_t C, uint64_t n_esc) {
  uint64_t nchunks = 0;
  for (uint32_t s = 0; s < nseg; ++s) {
    uint64_t len = seg_end(seg_off, s, n) - seg_begin(seg_off, s);
    nchunks += (len + C - 1) / C;
  }
  uint64_t off_escoff = ZC_HDR + round_up((uint64_t)ZC_SEGREC * nseg, ZC_ALIGN);
  uint64_t off_static = off_escoff + round_up(8u * (nchunks + 1), ZC_ALIGN);
  uint64_t off_esc = off_static + nchunks * zc_slot_bytes(C);
  return off_esc + round_up(n_esc, ZC_ALIGN);
}

/* [ZipCCL] 2.B for one element: split sign+mantissa from the 8-bit exponent,
 * look the exponent up in the 7-entry book. */
static unsigned zc_code_of(unsigned e, const uint8_t book[7]) {
  for (unsigned j = 0; j < 7; ++j)
    if (book[j] == e) return j + 1; /* codes 001..111 */
  return 0;                         /* 000: escape */
}

int ora_zc_encode_chunk(const uint16_t* x, uint32_t L, uint32_t C,
                        const uint8_t book[7], uint8_t* slot, uint8_t* esc,
                        uint32_t* n_esc, int* raw) {
  if (C < 1024u || (C % 1024u) != 0 || L > C) return ORA_E_ARG;
  uint64_t S = zc_slot_bytes(C);
  memset(slot, 0, S);
  uint8_t* sm = slot;
  uint8_t* plane[3] = {slot + C, slot + C + C / 8, slot + C + 2 * (C / 8)};
  uint32_t ne = 0;
  for (uint32_t i = 0; i < L; ++i) {
    uint16_t v = x[i];
    unsigned sign = (v >> 15) & 1u;
    unsigned e = (v >> 7) & 0xFFu;
    unsigned mant = v & 0x7Fu;
    sm[i] = (uint8_t)((sign << 7) | mant);
    unsigned code = zc_code_of(e, book);
    for (int k = 0; k < 3; ++k) set_bit(plane[k], i, (code >> k) & 1u);
    if (code == 0) esc[ne++] = (uint8_t)e;
  }
  /* raw fallback for a full chunk: fewer dynamic bytes than the escapes */
  const uint64_t raw_bytes = 2ull * L;
  const uint64_t raw_dyn = raw_bytes - S; /* 5C/8 when L = C */
  *raw = L == C && raw_dyn < ne;
  if (*raw) {
    for (uint64_t b = 0; b < raw_bytes; ++b) {
      const uint8_t byte = (uint8_t)(x[b / 2] >> (8 * (b % 2)));
      if (b < S) slot[b] = byte;
      else esc[b - S] = byte;
    }
    ne = (uint32_t)raw_dyn;
  }
  *n_esc = ne;
  return ORA_OK;
}

int ora_zc_encode(const uint16_t* x, uint64_t n, const uint64_t* seg_off,
                  uint32_t nseg, uint32_t C, const uint8_t* books, uint8_t* out,
                  uint64_t cap, uint64_t* out_bytes, uint8_t* books_used,
                  double* mus, double* sigmas) {
  int rc = zc_check_layout(n, nseg, seg_off, C);
  if (rc) return rc;
  uint64_t nchunks = 0;
  for (uint32_t s = 0; s < nseg; ++s) {
    uint64_t len = seg_end(seg_off, s, n) - seg_begin(seg_off, s);
    nchunks += (len + C - 1) / C;
  }
  const uint64_t S = zc_slot_bytes(C);
  const uint64_t off_seg = ZC_HDR;
  const uint64_t off_escoff = off_seg + round_up((uint64_t)ZC_SEGREC * nseg, ZC_ALIGN);
  const uint64_t off_static = off_escoff + round_up(8u * (nchunks + 1), ZC_ALIGN);
  const uint64_t off_esc = off_static + nchunks * S;
  if (cap < off_esc) return ORA_E_CAPACITY;
  memset(out, 0, off_esc);

  uint8_t* slot = (uint8_t*)malloc(S);
  uint8_t* esc = (uint8_t*)malloc(C);  /* escapes, or a raw chunk's remainder (< C) */
  if (!slot || !esc) {
    free(slot);
    free(esc);
    return ORA_E_ARG;
  }
  uint64_t esc_total = 0;
  uint64_t chunk = 0;
  for (uint32_t s = 0; s < nseg; ++s) {
    uint64_t b = seg_begin(seg_off, s), e = seg_end(seg_off, s, n);
    uint64_t len = e - b;
    uint8_t book[7];
    if (books) {
      memcpy(book, books + 7u * s, 7);
    } else {
      uint64_t cnt;
      double s1, s2, mu, sg;
      ora_zc_stats(x + b, len, &cnt, &s1, &s2);
      ora_zc_moments(cnt, s1, s2, &mu, &sg);
      ora_zc_predict(mu, sg, book);
      if (mus) mus[s] = mu;
      if (sigmas) sigmas[s] = sg;
    }
    if (books_used) memcpy(books_used + 7u * s, book, 7);
    uint64_t seg_chunks = (len + C - 1) / C;
    uint8_t* rec = out + off_seg + (uint64_t)ZC_SEGREC * s;
    wr64(rec + 0, b);
    wr64(rec + 8, len);
    wr64(rec + 16, chunk);
    wr64(rec + 24, seg_chunks);
    wr64(rec + 32, esc_total);
    uint64_t seg_esc0 = esc_total;
    for (int j = 0; j < 7; ++j) rec[48 + j] = book[j];
    for (uint64_t j = 0; j < seg_chunks; ++j, ++chunk) {
      uint64_t first = b + j * C;
      uint32_t L = (uint32_t)((e - first) < C ? (e - first) : C);
      uint32_t ne = 0;
      int raw = 0;
      ora_zc_encode_chunk(x + first, L, C, book, slot, esc, &ne, &raw);
      wr64(out + off_escoff + 8u * chunk, esc_total | ((uint64_t)raw << 63));
      memcpy(out + off_static + chunk * S, slot, S);
      if (off_esc + esc_total + ne > cap) {
        free(slot);
        free(esc);
        return ORA_E_CAPACITY;
      }
      memcpy(out + off_esc + esc_total, esc, ne);
      esc_total += ne;
    }
    wr64(rec + 40, esc_total - seg_esc0);
  }
  free(slot);
  free(esc);
  wr64(out + off_escoff + 8u * nchunks, esc_total);
  uint64_t total = off_esc + round_up(esc_total, ZC_ALIGN);
  if (total > cap) return ORA_E_CAPACITY;
  memset(out + off_esc + esc_total, 0, total - off_esc - esc_total);

  memset(out, 0, ZC_HDR);
  wr32(out + 0, ZC_MAGIC);
  wr16(out + 4, 1);
  wr16(out + 6, ZC_HDR);
  wr32(out + 8, C);
  wr32(out + 12, nseg);
  wr64(out + 16, n);
  wr64(out + 24, nchunks);
  wr64(out + 32, esc_total);
  wr64(out + 40, off_seg);
  wr64(out + 48, off_escoff);
  wr64(out + 56, off_static);
  wr64(out + 64, off_esc);
  wr64(out + 72, total);
  *out_bytes = total;
  return ORA_OK;
}

int ora_zc_decode(const uint8_t* in, uint64_t in_bytes, uint16_t* y,
                  uint64_t y_cap, uint64_t* n_out) {
  if (in_bytes < ZC_HDR) return ORA_E_FORMAT;
  if (rd32(in) != ZC_MAGIC || rd16(in + 4) != 1 || rd16(in + 6) != ZC_HDR)
    return ORA_E_FORMAT;
  uint32_t C = rd32(in + 8);
  uint32_t nseg = rd32(in + 12);
  uint64_t n = rd64(in + 16), nchunks = rd64(in + 24), esc_total = rd64(in + 32);
  uint64_t off_seg = rd64(in + 40), off_escoff = rd64(in + 48);
  uint64_t off_static = rd64(in + 56), off_esc = rd64(in + 64);
  uint64_t total = rd64(in + 72);
  if (C < 1024u || C > 65536u || (C % 1024u) != 0 || nseg == 0) return ORA_E_FORMAT;
  if (total > in_bytes) return ORA_E_FORMAT;
  const uint64_t S = zc_slot_bytes(C);
  /* every offset must follow from the counts */
  if (off_seg != ZC_HDR) return ORA_E_FORMAT;
  if (nseg > (total - ZC_HDR) / ZC_SEGREC) return ORA_E_FORMAT;
  if (off_escoff != off_seg + round_up((uint64_t)ZC_SEGREC * nseg, ZC_ALIGN))
    return ORA_E_FORMAT;
  if (nchunks > total / 8u) return ORA_E_FORMAT;
  if (off_static != off_escoff + round_up(8u * (nchunks + 1), ZC_ALIGN))
    return ORA_E_FORMAT;
  if (nchunks > total / S + 1 || off_esc != off_static + nchunks * S)
    return ORA_E_FORMAT;
  if (off_esc > total || esc_total > total - off_esc ||
      total != off_esc + round_up(esc_total, ZC_ALIGN))
    return ORA_E_FORMAT;
  if (n > y_cap) return ORA_E_CAPACITY;

  uint64_t elem = 0, chunk = 0;
  for (uint32_t s = 0; s < nseg; ++s) {
    const uint8_t* rec = in + off_seg + (uint64_t)ZC_SEGREC * s;
    uint64_t b = rd64(rec), len = rd64(rec + 8), c0 = rd64(rec + 16);
    uint64_t segc = rd64(rec + 24);
    if (b != elem || c0 != chunk || len > n - elem) return ORA_E_FORMAT;
    if (segc != (len + C - 1) / C || segc > nchunks - chunk) return ORA_E_FORMAT;
    const uint8_t* book = rec + 48;
    for (uint64_t j = 0; j < segc; ++j, ++chunk) {
      uint64_t first = b + j * C;
      uint64_t L = (b + len - first) < C ? (b + len - first) : C;
      const uint8_t* slot = in + off_static + chunk * S;
      const uint8_t* plane[3] = {slot + C, slot + C + C / 8, slot + C + 2 * (C / 8)};
      const uint64_t e0 = rd64(in + off_escoff + 8u * chunk);
      const uint64_t e1 = rd64(in + off_escoff + 8u * (chunk + 1));
      const int raw = (int)(e0 >> 63);
      uint64_t ep = e0 & ~(1ull << 63);
      uint64_t ep_end = e1 & ~(1ull << 63);
      if (chunk + 1 == nchunks && (e1 >> 63)) return ORA_E_FORMAT;
      if (ep > ep_end || ep_end > esc_total) return ORA_E_FORMAT;
      if (raw) {
        /* the raw fallback: 2C bytes, the slot's first, then the remainder */
        const uint64_t rb = 2ull * L, rd = rb - S;
        if (L != C || ep_end - ep != rd) return ORA_E_FORMAT;
        for (uint64_t i = 0; i < L; ++i) {
          uint16_t v = 0;
          for (uint64_t h = 0; h < 2; ++h) {
            const uint64_t bb = 2 * i + h;
            const uint8_t byte = bb < S ? slot[bb] : in[off_esc + ep + (bb - S)];
            v |= (uint16_t)((unsigned)byte << (8 * h));
          }
          y[first + i] = v;
        }
        continue;
      }
      for (uint64_t i = 0; i < L; ++i) {
        unsigned smb = slot[i];
        unsigned code = 0;
        for (int k = 0; k < 3; ++k) code |= (unsigned)get_bit(plane[k], i) << k;
        unsigned e;
        if (code) {
          e = book[code - 1];
        } else {
          if (ep >= ep_end) return ORA_E_FORMAT;
          e = in[off_esc + ep];
          ep++;
        }
        y[first + i] = (uint16_t)(((smb & 0x80u) << 8) | (e << 7) | (smb & 0x7Fu));
      }
      if (ep != ep_end) return ORA_E_FORMAT;
    }
    elem += len;
  }
  if (elem != n || chunk != nchunks) return ORA_E_FORMAT;
  *n_out = n;
  return ORA_OK;
}

/* ============================================================ IBP
 *
 * Metadata "IBPM" ([IBP] Algoritmo Core step 1; fixed size, kept and reused):
 *     0 u32 magic 0x4D504249 ('I','B','P','M')  4 u16 version 1
 *     6 u16 header bytes 64   8 u32 chunk_bytes  12 u32 chunk bits B
 *    16 u32 m = popcount(Mask)  20 u32 mode  24 u64 N samples  32 u64 k
 *    40 f64 T   48 u64 FNV-1a-64 of (chunk_bytes as 4 LE bytes, Mask, Bitval)
 *    56 u64 zero
 *   Mask at 64 (chunk_bytes bytes), Bitval after it (chunk_bytes bytes);
 *   chunk bit j is bit j%8 of byte j/8.
 *
 * Stream "IBP1" ([IBP] steps 2-3):
 *   header 128 bytes:
 *     0 u32 magic 0x31504249 ('I','B','P','1')  4 u16 version 1
 *     6 u16 header bytes 128  8 u32 chunk_bytes  12 u32 m  16 u64 n_bytes
 *    24 u64 nchunks  32 u64 ngroups  40 u64 meta hash  48 u64 off_grp (=128)
 *    56 u64 off_payload  64 u64 payload bits  72 u64 total bytes  80.. zero
 *   group offsets at 128: u64 x (ngroups+1), bit offsets from the payload
 *     start (multiples of 128); padded to 128 bytes
 *   payload: group g = chunks 32g..32g+31:
 *     32 participation bits (bit t for chunk 32g+t; 0 past the last chunk),
 *     then the chunk bodies in order, then zero bits up to a multiple of 128.
 *     body with p=1: the bits at positions outside Mask, ascending;
 *     body with p=0: all the chunk's bits (a short last chunk is always p=0).
 *   Bit q of the payload is bit q%8 of byte q/8.
 */

#define IBPM_MAGIC 0x4D504249u
#define IBP1_MAGIC 0x31504249u
#define IBPM_HDR 64u
#define IBP1_HDR 128u

uint64_t ora_ibp_meta_bytes(uint32_t chunk_bytes) {
  return IBPM_HDR + 2ull * chunk_bytes;
}

uint64_t ora_fnv1a64(const uint8_t* p, size_t n) {
  uint64_t h = 0xcbf29ce484222325ull;
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 0x100000001b3ull;
  }
  return h;
}

static uint64_t ibp_meta_hash(uint32_t chunk_bytes, const uint8_t* mask,
                              const uint8_t* bitval) {
  uint64_t h = 0xcbf29ce484222325ull;
  uint8_t cb[4];
  wr32(cb, chunk_bytes);
  for (int i = 0; i < 4; ++i) {
    h ^= cb[i];
    h *= 0x100000001b3ull;
  }
  for (uint32_t i = 0; i < chunk_bytes; ++i) {
    h ^= mask[i];
    h *= 0x100000001b3ull;
  }
  for (uint32_t i = 0; i < chunk_bytes; ++i) {
    h ^= bitval[i];
    h *= 0x100000001b3ull;
  }
  return h;
}

static void ibp_write_meta_header(uint8_t* meta, uint32_t chunk_bytes, uint32_t m,
                                  int mode, uint64_t N, uint64_t k, double T) {
  memset(meta, 0, IBPM_HDR);
  wr32(meta + 0, IBPM_MAGIC);
  wr16(meta + 4, 1);
  wr16(meta + 6, IBPM_HDR);
  wr32(meta + 8, chunk_bytes);
  wr32(meta + 12, chunk_bytes * 8u);
  wr32(meta + 16, m);
  wr32(meta + 20, (uint32_t)mode);
  wr64(meta + 24, N);
  wr64(meta + 32, k);
  uint64_t tb;
  memcpy(&tb, &T, 8);
  wr64(meta + 40, tb);
  wr64(meta + 48, ibp_meta_hash(chunk_bytes, meta + IBPM_HDR,
                                meta + IBPM_HDR + chunk_bytes));
}

int ora_ibp_build_meta(const uint8_t* samples, uint64_t N, uint32_t chunk_bytes,
                       double T, int mode, uint8_t* meta) {
  if (chunk_bytes == 0 || (chunk_bytes % 4u) != 0 || N == 0) return ORA_E_ARG;
  if (!(T > 0.5 && T <= 1.0) || (mode != 0 && mode != 1)) return ORA_E_ARG;
  const uint64_t B = (uint64_t)chunk_bytes * 8u;
  const uint64_t k = (uint64_t)ceil(T * (double)N);
  uint64_t* ones = (uint64_t*)calloc(B, sizeof(uint64_t));
  if (!ones) return ORA_E_ARG;
  /* count, per bit position, the samples holding a 1 there */
  for (uint64_t s = 0; s < N; ++s) {
    const uint8_t* c = samples + s * chunk_bytes;
    for (uint64_t j = 0; j < B; ++j) ones[j] += (uint64_t)get_bit(c, j);
  }
  uint8_t* mask = meta + IBPM_HDR;
  uint8_t* bitval = meta + IBPM_HDR + chunk_bytes;
  memset(mask, 0, chunk_bytes);
  memset(bitval, 0, chunk_bytes);
  uint32_t m = 0;
  if (mode == 0) {
    /* a position is invariant when one value holds in at least k samples */
    for (uint64_t j = 0; j < B; ++j) {
      uint64_t agree = ones[j] > N - ones[j] ? ones[j] : N - ones[j];
      if (agree >= k) {
        set_bit(mask, j, 1);
        set_bit(bitval, j, ones[j] >= k);
        ++m;
      }
    }
  } else {
    /* joint reading: keep adding positions, most-agreeing first (ties: lower
     * position), while at least k samples match every kept position */
    uint64_t* cand = (uint64_t*)malloc(B * sizeof(uint64_t));
    uint8_t* alive = (uint8_t*)malloc(N);
    if (!cand || !alive) {
      free(cand);
      free(alive);
      free(ones);
      return ORA_E_ARG;
    }
    uint64_t nc = 0;
    for (uint64_t j = 0; j < B; ++j) {
      uint64_t agree = ones[j] > N - ones[j] ? ones[j] : N - ones[j];
      if (agree >= k) cand[nc++] = j;
    }
    /* insertion sort by (agreement descending, position ascending) */
    for (uint64_t a = 1; a < nc; ++a) {
      uint64_t j = cand[a];
      uint64_t aj = ones[j] > N - ones[j] ? ones[j] : N - ones[j];
      uint64_t b = a;
      while (b > 0) {
        uint64_t p = cand[b - 1];
        uint64_t ap = ones[p] > N - ones[p] ? ones[p] : N - ones[p];
        if (ap > aj || (ap == aj && p < j)) break;
        cand[b] = p;
        --b;
      }
      cand[b] = j;
    }
    for (uint64_t s = 0; s < N; ++s) alive[s] = 1;
    for (uint64_t a = 0; a < nc; ++a) {
      uint64_t j = cand[a];
      int v = ones[j] >= k;
      uint64_t cnt = 0;
      for (uint64_t s = 0; s < N; ++s)
        if (alive[s] && get_bit(samples + s * chunk_bytes, j) == v) ++cnt;
      if (cnt >= k) {
        set_bit(mask, j, 1);
        set_bit(bitval, j, v);
        ++m;
        for (uint64_t s = 0; s < N; ++s)
          if (alive[s] && get_bit(samples + s * chunk_bytes, j) != v) alive[s] = 0;
      }
    }
    free(cand);
    free(alive);
  }
  free(ones);
  ibp_write_meta_header(meta, chunk_bytes, m, mode, N, k, T);
  return ORA_OK;
}

int ora_ibp_make_meta(uint32_t chunk_bytes, const uint8_t* mask,
                      const uint8_t* bitval, uint8_t* meta) {
  if (chunk_bytes == 0 || (chunk_bytes % 4u) != 0) return ORA_E_ARG;
  uint32_t m = 0;
  for (uint64_t j = 0; j < (uint64_t)chunk_bytes * 8u; ++j) {
    int mk = get_bit(mask, j);
    set_bit(meta + IBPM_HDR, j, mk);
    set_bit(meta + IBPM_HDR + chunk_bytes, j, mk && get_bit(bitval, j));
    m += (uint32_t)mk;
  }
  ibp_write_meta_header(meta, chunk_bytes, m, 0, 0, 0, 1.0);
  return ORA_OK;
}

static int ibp_meta_ok(const uint8_t* meta) {
  return rd32(meta) == IBPM_MAGIC && rd16(meta + 4) == 1 &&
         rd16(meta + 6) == IBPM_HDR && rd32(meta + 8) != 0 &&
         (rd32(meta + 8) % 4u) == 0 && rd32(meta + 12) == rd32(meta + 8) * 8u;
}

int ora_ibp_chunk_p(const uint8_t* meta, const uint8_t* chunk) {
  uint32_t cb = rd32(meta + 8);
  uint32_t m = rd32(meta + 16);
  const uint8_t* mask = meta + IBPM_HDR;
  const uint8_t* bitval = meta + IBPM_HDR + cb;
  if (m == 0) return 0; /* nothing to drop: compression saves nothing */
  for (uint64_t j = 0; j < (uint64_t)cb * 8u; ++j)
    if (get_bit(mask, j) && get_bit(chunk, j) != get_bit(bitval, j)) return 0;
  return 1;
}

uint64_t ora_ibp_stream_bytes_bound(uint32_t chunk_bytes, uint64_t n_bytes) {
  uint64_t nch = (n_bytes + chunk_bytes - 1) / chunk_bytes;
  uint64_t ng = (nch + 31) / 32;
  uint64_t pay_bits = 0;
  for (uint64_t g = 0; g < ng; ++g) {
    uint64_t in_g = nch - 32 * g < 32 ? nch - 32 * g : 32;
    pay_bits += round_up(32 + in_g * (uint64_t)chunk_bytes * 8u, 128);
  }
  return IBP1_HDR + round_up(8 * (ng + 1), 128) + pay_bits / 8;
}

int ora_ibp_encode_group(const uint8_t* meta, const uint8_t* x, uint32_t nch,
                         uint32_t last_bytes, uint8_t* out, uint64_t cap,
                         uint64_t* bits) {
  if (!ibp_meta_ok(meta) || nch == 0 || nch > 32) return ORA_E_ARG;
  const uint32_t cb = rd32(meta + 8);
  const uint64_t B = (uint64_t)cb * 8u;
  const uint8_t* mask = meta + IBPM_HDR;
  if (last_bytes == 0) last_bytes = cb;
  if (last_bytes > cb || (last_bytes % 4u) != 0) return ORA_E_ARG;
  memset(out, 0, cap);
  int p[32];
  uint64_t q = 32;
  for (uint32_t t = 0; t < nch; ++t) {
    const uint8_t* c = x + (uint64_t)t * cb;
    int full = (t + 1 < nch) || last_bytes == cb;
    p[t] = full ? ora_ibp_chunk_p(meta, c) : 0;
    if (p[t]) {
      for (uint64_t j = 0; j < B; ++j) {
        if (get_bit(mask, j)) continue; /* invariant bit: dropped */
        if (q >= cap * 8u) return ORA_E_CAPACITY;
        set_bit(out, q++, get_bit(c, j));
      }
    } else {
      uint64_t len = full ? B : (uint64_t)last_bytes * 8u;
      for (uint64_t j = 0; j < len; ++j) {
        if (q >= cap * 8u) return ORA_E_CAPACITY;
        set_bit(out, q++, get_bit(c, j));
      }
    }
  }
  for (uint32_t t = 0; t < 32; ++t) set_bit(out, t, t < nch ? p[t] : 0);
  uint64_t padded = round_up(q, 128);
  if (padded > cap * 8u) return ORA_E_CAPACITY;
  *bits = padded;
  return ORA_OK;
}

int ora_ibp_encode(const uint8_t* meta, const uint8_t* x, uint64_t n_bytes,
                   uint8_t* out, uint64_t cap, uint64_t* out_bytes) {
  if (!ibp_meta_ok(meta) || (n_bytes % 4u) != 0) return ORA_E_ARG;
  const uint32_t cb = rd32(meta + 8);
  const uint64_t nch = (n_bytes + cb - 1) / cb;
  const uint64_t ng = (nch + 31) / 32;
  const uint64_t off_grp = IBP1_HDR;
  const uint64_t off_pay = off_grp + round_up(8 * (ng + 1), 128);
  if (cap < off_pay) return ORA_E_CAPACITY;
  memset(out, 0, off_pay);
  uint64_t gcap = 4u + 32ull * cb + 16u;
  uint8_t* gbuf = (uint8_t*)malloc(gcap);
  if (!gbuf) return ORA_E_ARG;
  uint64_t pos = 0; /* payload bits written */
  for (uint64_t g = 0; g < ng; ++g) {
    uint64_t c0 = 32 * g;
    uint32_t in_g = (uint32_t)(nch - c0 < 32 ? nch - c0 : 32);
    uint64_t last_first = (c0 + in_g - 1) * cb;
    uint32_t last_bytes = (uint32_t)(n_bytes - last_first < cb ? n_bytes - last_first : cb);
    uint64_t bits = 0;
    int rc = ora_ibp_encode_group(meta, x + c0 * cb, in_g, last_bytes, gbuf,
                                  gcap, &bits);
    if (rc) {
      free(gbuf);
      return rc;
    }
    wr64(out + off_grp + 8 * g, pos);
    if (off_pay + (pos + bits) / 8 > cap) {
      free(gbuf);
      return ORA_E_CAPACITY;
    }
    memcpy(out + off_pay + pos / 8, gbuf, bits / 8);
    pos += bits;
  }
  free(gbuf);
  wr64(out + off_grp + 8 * ng, pos);
  uint64_t total = off_pay + pos / 8;
  memset(out, 0, IBP1_HDR);
  wr32(out + 0, IBP1_MAGIC);
  wr16(out + 4, 1);
  wr16(out + 6, IBP1_HDR);
  wr32(out + 8, cb);
  wr32(out + 12, rd32(meta + 16));
  wr64(out + 16, n_bytes);
  wr64(out + 24, nch);
  wr64(out + 32, ng);
  wr64(out + 40, rd64(meta + 48));
  wr64(out + 48, off_grp);
  wr64(out + 56, off_pay);
  wr64(out + 64, pos);
  wr64(out + 72, total);
  *out_bytes = total;
  return ORA_OK;
}

int ora_ibp_decode(const uint8_t* meta, const uint8_t* in, uint64_t in_bytes,
                   uint8_t* y, uint64_t y_cap, uint64_t* n_out) {
  if (!ibp_meta_ok(meta)) return ORA_E_ARG;
  if (in_bytes < IBP1_HDR) return ORA_E_FORMAT;
  if (rd32(in) != IBP1_MAGIC || rd16(in + 4) != 1 || rd16(in + 6) != IBP1_HDR)
    return ORA_E_FORMAT;
  const uint32_t cb = rd32(in + 8);
  const uint32_t m = rd32(in + 12);
  const uint64_t n_bytes = rd64(in + 16), nch = rd64(in + 24), ng = rd64(in + 32);
  const uint64_t hash = rd64(in + 40), off_grp = rd64(in + 48);
  const uint64_t off_pay = rd64(in + 56), pay_bits = rd64(in + 64);
  const uint64_t total = rd64(in + 72);
  if (cb != rd32(meta + 8) || m != rd32(meta + 16) || hash != rd64(meta + 48))
    return ORA_E_META;
  if (total > in_bytes || off_grp != IBP1_HDR || (n_bytes % 4u) != 0)
    return ORA_E_FORMAT;
  if (nch != (n_bytes + cb - 1) / cb || ng != (nch + 31) / 32) return ORA_E_FORMAT;
  if (ng > total / 8u) return ORA_E_FORMAT;
  if (off_pay != off_grp + round_up(8 * (ng + 1), 128)) return ORA_E_FORMAT;
  if (off_pay > total || pay_bits % 128u != 0 || pay_bits / 8 != total - off_pay)
    return ORA_E_FORMAT;
  if (n_bytes > y_cap) return ORA_E_CAPACITY;
  const uint64_t B = (uint64_t)cb * 8u;
  const uint8_t* mask = meta + IBPM_HDR;
  const uint8_t* bitval = meta + IBPM_HDR + cb;
  const uint8_t* pay = in + off_pay;
  for (uint64_t g = 0; g < ng; ++g) {
    uint64_t g0 = rd64(in + off_grp + 8 * g), g1 = rd64(in + off_grp + 8 * (g + 1));
    if (g0 > g1 || g1 > pay_bits || g0 % 128u != 0) return ORA_E_FORMAT;
    uint64_t q = g0 + 32;
    for (uint32_t t = 0; t < 32; ++t) {
      uint64_t c = 32 * g + t;
      int p = get_bit(pay, g0 + t);
      if (c >= nch) {
        if (p) return ORA_E_FORMAT;
        continue;
      }
      uint64_t first = c * cb;
      uint64_t len = n_bytes - first < cb ? n_bytes - first : cb;
      uint8_t* out = y + first;
      if (p) {
        if (len != cb || m == 0) return ORA_E_FORMAT;
        /* [IBP] step 3: put the Bitval bits back at the invariant positions */
        for (uint64_t j = 0; j < B; ++j) {
          if (get_bit(mask, j)) {
            set_bit(out, j, get_bit(bitval, j));
          } else {
            if (q >= g1) return ORA_E_FORMAT;
            set_bit(out, j, get_bit(pay, q++));
          }
        }
      } else {
        for (uint64_t j = 0; j < len * 8u; ++j) {
          if (q >= g1) return ORA_E_FORMAT;
          set_bit(out, j, get_bit(pay, q++));
        }
      }
    }
    if (round_up(q, 128) != g1) return ORA_E_FORMAT;
  }
  if (ng && rd64(in + off_grp + 8 * ng) != pay_bits) return ORA_E_FORMAT;
  *n_out = n_bytes;
  return ORA_OK;
}

/* ---------------- IBP in-place slots ([IBP] Integrazione del Sistema) ---- */

uint32_t ora_ibp_slot_read_bytes(const uint8_t* meta, int p, uint32_t len) {
  const uint64_t B = (uint64_t)rd32(meta + 8) * 8u;
  const uint64_t m = rd32(meta + 16);
  return p ? (uint32_t)(4u * ((B - m + 31u) / 32u)) : len;
}

int ora_ibp_slot_encode(const uint8_t* meta, const uint8_t* chunk, uint32_t len,
                        uint8_t* slot, int* p) {
  if (!ibp_meta_ok(meta)) return ORA_E_ARG;
  const uint32_t cb = rd32(meta + 8);
  if (len == 0 || len > cb || (len % 4u) != 0) return ORA_E_ARG;
  const uint64_t B = (uint64_t)cb * 8u;
  const uint8_t* mask = meta + IBPM_HDR;
  /* [IBP] step 2's predicate; a short chunk is kept raw */
  *p = len == cb ? ora_ibp_chunk_p(meta, chunk) : 0;
  if (!*p) {
    memmove(slot, chunk, len);
    return ORA_OK;
  }
  /* the kept bits, one at a time, into a scratch body, then the body's
   * words over the start of the slot */
  const uint32_t rb = ora_ibp_slot_read_bytes(meta, 1, cb);
  uint8_t* body = (uint8_t*)calloc(rb ? rb : 1, 1);
  if (!body) return ORA_E_ARG;
  uint64_t q = 0;
  for (uint64_t j = 0; j < B; ++j) {
    if (get_bit(mask, j)) continue;
    set_bit(body, q++, get_bit(chunk, j));
  }
  memcpy(slot, body, rb);
  free(body);
  return ORA_OK;
}

int ora_ibp_slot_decode(const uint8_t* meta, const uint8_t* slot, uint32_t len,
                        int p, uint8_t* chunk) {
  if (!ibp_meta_ok(meta)) return ORA_E_ARG;
  const uint32_t cb = rd32(meta + 8);
  if (len == 0 || len > cb || (len % 4u) != 0) return ORA_E_ARG;
  if (!p) {
    memmove(chunk, slot, len);
    return ORA_OK;
  }
  if (len != cb || rd32(meta + 16) == 0) return ORA_E_FORMAT;
  const uint64_t B = (uint64_t)cb * 8u;
  const uint8_t* mask = meta + IBPM_HDR;
  const uint8_t* bitval = meta + IBPM_HDR + cb;
  uint8_t* out = (uint8_t*)calloc(cb, 1);
  if (!out) return ORA_E_ARG;
  uint64_t q = 0;
  for (uint64_t j = 0; j < B; ++j) {
    /* [IBP] step 3: Bitval at the invariant positions, kept bits in order */
    if (get_bit(mask, j)) set_bit(out, j, get_bit(bitval, j));
    else set_bit(out, j, get_bit(slot, q++));
  }
  memcpy(chunk, out, cb);
  free(out);
  return ORA_OK;
}
