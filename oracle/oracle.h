/*
 * oracle.h -- bit-serial CPU oracle for the two lossless codecs.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path includes, links or
 * calls this code; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no header, table or helper with the CUDA
 * library: every constant of the stream formats is written out here again on
 * purpose.
 *
 * Sources (gist.science summaries; cited by page title and section):
 *   [ZipCCL] "ZipCCL: Efficient Lossless Data Compression of Communication
 *            Collectives for Accelerating LLM Training", section
 *            "2. Metodologia", parts A (Gaussian insight, top-7 exponents,
 *            closed-form codebook from sigma), B (exponent coding: 3-bit codes
 *            001-111, escape code 000 with the full 8-bit exponent kept in a
 *            separate array, 16 -> 11 bits), C (128-byte padding, three 1-bit
 *            planes), D (static part first, dynamic part after).
 *   [IBP]    "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria
 *            GPU con la Compressione Lossless per il ML", section
 *            "Metodologia: Invariant Bit Packing (IBP)" -> "Algoritmo Core",
 *            steps 1 (Mask/Bitval from positions invariant over a fraction T of
 *            sampled tensors), 2 (per-chunk match, drop invariant bits, one
 *            participation bit per chunk), 3 (warp prefix scan of chunk bit
 *            lengths, re-insert Bitval bits).
 *
 * The byte layouts of both streams are this project's own readings of those
 * sections (the pages print no bitstream); they are stated in the repository's
 * design notes and restated next to each function below.
 *
 * Parity status of each function (what pins it other than itself) is listed in
 * the design notes; every function here is pinned by at least one test.
 *
 * All multi-byte integers in every stream are little-endian.
 * Return values: 0 on success, negative on error (see ORA_E_*).
 */
#ifndef LBB16_ORACLE_H
#define LBB16_ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORA_OK 0
#define ORA_E_ARG (-1)
#define ORA_E_CAPACITY (-2)
#define ORA_E_FORMAT (-3)
#define ORA_E_META (-4)

/* ---------------- ZipCCL exponent coding of bf16 ---------------- */

/* Sums over the finite elements (exponent field != 255) of a bf16 array, in
 * fp64, one element at a time in index order ([ZipCCL] 2.A: the codebook is
 * derived from the standard deviation of the values). */
void ora_zc_stats(const uint16_t* x, uint64_t n, uint64_t* cnt, double* sum,
                  double* sumsq);

/* Mean and population standard deviation from the sums. cnt == 0 gives 0, 0. */
void ora_zc_moments(uint64_t cnt, double sum, double sumsq, double* mu,
                    double* sigma);

/* Gaussian probability mass of exponent field f (1..254) for N(mu, sigma):
 * P(2^(f-127) <= |X| < 2^(f-126)); values below 1e-300 read as 0. */
double ora_zc_mass(double mu, double sigma, int f);

/* The 7-entry codebook (ascending exponent fields) predicted from (mu, sigma):
 * the 7 fields with the largest mass, ties toward the smaller field; sigma == 0
 * gives the window of 7 fields centred on the field of mu. */
void ora_zc_predict(double mu, double sigma, uint8_t book[7]);

/* Size of the stream for the given layout and escape count. */
uint64_t ora_zc_stream_bytes(uint64_t n, uint32_t nseg, const uint64_t* seg_off,
                             uint32_t chunk_elems, uint64_t n_esc);

/* Encode n bf16 values (bit patterns) split at seg_off[0..nseg] (NULL: one
 * segment) into a ZCC1 stream.  books: 7*nseg fields, or NULL to predict each
 * segment's book from its own statistics (mu/sigma out arrays may be NULL). */
int ora_zc_encode(const uint16_t* x, uint64_t n, const uint64_t* seg_off,
                  uint32_t nseg, uint32_t chunk_elems, const uint8_t* books,
                  uint8_t* out, uint64_t cap, uint64_t* out_bytes,
                  uint8_t* books_used, double* mus, double* sigmas);

/* Decode a ZCC1 stream; *n_out receives the element count. */
int ora_zc_decode(const uint8_t* in, uint64_t in_bytes, uint16_t* y,
                  uint64_t y_cap, uint64_t* n_out);

/* One chunk on its own: L real elements (L <= C), the static slot (11*C/8
 * bytes) and the chunk's dynamic bytes (escapes, or a raw chunk's last 5C/8
 * bytes); *raw is set when the (full) chunk is stored raw. */
int ora_zc_encode_chunk(const uint16_t* x, uint32_t L, uint32_t chunk_elems,
                        const uint8_t book[7], uint8_t* slot, uint8_t* esc,
                        uint32_t* n_esc, int* raw);

/* ---------------- IBP invariant bit packing ---------------- */

uint64_t ora_ibp_meta_bytes(uint32_t chunk_bytes);

/* FNV-1a (64-bit) over a byte string. */
uint64_t ora_fnv1a64(const uint8_t* p, size_t n);

/* Build the IBPM metadata blob from N sample chunks laid end to end
 * ([IBP] Algoritmo Core, step 1).  mode 0: per-position threshold;
 * mode 1: joint greedy (see the design notes).  T in (0.5, 1]. */
int ora_ibp_build_meta(const uint8_t* samples, uint64_t n_samples,
                       uint32_t chunk_bytes, double T, int mode, uint8_t* meta);

/* Make a blob directly from a given Mask and Bitval (Bitval is ANDed with
 * Mask); mode/N/T are recorded as given. */
int ora_ibp_make_meta(uint32_t chunk_bytes, const uint8_t* mask,
                      const uint8_t* bitval, uint8_t* meta);

/* Participation bit of one full chunk ([IBP] step 2). */
int ora_ibp_chunk_p(const uint8_t* meta, const uint8_t* chunk);

uint64_t ora_ibp_stream_bytes_bound(uint32_t chunk_bytes, uint64_t n_bytes);

/* Encode n_bytes (multiple of 4) into an IBP1 stream. */
int ora_ibp_encode(const uint8_t* meta, const uint8_t* x, uint64_t n_bytes,
                   uint8_t* out, uint64_t cap, uint64_t* out_bytes);

/* Decode an IBP1 stream with the matching metadata. */
int ora_ibp_decode(const uint8_t* meta, const uint8_t* in, uint64_t in_bytes,
                   uint8_t* y, uint64_t y_cap, uint64_t* n_bytes);

/* One group on its own: nch (1..32) chunks starting at x (the last one may be
 * short: last_bytes, a multiple of 4, else chunk_bytes).  Writes the group's
 * padded payload (zeroed first, cap bytes) and its length in bits. */
int ora_ibp_encode_group(const uint8_t* meta, const uint8_t* x, uint32_t nch,
                         uint32_t last_bytes, uint8_t* out, uint64_t cap,
                         uint64_t* bits);

/* ---------------- IBP in-place slots ([IBP] Integrazione del Sistema) ------
 *
 * Tensors kept in host memory for transfer: chunk s of the input owns a fixed
 * slot of chunk_bytes at slot_base + s*chunk_bytes (the last slot is as long
 * as the last chunk).  When the chunk participates (the predicate of step 2)
 * the slot starts with its body -- the B - m kept bits in ascending position
 * order, zero bits up to a whole 32-bit word -- and the slot's later bytes are
 * left as they were (compression in place); otherwise the slot holds the raw
 * chunk.  A bitmask (bit s % 32 of 32-bit word s / 32) records which slots
 * are compressed.  Reading a slot reads only its first
 * ora_ibp_slot_read_bytes bytes. */

/* Bytes of a slot that hold the chunk: 4*ceil((B - m)/32) when compressed,
 * else len. */
uint32_t ora_ibp_slot_read_bytes(const uint8_t* meta, int p, uint32_t len);

/* Slot form of one chunk of len bytes (a multiple of 4, at most chunk_bytes):
 * *p receives its participation bit; the slot's first read_bytes bytes are
 * written, the rest of the slot is not touched. */
int ora_ibp_slot_encode(const uint8_t* meta, const uint8_t* chunk, uint32_t len,
                        uint8_t* slot, int* p);

/* The chunk (len bytes) back from its slot and participation bit. */
int ora_ibp_slot_decode(const uint8_t* meta, const uint8_t* slot, uint32_t len,
                        int p, uint8_t* chunk);

#ifdef __cplusplus
}
#endif
#endif
