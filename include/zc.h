/*
 * zc.h -- C ABI of liblbb16.so: lossless bit-level codecs for ML tensors on
 * one GB300 GPU (sm_103a).
 *
 * Two codecs, both from gist.science page summaries:
 *
 *  [ZipCCL]  "ZipCCL: Efficient Lossless Data Compression of Communication
 *            Collectives for Accelerating LLM Training".
 *            2. Metodologia A: LLM tensors are near-Gaussian, so the 7 most
 *            frequent bf16 exponents cover > 97 % of values and can be
 *            predicted from the standard deviation, without a histogram.
 *            2. Metodologia B: each value splits into sign+mantissa and an
 *            8-bit exponent; a top-7 exponent becomes a 3-bit code 001..111,
 *            any other gets code 000 and its full exponent goes to a separate
 *            escape array (16 -> 11 bits for most values).
 *            2. Metodologia C: 128-byte padded blocks, 1-bit code planes,
 *            asynchronous global->shared staging.
 *            2. Metodologia D: fixed-size ("static") parts sent before the
 *            variable ("dynamic") parts.
 *  [IBP]     "Riepilogo Tecnico: Riduzione del Collo di Bottiglia della Memoria
 *            GPU con la Compressione Lossless per il ML", Metodologia:
 *            Invariant Bit Packing (IBP), Algoritmo Core:
 *            1 (Preprocessing): Mask and Bitval of bit positions invariant over
 *              a fraction T of sampled tensors, kept on the GPU and reused;
 *            2 (Compressione): per chunk, if the invariant positions match
 *              Bitval the invariant bits are dropped and the rest closed up; a
 *              participation bit marks compressed chunks;
 *            3 (Decompressione): warps read a compressed segment, a warp prefix
 *              scan gives every chunk's start bit, Bitval bits are re-inserted.
 *
 * Conventions for every call:
 *  - d_* arguments are device pointers, h_* host pointers.  The caller owns
 *    all data buffers and workspaces (allocated with cudaMalloc or PyTorch);
 *    the library keeps no pointer to them after the call returns.
 *  - Calls that take a stream are asynchronous on it: they validate what the
 *    host knows, enqueue kernels and return.  Nothing synchronises unless the
 *    description says so.  Output sizes go to device words (no hidden sync).
 *  - Errors the host can see are returned (ZC_OK = 0, negative otherwise).
 *    Errors only the GPU can see (corrupt stream, full output buffer,
 *    metadata mismatch, a scan wait that ran out) are written to the status
 *    word at the start of the workspace; read it with zc_status().  The first
 *    error of a call wins; each call clears the word when it starts.  No
 *    kernel traps or asserts; a failing kernel stops writing and returns.
 *  - Workspaces must be 256-byte aligned; sizes come from the *_workspace_bytes
 *    functions.  Two calls in flight at once must not share a workspace.
 *  - Stream formats (byte layouts) are described in the repository's design
 *    notes; all integers are little-endian, bit q of a bit string is bit q%8
 *    of byte q/8.
 */
#ifndef LBB16_ZC_H
#define LBB16_ZC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (ABI-identical to cudaStream_t; NULL = the legacy default). */
typedef struct CUstream_st* zc_stream_t;

enum {
  ZC_OK = 0,
  ZC_ERR_ARG = -1,           /* bad argument (host check)                     */
  ZC_ERR_CAPACITY = -2,      /* output or workspace buffer too small          */
  ZC_ERR_FORMAT = -3,        /* stream header/tables inconsistent (device)    */
  ZC_ERR_META_MISMATCH = -4, /* IBP stream made with other metadata (device)  */
  ZC_ERR_TIMEOUT = -5,       /* a bounded inter-block wait ran out (device)   */
  ZC_ERR_CUDA = -6,          /* a CUDA runtime call failed                    */
  ZC_ERR_UNSUPPORTED = -7,   /* legal in the format, not handled by this GPU path */
  ZC_ERR_NOMEM = -8          /* host or plan allocation failed                */
};

/* Text for an error code (static storage). */
const char* zc_strerror(int code);

/* Library version as an integer (major*10000 + minor*100 + patch). */
int zc_version(void);

/* TEST ONLY -- for checking that the encoders' bounded waits end; the pages
 * have no counterpart.  Every later zc_compress / ibp_compress call of this
 * process (until switched off) leaves out the scan state of tile `tile` --
 * the tile whose stream length or escape count the later tiles wait for: an
 * 8192-slot ticket of the ZipCCL encoder, a tile of the IBP encoder (16 KB
 * of input up to 512-byte chunks, one group at 1024 and 2048 bytes, 4096
 * groups of the offsets pass for the other chunk sizes up to 2048 bytes and
 * in the three-launch encode, one group above) -- and limits every wait between thread
 * blocks to `max_spins` polls (0: the normal limit, about one second).  The
 * waits behind the missing state run out, the call sets ZC_ERR_TIMEOUT in
 * its status word and returns with a stream that must not be used; nothing
 * faults or hangs.  tile = UINT64_MAX with max_spins = 0 switches it off
 * (the default).  Process-wide; not for use while other threads compress.
 * Returns ZC_OK. */
int zc_test_wait_fault(uint64_t tile, uint32_t max_spins);

/* TEST ONLY -- the pages have no counterpart.  ibp_compress of chunks up to
 * 512 bytes, and of 1024 and 2048 bytes, normally runs one cooperative kernel
 * (its blocks wait for each other's tile lengths, so the driver must place
 * the whole grid at once); when the driver refuses that launch it takes the
 * three-launch encode instead.
 * enable = 0 makes every such call take the three-launch encode (so tests can
 * check it), 1 restores the default.  Process-wide.  Returns ZC_OK. */
int zc_test_ibp_single_pass(int enable);

/* Read the status word of a workspace: synchronises the stream, copies the
 * word to *h_status (ZC_OK or a negative code).  Returns ZC_OK or ZC_ERR_CUDA. */
int zc_status(const void* d_ws, zc_stream_t stream, int* h_status);

/* ======================================================== ZipCCL, bf16
 *
 * A plan fixes the layout: n elements split at h_seg_off[0..nseg]
 * (h_seg_off[0] = 0, non-decreasing, h_seg_off[nseg] = n; NULL with nseg = 1
 * means one segment) and chunked with chunk_elems (multiple of 1024, at most
 * 65536) inside each segment.  Each segment gets its own 7-entry codebook.
 * The plan object and its small device tables (per-segment layout, codebooks,
 * statistics) are owned by the library.
 */
typedef struct zc_plan_s* zc_plan_t;

/* Create a plan on the current device.  Host-side and synchronous: copies the
 * segment table to device memory the plan allocates (about 64 bytes per
 * segment).  Not stream-ordered; call it once per layout. */
int zc_plan_create(uint64_t n, const uint64_t* h_seg_off, uint32_t nseg,
                   uint32_t chunk_elems, zc_plan_t* out_plan);

/* Free a plan (waits for nothing: the caller must make sure no enqueued
 * work still uses it, e.g. by synchronising the streams it was used on). */
void zc_plan_destroy(zc_plan_t plan);

/* Workspace bytes zc_plan and zc_compress need for this plan. */
size_t zc_workspace_bytes(zc_plan_t plan);

/* Upper bound of the stream size for this plan: the fixed part plus, per
 * chunk, at most 5C/8 dynamic bytes (an incompressible full chunk is stored
 * raw: 2C bytes in all) and one escape per element of a short last chunk. */
uint64_t zc_max_compressed_bytes(zc_plan_t plan);

/* Statistics and codebooks, [ZipCCL] 2.A: per segment, the count, sum and
 * sum of squares of the finite values of d_x (n bf16 bit patterns), then
 * mu, sigma (population) and the 7 exponent fields with the largest Gaussian
 * probability mass, into the plan's device tables.  Enqueues two kernels. */
int zc_plan(zc_plan_t plan, const uint16_t* d_x, void* d_ws, size_t ws_bytes,
            zc_stream_t stream);

/* Replace the plan's codebooks with h_books (7 fields per segment, strictly
 * ascending).  Synchronous copy.  Lets a caller reuse a known codebook. */
int zc_plan_set_books(zc_plan_t plan, const uint8_t* h_books);

/* Copy the plan's codebooks (7*nseg bytes) and/or mu, sigma (2*nseg doubles,
 * interleaved) to the host; either pointer may be NULL.  Synchronises
 * `stream` (the stream zc_plan ran on) first, then copies. */
int zc_plan_info(zc_plan_t plan, zc_stream_t stream, uint8_t* h_books,
                 double* h_mu_sigma);

/* Encode d_x (n bf16 bit patterns, the plan's layout) into a ZCC1 stream at
 * d_out ([ZipCCL] 2.B-2.D).  out_cap must cover at least the fixed part of
 * the stream (header, tables and slots); escapes that do not fit set
 * ZC_ERR_CAPACITY in the status word.  *d_out_bytes (device, may be NULL)
 * receives the stream size.  One memset and one kernel on the stream. */
int zc_compress(zc_plan_t plan, const uint16_t* d_x, void* d_out,
                uint64_t out_cap, uint64_t* d_out_bytes, void* d_ws,
                size_t ws_bytes, zc_stream_t stream);

/* zc_compress and the statistics of zc_plan from one read of d_x: the
 * stream is the one zc_compress writes with the plan's codebooks as they are
 * when the call starts; from the same loads the encoder sums each chunk's
 * finite values and their squares, and a second kernel then replaces the
 * plan's mu, sigma and codebooks with those of d_x ([ZipCCL] 2.A: the
 * codebook comes from sigma, with no separate statistics pass) -- ready for
 * the next call, as when consecutive tensors of a training run keep their
 * distribution.  The sums are fp32 (sum, error) pairs of per-lane partial
 * sums, so mu and sigma agree with zc_plan's to a few fp32 units in the last
 * place and the codebooks are the same except at a near-tie.  Workspace:
 * zc_workspace_bytes.  One memset, two kernels. */
int zc_compress_fit(zc_plan_t plan, const uint16_t* d_x, void* d_out,
                    uint64_t out_cap, uint64_t* d_out_bytes, void* d_ws,
                    size_t ws_bytes, zc_stream_t stream);

/* zc_compress without a workspace.  The ZipCCL pages have no counterpart:
 * this is an interface for callers that cannot allocate at the point where
 * they compress -- e.g. a communication library's progress thread, where a
 * cudaMalloc would synchronise the device and stall transfers in flight, or
 * a program whose device memory is all held by a pool it cannot reach from
 * here -- and so cannot size or keep a workspace.  The encoder's scratch
 * (status block and look-back words) is instead a fixed 1 MiB array in
 * device memory owned by the library, which limits the plan to 130,024 tiles
 * of 8192 slots (1,065,156,608 slots, chunk padding included); a larger plan
 * returns ZC_ERR_CAPACITY.  Nothing is allocated by this call (the plan
 * itself was allocated by zc_plan_create).
 *
 * Arguments, layout and the stream bytes are those of zc_compress.  d_status
 * (device, 4-byte aligned, may be NULL) receives the status word
 * (ZC_OK or a ZC_ERR_* code) once the kernel is done.  Enqueues one memset,
 * the encode kernel and a 4-byte device copy on `stream`.
 *
 * Each call made outside a stream capture looks up the array's address on
 * the current device (a device reset reloads the library and may move it); a
 * call during a capture uses the address the last such call found, so make
 * one call on the device before any stream capture.  All calls on a device
 * share the one array: calls whose GPU work overlaps (other streams, other
 * threads) race and corrupt each other's streams, so order them on one
 * stream or with events. */
int zc_compress_static(zc_plan_t plan, const uint16_t* d_x, void* d_out,
                       uint64_t out_cap, uint64_t* d_out_bytes, int* d_status,
                       zc_stream_t stream);

/* Workspace bytes zc_decompress needs (a constant). */
size_t zc_decompress_workspace_bytes(void);

/* Decode the ZCC1 stream at d_in (in_bytes readable) into d_y (room for
 * y_cap_elems bf16).  The stream is validated on the device; any
 * inconsistency sets ZC_ERR_FORMAT (or ZC_ERR_CAPACITY when y is too small)
 * in the status word and nothing is written past what was checked.
 * One memset and one kernel on the stream. */
int zc_decompress(const void* d_in, uint64_t in_bytes, uint16_t* d_y,
                  uint64_t y_cap_elems, void* d_ws, size_t ws_bytes,
                  zc_stream_t stream);

/* ======================================================== IBP
 *
 * Chunks are chunk_bytes long (any multiple of 4, 4..4096: multiples of 16
 * up to 2048 run on the TMA-pipelined kernels, the rest on word-granular
 * ones); the last chunk of an input may be shorter (a multiple of 4 bytes)
 * and is stored raw.
 */

/* Size of an IBPM metadata blob: 64 + 2*chunk_bytes. */
uint64_t ibp_meta_bytes(uint32_t chunk_bytes);

/* Workspace bytes for ibp_build_meta (n_samples chunks), ibp_compress and
 * ibp_decompress (n_bytes of uncompressed data). */
size_t ibp_workspace_bytes(uint32_t chunk_bytes, uint64_t n_bytes,
                           uint64_t n_samples);

/* Upper bound of the IBP1 stream size for n_bytes of input. */
uint64_t ibp_max_compressed_bytes(uint32_t chunk_bytes, uint64_t n_bytes);

/* [IBP] step 1: count the ones at every bit position over the n_samples
 * chunks at d_samples (laid end to end), then write the IBPM blob to d_meta
 * (ibp_meta_bytes(chunk_bytes), device): position j is invariant when at
 * least k = ceil(T * n_samples) samples agree on it, T in (0.5, 1].
 * mode 0: every such position (the page's per-position rule);
 * mode 1: joint -- positions are taken most-agreeing first (ties: lower
 * position) while at least k samples still match every taken position
 * (chunk_bytes <= 2048 in this mode). */
int ibp_build_meta(const void* d_samples, uint64_t n_samples,
                   uint32_t chunk_bytes, double T, int mode, void* d_meta,
                   void* d_ws, size_t ws_bytes, zc_stream_t stream);

/* [IBP] step 2: encode n_bytes (multiple of 4) at d_x into an IBP1 stream at
 * d_out using the metadata at d_meta (its chunk size must be chunk_bytes;
 * checked on the device).  *d_out_bytes (device, may be NULL) receives the
 * stream size; a stream larger than out_cap sets ZC_ERR_CAPACITY and nothing
 * is written past out_cap.  For chunk_bytes <= 512 (multiples of 16): one
 * memset and one cooperative kernel that reads the input from device memory
 * once (tiles are matched, their stream lengths published in the workspace
 * and their offsets resolved a few tiles later, while the input is still in
 * L2); if the driver cannot place its whole grid at once, the three kernels
 * below instead.  For chunk_bytes 1024 and 2048 the same, with a whole group
 * per tile moved through shared memory 16 KB at a time (the workspace holds
 * one stream length per group).  For the other chunk_bytes <= 2048: one
 * memset and three kernels (a read-only pass that decides every
 * chunk's participation bit, a scan of the group lengths into the stream's
 * group-offset table, the packing pass); the workspace holds one
 * participation word per group between them.  Larger chunks: one memset and
 * one kernel.  The workspace size is ibp_workspace_bytes().  With a
 * host-resident d_x or d_out (see below) the single-kernel encoder runs.
 * d_x and d_out may be pinned host
 * memory ([IBP] Algoritmo Core step 2: the GPU compresses through zero-copy
 * unified memory); a host-resident d_x is read with plain loads by the
 * single-kernel encoder.  Other host memory returns ZC_ERR_ARG. */
int ibp_compress(const void* d_meta, uint32_t chunk_bytes, const void* d_x,
                 uint64_t n_bytes, void* d_out, uint64_t out_cap,
                 uint64_t* d_out_bytes, void* d_ws, size_t ws_bytes,
                 zc_stream_t stream);

/* [IBP] step 3: decode the IBP1 stream at d_in into d_y (y_cap bytes).  A
 * stream made with other metadata sets ZC_ERR_META_MISMATCH.  d_in may be
 * device memory or pinned host memory (cudaHostAlloc / cudaHostRegister): a
 * host-resident stream is read in place over the host link, as in [IBP]
 * Algoritmo Core step 3 (warps read the compressed segment from CPU memory)
 * and Integrazione del Sistema (tensors kept compressed in CPU memory), with
 * no separate copy.  d_y may be pinned host memory too.  Other host memory
 * returns ZC_ERR_ARG.  d_meta and d_ws are device memory. */
int ibp_decompress(const void* d_meta, uint32_t chunk_bytes, const void* d_in,
                   uint64_t in_bytes, void* d_y, uint64_t y_cap, void* d_ws,
                   size_t ws_bytes, zc_stream_t stream);

/* ======================================================== IBP in-place slots
 *
 * [IBP] Integrazione del Sistema (PCIe transfer compression): tensors are
 * compressed in CPU memory before they are transferred; a compressed tensor
 * stays in place in a buffer of fixed size, of which only the compressed
 * part is read, and a bitmask in GPU memory records which tensors are
 * compressed.  Here a tensor is one chunk: chunk s of the data owns the slot
 * of chunk_bytes at d_slots + s * chunk_bytes (the last slot is as long as
 * the last chunk, a multiple of 4 bytes).  A compressed slot -- the chunk's
 * participation bit of [IBP] step 2 is set -- starts with the chunk's body
 * (its B - m kept bits in ascending position order, LSB first, zero bits up
 * to a whole 32-bit word: 4*ceil((B - m)/32) bytes) and its later bytes are
 * not written; every other slot holds the raw chunk.  Bit s % 32 of
 * d_bitmask word s / 32 is set when slot s is compressed (the same bits as
 * the IBP1 stream's group participation words).
 */

/* Write the slot form of the n_bytes (a multiple of 4) at d_x into d_slots
 * (n_bytes long; d_x may be d_slots itself: compression in place, each chunk
 * read whole before its slot is written; otherwise the two must not overlap)
 * and the bitmask into d_bitmask (ceil(ceil(n_bytes/chunk_bytes)/32) words,
 * device memory).  d_x and d_slots may be pinned host memory, read and
 * written in place over the host link ([IBP] step 2: the GPU compresses
 * through zero-copy access to CPU memory); other host memory returns
 * ZC_ERR_ARG.  4-byte alignment.  d_ws: 256 bytes (status word).  One memset
 * and one kernel; metadata made for another chunk size sets
 * ZC_ERR_META_MISMATCH. */
int ibp_slots_compress(const void* d_meta, uint32_t chunk_bytes, const void* d_x,
                       uint64_t n_bytes, void* d_slots, uint32_t* d_bitmask,
                       void* d_ws, size_t ws_bytes, zc_stream_t stream);

/* Gather: row i of d_y (chunk_bytes each; a short last chunk fills only its
 * length) receives chunk d_idx[i] (u64 slot indices, device memory, any
 * order, repeats allowed), read from its slot -- only the slot's stored part
 * -- and decoded ([IBP] step 3: a warp reads the segment from CPU memory into
 * shared memory and puts the Bitval bits back).  d_slots may be pinned host
 * memory; d_y device or pinned host memory.  *d_read_bytes (device, may be
 * NULL) receives the bytes read from the slots.  An index past the last
 * chunk sets ZC_ERR_ARG in the status word and its row is not written; a set
 * bit on a slot that cannot hold a body (the short last one, or m = 0) sets
 * ZC_ERR_FORMAT.  Up to two memsets and one kernel. */
int ibp_slots_gather(const void* d_meta, uint32_t chunk_bytes, const void* d_slots,
                     uint64_t n_bytes, const uint32_t* d_bitmask, const uint64_t* d_idx,
                     uint64_t n_idx, void* d_y, uint64_t* d_read_bytes, void* d_ws,
                     size_t ws_bytes, zc_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* LBB16_ZC_H */
