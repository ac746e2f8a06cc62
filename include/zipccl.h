/*
 * zipccl.h -- C ABI of the GB300 (sm_103a) ZipCCL BF16 exponent-coding path.
 *
 * The operations follow "ZipCCL: Efficient Lossless Data Compression of
 * Communication Collectives for Accelerating LLM Training":
 *   - abstract, technique (1) and the shd-paper summary's key design: BF16
 *     communication tensors are near-Gaussian, so the 8-bit exponent is
 *     entropy-coded with a code derived from the Gaussian density, with no
 *     online statistics;  Fig. 6 caption: sign and mantissa stay raw and a
 *     value shrinks to about 11 bits;
 *   - abstract, technique (2): GPU compressor/decompressor kernels with a
 *     communication-aware data layout -- here one self-contained compressed
 *     chunk per destination rank, back to back in one buffer;
 *   - Fig. 3 and Fig. 5 captions: the receive side of zipcclReduceScatter
 *     decompresses the peers' chunks and reduces them.
 * The stream format (v1) is defined by this library; the pages fix none.
 *
 * Conventions for every call:
 *   - Pointers named d_* are device memory on the current CUDA device, owned
 *     by the caller.  The library allocates and frees nothing on the device.
 *   - d_* base pointers must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void*.  Calls are asynchronous and
 *     stream-ordered; they never synchronize unless the name says so.
 *   - Argument errors are returned synchronously, before any launch.
 *   - Data-dependent errors (a corrupt stream, a look-back that timed out)
 *     are recorded by the kernels in a status word at the start of the
 *     workspace; zipccl_get_device_status reads it and reports the last
 *     call made on that workspace, so read it after the call you want to
 *     check.  A compress call clears it first; a decompress or
 *     decompress_reduce call does not clear anything but tags its errors
 *     with a 56-bit number of its own, so that an earlier call's code (or
 *     whatever the memory held) never reads as its status.  No
 *     initialisation of a workspace is needed.  On such an error outputs
 *     are undefined but every access stays inside the caller's buffers.
 *   - A workspace must not be shared by calls that may run concurrently.
 */
#ifndef ZIPCCL_H
#define ZIPCCL_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZIPCCL_OK = 0,
    ZIPCCL_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, sum mismatch */
    ZIPCCL_ERR_CAPACITY = 2,    /* output or workspace smaller than required */
    ZIPCCL_ERR_CORRUPT = 3,     /* stream fails validation (device status) */
    ZIPCCL_ERR_VERSION = 4,     /* stream written by another format version */
    ZIPCCL_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (device status) */
    ZIPCCL_ERR_CUDA = 6         /* a CUDA runtime call failed */
} zipccl_status;

/* Format version written and read by this library (1). */
int zipccl_format_version(void);

/* Static, human-readable name of a status code. */
const char *zipccl_status_string(int status);

/*
 * Passage: abstract, technique (3) (collectives fall back to uncompressed
 * operation) -- read as a per-tile raw fallback, so the expansion is bounded.
 * Exact worst-case compressed size of a chunk layout: every tile stored with
 * raw exponents (bounded expansion).  chunk_elems: host array of n_chunks
 * element counts.  *out_bytes receives the bound.  Host only.
 */
zipccl_status zipccl_max_compressed_bytes(const uint64_t *chunk_elems, uint32_t n_chunks,
                                          uint64_t *out_bytes);

/*
 * Workspace sizes, one call per operation (each sizes only what its kernels
 * use): compress needs per-chunk code tables and per-tile records, the
 * decoders per-chunk decode tables.  Host only.
 */
/* Workspace bytes needed by zipccl_compress for this chunk layout. */
zipccl_status zipccl_compress_workspace_bytes(const uint64_t *chunk_elems, uint32_t n_chunks,
                                              uint64_t *out_bytes);

/* Workspace bytes needed by zipccl_decompress for n elements in n_chunks chunks. */
zipccl_status zipccl_decompress_workspace_bytes(uint64_t n, uint32_t n_chunks, uint64_t *out_bytes);

/* Workspace bytes needed by zipccl_decompress_reduce for k peers. */
zipccl_status zipccl_reduce_workspace_bytes(uint32_t k, uint64_t *out_bytes);

/*
 * Passages: abstract, technique (1) (exponent coding from the Gaussian law,
 * no expensive online statistics) and technique (2) (GPU compressor with a
 * communication-aware data layout); shd-paper key-design paragraph
 * (frequent exponents get short codes); Fig. 6 caption (about 11 bits per
 * value: sign and mantissa raw).
 * Compress n BF16 words (d_in, bit patterns as uint16) split into n_chunks
 * per-destination chunks: chunk c is the next chunk_elems[c] words (host
 * array, sum == n, n_chunks >= 1, each chunk < 2^31 words; empty chunks are
 * allowed and produce a header-only chunk).
 * sigma_hint: host array of n_chunks floats or NULL.  A value > 0 fixes the
 * Gaussian scale of that chunk's code; otherwise the scale is taken from a
 * fixed sample of the chunk's exponents (no histogram pass).
 * d_out receives the chunks back to back, each a self-contained stream that
 * can be sent alone; out_capacity must be >= zipccl_max_compressed_bytes.
 * d_chunk_offsets (device, n_chunks + 1 uint64) receives each chunk's byte
 * offset in d_out and, last, the total size.  d_ws: workspace of at least
 * zipccl_compress_workspace_bytes bytes.
 * The tiles are coded by one persistent kernel whose CTAs (one per SM) must
 * all be resident at once, so it is issued as a cooperative launch; where the
 * device or context cannot make that launch the call returns ZIPCCL_ERR_CUDA.
 * The first call on a device sets the kernel's shared-memory limit and reads
 * its occupancy; later calls reuse them.
 */
zipccl_status zipccl_compress(const uint16_t *d_in, uint64_t n, const uint64_t *chunk_elems,
                              uint32_t n_chunks, const float *sigma_hint, void *d_out,
                              uint64_t out_capacity, uint64_t *d_chunk_offsets, void *d_ws,
                              uint64_t ws_bytes, void *stream);

/*
 * Passages: abstract (the compressor and decompressor kernels overlap
 * compression with memory access through a pipeline); Fig. 5 caption
 * (minimize kernel launch overhead, overlap compression with memory access);
 * abstract, technique (2) (communication-aware layout: one chunk per
 * destination rank).
 * zipccl_compress that also writes every chunk into d_send, the buffer a
 * transport would send from, and posts each chunk as soon as it is complete
 * while later chunks are still being coded.  In the same kernel: each tile's
 * image leaves shared memory by two TMA stores, one to d_out and one to the
 * same offset in d_send (the send costs HBM writes, no reads); the store
 * warps count the stored tiles of each chunk (release at GPU scope); one
 * warp in the first CTA, the stand-in for the proxy that hands chunks to
 * the network, waits for each chunk's count in chunk order (acquire, bounded
 * by 2 s) and posts it: it writes %globaltimer into d_chunk_ready[c].
 * d_chunk_ready[n_chunks] receives the kernel's start on the same clock.
 * The exchange itself is outside this library.
 *   d_send: device, 16-byte aligned, not d_out, send_capacity >=
 *     zipccl_max_compressed_bytes; afterwards d_send[0, offsets[n_chunks])
 *     equals d_out over the same range.
 *   d_chunk_ready: device, n_chunks + 1 uint64, 8-byte aligned, or NULL.
 * A wait that gives up records ZIPCCL_ERR_TIMEOUT; an error of the coding
 * warps ends the posting; read either with zipccl_get_device_status.  Other
 * arguments as zipccl_compress.
 */
zipccl_status zipccl_compress_send(const uint16_t *d_in, uint64_t n, const uint64_t *chunk_elems,
                                   uint32_t n_chunks, const float *sigma_hint, void *d_out,
                                   uint64_t out_capacity, uint64_t *d_chunk_offsets, void *d_send,
                                   uint64_t send_capacity, uint64_t *d_chunk_ready, void *d_ws,
                                   uint64_t ws_bytes, void *stream);

/*
 * Passages: Fig. 6 caption (the decompressor restores each value from its
 * raw sign/mantissa byte and its decoded exponent); pith summary (lossless:
 * every byte restored).
 * Decompress n_chunks chunks from d_stream into n BF16 words at d_out,
 * bit-identical to the compressed input.  d_chunk_offsets (device,
 * n_chunks + 1) are the offsets compress wrote; the stream must hold
 * d_chunk_offsets[n_chunks] bytes.  The chunks' element counts are read from
 * their headers and must sum to n (else ZIPCCL_ERR_CORRUPT in the device
 * status).  d_ws: at least zipccl_decompress_workspace_bytes bytes.
 */
zipccl_status zipccl_decompress(const void *d_stream, const uint64_t *d_chunk_offsets,
                                uint32_t n_chunks, uint16_t *d_out, uint64_t n, void *d_ws,
                                uint64_t ws_bytes, void *stream);

/*
 * Passages: Fig. 3 and Fig. 5 captions (zipcclReduceScatter: the receiver
 * decompresses the peers' chunks and reduces them).
 * Receive side of a reduce-scatter: d_peer_chunks is a host array of k
 * (1 <= k <= 16) device pointers, in rank order, each to one compressed
 * chunk of n elements and peer_chunk_bytes[p] bytes (host array; every read
 * of peer p stays inside those bytes, so a truncated or corrupt chunk gives
 * ZIPCCL_ERR_CORRUPT instead of a read past it).
 * d_out[i] = bf16_rne(((x0[i] + x1[i]) + x2[i]) ... + x_{k-1}[i]) with every
 * addition in fp32 (round to nearest even, subnormals kept); a NaN result is
 * written as 0x7FC0.  d_ws: at least zipccl_reduce_workspace_bytes bytes.
 */
zipccl_status zipccl_decompress_reduce(const void *const *d_peer_chunks,
                                       const uint64_t *peer_chunk_bytes, uint32_t k, uint64_t n,
                                       uint16_t *d_out, void *d_ws, uint64_t ws_bytes,
                                       void *stream);

/*
 * Passages: none; this call has no counterpart in the paper.
 * zipccl_decompress_reduce for callers that may not allocate device memory
 * at the point of the call: code that runs inside a device allocator's own
 * hook or callback (allocating there would re-enter the allocator), and
 * processes whose device memory is all reserved up front by a caching
 * allocator, where a new allocation would fail or force the cache to be
 * emptied.  Same kernels, same results; the workspace is a scratch area
 * compiled into this library (one per device) instead of a caller buffer, and
 * no call allocates or frees anything.  The paper has no counterpart to this
 * call: it serves only such callers.
 *   - The scratch holds ZIPCCL_NOALLOC_SCRATCH_BYTES bytes per device, the
 *     workspace of k = ZIPCCL_NOALLOC_MAX_PEERS (16) peers.  k == 0 or
 *     k > 16 returns ZIPCCL_ERR_INVALID_ARG before anything is launched.
 *   - The first call on a device, made with that device current, does a
 *     one-time set-up: it looks up the scratch's device address, which may
 *     load this library's kernels onto the device.  Make that first call
 *     before any stream capture begins.  A failed lookup returns
 *     ZIPCCL_ERR_CUDA.  The address is kept for the life of the process:
 *     do not call this after cudaDeviceReset on that device, or from a
 *     context other than the device's primary context; the library's module,
 *     and the scratch with it, may then sit at another address.
 *   - Each call first clears the scratch's 256-byte status header on
 *     `stream` (cudaMemsetAsync); the rest of the scratch is written before
 *     it is read, so nothing else must start at zero.
 *   - One scratch per device is shared by every call on that device: calls
 *     that may overlap (other streams, host threads, or processes sharing the
 *     context) race on it and must be ordered by the caller, e.g. on one
 *     stream.
 *   - d_scratch (may be NULL) receives the scratch's device address; pass it
 *     to zipccl_get_device_status to read the device status of the call.
 */
#define ZIPCCL_NOALLOC_MAX_PEERS 16
#define ZIPCCL_NOALLOC_SCRATCH_BYTES (256u + 1024u + 16u * 4096u)
zipccl_status zipccl_decompress_reduce_noalloc(const void *const *d_peer_chunks,
                                               const uint64_t *peer_chunk_bytes, uint32_t k,
                                               uint64_t n, uint16_t *d_out, void **d_scratch,
                                               void *stream);

/*
 * Synchronizes `stream`, then returns the status the kernels of the last call
 * on this workspace recorded (ZIPCCL_OK, ZIPCCL_ERR_CORRUPT,
 * ZIPCCL_ERR_VERSION, ZIPCCL_ERR_TIMEOUT), or ZIPCCL_ERR_CUDA.
 */
zipccl_status zipccl_get_device_status(const void *d_ws, void *stream);

/*
 * Self-test of the bounded device waits: which = 0 runs the compressor's
 * look-back for a tile whose predecessor never publishes its state; which =
 * 1 waits for an mbarrier phase that never completes (the wait used for the
 * decoders' payload copies); which = 2 runs the compress-and-send sender's
 * wait for a chunk whose tiles are never stored (no encoder runs).  The wait
 * gives up after its limit (2 s) and the kernel records ZIPCCL_ERR_TIMEOUT
 * in the workspace status, read with zipccl_get_device_status; nothing
 * faults and the context stays usable.  d_ws: 256-byte aligned, at least
 * 272 bytes (which 0, 1) or 336 bytes (which 2).  Asynchronous on `stream`.
 */
zipccl_status zipccl_selftest_bounded_wait(int which, void *d_ws, uint64_t ws_bytes, void *stream);

/*
 * Measurement hook, for timing the encode kernel on its own.  While a pair
 * of events is set, every zipccl_compress and zipccl_compress_send call
 * records ev_before (a cudaEvent_t) on its stream immediately before it
 * launches its encode kernel and ev_after immediately after, so that
 * cudaEventElapsedTime(ev_before, ev_after) is that kernel's duration (the
 * select kernel before it excluded).  The events belong to the caller, who
 * creates them with timing enabled; two NULLs turn the hook off.  One NULL
 * and one event: ZIPCCL_ERR_INVALID_ARG.  The setting is process-wide and
 * meant for a benchmark driving calls from one host thread.
 */
zipccl_status zipccl_profile_encode_events(void *ev_before, void *ev_after);

/*
 * Cost model of the switch between compressed and plain exchange ("ZipCCL:
 * Efficient Lossless Data Compression of Communication Collectives for
 * Accelerating LLM Training", abstract, technique (3): collectives switch
 * between compressed and uncompressed operation from workload and system
 * characteristics).  Host only; nothing is launched.
 *
 * zipccl_predict_chunk_bytes: the size in bytes of the stream of one chunk
 * of n values drawn from N(0, sigma^2) and compressed with a sigma hint of
 * `sigma`: the format's header, tile table and tile headers, the raw
 * sign/mantissa plane, and per tile an exponent region of
 * ceil(n_t * E / 32) words plus the segment table, E being the expected code
 * bits of one exponent under that code (closed-form masses); raw exponent
 * bytes where those are not larger.  out_bits_per_value (nullable): 8 x
 * bytes / n.  sigma <= 0, not finite, or n above the per-chunk limit give
 * ZIPCCL_ERR_INVALID_ARG.
 *
 * zipccl_choose_compressed: with link, compress and decompress throughputs
 * in GB/s of their input, sending n values raw takes 2n / link; compressed,
 * 2n / compress + bytes / link + 2n / decompress (stages in sequence, bytes
 * as predicted above).  *use_compressed = 1 when raw time / compressed time
 * > 1 + margin; predicted_speedup (nullable) receives that ratio.
 * Non-positive throughputs or a negative margin give ZIPCCL_ERR_INVALID_ARG.
 */
zipccl_status zipccl_predict_chunk_bytes(uint64_t n, float sigma, uint64_t *out_bytes, double *out_bits_per_value);
zipccl_status zipccl_choose_compressed(uint64_t n, float sigma, double link_gbs, double compress_gbs,
                                       double decompress_gbs, double margin, int *use_compressed,
                                       double *predicted_speedup);

/*
 * The code this library uses for scale phase r = q mod 16 (0..15), frozen
 * in format v1: the window start relative to floor(q/16) + 127 and the 16
 * code lengths (symbols 0..14 = window exponents, 15 = escape).  Host only.
 */
zipccl_status zipccl_codebook_phase(int phase, int *base_offset, uint8_t *lens16);

/*
 * Passages: abstract, technique (1); shd-paper key-design paragraph (the
 * code comes from the Gaussian density).
 * The same table as zipccl_codebook_phase, derived again from the
 * closed-form masses at sigma = 2^(phase/16) (exact dynamic program over
 * Kraft sums, libm erf/erfc).  The library codes only with the frozen
 * tables of format v1; this call lets a test check that they still equal
 * their derivation.  Host only.
 */
zipccl_status zipccl_codebook_rebuild_phase(int phase, int *base_offset, uint8_t *lens16);

#ifdef __cplusplus
}
#endif

#endif /* ZIPCCL_H */
