/*
 * zc.h -- C ABI of the GB300 lossless BF16 exponent codec.
 *
 * The operation is the exponent coding of "ZipCCL: Efficient Lossless Data Compression of
 * Communication Collectives for Accelerating LLM Training" (SIGCOMM scribe notes), section
 * "Key idea and contribution", first technique: the frequent-exponent window is taken
 * directly from the tensor's standard deviation (no histogram, no sort), in-window exponents
 * are stored in 3 bits instead of 8, out-of-window exponents keep their full 8 bits in a
 * separate store so that reconstruction is exact, and sign and mantissa travel unchanged --
 * about 11 bits per value instead of 16.  The separate store of a chunk is a list of
 * (position, exponent) pairs, or, when more than a third of the chunk escapes, a plane of all
 * its exponents, whichever is smaller (the same section's third technique switches to the
 * uncompressed form where coding does not pay).  The second technique of the same section
 * (kernels tuned for the GPU: a layout shaped by the communication, aligned global and shared
 * memory access, data movement pipelined with compute) is what the
 * kernels behind these calls implement for sm_103a.
 *
 * Stream format "ZCB1", version 4 (little-endian, every section zero-padded to 16 bytes):
 *   header    32 B  "ZCB1", u16 version = 4, u8 form, u8 e0, u64 n, u64 N, u64 total_bytes.
 *             form = 12 (log2 of the chunk size) for the coded form, 0 for the raw form.
 * Coded form (N = ceil(n / 4096) chunks):
 *   offsets   u64[N+1]: absolute byte offset of each chunk's escape section; offsets[N] =
 *             total_bytes.  Zero padding to R0 = pad16(32 + 8 (N+1)).
 *   fixed     for chunk c (m values), at R0 + 5632 c: 3-bit codes, code i at bits [3i, 3i+3)
 *             least significant bit first (pad16(ceil(3m/8)) B), then one sign|mantissa byte
 *             per value, (x >> 8 & 0x80) | (x & 0x7F) (pad16(m) B).  The place of every fixed
 *             part follows from n alone (a layout shaped by the communication: it can be sent
 *             before any size is exchanged).
 *   escapes   after the last fixed part, in chunk order, one section per chunk.  For a chunk
 *             of m values with k escapes (k = the number of code-7 values): if 3k <= m, u16
 *             positions then u8 full exponents in ascending position order (pad16(3k) B);
 *             otherwise the u8 exponents of all m values in value order (pad16(m) B).
 *   Code c < 7 means exponent e0 + c; code 7 means "escape".  e0 is in [0, 249].
 * Raw form (N = 0): the n values as they are (2n B), zero padding; total_bytes =
 *   32 + pad16(2n).  A tensor whose coded form would be longer than its raw form is stored raw
 *   (the same section's third technique switches a transfer to the native path where
 *   compressing does not pay); ties keep the coded form.  So no stream is longer than its
 *   values plus 32 bytes (and 15 of padding).
 * A full chunk without escapes costs 5632 B for 4096 values: 11 bits per value.  A full coded
 * chunk costs at most 9728 B (a plane), but a coded stream is never longer than the raw form.
 *
 * All entry points are host functions.  Pointers called "device" may be any address the GPU
 * can dereference (cudaMalloc, managed, or mapped pinned memory).  Every call is
 * asynchronous in the order of `stream` and never synchronizes, except where stated.
 */
#ifndef ZC_H
#define ZC_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* cudaStream_t; /* the CUDA runtime's own stream handle type */

/* ------------------------------------------------------------------ status codes */
#define ZC_OK 0
#define ZC_ERR_INVALID_ARG 1   /* null pointer, base outside [0,249] and not ZC_BASE_AUTO,
                                  n > ZC_MAX_N, overlapping buffers                        */
#define ZC_ERR_MISALIGNED 2    /* in/out not 16-byte aligned, out_bytes not 8-byte aligned  */
#define ZC_ERR_CUDA 3          /* a CUDA runtime call or a launch failed                    */
#define ZC_ERR_CORRUPT 4       /* device-side: the stream is not one the encoder writes     */
#define ZC_ERR_SIZE_MISMATCH 5 /* device-side: the stream holds a different n               */
#define ZC_ERR_TIMEOUT 6       /* device-side: a bounded wait inside a kernel ran out       */

#define ZC_BASE_AUTO (-1)               /* choose the window base from the data */
#define ZC_MAX_N ((size_t)1 << 40)      /* largest supported number of values   */
#define ZC_CHUNK_VALUES 4096

/* ------------------------------------------------------------------ sizes */

/* Bytes the caller must provide at `out` for zc_compress of n values: zc_max_stream_bytes(n),
 * rounded up to 256, followed by the call's workspace (scan state, 8 B per chunk, and a
 * 16.25 KiB control block).  Pure host function; makes no CUDA call.  Returns 0 when
 * n > ZC_MAX_N. */
size_t zc_max_compressed_bytes(size_t n);

/* Bytes of `out` that the stream may occupy while it is written: the larger of the raw form's
 * length, 32 + pad16(2n) (no stream is longer), and the end of the coded fixed parts, which
 * are written before the form is known (larger only for n below about 100).  Pure host
 * function.  Returns 0 when n > ZC_MAX_N. */
size_t zc_max_stream_bytes(size_t n);

/* ------------------------------------------------------------------ compress */

/* Compress n BF16 values (raw bit patterns) into one "ZCB1" stream.
 *   in            device, n x u16, 16-byte aligned, read only.
 *   n             number of values, 0 <= n <= ZC_MAX_N.  n = 0 gives a 32-byte (raw) stream.
 *   base_or_auto  ZC_BASE_AUTO: e0 = floor(log2(sigma * c)) + 127 clamped to [0, 249], with
 *                 sigma the root mean square of the finite values and c^2 =
 *                 0x1.79a1e790e0f01p-10 (the window with the fewest expected escapes for a
 *                 Gaussian: the window comes from the standard deviation alone, with no
 *                 histogram or sort).  0..249: use that e0.  The stream depends only on
 *                 (input bits, e0): both modes give identical bytes for the same e0.
 *   out           device, zc_max_compressed_bytes(n) bytes, 16-byte aligned, must not overlap
 *                 `in`.  The stream is written from out[0]: the coded form, or the raw form
 *                 when that is shorter.  The form is decided on the device from the coded
 *                 form's exact length, with no host synchronization.  A tensor of up to 2^25
 *                 values compresses in one launch (a thread-block cluster or a cooperative
 *                 grid, every CTA resident from the start), which knows every chunk's escape
 *                 count before it writes a section.  A larger one runs the encode kernel; in
 *                 auto mode that kernel first guesses e0 from a 4096-value sample, codes with
 *                 the guess and checks it against the rule on the whole tensor's sum of
 *                 squares, which it takes while coding (the input is read once).  When the
 *                 sample is not trusted or the guess does not hold, a statistics kernel and the
 *                 encode kernel run again after it (they return at once otherwise): the form is
 *                 then decided after the encoder's scan, or, when an exponent sample of the
 *                 statistics pass predicts a raw stream, by a pass that counts every chunk's
 *                 escapes while it copies the values to the raw form.  The bytes past
 *                 *out_bytes, including the workspace tail, are unspecified afterwards.  The
 *                 library keeps no per-call state outside `out`, so calls on different streams
 *                 with different buffers may run concurrently.  The encode kernel's CTAs wait
 *                 on one another (bounded) only for work that a CTA already running has taken,
 *                 so a concurrent kernel that delays some of them slows the call but does not
 *                 make it fail.  The host picks the route from n and base_or_auto alone and
 *                 the kernels reset their own state, so a call whose out_bytes is not pageable
 *                 can be captured in a CUDA graph (after a first call on the device, which loads
 *                 the kernels) and replayed on new contents of the same buffers.
 *   out_bytes     receives the stream length.  Device, managed or pinned host memory is
 *                 written by the last kernel (asynchronously).  Pageable host memory is also
 *                 accepted: the call then copies the length back and synchronizes `stream`.
 * The chosen e0 is byte 7 of the stream.  Returns ZC_OK or a host-side error code
 * (ZC_ERR_INVALID_ARG, ZC_ERR_MISALIGNED, ZC_ERR_CUDA); device-side errors
 * (ZC_ERR_TIMEOUT) are reported through zc_status. */
int zc_compress(const void* in, size_t n, int base_or_auto, void* out, size_t* out_bytes,
                cudaStream_t stream);

/* ------------------------------------------------------------------ decompress */

/* Decompress a "ZCB1" stream back into n BF16 bit patterns (the exact input of compress).
 *   in      device, 16-byte aligned.  The kernel first reads the 32-byte header and checks it
 *           against n: magic, version, base, n, N, and the start of the escape region (a
 *           function of n alone) <= total_bytes (header bytes 24..31) <= the largest stream n
 *           values can produce.  Only after that check
 *           does it read further, and every later read lies inside [0, total_bytes): offsets and
 *           section sizes are checked against the header and against each other before use.
 *           So `in` must hold max(32, total_bytes) readable bytes; a wrong n or a short
 *           total_bytes is reported, never read past.
 *   out     device, n x u16, 16-byte aligned, must not overlap `in`.
 *   n       the number of values the caller expects; a stream holding another n sets
 *           ZC_ERR_SIZE_MISMATCH.
 * Any stream the encoder could not have written (bad magic, version, form, base, offsets,
 * sizes, escape positions or exponents, nonzero padding, a coded stream longer than the raw
 * form) sets ZC_ERR_CORRUPT; `out` is then unspecified.  A raw stream is checked byte for byte
 * (header, length, padding), but whether its coded form would have been shorter is not
 * recomputed.  Device-side errors are read with zc_status. */
int zc_decompress(const void* in, void* out, size_t n, cudaStream_t stream);

/* ------------------------------------------------------------------ loopback pipeline */

/* Bytes the caller must provide at `out` for zc_loopback of n values: the longest coded form
 * (every chunk with a plane of exponents, 9,728 B per full chunk), since the loopback writes every
 * escape section before the stream's form is chosen, rounded up to 256, then the workspace.
 * Pure host function.  Returns 0 when n > ZC_MAX_N. */
size_t zc_loopback_bytes(size_t n);

/* Compress n values into a stream and decompress that stream into `values`, in one launch, as a
 * sender and a receiver on one GPU would: a chunk is decoded as soon as its own bytes are in the
 * stream -- its fixed part (whose place follows from n) and its escape section (once the
 * device-wide scan has placed it and it has been written) -- while later chunks are still being
 * coded.  This is the compress -> exchange sizes -> send -> decompress workflow of the same page
 * (Figure 5(b), Design-1) and UCCL-Zip's split-send pipeline (data transmissible as early as
 * possible, compression overlapped with the transfer), with the transfer taken out: the decoder
 * reads the stream where the encoder wrote it.
 *   in, n, base_or_auto, out_bytes, stream   as for zc_compress.
 *   out     device, zc_loopback_bytes(n) bytes, 16-byte aligned, not overlapping `in` or
 *           `values`; afterwards it holds the same stream zc_compress writes (the raw form when
 *           that is shorter, which is decided after the decoding, from the coded form).
 *   values  device, n x u16, 16-byte aligned: receives the decoded values, equal to `in`.
 * Returns ZC_OK or a host-side error code; device-side errors (a stream section that fails the
 * decoder's checks: ZC_ERR_CORRUPT; a bounded wait that ran out: ZC_ERR_TIMEOUT) are read with
 * zc_status.  The pages have no counterpart of this entry point as an interface. */
int zc_loopback(const void* in, size_t n, int base_or_auto, void* out, size_t* out_bytes, void* values,
                cudaStream_t stream);

/* ------------------------------------------------------------------ status */

/* Synchronize `stream`, then return the first device-side error recorded on the current
 * device since the last reset (ZC_OK if none).  The status word is shared by all streams of
 * the device; reset != 0 clears it.  Returns ZC_ERR_CUDA if the synchronization fails. */
int zc_status(cudaStream_t stream, int reset);

/* ------------------------------------------------------------------ kernel timing */

#define ZC_KERNEL_STATS 1
#define ZC_KERNEL_ENCODE 2
#define ZC_KERNEL_DECODE 3
#define ZC_KERNEL_RAW 4    /* the step that rewrites a stream in the raw form when that is shorter */
#define ZC_KERNEL_SMALL 5  /* the single launch that compresses a tensor of up to 64 chunks */
#define ZC_KERNEL_MEDIUM 6 /* the single cooperative launch that compresses a medium tensor */
#define ZC_KERNEL_FUSED 7  /* the single cooperative launch for a tensor of up to 2^25 values */
#define ZC_KERNEL_REFIT_STATS 8  /* larger tensors, auto mode: the statistics pass after the
                                    encode kernel's guess of e0 was not trusted or did not hold */
#define ZC_KERNEL_REFIT_ENCODE 9 /* ... and the encode kernel again, after it */

/* enable != 0: bracket every kernel the library launches from now on with CUDA events on the
 * kernel's own stream.  enable == 0: stop recording.  Returns ZC_OK or ZC_ERR_CUDA. */
int zc_timing_enable(int enable);

/* Wait for the recorded events, write up to `max` (kernel id, milliseconds) pairs, oldest
 * first, drop them from the record and return how many were written (negative ZC_ERR_CUDA on
 * failure).  Records beyond `max` are dropped too. */
int zc_timing_collect(int* kernel_ids, float* ms, int max);

/* ------------------------------------------------------------------ compress without allocation */

/* Largest n zc_compress_static_scratch accepts: its workspace must fit a fixed 2 MiB array. */
#define ZC_STATIC_SCRATCH_MAX_N ((size_t)1065222144)

/* zc_compress for callers that cannot allocate device memory, such as a communication layer
 * whose send buffers are registered once at exactly the worst-case stream size and that may
 * not call cudaMalloc on its progress path.  The paper has no counterpart: it is an interface
 * for such callers.
 * Arguments, stream and results are those of zc_compress, except:
 *   - `out` needs only zc_max_stream_bytes(n) bytes (about the size of the input): the
 *     call's workspace lives in a
 *     file-scope 2 MiB device array of the library instead of the tail of `out`.  That array
 *     exists on every GPU that loads the library until the process exits.
 *   - n > ZC_STATIC_SCRATCH_MAX_N returns ZC_ERR_INVALID_ARG.
 *   - The call allocates nothing (no cudaMalloc, no cudaFree, no allocating library call).
 *   - All calls on a device share the array; calls whose work overlaps on the GPU (for
 *     example on two streams running at the same time) corrupt each other, so order them
 *     (one stream, or events).  Each call clears the part of the array that must start at
 *     zero before its kernels run.
 *   - The first call on a device looks up the array's device address (once per device, with
 *     that device current); make that first call before any stream capture. */
int zc_compress_static_scratch(const void* in, size_t n, int base_or_auto, void* out, size_t* out_bytes,
                               cudaStream_t stream);

/* ------------------------------------------------------------------ test hook */

/* zc_compress with a planted stall, for testing the bounded waits: chunk `stalled_chunk` never
 * publishes its escape-list size, so the device-wide scan cannot pass it; the waits for it run
 * out after about `spin_limit` polls and the call reports ZC_ERR_TIMEOUT through zc_status
 * instead of hanging.  The stream written is then incomplete.  No counterpart on the pages. */
int zc_compress_stall_test(const void* in, size_t n, int base_or_auto, void* out,
                           size_t* out_bytes, cudaStream_t stream, size_t stalled_chunk,
                           unsigned spin_limit);

/* zc_loopback with the same planted stall as zc_compress_stall_test: chunk `stalled_chunk` never
 * publishes its escape-section size, so neither the scan nor the chunks' decoding can pass it;
 * the waits run out after about `spin_limit` polls and zc_status reports ZC_ERR_TIMEOUT.  No
 * counterpart on the pages. */
int zc_loopback_stall_test(const void* in, size_t n, int base_or_auto, void* out, size_t* out_bytes, void* values,
                           cudaStream_t stream, size_t stalled_chunk, unsigned spin_limit);

#ifdef __cplusplus
}
#endif

#endif /* ZC_H */
