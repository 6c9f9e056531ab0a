/*
 * zc_oracle.h -- plain, single-threaded reference of the lossless BF16 exponent codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path includes, links or calls this
 * code: only the test suite, the package's smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no source, header, table or constant generator with the CUDA
 * library; the two meet only through byte buffers.
 *
 * What it computes follows "ZipCCL: Efficient Lossless Data Compression of Communication
 * Collectives for Accelerating LLM Training" (SIGCOMM scribe notes), section "Key idea and
 * contribution", first technique (theoretically grounded exponent coding): a window of
 * frequent exponents is taken directly from the tensor's standard deviation, in-window
 * exponents are stored in 3 bits, out-of-window exponents are kept whole in a separate
 * list, and sign and mantissa travel unchanged, for roughly 11 bits per value; where that
 * coding does not pay, the tensor travels in its native form (third technique).  The page
 * fixes neither the window rule's constant nor a byte layout; the readings used here are
 * stated beside each function in zc_oracle.c.
 *
 * Parity status:
 *   zco_sum_squares / zco_select_e0 / zco_choose_e0 -- pinned (correctly rounded sum checked
 *       against math.fsum; window rule checked against a Gaussian escape-rate argmin; the
 *       constant re-derived with mpmath).
 *   zco_compress / zco_decompress -- pinned against the format readings (hand-derived
 *       stream fixtures of the coded form with a list and with a plane, and of the raw form;
 *       closed-form size; exhaustive round trips; bijection under byte flips); the byte
 *       layout itself has no counterpart on the pages.
 */
#ifndef ZC_ORACLE_H
#define ZC_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status values.  They carry the same numbers as the library's public codes so that a test
 * can compare the two, but they are defined here on their own. */
#define ZCO_OK 0
#define ZCO_ERR_INVALID_ARG 1
#define ZCO_ERR_CORRUPT 4
#define ZCO_ERR_SIZE_MISMATCH 5
#define ZCO_ERR_CAPACITY 7

/* Layout helpers (pure).  records_base: start of the fixed-part region (after the header and
 * the escape-offset table); record_bytes: what a chunk of m values with k escapes adds to the
 * stream (its fixed part plus its escape section: a list of k pairs, or all m exponents when
 * 3k > m). */
uint64_t zco_num_chunks(uint64_t n);
uint64_t zco_records_base(uint64_t n);
uint64_t zco_record_bytes(uint64_t m, uint64_t k);
uint64_t zco_max_stream_bytes(uint64_t n); /* the longest stream: the raw form's length */
uint64_t zco_raw_stream_bytes(uint64_t n); /* 32-byte header + n values, zero-padded to 16 */

/* The constant c^2 of the window rule (fp64). */
double zco_window_constant(void);

/* Exact sum of squares of the finite values, rounded once to the nearest fp64 (ties to
 * even).  n_f receives the number of finite values.  Returns ZCO_OK. */
int zco_sum_squares(const uint16_t* x, uint64_t n, double* S_d, uint64_t* n_f);

/* Window base e0 in [0, 249] from (S_d, n_f). */
int zco_select_e0(double S_d, uint64_t n_f);

/* zco_select_e0 applied to zco_sum_squares of x. */
int zco_choose_e0(const uint16_t* x, uint64_t n);

/* Compress n BF16 bit patterns.  base_or_auto is -1 (choose e0 from the data) or a base in
 * [0, 249].  Writes the stream to out (capacity cap bytes) and returns its length, or a
 * negative status (-ZCO_ERR_...).  The stream is the coded form, or the raw form when the
 * coded one would be longer. */
int64_t zco_compress(const uint16_t* x, uint64_t n, int base_or_auto, uint8_t* out, uint64_t cap);

/* Decompress a stream of in_bytes bytes into n BF16 bit patterns.  Returns ZCO_OK, or
 * ZCO_ERR_SIZE_MISMATCH when the stream holds another n, or ZCO_ERR_CORRUPT for any stream
 * that the encoder could not have written. */
int zco_decompress(const uint8_t* in, uint64_t in_bytes, uint16_t* out, uint64_t n);

#ifdef __cplusplus
}
#endif

#endif /* ZC_ORACLE_H */
