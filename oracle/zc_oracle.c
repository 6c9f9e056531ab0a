/*
 * zc_oracle.c -- plain, single-threaded reference of the lossless BF16 exponent codec.
 *
 * TEST INFRASTRUCTURE ONLY (see zc_oracle.h).  Written for clarity, not speed: one value at
 * a time, in index order, with no blocking or reordering beyond what the definitions state.
 *
 * Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution", first technique.
 *   - the frequent exponent range comes directly from the tensor standard deviation,
 *     with no histogram and no sort;
 *   - for BF16, frequent exponents go from 8 bits to 3 bits;
 *   - infrequent exponents keep their full 8 bits in a separate store (lossless);
 *   - sign and mantissa are kept as they are, so an in-window value costs 1 + 7 + 3 bits.
 *
 * Readings taken where the page is silent (each one is also listed in the design notes):
 *   R1  sigma is the root mean square about zero over the finite values; Inf and NaN are
 *       left out of both the sum and the count.
 *   R2  the sum of squares is exact and then rounded once to fp64 (nearest, ties to even);
 *       q = S/n_f and y = q*C are single fp64 operations rounded to nearest.
 *   R3  the window holds 7 consecutive exponents [e0, e0+6]; 3-bit codes 0..6 name them and
 *       code 7 marks an escape.
 *   R4  e0 = floor(log2(sigma*c)) + 127, clamped to [0, 249], where c = 2u and u solves
 *       f(u) = f(2u) for f(t) = P(|Z| < t) + P(|Z| >= 128 t), Z ~ N(0,1).  For a Gaussian
 *       of standard deviation sigma this picks the 7-binade window with the fewest expected
 *       escapes.  It is evaluated as floor(ilogb(q*c^2)/2) + 127.
 *   R5  byte layout of the coded form ("ZCB1", version 4), read from the data layout shaped by the
 *       communication in the second technique and the compress / exchange sizes / send workflow (Figure 5(b),
 *       Design-1): every chunk's fixed-size part (3-bit codes, then the sign|mantissa plane) sits
 *       at an offset that follows from n alone, so it can be sent before any size is known;
 *       only the variable escape sections (R6) are compacted, behind a table of their offsets.
 *       32-byte header, u64 escape-offset table, fixed parts in chunk order, escape sections in
 *       chunk order; every section padded with zeros to 16 bytes; little-endian.
 *   R6  the separate store of a chunk's infrequent exponents (first technique: they keep their
 *       complete information apart from the codes) takes whichever of two lossless forms is
 *       smaller, in the spirit of the third technique's switch to the native path where
 *       compression does not pay: with k escapes among m values, a list of k (u16 position,
 *       u8 exponent) pairs when 3k <= m, else the chunk's m exponent bytes in value order (an
 *       exponent plane).  The form follows from k, which the codes give, so the stream needs
 *       no flag; the codes are the same in both forms.
 *   R7  stream form: the third technique also switches a whole transfer between the compressed
 *       path and the native one, by the benefit of compressing.  A tensor whose coded stream
 *       (R5, R6) would be longer than its native form -- the 32-byte header followed by the n
 *       values as they are, zero-padded to 16 bytes -- is stored in that native ("raw") form:
 *       header byte 6 (the chunk size field) is 0, N is 0, and the values follow the header as
 *       little-endian u16.  Ties keep the coded form.  The decoder checks a raw stream's bytes
 *       (header, length, padding) but does not recompute whether the coded form would have been
 *       shorter.  Format version 4.
 */
#include "zc_oracle.h"

#include <math.h>
#include <stddef.h>
#include <string.h>

#define CHUNK 4096u
#define HEADER_BYTES 32u
#define FORMAT_VERSION 4u
#define LOG2_CHUNK 12u
#define RAW_FORM 0u /* header byte 6 of a raw stream (R7) */
#define E0_MAX 249
#define WINDOW 7

/* c^2 for the rule R4; its derivation is re-done in the test suite with mpmath. */
static const double WINDOW_C2 = 0x1.79a1e790e0f01p-10;

static uint64_t pad16(uint64_t v) { return (v + 15u) & ~(uint64_t)15u; }

/* ---------------------------------------------------------------- little-endian I/O */

static void put_u16(uint8_t* p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xFFu);
  p[1] = (uint8_t)(v >> 8);
}
static void put_u64(uint8_t* p, uint64_t v) {
  for (int i = 0; i < 8; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint64_t get_u64(const uint8_t* p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}

/* ---------------------------------------------------------------- BF16 fields */

static unsigned bf16_exponent(uint16_t x) { return (x >> 7) & 0xFFu; }
static unsigned bf16_mantissa(uint16_t x) { return x & 0x7Fu; }
static unsigned bf16_sign(uint16_t x) { return (x >> 15) & 1u; }

/* ---------------------------------------------------------------- layout (R5) */

uint64_t zco_num_chunks(uint64_t n) { return (n + CHUNK - 1) / CHUNK; }

static uint64_t chunk_len(uint64_t n, uint64_t c) { return n - c * CHUNK < CHUNK ? n - c * CHUNK : CHUNK; }

/* Start of the fixed region: after the header and the N+1 escape offsets. */
uint64_t zco_records_base(uint64_t n) {
  return pad16(HEADER_BYTES + 8u * (zco_num_chunks(n) + 1u));
}

/* Fixed part of a chunk of m values: 3-bit code section, then the sign|mantissa plane. */
static uint64_t fixed_bytes(uint64_t m) { return pad16((3u * m + 7u) / 8u) + pad16(m); }

/* R6: a chunk keeps its escapes as a list of k (position, exponent) pairs when 3k <= m, else as
 * a plane of all m exponents. */
static int exponent_plane(uint64_t m, uint64_t k) { return 3u * k > m; }

/* Size of a chunk's escape section (list or plane), zero-padded to 16 bytes. */
static uint64_t escape_bytes(uint64_t m, uint64_t k) { return exponent_plane(m, k) ? pad16(m) : pad16(3u * k); }

/* Bytes a chunk of m values with k escapes contributes: its fixed part and its escape section. */
uint64_t zco_record_bytes(uint64_t m, uint64_t k) { return fixed_bytes(m) + escape_bytes(m, k); }

/* Where chunk c's fixed part starts: every earlier chunk is full. */
static uint64_t fixed_offset(uint64_t n, uint64_t c) { return zco_records_base(n) + c * fixed_bytes(CHUNK); }

/* Start of the escape region: after every fixed part. */
static uint64_t escape_base(uint64_t n) {
  uint64_t N = zco_num_chunks(n);
  return N ? fixed_offset(n, N - 1) + fixed_bytes(chunk_len(n, N - 1)) : zco_records_base(n);
}

/* Length of the coded form (R5, R6) of x under e0. */
static uint64_t coded_bytes(const uint16_t* x, uint64_t n, int e0);

/* Length of the raw form (R7): header, n values, zero padding. */
uint64_t zco_raw_stream_bytes(uint64_t n) { return HEADER_BYTES + pad16(2u * n); }

/* Every stream is at most as long as the raw form (R7). */
uint64_t zco_max_stream_bytes(uint64_t n) { return zco_raw_stream_bytes(n); }

double zco_window_constant(void) { return WINDOW_C2; }

/* ---------------------------------------------------------------- exact sum (R1, R2) */

/* A finite BF16 value is +-sig * 2^(Ep-134) with sig = 128+mantissa, Ep = E for E >= 1,
 * and sig = mantissa, Ep = 1 for E = 0.  Its square is sig^2 * 2^(2Ep-268), so
 * S * 2^266 = sum of sig^2 * 2^(2Ep-2): an integer below 2^(16+506+44) for n <= 2^44.
 * Nine 64-bit limbs (576 bits) hold it exactly. */
#define LIMBS 9

static void big_add_shifted(uint64_t acc[LIMBS], uint64_t v, unsigned shift) {
  unsigned li = shift / 64u, sh = shift % 64u;
  uint64_t lo = v << sh;
  uint64_t hi = sh ? (v >> (64u - sh)) : 0u;
  uint64_t old = acc[li];
  acc[li] = old + lo;
  uint64_t carry = acc[li] < old ? 1u : 0u;
  for (unsigned i = li + 1; i < LIMBS && (hi != 0 || carry != 0); ++i) {
    uint64_t add = hi + carry; /* hi < 2^16, no overflow */
    old = acc[i];
    acc[i] = old + add;
    carry = acc[i] < old ? 1u : 0u;
    hi = 0;
  }
}

static int big_bit(const uint64_t acc[LIMBS], int i) {
  return (int)((acc[i / 64] >> (i % 64)) & 1u);
}

/* Round acc * 2^-266 to the nearest fp64, ties to even. */
static double big_to_double_rn(const uint64_t acc[LIMBS]) {
  int top = -1;
  for (int i = LIMBS - 1; i >= 0 && top < 0; --i) {
    if (acc[i] != 0) {
      for (int b = 63; b >= 0; --b) {
        if ((acc[i] >> b) & 1u) {
          top = 64 * i + b;
          break;
        }
      }
    }
  }
  if (top < 0) return 0.0;
  if (top <= 52) return ldexp((double)acc[0], -266); /* exact: at most 53 bits */

  int shift = top - 52; /* keep bits [shift, top] */
  uint64_t M = 0;
  for (int b = top; b >= shift; --b) M = (M << 1) | (uint64_t)big_bit(acc, b);
  int round = big_bit(acc, shift - 1);
  int sticky = 0;
  for (int b = shift - 2; b >= 0 && !sticky; --b) sticky = big_bit(acc, b);
  if (round && (sticky || (M & 1u))) {
    M += 1u;
    if (M == ((uint64_t)1 << 53)) {
      M >>= 1;
      shift += 1;
    }
  }
  return ldexp((double)M, shift - 266);
}

int zco_sum_squares(const uint16_t* x, uint64_t n, double* S_d, uint64_t* n_f) {
  uint64_t acc[LIMBS];
  memset(acc, 0, sizeof acc);
  uint64_t finite = 0;
  for (uint64_t i = 0; i < n; ++i) {
    unsigned E = bf16_exponent(x[i]);
    if (E == 255u) continue; /* Inf or NaN: not part of the statistic (R1) */
    finite += 1;
    uint64_t sig = (E == 0u) ? bf16_mantissa(x[i]) : 128u + bf16_mantissa(x[i]);
    unsigned Ep = (E == 0u) ? 1u : E;
    big_add_shifted(acc, sig * sig, 2u * Ep - 2u);
  }
  *S_d = big_to_double_rn(acc);
  *n_f = finite;
  return ZCO_OK;
}

/* ---------------------------------------------------------------- window base (R3, R4) */

static int floor_half(int v) { return v >= 0 ? v / 2 : -((-v + 1) / 2); }

int zco_select_e0(double S_d, uint64_t n_f) {
  if (n_f == 0 || S_d == 0.0) return 0;
  double q = S_d / (double)n_f; /* mean square, one rounding */
  double y = q * WINDOW_C2;     /* (sigma*c)^2, one rounding */
  int e = floor_half(ilogb(y)) + 127;
  if (e < 0) e = 0;
  if (e > E0_MAX) e = E0_MAX;
  return e;
}

int zco_choose_e0(const uint16_t* x, uint64_t n) {
  double S_d;
  uint64_t n_f;
  zco_sum_squares(x, n, &S_d, &n_f);
  return zco_select_e0(S_d, n_f);
}

/* ---------------------------------------------------------------- encode (R3, R5) */

static unsigned exponent_code(unsigned E, int e0) {
  int d = (int)E - e0;
  return (d >= 0 && d < WINDOW) ? (unsigned)d : 7u;
}

static void set_bit(uint8_t* base, uint64_t bit) { base[bit / 8] |= (uint8_t)(1u << (bit % 8)); }
static unsigned get_bit(const uint8_t* base, uint64_t bit) { return (base[bit / 8] >> (bit % 8)) & 1u; }

static uint64_t coded_bytes(const uint16_t* x, uint64_t n, int e0) {
  uint64_t total = escape_base(n);
  for (uint64_t c = 0; c < zco_num_chunks(n); ++c) {
    uint64_t m = chunk_len(n, c), k = 0;
    for (uint64_t i = 0; i < m; ++i) k += exponent_code(bf16_exponent(x[c * CHUNK + i]), e0) == 7u;
    total += escape_bytes(m, k);
  }
  return total;
}

static void put_header(uint8_t* out, unsigned form, int e0, uint64_t n, uint64_t N, uint64_t total) {
  out[0] = 'Z';
  out[1] = 'C';
  out[2] = 'B';
  out[3] = '1';
  put_u16(out + 4, FORMAT_VERSION);
  out[6] = (uint8_t)form;
  out[7] = (uint8_t)e0;
  put_u64(out + 8, n);
  put_u64(out + 16, N);
  put_u64(out + 24, total);
}

int64_t zco_compress(const uint16_t* x, uint64_t n, int base_or_auto, uint8_t* out, uint64_t cap) {
  if (base_or_auto < -1 || base_or_auto > E0_MAX) return -ZCO_ERR_INVALID_ARG;
  if (n > 0 && (x == NULL || out == NULL)) return -ZCO_ERR_INVALID_ARG;
  int e0 = base_or_auto == -1 ? zco_choose_e0(x, n) : base_or_auto;

  /* First pass: the coded length, so that the form (R7) and the capacity are settled before
   * any write. */
  const uint64_t coded = coded_bytes(x, n, e0);
  const uint64_t raw = zco_raw_stream_bytes(n);
  const int raw_form = coded > raw; /* R7: ties keep the coded form */
  const uint64_t total = raw_form ? raw : coded;
  if (out == NULL || total > cap) return -ZCO_ERR_CAPACITY;
  memset(out, 0, (size_t)total);

  if (raw_form) { /* R7: the native form */
    put_header(out, RAW_FORM, e0, n, 0, total);
    for (uint64_t i = 0; i < n; ++i) put_u16(out + HEADER_BYTES + 2u * i, x[i]);
    return (int64_t)total;
  }

  uint64_t N = zco_num_chunks(n);
  put_header(out, LOG2_CHUNK, e0, n, N, total);
  uint64_t esc_pos = escape_base(n);
  for (uint64_t c = 0; c < N; ++c) {
    const uint16_t* xc = x + c * CHUNK;
    uint64_t m = chunk_len(n, c);
    uint8_t* codes = out + fixed_offset(n, c);
    uint8_t* sm = codes + pad16((3u * m + 7u) / 8u);
    uint8_t* esc = out + esc_pos;
    put_u64(out + HEADER_BYTES + 8u * c, esc_pos);

    uint64_t k = 0;
    for (uint64_t i = 0; i < m; ++i) k += exponent_code(bf16_exponent(xc[i]), e0) == 7u;
    const int plane = exponent_plane(m, k);

    uint64_t r = 0;
    for (uint64_t i = 0; i < m; ++i) {
      unsigned E = bf16_exponent(xc[i]);
      unsigned code = exponent_code(E, e0);
      for (unsigned b = 0; b < 3; ++b)
        if ((code >> b) & 1u) set_bit(codes, 3u * i + b); /* code i at bits [3i, 3i+3) */
      sm[i] = (uint8_t)((bf16_sign(xc[i]) << 7) | bf16_mantissa(xc[i]));
      if (plane) {
        esc[i] = (uint8_t)E; /* every exponent, in value order */
      } else if (code == 7u) {
        put_u16(esc + 2u * r, (uint16_t)i); /* positions, ascending */
        esc[2u * k + r] = (uint8_t)E;       /* full exponents, same order */
        r += 1;
      }
    }
    esc_pos += escape_bytes(m, k);
  }
  put_u64(out + HEADER_BYTES + 8u * N, esc_pos);
  return (int64_t)total;
}

/* ---------------------------------------------------------------- decode (R5, inverse) */

static int all_zero(const uint8_t* p, uint64_t len) {
  for (uint64_t i = 0; i < len; ++i)
    if (p[i] != 0) return 0;
  return 1;
}

int zco_decompress(const uint8_t* in, uint64_t in_bytes, uint16_t* out, uint64_t n) {
  if (in == NULL || (n > 0 && out == NULL)) return ZCO_ERR_INVALID_ARG;
  if (in_bytes < HEADER_BYTES) return ZCO_ERR_CORRUPT;
  if (in[0] != 'Z' || in[1] != 'C' || in[2] != 'B' || in[3] != '1') return ZCO_ERR_CORRUPT;
  if (get_u16(in + 4) != FORMAT_VERSION || (in[6] != LOG2_CHUNK && in[6] != RAW_FORM)) return ZCO_ERR_CORRUPT;
  int e0 = in[7];
  if (e0 > E0_MAX) return ZCO_ERR_CORRUPT;
  if (get_u64(in + 8) != n) return ZCO_ERR_SIZE_MISMATCH;
  uint64_t total = get_u64(in + 24);

  if (in[6] == RAW_FORM) { /* R7: header, the values as they are, zero padding */
    if (get_u64(in + 16) != 0 || total != zco_raw_stream_bytes(n) || total > in_bytes) return ZCO_ERR_CORRUPT;
    for (uint64_t i = 0; i < n; ++i) out[i] = get_u16(in + HEADER_BYTES + 2u * i);
    if (!all_zero(in + HEADER_BYTES + 2u * n, total - HEADER_BYTES - 2u * n)) return ZCO_ERR_CORRUPT;
    return ZCO_OK;
  }

  uint64_t N = zco_num_chunks(n);
  if (get_u64(in + 16) != N) return ZCO_ERR_CORRUPT;
  uint64_t base = zco_records_base(n);
  /* a coded stream is never longer than the raw form (R7), nor shorter than its fixed parts */
  if (total > in_bytes || total > zco_raw_stream_bytes(n) || total < escape_base(n)) return ZCO_ERR_CORRUPT;
  if (!all_zero(in + HEADER_BYTES + 8u * (N + 1), base - (HEADER_BYTES + 8u * (N + 1))))
    return ZCO_ERR_CORRUPT;

  uint64_t esc_pos = escape_base(n);
  for (uint64_t c = 0; c < N; ++c) {
    uint64_t m = chunk_len(n, c);
    if (get_u64(in + HEADER_BYTES + 8u * c) != esc_pos) return ZCO_ERR_CORRUPT;
    const uint8_t* codes = in + fixed_offset(n, c);
    uint64_t code_bytes = pad16((3u * m + 7u) / 8u);
    const uint8_t* sm = codes + code_bytes;

    uint64_t k = 0; /* the escape count follows from the codes */
    for (uint64_t i = 0; i < m; ++i)
      k += (get_bit(codes, 3u * i) & get_bit(codes, 3u * i + 1) & get_bit(codes, 3u * i + 2));
    const int plane = exponent_plane(m, k);
    const uint64_t section = escape_bytes(m, k);
    if (esc_pos + section > total) return ZCO_ERR_CORRUPT;
    const uint8_t* esc = in + esc_pos;

    uint64_t r = 0;
    for (uint64_t i = 0; i < m; ++i) {
      unsigned code = get_bit(codes, 3u * i) | (get_bit(codes, 3u * i + 1) << 1) |
                      (get_bit(codes, 3u * i + 2) << 2);
      unsigned E;
      if (plane) {
        E = esc[i];
        if (exponent_code(E, e0) != code) return ZCO_ERR_CORRUPT; /* the plane must agree with the codes */
      } else if (code < 7u) {
        E = (unsigned)e0 + code;
      } else {
        if (get_u16(esc + 2u * r) != i) return ZCO_ERR_CORRUPT; /* positions ascending, exact */
        E = esc[2u * k + r];
        if (exponent_code(E, e0) != 7u) return ZCO_ERR_CORRUPT; /* an escape must lie outside */
        r += 1;
      }
      out[c * CHUNK + i] = (uint16_t)(((unsigned)(sm[i] >> 7) << 15) | (E << 7) | (sm[i] & 0x7Fu));
    }
    for (uint64_t b = 3u * m; b < 8u * code_bytes; ++b)
      if (get_bit(codes, b)) return ZCO_ERR_CORRUPT;
    if (!all_zero(sm + m, pad16(m) - m)) return ZCO_ERR_CORRUPT;
    const uint64_t used = plane ? m : 3u * k;
    if (!all_zero(esc + used, section - used)) return ZCO_ERR_CORRUPT;
    esc_pos += section;
  }
  if (get_u64(in + HEADER_BYTES + 8u * N) != esc_pos || esc_pos != total) return ZCO_ERR_CORRUPT;
  return ZCO_OK;
}
