// zc_stats_core.cuh -- the arithmetic of the window base e0, shared by the statistics kernel and
// the small-tensor kernel: fp32 block sums of squares with a rigorous error bound, the window rule,
// and the exact fallback (per-exponent integer sums rounded once to fp64).
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution", first technique: the
// window of frequent exponents is taken from the tensor's standard deviation alone, with no
// histogram and no sort.  e0 = floor(log2(sigma * c)) + 127 clamped to [0, 249], sigma^2 = S / n_f,
// where S is the exact sum of squares rounded once to fp64 and c^2 = 0x1.79a1e790e0f01p-10 (the
// base whose 7-binade window has the fewest expected escapes under a Gaussian).
//
// Every block sum of 64 values carries a relative error below 2^-18 (at most 17 roundings, or 64
// for the last n % 8 values, summed one by one), so a total over blocks lies within 2^-17 of the
// exact sum; decide_e0_pair then settles e0 exactly for all but ~4e-5 of random tensors, and the
// exact fallback decides the rest.
#pragma once

#include "zc_common.cuh"

namespace zc {
namespace {

constexpr double kWindowC2 = 0x1.79a1e790e0f01p-10;

// floor(log2(y)) for a positive finite double, from its bit pattern.
__device__ __forceinline__ int ilogb_pos(double y) {
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(y));
  const int ex = static_cast<int>((b >> 52) & 0x7FF);
  if (ex != 0) return ex - 1023;
  const unsigned long long mant = b & ((1ull << 52) - 1);
  return (63 - __clzll(static_cast<long long>(mant))) - 1074;
}

__device__ __forceinline__ int floor_half(int v) { return v >= 0 ? v / 2 : -((-v + 1) / 2); }

// The window rule at a given fp64 sum of squares.
__device__ int select_e0(double S, unsigned long long n_f) {
  if (n_f == 0 || S == 0.0) return 0;
  const double q = __ddiv_rn(S, static_cast<double>(n_f));
  const double y = __dmul_rn(q, kWindowC2);
  int e = floor_half(ilogb_pos(y)) + 127;
  return e < 0 ? 0 : (e > kE0Max ? kE0Max : e);
}

// The window rule in fp32, for a guess only (the exact rule decides what is kept): the binary
// exponent of S taken out first, so nothing overflows or underflows; a few fp32 operations
// where select_e0's fp64 division takes far longer on this part.
__device__ __forceinline__ int rough_e0(double S, unsigned long long n_f) {
  if (n_f == 0 || !(S > 0.0)) return 0;
  const int kS = ilogb_pos(S);  // S = Sn 2^kS, Sn in [1, 2)
  const float Sn = static_cast<float>(S * __longlong_as_double(static_cast<long long>(1023 - kS) << 52));
  const float y = Sn / static_cast<float>(n_f) * static_cast<float>(kWindowC2);  // the rule's y, times 2^-kS
  const int e = floor_half(static_cast<int>((__float_as_uint(y) >> 23) & 0xFF) - 127 + kS) + 127;
  return e < 0 ? 0 : (e > kE0Max ? kE0Max : e);
}

// Careful block sum for 64 values (32 words), one by one (used for the last n % 8 values): skips
// Inf/NaN, and scales every square by 4^-(Emax'-E') relative to the largest exponent present, so
// no fp32 overflow or underflow matters.  Returns the fp64 value of the block sum and adds the
// non-finite count.
__device__ __forceinline__ double careful_block(const uint32_t (&w)[32], unsigned* nonfinite) {
  int emax = 0;
  unsigned nf = 0;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const uint32_t x = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
    const int E = (x >> 7) & 0xFF;
    if (E == 255) {
      ++nf;
    } else if (x & 0x7FFFu) {
      emax = max(emax, max(E, 1));
    }
  }
  *nonfinite += nf;
  if (emax == 0) return 0.0;  // only zeros (and non-finite values)
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const uint32_t x = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
    const int E = (x >> 7) & 0xFF;
    if (E == 255 || (x & 0x7FFFu) == 0) continue;
    const int sig = E ? 128 + static_cast<int>(x & 0x7F) : static_cast<int>(x & 0x7F);
    const int d2 = 2 * (emax - max(E, 1));
    if (d2 > 126) continue;  // below 2^-110 of the block's largest square
    s = fmaf(static_cast<float>(sig * sig), __int_as_float((127 - d2) << 23), s);
  }
  // The block sum is s * 2^(2 emax - 268); emax in [1, 254] keeps the scale a normal double.
  const double scale = __longlong_as_double(static_cast<long long>(755 + 2 * emax) << 52);
  return static_cast<double>(s) * scale;
}

// The last n % 8 values, zero-padded (a zero adds nothing and is not counted as non-finite).
__device__ __noinline__ double tail_block(const uint16_t* tail, unsigned count, unsigned* nonfinite) {
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) w[i] = 0;
  for (unsigned i = 0; i < count; ++i) w[i >> 1] |= static_cast<uint32_t>(tail[i]) << (16 * (i & 1));
  return careful_block(w, nonfinite);
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Block sum of 2W values (this lane's block, W = 32 or 16 words; `w` is consumed).  Bit
// patterns with the sign cleared order like magnitudes, so one packed 16-bit max finds the
// block's largest, and it decides, per warp, between the plain sum (every lane's largest biased
// exponent in [87, 187): no square reaches 2^122 and the block sum is at least 2^-80, so the at
// most 64 squares, at most 17 roundings, stay within 2^-19 of the exact sum) and a sum with every
// lane's values scaled by 2^(126 - Es), Es = E clamped to [1, 252] (1 for lanes that need no
// scaling), which puts the largest magnitude in [2^-8, 4): no square overflows and what
// underflows is under 2^-120 of the block sum.  The decision is one warp vote, so a warp runs one
// of the two loops (every lane of the warp must call).  A lane whose block holds Inf or NaN (its
// largest pattern is at or above 0x7F80) first counts them and clears them to zero, which adds
// nothing to the sum, and takes the largest of the rest; its warp then sums scaled.
template <int W>
__device__ __forceinline__ void block_sum(uint32_t (&w)[W], double* acc, unsigned* nonfinite) {
  static_assert(W == 32 || W == 16, "blocks of 64 or 32 values");
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < W; ++i) mx = max_u16x2(mx, w[i] & 0x7FFF7FFFu);
  unsigned m = max(mx & 0xFFFFu, mx >> 16);
  bool odd = m != 0 && (m >> 7 >= 187u || m >> 7 < 87u);  // Inf and NaN included (E = 255)
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (!__any_sync(0xFFFFFFFFu, odd)) {
#pragma unroll
    for (int i = 0; i < W; i += 2) {
      const float l0 = __uint_as_float(w[i] << 16), h0 = __uint_as_float(w[i] & 0xFFFF0000u);
      const float l1 = __uint_as_float(w[i + 1] << 16), h1 = __uint_as_float(w[i + 1] & 0xFFFF0000u);
      a0 = fmaf(l0, l0, a0);
      a1 = fmaf(h0, h0, a1);
      a2 = fmaf(l1, l1, a2);
      a3 = fmaf(h1, h1, a3);
    }
    *acc += static_cast<double>((a0 + a1) + (a2 + a3));
    return;
  }
  if (m >= 0x7F80u) {
    // A 16-bit magnitude a is at or above 0x7F80 exactly when a + 0x80 reaches bit 15 (a <= 0x7FFF,
    // so nothing carries into the other half).
    unsigned nf = 0;
    mx = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const uint32_t t = ((w[i] & 0x7FFF7FFFu) + 0x00800080u) & 0x80008000u;  // bit 15 of each non-finite half
      nf += __popc(t);
      w[i] &= ~(t | (t - (t >> 15)));  // clear those halves
      mx = max_u16x2(mx, w[i] & 0x7FFF7FFFu);
    }
    *nonfinite += nf;
    m = max(mx & 0xFFFFu, mx >> 16);
    odd = m != 0 && (m >> 7 >= 187u || m >> 7 < 87u);
  }
  const int Es = odd ? min(max(static_cast<int>(m >> 7), 1), 252) : 126;
  const float sc = __int_as_float((253 - Es) << 23);
#pragma unroll
  for (int i = 0; i < W; i += 2) {
    const float l0 = __uint_as_float(w[i] << 16) * sc, h0 = __uint_as_float(w[i] & 0xFFFF0000u) * sc;
    const float l1 = __uint_as_float(w[i + 1] << 16) * sc, h1 = __uint_as_float(w[i + 1] & 0xFFFF0000u) * sc;
    a0 = fmaf(l0, l0, a0);
    a1 = fmaf(h0, h0, a1);
    a2 = fmaf(l1, l1, a2);
    a3 = fmaf(h1, h1, a3);
  }
  const float blk = (a0 + a1) + (a2 + a3);
  *acc += static_cast<double>(blk) * __longlong_as_double(static_cast<long long>(1023 + 2 * Es - 252) << 52);
}

// The e0 both ends of decide_e0_pair's interval give, found in fp32 when it can be: with
// Sn = S_est 2^-kS in [1, 2), y = Sn / n_f c^2 in fp32 is within 6 roundings (below 2^-21.4) of
// its exact value, so y (1 -+ 2^-12) brackets the rule's fp64 y at S_est (1 -+ 2^-16) (each within
// 2^-52 of exact) with room to spare; when both brackets fall in one bin of the rule (one power
// of 4 of y), that bin's e0 is what the fp64 ends give.  Returns -1 otherwise (a bracket straddles
// a switching point: the fp64 ends decide).
__device__ __forceinline__ int settled_e0_fp32(double S_est, unsigned long long n_f) {
  if (n_f == 0 || S_est == 0.0) return 0;  // as select_e0
  const int kS = ilogb_pos(S_est);
  const float Sn = static_cast<float>(S_est * __longlong_as_double(static_cast<long long>(1023 - kS) << 52));
  const float y = Sn / static_cast<float>(n_f) * static_cast<float>(kWindowC2);  // the rule's y, times 2^-kS
  int e[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const float yt = y * (t == 0 ? 1.0f - 0x1p-12f : 1.0f + 0x1p-12f);
    const int v = floor_half(static_cast<int>((__float_as_uint(yt) >> 23) & 0xFF) - 127 + kS) + 127;
    e[t] = v < 0 ? 0 : (v > kE0Max ? kE0Max : v);
  }
  return e[0] == e[1] ? e[0] : -1;
}

// The window rule at an fp64 estimate S_est of the sum of squares that lies within 2^-17 of the
// exact sum: evaluated at S_est (1 -+ 2^-16), rounded outward, both ends give the exact e0 when
// they agree (the rule is monotone in S).  Returns false when they do not: the exact sum decides.
// Lanes 0 and 1 of a warp call it together, with the same S_est and n_f, and both get the result;
// *e0 is the lower end's.  Most estimates are settled by settled_e0_fp32; otherwise each lane
// evaluates one end in fp64 (their divisions in parallel).
__device__ __forceinline__ bool decide_e0_pair(double S_est, unsigned long long n_f, int* e0) {
  const int quick = settled_e0_fp32(S_est, n_f);
  if (quick >= 0) {
    *e0 = quick;
    return true;
  }
  const int e =
      select_e0((threadIdx.x & 1) == 0 ? __dmul_rd(S_est, 1.0 - 0x1p-16) : __dmul_ru(S_est, 1.0 + 0x1p-16), n_f);
  const int lo = __shfl_sync(0x3u, e, 0), hi = __shfl_sync(0x3u, e, 1);
  *e0 = lo;
  return lo == hi;
}

// The speculative routes' guess of e0 from a sample, by a group of kThreads threads (whole warps)
// each holding W words (2W values) of it, `vals` of them real (the rest zero, at the end).  Per
// warp: squares and fourth powers in fp32, scaled by 2^(126 - Es) from the warp's largest finite
// magnitude (so no power overflows); Inf and NaN are counted out.  Thread 0 combines the warps in
// fp64 and evaluates the rule (in fp32, the binary exponent taken out first) at the sample's mean
// square q and at q (1 -+ d), d = 1/32 + 4 r (at most 3/4), r the mean square's relative standard
// error estimated from the fourth powers; *guess is the e0 at q, *confident whether the three
// agree and the sample has a finite nonzero value.  For a guess only: no error bound is claimed,
// and the group's every thread sees the same answer after bar().  g2, g4, gk, gf: per-warp scratch.
template <int kThreads, int W, typename Bar>
__device__ void guess_e0(const uint32_t (&w)[W], unsigned vals, float* g2, float* g4, int* gk, unsigned* gf,
                         int* guess, int* confident, Bar bar) {
  constexpr int kWarpsG = kThreads / 32;
  const unsigned tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kVals = 2 * W;
  unsigned mx = 0, nonfinite = 0;
#pragma unroll
  for (int i = 0; i < kVals; ++i) {
    const unsigned a = (w[i >> 1] >> (16 * (i & 1))) & 0x7FFFu;
    if (a >= 0x7F80u) ++nonfinite;
    else mx = max(mx, a);
  }
  mx = __reduce_max_sync(0xFFFFFFFFu, mx);
  const int Es = min(max(static_cast<int>(mx >> 7), 1), 252);
  const float sc = __int_as_float((253 - Es) << 23);  // 2^(126 - Es)
  float a2 = 0.f, a4 = 0.f, b2 = 0.f, b4 = 0.f;
#pragma unroll
  for (int i = 0; i < kVals; ++i) {
    const uint32_t h = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
    const float x = (h & 0x7FFFu) >= 0x7F80u ? 0.f : __uint_as_float(h << 16) * sc;
    const float x2 = x * x;
    if (i & 1) {
      b2 += x2;
      b4 = fmaf(x2, x2, b4);
    } else {
      a2 += x2;
      a4 = fmaf(x2, x2, a4);
    }
  }
  float s2 = a2 + b2, s4 = a4 + b4;
  unsigned fin = vals - nonfinite;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, o);
    s4 += __shfl_xor_sync(0xFFFFFFFFu, s4, o);
    fin += __shfl_xor_sync(0xFFFFFFFFu, fin, o);
  }
  if (lane == 0) {
    g2[warp] = s2;
    g4[warp] = s4;
    gk[warp] = Es - 126;
    gf[warp] = fin;
  }
  bar();
  if (tid == 0) {
    double Sd = 0.0, Qd = 0.0;  // the true sums: x^2 and x^4 times 2^(2k), 2^(4k)
    unsigned m = 0;
    for (int i = 0; i < kWarpsG; ++i) {
      Sd += static_cast<double>(g2[i]) * __longlong_as_double(static_cast<long long>(1023 + 2 * gk[i]) << 52);
      Qd += static_cast<double>(g4[i]) * __longlong_as_double(static_cast<long long>(1023 + 4 * gk[i]) << 52);
      m += gf[i];
    }
    int e_at[3] = {0, 0, 0};
    bool conf = false;
    if (m > 0 && Sd > 0.0) {
      const int kS = ilogb_pos(Sd);  // Sd = Sn 2^kS, Sn in [1, 2)
      const float Sn = static_cast<float>(Sd * __longlong_as_double(static_cast<long long>(1023 - kS) << 52));
      const float Qn = static_cast<float>(Qd * __longlong_as_double(static_cast<long long>(1023 - 2 * kS) << 52));
      const float fm = static_cast<float>(m);
      const float d = fminf(1.0f / 32 + 4.0f * sqrtf(fmaxf(Qn / (Sn * Sn) * fm - 1.0f, 0.0f) / fm), 0.75f);
      const float y = Sn / fm * static_cast<float>(kWindowC2);  // the rule's y, times 2^-kS
#pragma unroll
      for (int t = 0; t < 3; ++t) {
        const float yt = y * (t == 0 ? 1.0f - d : t == 1 ? 1.0f : 1.0f + d);
        const int e = floor_half(static_cast<int>((__float_as_uint(yt) >> 23) & 0xFF) - 127 + kS) + 127;
        e_at[t] = e < 0 ? 0 : (e > kE0Max ? kE0Max : e);
      }
      conf = e_at[0] == e_at[1] && e_at[2] == e_at[1];
    }
    *guess = e_at[1];
    *confident = conf;
  }
  bar();
}

// Exact sums of squares, one thread: sig^2 4^d, d = E - Eb, of the values whose exponent E
// (subnormals at 1) lies in the window [Eb, Eb + 24), in a 96-bit integer (a0, a1, a2); a finite
// nonzero value outside the window adds sig^2 to bins[E] instead (shared memory).  Two values of
// a word at a time: E and d in packed 16-bit halves, d clamped to the window's width; sig as
// y + 128 - 128 E from the magnitude y (128 + m for E >= 1, m for E = 0); the term as
// (sig << d)^2 (below 2^62) by one widening multiply, added by a carry chain.  A value outside
// the window has its sig masked to zero in that step and takes a branch to its bin; a zero stays
// inside and adds nothing, and Inf/NaN (E = 255) are outside and skipped there.  No atomics on
// the common path: a tensor's values share a handful of exponents, which per-value atomics on
// their bins would serialise.
constexpr int kExactWindow = 24;
struct ExactWindow {
  uint32_t neg_eb;  // -Eb in both halves
  unsigned a0 = 0, a1 = 0, a2 = 0;
  __device__ explicit ExactWindow(int Eb) : neg_eb(((0x10000u - static_cast<unsigned>(Eb)) & 0xFFFFu) * 0x00010001u) {}
  __device__ __forceinline__ void add_word(uint32_t w, unsigned long long* bins) {
    const uint32_t y = w & 0x7FFF7FFFu;
    const uint32_t Ep = max_u16x2((w >> 7) & 0x00FF00FFu, 0x00010001u);
    const uint32_t d = min_u16x2(add_u16x2(Ep, neg_eb), kExactWindow * 0x00010001u);
    // bit 15 of a half: d reached the window's width, and y is not zero
    const uint32_t outside = ((d + (0x8000u - kExactWindow) * 0x00010001u) & (y + 0x7FFF7FFFu) & 0x80008000u) >> 15;
    const uint32_t sig = (y + 0x00800080u - (Ep << 7)) & ~(outside * 0xFFFFu);
    const uint32_t u0 = (sig & 0xFFFFu) << (d & 0xFFFFu), u1 = (sig >> 16) << (d >> 16);  // < 2^31
    const unsigned long long t = static_cast<unsigned long long>(u0) * u0 + static_cast<unsigned long long>(u1) * u1;
    asm("add.cc.u32 %0, %0, %3;\n\taddc.cc.u32 %1, %1, %4;\n\taddc.u32 %2, %2, 0;"
        : "+r"(a0), "+r"(a1), "+r"(a2)
        : "r"(static_cast<unsigned>(t)), "r"(static_cast<unsigned>(t >> 32)));
    if (outside) {
      if (outside & 1u) to_bin(w & 0xFFFFu, bins);
      if (outside >> 16) to_bin(w >> 16, bins);
    }
  }
  __device__ static void to_bin(unsigned b, unsigned long long* bins) {
    const unsigned E = (b >> 7) & 0xFF;
    if (E == 255 || (b & 0x7FFF) == 0) return;
    const unsigned sig = E ? 128 + (b & 0x7F) : (b & 0x7F);
    atomicAdd(bins + (E ? E : 1), static_cast<unsigned long long>(sig * sig));
  }
};

// Per-exponent integer sums of sig^2 of the finite values x[0..count), the thread taking words
// (value pairs) start, start + stride, .., added into bins[E] (shared, 256 words; E = 0 and 1
// share bin 1; x 4-byte aligned).  Called by every thread of the CTA alike (warp reductions).
// The values in the 24-binade window from Eb = anchor_e0 - 12 (around a Gaussian's typical
// exponent; clamped to [1, 214]) are summed exactly in registers (ExactWindow); the thread's
// 96-bit sum goes to the bins as six 16-bit pieces, each summed over the warp: piece j weighs
// 2^(16 j) 4^(E - Eb), which is the weight of bin Eb + 8 j (bin e counts 4^e).  anchor_e0 only
// steers speed: any value gives the same bins' total.
__device__ __forceinline__ void add_exponent_sums(const uint16_t* x, uint64_t count, uint64_t start, uint64_t stride,
                                                  unsigned long long* bins, int anchor_e0) {
  int Eb = anchor_e0 - 12;
  Eb = Eb < 1 ? 1 : (Eb > 214 ? 214 : Eb);
  ExactWindow ew(Eb);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(x);
  for (uint64_t i = start; i < count / 2; i += stride) ew.add_word(w[i], bins);
  if ((count & 1) && start == 0) ew.add_word(x[count - 1], bins);  // an odd last value
  const unsigned piece[6] = {ew.a0 & 0xFFFFu, ew.a0 >> 16, ew.a1 & 0xFFFFu, ew.a1 >> 16, ew.a2 & 0xFFFFu, ew.a2 >> 16};
#pragma unroll
  for (int j = 0; j < 6; ++j) {
    const unsigned s = __reduce_add_sync(0xFFFFFFFFu, piece[j]);  // 32 pieces below 2^16
    if ((threadIdx.x & 31) == 0 && s) atomicAdd(bins + Eb + 8 * j, static_cast<unsigned long long>(s));
  }
}

// Add t * 2^s (t < 2^64, s + 64 < 576) into a 576-bit integer.
__device__ __forceinline__ void add_shifted_576(unsigned long long (&limb)[9], unsigned long long t, int s) {
  if (t == 0) return;
  const int li = s >> 6, sh = s & 63;
  const unsigned long long add[2] = {t << sh, sh ? t >> (64 - sh) : 0ull};
  unsigned long long carry = 0;
  for (int j = li; j < 9; ++j) {
    const unsigned long long a = (j - li < 2 ? add[j - li] : 0ull);
    const unsigned long long before = limb[j];
    unsigned long long sum = before + a;
    unsigned long long c1 = sum < before;
    sum += carry;
    c1 += sum < carry;
    limb[j] = sum;
    carry = c1;
    if (j - li >= 1 && carry == 0) break;
  }
}

// The 576-bit integer sum_E T_E 2^(2E-2) (= S 2^266) of per-exponent sums T_E (each below 2^56),
// plus, when `pieces` is given, sum_k pieces[k] 2^(32k + 2 Eb - 2) (window sums relative to the
// exponent Eb), rounded once to fp64, nearest-even: the exact sum of squares S rounded correctly.
// One thread.
__device__ __noinline__ double exact_from_bins(const unsigned long long* bins,
                                               const unsigned long long* pieces = nullptr, int Eb = 1) {
  unsigned long long limb[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
  for (int e = 1; e < 255; ++e) add_shifted_576(limb, bins[e], 2 * e - 2);
  if (pieces)
    for (int k = 0; k < 4; ++k) add_shifted_576(limb, pieces[k], 32 * k + 2 * Eb - 2);
  int top = -1;
  for (int j = 8; j >= 0 && top < 0; --j)
    if (limb[j]) top = 64 * j + 63 - __clzll(static_cast<long long>(limb[j]));
  if (top < 0) return 0.0;
  auto bit = [&](int i) -> unsigned long long { return (limb[i >> 6] >> (i & 63)) & 1ull; };
  int shift = top > 52 ? top - 52 : 0;
  unsigned long long M = 0;
  for (int b = top; b >= shift; --b) M = (M << 1) | bit(b);
  if (shift > 0) {
    const unsigned long long half = bit(shift - 1);
    bool sticky = false;
    for (int b = shift - 2; b >= 0 && !sticky; --b) sticky = bit(b) != 0;
    if (half && (sticky || (M & 1ull))) {
      ++M;
      if (M == (1ull << 53)) {
        M >>= 1;
        ++shift;
      }
    }
  }
  // M * 2^(shift - 266): M < 2^53 and the exponent stays inside the normal range.
  return static_cast<double>(M) * __longlong_as_double(static_cast<long long>(1023 + shift - 266) << 52);
}

}  // namespace
}  // namespace zc
