// zc_stats.cu -- statistics pass: sum of squares of the finite values, count of the
// non-finite ones, and the window base e0 derived from them.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution", first technique: the
// window of frequent exponents is taken from the tensor's standard deviation alone, with no
// histogram and no sort.  e0 = floor(log2(sigma * c)) + 127 clamped to [0, 249], sigma^2 = S / n_f, where S is
// the exact sum of squares rounded once to fp64 and c^2 = 0x1.79a1e790e0f01p-10 (the base
// whose 7-binade window has the fewest expected escapes under a Gaussian).
//
// GB300 design.  The pass is HBM-bound (it reads 2n bytes), and GB300's fp64 rate is far below
// what one fp64 operation per value would need, so values are summed in fp32 blocks of 64 with
// four FFMA chains, and only block sums go to fp64.  Each block's largest magnitude decides
// whether its plain fp32 sum is safe; when a lane's is not, its warp sums with every value
// scaled by a power of two from that magnitude (1 in lanes that need none), so no bit pattern
// of the BF16 range overflows or loses the block's sum to underflow and the warp runs one
// loop; only blocks holding Inf or NaN take a careful path that skips them.  Every block sum carries a relative error below 2^-18 (at most 17 roundings, or
// 64 on the careful path), so the grid total S_est
// satisfies |S_est - S| < 2^-17 S.  The last CTA evaluates the rule at S_est (1 -+ 2^-16),
// rounded outward; when both ends give the same e0 (all but ~4e-5 of random tensors) that e0
// is exactly the one the correctly rounded S gives, because the rule is monotone in S.
// Otherwise the same CTA recomputes S exactly with per-exponent integer sums.
#include "zc_common.cuh"

namespace zc {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 4;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerLane = 8;               // 8 x 16 B = 64 values per lane per block
constexpr int kVecPerWarpBlock = 32 * kVecPerLane;
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

// Careful block sum for 64 values (32 words): skips Inf/NaN, and scales every square by
// 4^-(Emax'-E') relative to the largest exponent present, so no fp32 overflow or underflow
// matters.  Returns the fp64 value of the block sum and adds the non-finite count.
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

// A block holding Inf or NaN, reloaded from memory (so that the fast path's registers need not
// survive the call) and summed by the careful path.
__device__ __noinline__ double careful_block_at(const uint4* in, uint64_t wb, uint64_t nv, unsigned lane,
                                                unsigned* nonfinite) {
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint64_t idx = wb + 32 * j + lane;
    const uint4 v = idx < nv ? __ldg(in + idx) : make_uint4(0, 0, 0, 0);
    w[4 * j] = v.x;
    w[4 * j + 1] = v.y;
    w[4 * j + 2] = v.z;
    w[4 * j + 3] = v.w;
  }
  return careful_block(w, nonfinite);
}

// Block sum of 64 values.  Bit patterns with the sign cleared order like magnitudes, so one
// packed 16-bit max finds the block's largest, and it decides, per warp, between the plain sum
// (every lane's largest biased exponent in [87, 187): no square reaches 2^122 and the block sum
// is at least 2^-80, so the 64 squares, 17 roundings, stay within 2^-19 of the exact sum) and a
// sum with every lane's values scaled by 2^(126 - Es), Es = E clamped to [1, 252] (1 for lanes
// that need no scaling), which puts the largest magnitude in [2^-8, 4): no square overflows and
// what underflows is under 2^-120 of the block sum.  The decision is one warp vote, so a warp runs one of the two loops.
// Blocks holding Inf or NaN take the careful path.
__device__ __forceinline__ void block_sum(const uint32_t (&w)[32], const uint4* in, uint64_t wb, uint64_t nv,
                                          unsigned lane, double* acc, unsigned* nonfinite) {
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) mx = max_u16x2(mx, w[i] & 0x7FFF7FFFu);
  const unsigned m = max(mx & 0xFFFFu, mx >> 16);
  const unsigned E = m >> 7;
  const bool nonfin = m >= 0x7F80u;
  const bool odd = m != 0 && (E >= 187u || E < 87u);
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (!__any_sync(0xFFFFFFFFu, nonfin || odd)) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
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
  if (nonfin) {
    *acc += careful_block_at(in, wb, nv, lane, nonfinite);
    return;
  }
  const int Es = odd ? min(max(static_cast<int>(E), 1), 252) : 126;
  const float sc = __int_as_float((253 - Es) << 23);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
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

struct StatsParams {
  const uint4* in;
  uint64_t n;
  Control* ctrl;
  StatsPartial* partials;
  int* status;
};

// Exact fallback, run by the last CTA alone: per-exponent integer sums of sig^2, then the
// 576-bit integer sum_E T_E 2^(2E-2) (= S 2^266), rounded once to fp64, nearest-even.
__device__ __noinline__ double exact_sum_of_squares(const uint16_t* x, uint64_t n, unsigned long long* bins) {
  const unsigned warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kWarps * 256; i += kThreads) bins[i] = 0;
  __syncthreads();
  unsigned long long* mine = bins + 256 * warp;
  for (uint64_t i = threadIdx.x; i < n; i += kThreads) {
    const unsigned v = x[i];
    const unsigned E = (v >> 7) & 0xFF;
    if (E == 255 || (v & 0x7FFF) == 0) continue;
    const unsigned sig = E ? 128 + (v & 0x7F) : (v & 0x7F);
    atomicAdd(mine + (E ? E : 1), static_cast<unsigned long long>(sig * sig));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 256; e += kThreads) {
    unsigned long long t = 0;
    for (int w = 0; w < kWarps; ++w) t += bins[256 * w + e];
    bins[e] = t;
  }
  __syncthreads();
  double result = 0.0;
  if (threadIdx.x == 0) {
    unsigned long long limb[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    for (int e = 1; e < 255; ++e) {
      const unsigned long long t = bins[e];  // < 2^56
      if (t == 0) continue;
      const int s = 2 * e - 2, li = s >> 6, sh = s & 63;
      unsigned long long add[2] = {t << sh, sh ? t >> (64 - sh) : 0ull};
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
    int top = -1;
    for (int j = 8; j >= 0 && top < 0; --j)
      if (limb[j]) top = 64 * j + 63 - __clzll(static_cast<long long>(limb[j]));
    if (top >= 0) {
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
      result = static_cast<double>(M) *
               __longlong_as_double(static_cast<long long>(1023 + shift - 266) << 52);
    }
  }
  return result;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) stats_kernel(StatsParams p) {
  // The encode kernel that follows may start now (it waits for this kernel before it reads e0).
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ double red_sum[kWarps];
  __shared__ unsigned long long red_nf[kWarps];
  __shared__ unsigned long long bins[kWarps * 256];
  __shared__ int is_last;

  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t nv = p.n >> 3;  // whole 16-byte vectors
  const uint64_t warps_total = static_cast<uint64_t>(gridDim.x) * kWarps;
  double acc = 0.0;
  unsigned nonfinite = 0;

  for (uint64_t wb = (static_cast<uint64_t>(blockIdx.x) * kWarps + warp) * kVecPerWarpBlock; wb < nv;
       wb += warps_total * kVecPerWarpBlock) {
    uint32_t w[32];
    const bool full = wb + kVecPerWarpBlock <= nv;
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
      const uint64_t idx = wb + 32 * j + lane;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (full || idx < nv) v = __ldg(p.in + idx);
      w[4 * j] = v.x;
      w[4 * j + 1] = v.y;
      w[4 * j + 2] = v.z;
      w[4 * j + 3] = v.w;
    }
    block_sum(w, p.in, wb, nv, lane, &acc, &nonfinite);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && (p.n & 7))
    acc += tail_block(reinterpret_cast<const uint16_t*>(p.in) + (nv << 3), static_cast<unsigned>(p.n & 7), &nonfinite);

  // CTA reduction in a fixed order.
  unsigned long long nf = nonfinite;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    acc += __shfl_down_sync(0xFFFFFFFFu, acc, o);
    nf += __shfl_down_sync(0xFFFFFFFFu, nf, o);
  }
  if (lane == 0) {
    red_sum[warp] = acc;
    red_nf[warp] = nf;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    unsigned long long c = 0;
    for (int i = 0; i < kWarps; ++i) {
      s += red_sum[i];
      c += red_nf[i];
    }
    p.partials[blockIdx.x].sum = s;
    p.partials[blockIdx.x].nonfinite = c;
    __threadfence();
    const unsigned ticket = atomicAdd(&p.ctrl->stats_done, 1u);
    is_last = (ticket == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // Last CTA: combine the partials in index order (fixed tree), then pick e0.
  double s = 0.0;
  unsigned long long c = 0;
  for (unsigned i = threadIdx.x; i < gridDim.x; i += kThreads) {
    s += __ldcg(&p.partials[i].sum);
    c += __ldcg(&p.partials[i].nonfinite);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_down_sync(0xFFFFFFFFu, s, o);
    c += __shfl_down_sync(0xFFFFFFFFu, c, o);
  }
  __syncthreads();
  if (lane == 0) {
    red_sum[warp] = s;
    red_nf[warp] = c;
  }
  __syncthreads();
  __shared__ int need_exact;
  __shared__ unsigned long long n_finite;
  if (threadIdx.x == 0) {
    double S = 0.0;
    unsigned long long nonfin = 0;
    for (int i = 0; i < kWarps; ++i) {
      S += red_sum[i];
      nonfin += red_nf[i];
    }
    const unsigned long long n_f = p.n - nonfin;
    n_finite = n_f;
    need_exact = 0;
    int e0 = 0;
    if (n_f != 0 && S != 0.0) {
      const double lo = __dmul_rd(S, 1.0 - 0x1p-16);
      const double hi = __dmul_ru(S, 1.0 + 0x1p-16);
      const int elo = select_e0(lo, n_f), ehi = select_e0(hi, n_f);
      if (elo == ehi) {
        e0 = elo;
      } else {
        need_exact = 1;
      }
    }
    p.ctrl->e0 = e0;
  }
  __syncthreads();
  if (need_exact) {
    const double S = exact_sum_of_squares(reinterpret_cast<const uint16_t*>(p.in), p.n, bins);
    if (threadIdx.x == 0) {
      p.ctrl->e0 = select_e0(S, n_finite);
      p.ctrl->exact_path = 1;
    }
  }
}

}  // namespace

cudaError_t stats_occupancy(int* per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, stats_kernel, kThreads, 0);
}

cudaError_t launch_stats(const uint16_t* in, uint64_t n, uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream) {
  StatsParams p;
  p.in = reinterpret_cast<const uint4*>(in);
  p.n = n;
  p.ctrl = reinterpret_cast<Control*>(ws);
  p.partials = reinterpret_cast<StatsPartial*>(ws + kWsControlBytes);
  p.status = dev.status;
  const uint64_t nv = n >> 3;
  const uint64_t blocks_needed = (nv + kVecPerWarpBlock * kWarps - 1) / (kVecPerWarpBlock * kWarps);
  const int per_sm = dev.stats_per_sm;
  uint64_t grid = static_cast<uint64_t>(per_sm > 0 ? per_sm : 1) * dev.sm_count;  // one wave
  if (grid > blocks_needed) grid = blocks_needed;
  if (grid < 1) grid = 1;
  if (grid > kStatsMaxCtas) grid = kStatsMaxCtas;
  TimingRecord t = timing_begin(ZC_KERNEL_STATS, stream);
  stats_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
  timing_end(t, stream);
  return cudaGetLastError();
}

}  // namespace zc
