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
// loop; a lane whose block holds Inf or NaN clears and counts them first (they add nothing).
// Every block sum carries a relative error below 2^-18 (at most 17 roundings, or 64 for the last
// n % 8 values, summed one by one), so the grid total S_est satisfies |S_est - S| < 2^-17 S.
// The last CTA evaluates the rule at S_est (1 -+ 2^-16), rounded outward; when both ends give
// the same e0 (all but ~4e-5 of random tensors) that e0 is exactly the one the correctly
// rounded S gives, because the rule is monotone in S.
// Otherwise the encode kernel's first phase recomputes S exactly with per-exponent integer sums
// over the whole grid.
//
// Stream form (the third technique: send the data natively when coding does not pay).  The pass
// also counts the exponents of a sample, two values in every 256, and the last CTA predicts the
// coded stream's length from the sample's share of escapes p under the chosen e0: the fixed
// parts plus min(3p, 1) bytes per value (a list of 3-byte entries, or a plane of one byte per
// value once that is smaller).  When that prediction is clearly past the raw form's length, the
// encode kernel takes the raw pass first: it counts every chunk's escapes exactly, so the form it
// keeps is the one the rule gives, while it copies the values to their place in the raw form.
// A prediction only chooses the route; a wrong one costs time, never a different stream.
#include "zc_common.cuh"
#include "zc_stats_core.cuh"

namespace zc {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 4;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerLane = 8;               // 8 x 16 B = 64 values per lane per block
constexpr int kVecPerWarpBlock = 32 * kVecPerLane;
static_assert(kThreads == 256, "one thread per exponent of the sample");
struct StatsParams {
  const uint4* in;
  uint64_t n;
  Control* ctrl;
  StatsPartial* partials;
  unsigned long long* sample;  // 256 exponent counts of the sample
  int* status;
  int predict;                 // sample the exponents and predict the stream form
  int gated;                   // after the speculative path: run only when it fell back
};

// The prediction: the coded stream's length with min(3p, 1) escape bytes per value (p the
// sample's share of escapes under e0), against the raw form's length with a margin of 1/32.
__device__ bool predict_raw(uint64_t n, unsigned long long sampled, unsigned long long escapes) {
  if (sampled == 0) return false;
  const double per_value = fmin(3.0 * static_cast<double>(escapes) / static_cast<double>(sampled), 1.0);
  const double coded = static_cast<double>(escape_base(n)) + per_value * static_cast<double>(n);
  return coded > static_cast<double>(raw_stream_bytes(n)) * (1.0 + 1.0 / 32);
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) stats_kernel(StatsParams p) {
  // The encode kernel that follows may start now (it waits for this kernel before it reads e0).
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ double red_sum[kWarps];
  __shared__ unsigned long long red_nf[kWarps], red_win[kWarps];
  __shared__ unsigned hist[256];  // the CTA's exponent sample
  __shared__ int is_last, settled_e0;
  if (p.gated) {  // the steps before it (the speculative coding pass, the reset) are done first
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (__ldcg(&p.ctrl->fallback) == 0) return;
  }

  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  hist[threadIdx.x] = 0;
  __syncthreads();
  const uint64_t nv = p.n >> 3;  // whole 16-byte vectors
  const uint64_t warps_total = static_cast<uint64_t>(gridDim.x) * kWarps;
  double acc = 0.0;
  unsigned nonfinite = 0;

  unsigned turn = lane;  // the sample: a quarter of the lanes per block, in turn
  for (uint64_t wb = (static_cast<uint64_t>(blockIdx.x) * kWarps + warp) * kVecPerWarpBlock; wb < nv;
       wb += warps_total * kVecPerWarpBlock, ++turn) {
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
    if (p.predict && (turn & 3) == 0) {  // the first value of the lane's first vector, the last of its last
      if (full || wb + lane < nv) atomicAdd(&hist[(w[0] >> 7) & 0xFF], 1u);
      if (full || wb + 32 * (kVecPerLane - 1) + lane < nv) atomicAdd(&hist[(w[31] >> 23) & 0xFF], 1u);
    }
    block_sum(w, &acc, &nonfinite);
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
  if (warp == 0) {
    // Warp 0 reports: lane 0 the partials, every lane eight of the sample's counts; each lane's
    // fence makes its own writes visible before lane 0 takes the completion ticket.
    if (p.predict)
      for (unsigned b = lane; b < 256; b += 32)
        if (hist[b]) atomicAdd(p.sample + b, static_cast<unsigned long long>(hist[b]));
    if (lane == 0) {
      double s = 0.0;
      unsigned long long c = 0;
      for (int i = 0; i < kWarps; ++i) {
        s += red_sum[i];
        c += red_nf[i];
      }
      p.partials[blockIdx.x].sum = s;
      p.partials[blockIdx.x].nonfinite = c;
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) is_last = atomicAdd(&p.ctrl->stats_done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const unsigned long long bin = p.predict ? __ldcg(p.sample + threadIdx.x) : 0ull;

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
  if (threadIdx.x == 0) {
    double S = 0.0;
    unsigned long long nonfin = 0;
    for (int i = 0; i < kWarps; ++i) {
      S += red_sum[i];
      nonfin += red_nf[i];
    }
    const unsigned long long n_f = p.n - nonfin;
    int e0 = 0;
    const bool settled = decide_e0(S, n_f, &e0);
    p.ctrl->e0 = e0;  // when not settled: the lower end's e0, the exact sums' window anchor
    p.ctrl->n_finite = n_f;
    p.ctrl->exact_path = settled ? 0u : 1u;  // the encode kernel's first phase decides then
    settled_e0 = settled ? e0 : -1;
  }
  if (!p.predict) return;
  __syncthreads();
  const int e0 = settled_e0;
  if (e0 < 0) return;  // the exact fallback decides e0; no prediction then
  // the sample's size and its values inside the window [e0, e0 + 6]
  unsigned long long tot = bin, win = threadIdx.x - static_cast<unsigned>(e0) < 7u ? bin : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_down_sync(0xFFFFFFFFu, tot, o);
    win += __shfl_down_sync(0xFFFFFFFFu, win, o);
  }
  if (lane == 0) {
    red_nf[warp] = tot;
    red_win[warp] = win;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long T = 0, W = 0;
    for (int i = 0; i < kWarps; ++i) {
      T += red_nf[i];
      W += red_win[i];
    }
    p.ctrl->raw_predicted = predict_raw(p.n, T, T - W) ? 1u : 0u;
  }
}

// ------------------------------------------------------------------ the sample pass
//
// The speculative path codes the tensor with the e0 of a sample and checks it afterwards against
// the e0 of the whole tensor, which the coding pass sums as it goes (so the input is read once
// on that path, not twice).  The sample: one 16-byte vector (8 values) of every full chunk, the
// vector (37 c + 11) mod 512 of chunk c, so that a structure repeating with the chunks is not
// sampled at one place only.  Lane L of global warp g takes chunks 256 g + 32 j + L, j < 8: 64
// values, whose sums of squares and of fourth powers it takes (in fp32, scaled by a power of two
// from the lane's largest magnitude); the first value of each vector goes to an exponent
// histogram.  The last CTA takes
// the sample's e0 as the guess, and declares the guess confident only when (a) the rule gives the
// same e0 at the sample's mean square times 1 -+ (4 r + 1/32), r the mean square's relative
// standard error estimated from the fourth powers -- so a tensor near a switching point, or one
// whose sum of squares a few large values dominate (which a sample estimates badly), goes the
// safe way --, (b) the stream the sample predicts under that e0 (the fixed parts plus min(3p, 1)
// bytes per value, p the sample's share of escapes) is shorter than 0.95 of the raw form (a
// stream that may come out raw goes the way that predicts it exactly) and (c) the sample has a
// finite nonzero value.  Otherwise it sets the fallback word, and the statistics and encode
// kernels do the job as without the speculation.  A guess only chooses the route: the coding
// pass's exact check decides.
constexpr int kSampleThreads = 128;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr uint64_t kSampleChunksPerCta = 32ull * 8 * kSampleWarps;  // 1024

// Sums of squares and of fourth powers of a lane's 64 values (32 words) in fp32, every value
// scaled by 2^(126 - Es), Es the lane's largest biased exponent clamped to [1, 252] (so no power
// overflows, and what underflows is negligible beside the largest); Inf and NaN are counted and
// left out.  For the sample's guess only: no error bound is claimed.
__device__ void lane_moments(const uint32_t (&w)[32], double* s2, double* s4, unsigned* nonfinite) {
  unsigned mx = 0, nf = 0;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const unsigned a = (w[i >> 1] >> (16 * (i & 1))) & 0x7FFFu;
    if (a >= 0x7F80u) ++nf;
    else mx = max(mx, a);
  }
  *nonfinite += nf;
  if (mx == 0) return;
  const int Es = min(max(static_cast<int>(mx >> 7), 1), 252);
  const float sc = __int_as_float((253 - Es) << 23);
  float a2 = 0.f, a4 = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const uint32_t h = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
    if ((h & 0x7FFFu) >= 0x7F80u) continue;
    const float x = __uint_as_float(h << 16) * sc;
    const float x2 = x * x;
    a2 += x2;
    a4 = fmaf(x2, x2, a4);
  }
  *s2 += static_cast<double>(a2) * __longlong_as_double(static_cast<long long>(1023 + 2 * Es - 252) << 52);
  *s4 += static_cast<double>(a4) * __longlong_as_double(static_cast<long long>(1023 + 4 * Es - 504) << 52);
}

struct SampleParams {
  const uint4* in;
  uint64_t n;
  Control* ctrl;
  unsigned long long* bins;  // 256 exponent counts of the sample (cleared)
};

__global__ void __launch_bounds__(kSampleThreads) sample_kernel(SampleParams p) {
  asm volatile("griddepcontrol.launch_dependents;");  // the coding pass takes its tickets meanwhile
  __shared__ unsigned hist[256];
  __shared__ double red_sum[kSampleWarps], red_sum4[kSampleWarps];
  __shared__ unsigned long long red_cnt[kSampleWarps];
  __shared__ int is_last;
  __shared__ int e_at[3];
  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (unsigned b = threadIdx.x; b < 256; b += kSampleThreads) hist[b] = 0;
  __syncthreads();
  const uint64_t full = p.n / kChunk;
  const uint64_t c0 = (static_cast<uint64_t>(blockIdx.x) * kSampleWarps + warp) * 256 + lane;
  uint32_t w[32];
  unsigned valid = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint64_t c = c0 + 32 * j;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (c < full) {
      v = __ldg(p.in + c * (kChunk / 8) + ((37 * c + 11) & (kChunk / 8 - 1)));
      valid += 8;
    }
    w[4 * j] = v.x;
    w[4 * j + 1] = v.y;
    w[4 * j + 2] = v.z;
    w[4 * j + 3] = v.w;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)  // the histogram takes the first value of each vector (few atomics on few bins)
    if (c0 + 32 * j < full) atomicAdd(&hist[(w[4 * j] >> 7) & 0xFF], 1u);
  double acc = 0.0, acc4 = 0.0;
  unsigned nonfinite = 0;
  lane_moments(w, &acc, &acc4, &nonfinite);
  unsigned long long fin = valid - nonfinite;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    acc += __shfl_down_sync(0xFFFFFFFFu, acc, o);
    acc4 += __shfl_down_sync(0xFFFFFFFFu, acc4, o);
    fin += __shfl_down_sync(0xFFFFFFFFu, fin, o);
  }
  if (lane == 0) {
    red_sum[warp] = acc;
    red_sum4[warp] = acc4;
    red_cnt[warp] = fin;
  }
  __syncthreads();
  for (unsigned b = threadIdx.x; b < 256; b += kSampleThreads)
    if (hist[b]) atomicAdd(p.bins + b, static_cast<unsigned long long>(hist[b]));
  if (threadIdx.x == 0) {
    double s = 0.0, s4 = 0.0;
    unsigned long long f = 0;
    for (int i = 0; i < kSampleWarps; ++i) {
      s += red_sum[i];
      s4 += red_sum4[i];
      f += red_cnt[i];
    }
    atomicAdd(&p.ctrl->sample_sum, s);
    atomicAdd(&p.ctrl->sample_sum4, s4);
    atomicAdd(&p.ctrl->sample_finite, f);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    is_last = atomicAdd(&p.ctrl->sample_done, 1u) == gridDim.x - 1;
    __threadfence();
  }
  __syncthreads();
  if (!is_last) return;
  const double S = __ldcg(&p.ctrl->sample_sum), Q = __ldcg(&p.ctrl->sample_sum4);
  const unsigned long long nf = __ldcg(&p.ctrl->sample_finite);
  if (threadIdx.x < 3) {  // the rule at S (1 - d), S and S (1 + d), one per thread
    float d = 1.0f / 32;
    if (nf > 0 && S > 0.0) {  // 4 relative standard errors of the mean square: r^2 = (Q m / S^2 - 1) / m
      const float m = static_cast<float>(nf), ratio = static_cast<float>(Q * static_cast<double>(nf) / (S * S));
      d += 4.0f * sqrtf(fmaxf(ratio - 1.0f, 0.0f) / m);
    }
    d = fminf(d, 0.75f);
    e_at[threadIdx.x] =
        select_e0(S * (threadIdx.x == 0 ? 1.0 - d : threadIdx.x == 1 ? 1.0 : 1.0 + static_cast<double>(d)), nf);
  }
  __syncthreads();
  const int e0 = e_at[1];
  // the sample's size and its values inside the window [e0, e0 + 6]
  const unsigned long long bin0 = __ldcg(p.bins + threadIdx.x), bin1 = __ldcg(p.bins + threadIdx.x + 128);
  unsigned long long tot = bin0 + bin1;
  unsigned long long win = (threadIdx.x - static_cast<unsigned>(e0) < 7u ? bin0 : 0ull) +
                           (threadIdx.x + 128 - static_cast<unsigned>(e0) < 7u ? bin1 : 0ull);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_down_sync(0xFFFFFFFFu, tot, o);
    win += __shfl_down_sync(0xFFFFFFFFu, win, o);
  }
  if (lane == 0) {
    red_cnt[warp] = tot;
    red_sum[warp] = static_cast<double>(win);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long T = 0, W = 0;
    for (int i = 0; i < kSampleWarps; ++i) {
      T += red_cnt[i];
      W += static_cast<unsigned long long>(red_sum[i]);
    }
    bool confident = S > 0.0 && nf > 0 && T > 0 && e_at[0] == e0 && e_at[2] == e0;
    if (confident) {
      const double per_value = fmin(3.0 * static_cast<double>(T - W) / static_cast<double>(T), 1.0);
      const double coded = static_cast<double>(escape_base(p.n)) + per_value * static_cast<double>(p.n);
      confident = coded < 0.95 * static_cast<double>(raw_stream_bytes(p.n));
    }
    p.ctrl->e0_guess = e0;
    p.ctrl->fallback = confident ? 0u : 1u;
  }
}

}  // namespace

cudaError_t launch_sample(const uint16_t* in, uint64_t n, uint8_t* ws, cudaStream_t stream) {
  SampleParams p;
  p.in = reinterpret_cast<const uint4*>(in);
  p.n = n;
  p.ctrl = reinterpret_cast<Control*>(ws);
  p.bins = reinterpret_cast<unsigned long long*>(ws + kWsSampleOffset);
  const uint64_t full = n / kChunk;
  uint64_t grid = (full + kSampleChunksPerCta - 1) / kSampleChunksPerCta;
  if (grid < 1) grid = 1;
  TimingRecord t = timing_begin(ZC_KERNEL_SAMPLE, stream);
  sample_kernel<<<static_cast<unsigned>(grid), kSampleThreads, 0, stream>>>(p);
  timing_end(t, stream);
  return cudaGetLastError();
}

cudaError_t stats_occupancy(int* per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, stats_kernel, kThreads, 0);
}

cudaError_t launch_stats(const uint16_t* in, uint64_t n, uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream,
                         bool predict_raw, bool gated) {
  StatsParams p;
  p.in = reinterpret_cast<const uint4*>(in);
  p.n = n;
  p.ctrl = reinterpret_cast<Control*>(ws);
  p.partials = reinterpret_cast<StatsPartial*>(ws + kWsControlBytes);
  p.sample = reinterpret_cast<unsigned long long*>(ws + kWsSampleOffset);
  p.status = dev.status;
  p.predict = predict_raw ? 1 : 0;
  p.gated = gated ? 1 : 0;
  const uint64_t nv = n >> 3;
  const uint64_t blocks_needed = (nv + kVecPerWarpBlock * kWarps - 1) / (kVecPerWarpBlock * kWarps);
  const int per_sm = dev.stats_per_sm;
  uint64_t grid = static_cast<uint64_t>(per_sm > 0 ? per_sm : 1) * dev.sm_count;  // one wave
  if (grid > blocks_needed) grid = blocks_needed;
  if (grid < 1) grid = 1;
  if (grid > kStatsMaxCtas) grid = kStatsMaxCtas;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  // Gated, it follows our own kernels (it waits for them before it reads anything).
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = gated ? 1 : 0;
  TimingRecord t = timing_begin(ZC_KERNEL_STATS, stream);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, stats_kernel, p);
  timing_end(t, stream);
  return err;
}

}  // namespace zc
