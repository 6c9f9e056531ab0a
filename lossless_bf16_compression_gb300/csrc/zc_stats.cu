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
  int gated;                   // after the speculative encode kernel: run only when it fell back
  unsigned long long* flags;   // gated: the scan state, cleared here for the encode kernel after
  uint64_t flag_words;
};

// The prediction: the coded stream's length with min(3p, 1) escape bytes per value (p the
// sample's share of escapes under e0), against the raw form's length with a margin of 1/32.
__device__ bool predict_raw(uint64_t n, unsigned long long sampled, unsigned long long escapes) {
  if (sampled == 0) return false;
  const double per_value = fmin(3.0 * static_cast<double>(escapes) / static_cast<double>(sampled), 1.0);
  const double coded = static_cast<double>(escape_base(n)) + per_value * static_cast<double>(n);
  return coded > static_cast<double>(raw_stream_bytes(n)) * (1.0 + 1.0 / 32);
}

// Scratch of one 256-thread CTA of the statistics pass.
struct StatsScratch {
  double red_sum[kWarps];
  unsigned long long red_nf[kWarps], red_win[kWarps];
  unsigned hist[256];  // the CTA's exponent sample
  int is_last, settled_e0;
};

// CTA `cta` of `ctas`: block sums over its share of the input (and, predicting, the exponent
// sample); its partial goes to partials[cta] and its sample counts to the global sample bins.
__device__ void stats_share(const StatsParams& p, unsigned cta, unsigned ctas, StatsScratch& T) {
  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T.hist[threadIdx.x] = 0;
  __syncthreads();
  const uint64_t nv = p.n >> 3;  // whole 16-byte vectors
  const uint64_t warps_total = static_cast<uint64_t>(ctas) * kWarps;
  double acc = 0.0;
  unsigned nonfinite = 0;

  unsigned turn = lane;  // the sample: a quarter of the lanes per block, in turn
  for (uint64_t wb = (static_cast<uint64_t>(cta) * kWarps + warp) * kVecPerWarpBlock; wb < nv;
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
      if (full || wb + lane < nv) atomicAdd(&T.hist[(w[0] >> 7) & 0xFF], 1u);
      if (full || wb + 32 * (kVecPerLane - 1) + lane < nv) atomicAdd(&T.hist[(w[31] >> 23) & 0xFF], 1u);
    }
    block_sum(w, &acc, &nonfinite);
  }
  if (cta == 0 && threadIdx.x == 0 && (p.n & 7))
    acc += tail_block(reinterpret_cast<const uint16_t*>(p.in) + (nv << 3), static_cast<unsigned>(p.n & 7), &nonfinite);

  // CTA reduction in a fixed order.
  unsigned long long nf = nonfinite;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    acc += __shfl_down_sync(0xFFFFFFFFu, acc, o);
    nf += __shfl_down_sync(0xFFFFFFFFu, nf, o);
  }
  if (lane == 0) {
    T.red_sum[warp] = acc;
    T.red_nf[warp] = nf;
  }
  __syncthreads();
  if (warp == 0) {
    if (p.predict)
      for (unsigned b = lane; b < 256; b += 32)
        if (T.hist[b]) atomicAdd(p.sample + b, static_cast<unsigned long long>(T.hist[b]));
    if (lane == 0) {
      double s = 0.0;
      unsigned long long c = 0;
      for (int i = 0; i < kWarps; ++i) {
        s += T.red_sum[i];
        c += T.red_nf[i];
      }
      p.partials[cta].sum = s;
      p.partials[cta].nonfinite = c;
    }
  }
}

// The last CTA, with every partial and sample count published: combine the partials in index
// order (fixed tree), pick e0 (or ask for the exact sums), and predict the stream form.
__device__ void stats_settle(const StatsParams& p, unsigned ctas, StatsScratch& T) {
  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long bin = p.predict ? __ldcg(p.sample + threadIdx.x) : 0ull;
  double s = 0.0;
  unsigned long long c = 0;
  for (unsigned i = threadIdx.x; i < ctas; i += kThreads) {
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
    T.red_sum[warp] = s;
    T.red_nf[warp] = c;
  }
  __syncthreads();
  if (threadIdx.x < 2) {  // both the same sums; one end of the rule each
    double S = 0.0;
    unsigned long long nonfin = 0;
    for (int i = 0; i < kWarps; ++i) {
      S += T.red_sum[i];
      nonfin += T.red_nf[i];
    }
    const unsigned long long n_f = p.n - nonfin;
    int e0 = 0;
    const bool settled = decide_e0_pair(S, n_f, &e0);
    if (threadIdx.x == 0) {
      p.ctrl->e0 = e0;  // when not settled: the lower end's e0, the exact sums' window anchor
      p.ctrl->n_finite = n_f;
      p.ctrl->exact_path = settled ? 0u : 1u;  // the encode kernel's first phase decides then
      T.settled_e0 = settled ? e0 : -1;
    }
  }
  __syncthreads();
  if (!p.predict) return;
  const int e0 = T.settled_e0;
  if (e0 < 0) return;  // the exact fallback decides e0; no prediction then
  // the sample's size and its values inside the window [e0, e0 + 6]
  unsigned long long tot = bin, win = threadIdx.x - static_cast<unsigned>(e0) < 7u ? bin : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_down_sync(0xFFFFFFFFu, tot, o);
    win += __shfl_down_sync(0xFFFFFFFFu, win, o);
  }
  if (lane == 0) {
    T.red_nf[warp] = tot;
    T.red_win[warp] = win;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long Tn = 0, W = 0;
    for (int i = 0; i < kWarps; ++i) {
      Tn += T.red_nf[i];
      W += T.red_win[i];
    }
    p.ctrl->raw_predicted = predict_raw(p.n, Tn, Tn - W) ? 1u : 0u;
  }
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) stats_kernel(StatsParams p) {
  // The encode kernel that follows may start now (it waits for this kernel before it reads e0).
  if (!p.gated) asm volatile("griddepcontrol.launch_dependents;");
  __shared__ StatsScratch T;
  __shared__ int go;
  if (p.gated) {
    // After the speculative encode kernel: run only when it fell back, and then leave the
    // workspace as the encode kernel after this one expects it -- its tickets, counters, exact
    // sums and scan state back at zero (the speculative pass used them; this pass does not).
    if (threadIdx.x == 0) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      go = __ldcg(&p.ctrl->fallback) != 0;
    }
    __syncthreads();
    if (!go) return;  // the encode kernel after this one starts when this one is done
    if (blockIdx.x == 0) {
      if (threadIdx.x == 0) {
        Control& c = *p.ctrl;
        c.encode_ticket = c.role_ticket = c.decode_ticket = c.first_ticket = 0;
        c.first_done = c.first_ready = c.raw_done = 0;
        c.total = c.raw_escape_bytes = 0;
        for (int i = 0; i < 4; ++i) c.exact_pieces[i] = 0;
      }
      unsigned long long* bins = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(p.ctrl) +
                                                                       kWsExactBinsOffset);
      bins[threadIdx.x] = 0;  // 256 threads, 256 bins
    }
    for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < p.flag_words;
         i += static_cast<uint64_t>(gridDim.x) * kThreads)
      p.flags[i] = 0;
    // Only now may the encode kernel start: every CTA's share of the workspace is cleared and
    // visible device-wide before that kernel can take a ticket (it reads e0 only after waiting
    // for this kernel's completion).
    __threadfence();
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;");
  }
  stats_share(p, blockIdx.x, gridDim.x, T);
  if (threadIdx.x < 32) {  // warp 0's writes, then the completion ticket
    __threadfence();
    __syncwarp();
    if (threadIdx.x == 0) T.is_last = atomicAdd(&p.ctrl->stats_done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!T.is_last) return;
  __threadfence();
  stats_settle(p, gridDim.x, T);
}

}  // namespace

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
  p.flags = reinterpret_cast<unsigned long long*>(ws + kWsControlBytes + kWsPartialsBytes);
  p.flag_words = num_chunks(n);
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
  // Gated, it follows our own encode kernel (it waits for it before it touches anything).
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = gated ? 1 : 0;
  TimingRecord t = timing_begin(gated ? ZC_KERNEL_REFIT_STATS : ZC_KERNEL_STATS, stream);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, stats_kernel, p);
  timing_end(t, stream);
  return err;
}

}  // namespace zc
