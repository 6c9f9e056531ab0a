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
// n % 8 values, summed one by one), so the grid total S_est satisfies |S_est - S| < 2^-17 S.  The last CTA evaluates the rule at S_est (1 -+ 2^-16),
// rounded outward; when both ends give the same e0 (all but ~4e-5 of random tensors) that e0
// is exactly the one the correctly rounded S gives, because the rule is monotone in S.
// Otherwise a follow-on kernel recomputes S exactly with per-exponent integer sums over the
// whole grid.
//
// Stream form (the third technique: send the data natively when coding does not pay).  The pass
// also counts the exponents of a sample, two values in every 64, and the last CTA predicts the
// coded stream's length from the sample's share of escapes p under the chosen e0: the fixed
// parts plus min(3p, 1) bytes per value (a list of 3-byte entries, or a plane of one byte per
// value once that is smaller).  When that prediction is clearly past the raw form's length, the
// decide kernel takes the raw pass: it counts every chunk's escapes exactly, so the form it
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

  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  hist[threadIdx.x] = 0;
  __syncthreads();
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
    if (p.predict) {  // the sample: the first value of the lane's first vector, the last of its last
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
  if (p.predict) {  // the CTA's sample into the grid's counts, before this CTA reports
    if (hist[threadIdx.x]) atomicAdd(p.sample + threadIdx.x, static_cast<unsigned long long>(hist[threadIdx.x]));
    __threadfence();
    __syncthreads();
  }
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
    p.ctrl->e0 = e0;  // when not settled: the lower end's e0, the exact kernel's window anchor
    p.ctrl->n_finite = n_f;
    p.ctrl->exact_path = settled ? 0u : 1u;  // the exact kernel that follows decides then
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

// The exact fallback over the whole grid.  Every thread sums sig^2 4^d exactly in a 128-bit
// integer, d = E - Eb for the values whose exponent E lies in a 24-binade window from Eb (a window
// around the typical value, anchored on the statistics pass's estimate of e0; a term is below 2^62,
// so 2^66 of them fit); values outside it add sig^2 to their exponent's bin (shared atomics).  The
// window sums go to the control block in 32-bit pieces and the bins to the workspace (64-bit
// atomics; neither overflows), and the last CTA to finish rounds the 576-bit total once to fp64
// (exact_from_bins) and picks e0.
constexpr int kExactWindow = 24;

__device__ __noinline__ void exact_fallback(const uint16_t* x, uint64_t n, Control* ctrl, unsigned long long* gbins) {
  __shared__ unsigned long long bins[256];
  __shared__ unsigned long long pieces[4];
  __shared__ int is_last;
  const unsigned lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 256; i += kThreads) bins[i] = 0;
  if (threadIdx.x < 4) pieces[threadIdx.x] = 0;
  __syncthreads();
  int Eb = __ldcg(&ctrl->e0) - 12;  // e0 + 5 is about the typical exponent of a Gaussian tensor
  Eb = Eb < 1 ? 1 : (Eb > 254 - kExactWindow ? 254 - kExactWindow : Eb);
  unsigned long long lo = 0, hi = 0;
  auto add = [&](unsigned b) {
    const unsigned E = (b >> 7) & 0xFF;
    if (E == 255 || (b & 0x7FFF) == 0) return;
    const unsigned Ep = E ? E : 1, sig = E ? 128 + (b & 0x7F) : (b & 0x7F);
    const unsigned d = Ep - static_cast<unsigned>(Eb);
    if (d < static_cast<unsigned>(kExactWindow)) {
      const unsigned long long t = static_cast<unsigned long long>(sig * sig) << (2 * d);
      lo += t;
      hi += lo < t;
    } else {
      atomicAdd(bins + Ep, static_cast<unsigned long long>(sig * sig));
    }
  };
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads, nv = n / 8;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  constexpr int kUnroll = 4;  // 16-byte loads in flight per thread
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < nv; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = i + u * stride < nv ? __ldcs(xv + i + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) add((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
    }
  }
  if (blockIdx.x == 0)
    for (uint64_t i = 8 * nv + threadIdx.x; i < n; i += kThreads) add(x[i]);  // the last n % 8 values
  // the window sums in 32-bit pieces, summed over the warp, then the CTA
  unsigned long long pc[4] = {lo & 0xFFFFFFFFull, lo >> 32, hi & 0xFFFFFFFFull, hi >> 32};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pc[k] += __shfl_xor_sync(0xFFFFFFFFu, pc[k], o);
    if (lane == 0 && pc[k]) atomicAdd(pieces + k, pc[k]);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 256; e += kThreads)
    if (bins[e]) atomicAdd(gbins + e, bins[e]);
  if (threadIdx.x < 4 && pieces[threadIdx.x]) atomicAdd(&ctrl->exact_pieces[threadIdx.x], pieces[threadIdx.x]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&ctrl->exact_done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int e = threadIdx.x; e < 256; e += kThreads) bins[e] = __ldcg(gbins + e);
  if (threadIdx.x < 4) pieces[threadIdx.x] = __ldcg(&ctrl->exact_pieces[threadIdx.x]);
  __syncthreads();
  if (threadIdx.x == 0) ctrl->e0 = select_e0(exact_from_bins(bins, pieces, Eb), __ldcg(&ctrl->n_finite));
}


// The raw pass: one warp per chunk (16 vectors of 16 bytes per lane, in two halves).  Every value is copied to
// its place in the raw form (header, then the values, then zero padding to 16 bytes) and every
// chunk's escapes are counted under e0 as the encoder codes them, giving its escape section's
// size (a list of 3k bytes when 3k <= m, else a plane of m, padded to 16) and, summed over the
// grid, the coded stream's exact length.  The last CTA compares the two lengths: when the coded
// form is longer it finishes the raw form (the header and the length) and marks the stream done;
// otherwise (ties keep the coded form) the encode kernel writes the coded form over it.
constexpr int kRawVecPerLane = kChunk / 8 / 32;  // 16

// Escapes among the two values of w (codes7_x2 gives 7 << 7 exactly for them).
__device__ __forceinline__ unsigned escapes_x2(uint32_t w, uint32_t kadd, uint32_t keep = 0xFFFFFFFFu) {
  return __popc(((codes7_x2(w, kadd) & keep) + 0x00800080u) & 0x04000400u);
}

__device__ __noinline__ void raw_pass(const uint16_t* x, uint64_t n, Control* ctrl, uint8_t* out,
                                      unsigned long long* out_bytes) {
  __shared__ unsigned long long warp_bytes[kWarps];
  __shared__ int is_last;
  const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e0 = __ldcg(&ctrl->e0);
  const uint32_t kadd = ((256u - static_cast<unsigned>(e0)) << 7) * 0x00010001u;
  const uint64_t N = num_chunks(n), nv = n / 8, full_chunks = n / kChunk;
  const uint4* src = reinterpret_cast<const uint4*>(x);
  uint4* dst = reinterpret_cast<uint4*>(out + kHeaderBytes);
  unsigned long long bytes = 0;  // lane 0: the escape sections of this warp's chunks
  for (uint64_t c = static_cast<uint64_t>(blockIdx.x) * kWarps + warp; c < N;
       c += static_cast<uint64_t>(gridDim.x) * kWarps) {
    unsigned esc = 0, m = kChunk;
    if (c < full_chunks) {
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {  // two halves of 8 vectors per lane (64 registers in all)
        const uint64_t b = c * (kChunk / 8) + 32 * (kRawVecPerLane / 2) * h + lane;
        uint4 v[kRawVecPerLane / 2];
#pragma unroll
        for (int j = 0; j < kRawVecPerLane / 2; ++j) v[j] = __ldcs(src + b + 32 * j);
#pragma unroll
        for (int j = 0; j < kRawVecPerLane / 2; ++j) {
          __stcs(dst + b + 32 * j, v[j]);
          esc += escapes_x2(v[j].x, kadd) + escapes_x2(v[j].y, kadd) + escapes_x2(v[j].z, kadd) +
                 escapes_x2(v[j].w, kadd);
        }
      }
    } else {  // the ragged last chunk: its m values, the last vector completed with zeros
      m = static_cast<unsigned>(n - c * kChunk);
      for (unsigned i = lane; i < (m + 7) / 8; i += 32) {
        const uint64_t g = c * (kChunk / 8) + i;
        uint32_t w[4];
        if (g < nv) {
          const uint4 t = __ldcs(src + g);
          w[0] = t.x, w[1] = t.y, w[2] = t.z, w[3] = t.w;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint64_t v = 8 * g + 2 * q;
            w[q] = (v < n ? static_cast<uint32_t>(x[v]) : 0u) | (v + 1 < n ? static_cast<uint32_t>(x[v + 1]) << 16 : 0u);
          }
        }
        __stcs(dst + g, make_uint4(w[0], w[1], w[2], w[3]));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const unsigned v = 8 * i + 2 * q;
          esc += escapes_x2(w[q], kadd, (v < m ? 0x0000FFFFu : 0u) | (v + 1 < m ? 0xFFFF0000u : 0u));
        }
      }
    }
    const unsigned k = __reduce_add_sync(0xFFFFFFFFu, esc);
    if (lane == 0) bytes += 3 * k <= m ? pad16(3 * k) : pad16(m);
  }
  if (lane == 0) warp_bytes[warp] = bytes;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long sum = 0;
    for (int i = 0; i < kWarps; ++i) sum += warp_bytes[i];
    if (sum) atomicAdd(&ctrl->raw_escape_bytes, sum);
    __threadfence();
    is_last = atomicAdd(&ctrl->raw_pass_done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last || threadIdx.x != 0) return;
  __threadfence();
  const unsigned long long coded = escape_base(n) + __ldcg(&ctrl->raw_escape_bytes), raw = raw_stream_bytes(n);
  if (coded <= raw) return;
  unsigned long long* hdr = reinterpret_cast<unsigned long long*>(out);
  hdr[0] = kRawMagicWord | (static_cast<unsigned long long>(e0) << 56);
  hdr[1] = n;
  hdr[2] = 0;
  hdr[3] = raw;
  ctrl->total = raw;
  if (out_bytes) *out_bytes = raw;
  ctrl->raw_done = 1;
}

// After the statistics kernel in auto mode (a programmatic dependent launch): the exact fallback
// when that kernel's estimate could not settle e0, the raw pass when its sample predicted a raw
// stream, nothing otherwise (the two never meet: no prediction is made without a settled e0).
__global__ void __launch_bounds__(kThreads, 4) decide_kernel(const uint16_t* x, uint64_t n, Control* ctrl,
                                                          unsigned long long* gbins, uint8_t* out,
                                                          unsigned long long* out_bytes) {
  asm volatile("griddepcontrol.launch_dependents;");  // the encode kernel may start its copies
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the statistics kernel's verdict
  if (__ldcg(&ctrl->exact_path) != 0)
    exact_fallback(x, n, ctrl, gbins);
  else if (__ldcg(&ctrl->raw_predicted) != 0)
    raw_pass(x, n, ctrl, out, out_bytes);
}

}  // namespace

cudaError_t stats_occupancy(int* stats_per_sm, int* decide_per_sm) {
  const cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(stats_per_sm, stats_kernel, kThreads, 0);
  if (err != cudaSuccess) return err;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(decide_per_sm, decide_kernel, kThreads, 0);
}

cudaError_t launch_stats(const uint16_t* in, uint64_t n, uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream,
                         bool predict_raw) {
  StatsParams p;
  p.in = reinterpret_cast<const uint4*>(in);
  p.n = n;
  p.ctrl = reinterpret_cast<Control*>(ws);
  p.partials = reinterpret_cast<StatsPartial*>(ws + kWsControlBytes);
  p.sample = reinterpret_cast<unsigned long long*>(ws + kWsSampleOffset);
  p.status = dev.status;
  p.predict = predict_raw ? 1 : 0;
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

namespace zc {

cudaError_t launch_decide(const uint16_t* in, uint64_t n, uint8_t* out, unsigned long long* out_bytes, uint8_t* ws,
                          const DeviceInfo& dev, cudaStream_t stream) {
  const uint64_t blocks = (n + 8 * kThreads - 1) / (8 * kThreads);  // at least 8 values per thread
  uint64_t grid = static_cast<uint64_t>(dev.decide_per_sm > 0 ? dev.decide_per_sm : 1) * dev.sm_count;  // one wave
  if (grid > blocks) grid = blocks;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // after our own statistics kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TimingRecord t = timing_begin(ZC_KERNEL_DECIDE, stream);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, decide_kernel, in, n, reinterpret_cast<Control*>(ws),
                                             reinterpret_cast<unsigned long long*>(ws + kWsExactBinsOffset), out,
                                             out_bytes);
  timing_end(t, stream);
  return err;
}

}  // namespace zc
