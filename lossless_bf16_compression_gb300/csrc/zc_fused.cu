// zc_fused.cu -- compression of a tensor that fits the L2 in one cooperative launch: the
// statistics, an exact escape count per chunk, and the coding, each a pass over the input, the
// second and third served by the L2 (129 MB; a 2^25-value tensor is 64 MiB).
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution": the window base from the
// tensor's standard deviation, 3-bit codes with the full exponents of the others kept apart
// (first technique), and the native form where coding does not pay (third technique).
//
// GB300 design.  G CTAs of 128 threads, as many as the device holds at once, launched
// cooperatively so that all are resident; CTA r owns the contiguous chunks r J .. r J + J - 1.
//  1. Statistics: the statistics kernel's fp32 blocks of 64 values with the same error bound, one
//     partial per CTA, and the CTA's own e0 (the window rule at its own partial).
//  2. Count: one warp per chunk counts its escapes exactly as the coding does, giving the escape
//     section's size, under the CTA's own e0 in auto mode.  The last CTA to reach the barrier
//     adds the partials up in one fixed order and settles e0 for all, checks every CTA's own e0
//     against it, and turns the CTAs' totals into their sections' offsets (an exclusive scan)
//     and the stream's length, so the form is known before anything is written.  When some
//     CTA's own e0 was not the settled one -- or the bound straddles a switching point and the
//     exact per-exponent sums decide e0 after one more barrier -- the chunks are counted again
//     under e0 and another barrier places them.
//  3. Write: each chunk comes into a ring of four shared-memory slots by a bulk async copy, three
//     chunks ahead of the coding (the first three during the statistics pass); the CTA codes it
//     (a thread's 32 consecutive values, code32) and stores its fixed part, its escape section
//     and its offset straight to their places -- or, for the raw form, copies its values behind
//     the header.
// No scan state, look-back, retiring warp or second launch: every place is known before coding.
// The grid barriers count arrivals in the control block (cleared before the launch); every wait
// (the barriers, the copies) is bounded, and after a failed one the CTAs stop.
#include "zc_code_core.cuh"
#include "zc_common.cuh"
#include "zc_grid.cuh"
#include "zc_stats_core.cuh"

#ifndef ZC_FUSED_MAX_LOG2
// The largest tensor this path takes: 2^25 values (64 MiB).  Above it the input no longer stays
// in the L2 between the passes, and the three-kernel path is faster (at 2^26 values, 88 us
// against 95 us on a GB300).
#define ZC_FUSED_MAX_LOG2 25
#endif

namespace zc {
namespace {

constexpr int kThreads = kResidentThreads;  // 128: a chunk's coding threads, 32 values each
static_assert(32 * kThreads == kChunk, "a thread codes 32 consecutive values of a chunk");
constexpr unsigned kMaxPerCta = 64;         // chunks a CTA owns, at most
constexpr unsigned kRing = 4;               // shared-memory slots of the coding pass
constexpr unsigned kAhead = kRing - 1;      // chunks in flight ahead of the one being coded
constexpr unsigned kCopyWaitLimit = 1u << 22;
constexpr int kVecPerLane = 8;              // statistics: 8 x 16 B = 64 values per lane per block

struct FusedSmem {
  uint4 ring[kRing][kChunk / 8];            // input chunks of the coding pass, 8 KiB each
  uint64_t mbar[kRing];
  unsigned long long bins[256];             // exact fallback: this CTA's exponent sums
  unsigned size[kMaxPerCta];                // this CTA's chunks' escape-section bytes
  unsigned long long offset[kMaxPerCta];    // ... and their offsets in the stream
  double wsum[kResidentWarps];
  unsigned long long wnf[kResidentWarps], wtot[kResidentWarps];
  unsigned scan[2][kResidentWarps];          // the coding pass: warps' escape counts, by chunk parity
  int e0;
  int need_exact;
  int own;   // auto mode: this CTA's own e0 (the rule at its own partial), counted with at once
  int held;  // ... and whether every CTA's was the settled e0
};

struct FusedParams {
  const uint16_t* in;
  uint64_t n;
  int base;
  uint8_t* out;
  unsigned long long* out_bytes;
  uint8_t* ws;
  int* status;
};

// Escapes among the two values of w outside `keep`'s cleared halves (codes7_x2 gives exactly
// 7 << 7 for an escape, and 7 << 7 + 0x80 reaches bit 10).
__device__ __forceinline__ unsigned escapes_x2(uint32_t w, uint32_t kadd, uint32_t keep = 0xFFFFFFFFu) {
  return __popc(((codes7_x2(w, kadd) & keep) + 0x00800080u) & 0x04000400u);
}

// Values v .. v + 7 of x as one vector, zeros at and past n.
__device__ __forceinline__ uint4 tail_vector(const uint16_t* x, uint64_t n, uint64_t v) {
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint64_t a = v + 2 * q;
    w[q] = (a < n ? static_cast<uint32_t>(x[a]) : 0u) | (a + 1 < n ? static_cast<uint32_t>(x[a + 1]) << 16 : 0u);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One warp: chunk c's escape-section bytes (every lane).  A full chunk's 512 vectors are all in
// flight at once, 16 per lane.
__device__ unsigned count_chunk(const uint16_t* x, uint64_t n, uint64_t c, uint32_t kadd) {
  const unsigned lane = threadIdx.x & 31;
  const uint4* src = reinterpret_cast<const uint4*>(x) + c * (kChunk / 8);
  unsigned esc = 0, m = kChunk;
  if (c < n / kChunk) {
    uint4 v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __ldcg(src + lane + 32 * j);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      esc += escapes_x2(v[j].x, kadd) + escapes_x2(v[j].y, kadd) + escapes_x2(v[j].z, kadd) +
             escapes_x2(v[j].w, kadd);
  } else {  // the ragged last chunk: its m values (the zeros past them are no escapes)
    m = static_cast<unsigned>(n - c * kChunk);
    const unsigned whole = m / 8;
    for (unsigned i = lane; i < (m + 7) / 8; i += 32) {
      const uint4 t = i < whole ? __ldcg(src + i) : tail_vector(x, n, c * kChunk + 8 * i);
      const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const unsigned v = 8 * i + 2 * q;
        esc += escapes_x2(w[q], kadd, (v < m ? 0x0000FFFFu : 0u) | (v + 1 < m ? 0xFFFF0000u : 0u));
      }
    }
  }
  return escape_section_bytes(m, __reduce_add_sync(0xFFFFFFFFu, esc));
}

// Thread 0: chunk c's whole 16-byte vectors into ring slot s by one bulk async copy (none for a
// chunk of fewer than 8 values: the barrier's phase then completes at once).
__device__ __forceinline__ void issue_chunk(FusedSmem& S, const uint16_t* x, uint64_t n, uint64_t c, unsigned s) {
  const unsigned bytes = (2 * chunk_values(n, c)) & ~15u;
  mbar_arrive_expect_tx(&S.mbar[s], bytes);
  if (bytes) bulk_load(S.ring[s], x + c * kChunk, bytes, &S.mbar[s]);
}

__global__ void __launch_bounds__(kThreads, 6) fused_kernel(const FusedParams p) {
  __shared__ FusedSmem S;
  const unsigned G = gridDim.x, r = blockIdx.x;
  const unsigned tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint64_t n = p.n, N = num_chunks(n), nv = n / 8;
  const unsigned J = static_cast<unsigned>((N + G - 1) / G);
  const uint64_t first = static_cast<uint64_t>(r) * J;  // every CTA owns at least one chunk
  const unsigned mine = static_cast<unsigned>(N - first < J ? N - first : J);
  const uint64_t R0 = records_base(n), E0 = escape_base(n);
  Control* ctrl = reinterpret_cast<Control*>(p.ws);
  unsigned long long* gbins = reinterpret_cast<unsigned long long*>(p.ws + kWsExactBinsOffset);
  // The CTAs' partial sums in the scan-state slots (8 bytes per chunk; G <= N / 2); their escape
  // bytes, then offsets, in the statistics kernel's partials region (8 bytes per CTA); in auto
  // mode, the e0 each CTA counted with first in the exponent-sample region (a byte per CTA).
  StatsPartial* partials = reinterpret_cast<StatsPartial*>(p.ws + kWsControlBytes + kWsPartialsBytes);
  unsigned long long* totals = reinterpret_cast<unsigned long long*>(p.ws + kWsControlBytes);
  unsigned char* guesses = p.ws + kWsSampleOffset;
  unsigned barriers = 0;
  auto sync_last = [&](auto work) {
    ++barriers;
    return grid_barrier_last(&ctrl->grid_arrivals, barriers * G, &ctrl->grid_release, barriers, p.status,
                             kDefaultSpinLimit, work);
  };
  // Before leaving early: wait (bounded) for the copies of chunks lo .. hi - 1, issued and not yet
  // waited for, so that none is left writing to this CTA's shared memory.
  auto abandon = [&](unsigned lo, unsigned hi) {
    if (tid == 0)
      for (unsigned i = lo; i < hi && i < mine; ++i) mbar_wait(&S.mbar[i % kRing], (i / kRing) & 1, kCopyWaitLimit);
  };

  // the coding pass's first chunks start arriving now, while the statistics pass runs
  if (tid == 0) {
    for (unsigned s = 0; s < kRing; ++s) mbar_init(&S.mbar[s], 1);
    fence_mbar_init();
    for (unsigned j = 0; j < kAhead && j < mine; ++j) issue_chunk(S, p.in, n, first + j, j);
  }
  if (r == 0)  // before the first barrier; only the exact path adds to them, after it
    for (unsigned e = tid; e < 256; e += kThreads) gbins[e] = 0;

  // ---- 1. statistics over this CTA's chunks (vectors vb .. ve), then e0
  const uint64_t vb = first * (kChunk / 8);
  const uint64_t ve = (first + mine) * (kChunk / 8) < nv ? (first + mine) * (kChunk / 8) : nv;
  int e0 = p.base;
  if (p.base < 0) {
    double acc = 0.0;
    unsigned nonfinite = 0;
    for (uint64_t wb = vb + 256ull * warp; wb < ve; wb += 256ull * kResidentWarps) {
      uint32_t w[32];
      const bool full = wb + 256 <= ve;
#pragma unroll
      for (int j = 0; j < kVecPerLane; ++j) {
        const uint64_t idx = wb + 32 * j + lane;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (full || idx < ve) v = __ldcg(reinterpret_cast<const uint4*>(p.in) + idx);
        w[4 * j] = v.x;
        w[4 * j + 1] = v.y;
        w[4 * j + 2] = v.z;
        w[4 * j + 3] = v.w;
      }
      block_sum(w, &acc, &nonfinite);
    }
    if (tid == 0 && first + mine == N && (n & 7))  // the last n % 8 values
      acc += tail_block(p.in + (nv << 3), static_cast<unsigned>(n & 7), &nonfinite);
    const double s = cta_sum(acc, S.wsum);
    const unsigned long long nf = cta_sum(static_cast<unsigned long long>(nonfinite), S.wnf);
    if (tid == 0) {
      partials[r].sum = s;
      partials[r].nonfinite = nf;
      const uint64_t end = (first + mine) * kChunk < n ? (first + mine) * kChunk : n;
      S.own = rough_e0(s, end - first * kChunk - nf);  // the rule at this CTA's own values
    }
    bar_cta();
  }

  // ---- 2. every chunk's escape-section size under e, exactly; this CTA's total.  The chunks in
  // the reverse order of the first pass: the last ones read are the likeliest still in the L2.
  auto count_pass = [&](int e) {
    const uint32_t ka = ((256u - static_cast<unsigned>(e)) << 7) * 0x00010001u;
    unsigned long long mytotal = 0;  // lane 0 of each warp
    for (unsigned jj = warp; jj < mine; jj += kResidentWarps) {
      const unsigned j = mine - 1 - jj;
      const unsigned sz = count_chunk(p.in, n, first + j, ka);
      if (lane == 0) {
        S.size[j] = sz;
        mytotal += sz;
      }
    }
    if (lane == 0) S.wtot[warp] = mytotal;
    bar_cta();
    if (tid == 0) {
      unsigned long long t = 0;
      for (int w = 0; w < kResidentWarps; ++w) t += S.wtot[w];
      totals[r] = t;
    }
  };

  // Auto mode: count at once with this CTA's own e0; the barrier whose last CTA settles the
  // tensor's e0 also checks every CTA's own e0 against it and turns the totals into offsets.  When
  // every CTA's was the settled one, that barrier did for both (a grid barrier costs a few
  // microseconds); otherwise the exact sums (when needed) and a second count and barrier follow.
  bool counted = false;
  if (p.base < 0) {
    count_pass(S.own);
    if (tid == 0) guesses[r] = static_cast<unsigned char>(S.own);
    if (!sync_last([&] { settle_scan_work(partials, guesses, totals, G, n, ctrl, S.wsum, S.wnf, S.wtot, &S.own); }))
      return abandon(0, kAhead);
    if (tid == 0) {
      S.e0 = __ldcg(&ctrl->grid_e0);
      S.need_exact = static_cast<int>(__ldcg(&ctrl->grid_exact));
      S.held = !S.need_exact && __ldcg(&ctrl->grid_guesses_held) != 0;
    }
    bar_cta();
    counted = S.held != 0;
    if (S.need_exact) {  // the same in every CTA: exact per-exponent sums over the grid
      for (unsigned e = tid; e < 256; e += kThreads) S.bins[e] = 0;
      bar_cta();
      add_exponent_sums(p.in + vb * 8, (ve - vb) * 8, tid, kThreads, S.bins, S.own);
      if (first + mine == N && (n & 7)) add_exponent_sums(p.in + (nv << 3), n & 7, tid, kThreads, S.bins, S.own);
      bar_cta();
      for (unsigned e = tid; e < 256; e += kThreads)
        if (S.bins[e]) atomicAdd(gbins + e, S.bins[e]);
      if (!sync_last([&] {
            for (unsigned e = tid; e < 256; e += kThreads) S.bins[e] = __ldcg(gbins + e);
            bar_cta();
            if (tid == 0) ctrl->grid_e0 = select_e0(exact_from_bins(S.bins), __ldcg(&ctrl->n_finite));
          }))
        return abandon(0, kAhead);
      if (tid == 0) S.e0 = __ldcg(&ctrl->grid_e0);
      bar_cta();
    }
    e0 = S.e0;
    if (r == 0 && tid == 0) {
      ctrl->e0 = e0;
      ctrl->exact_path = S.need_exact;
    }
  }
  const uint32_t kadd = ((256u - static_cast<unsigned>(e0)) << 7) * 0x00010001u;
  if (!counted) {
    count_pass(e0);
    // the last CTA turns the totals into offsets from the escape region (an exclusive scan)
    if (!sync_last([&] { scan_totals_work(totals, G, ctrl, S.wtot); }))
      return abandon(0, kAhead);
  }
  if (tid == 0) {
    unsigned long long at = E0 + __ldcg(totals + r);
    for (unsigned j = 0; j < mine; ++j) {
      S.offset[j] = at;
      at += S.size[j];
    }
  }
  const unsigned long long coded = E0 + __ldcg(&ctrl->grid_escape_bytes), raw = raw_stream_bytes(n);
  const bool raw_form = coded > raw;
  bar_cta();

  // ---- 3. the stream: chunk by chunk through the ring, one CTA barrier per chunk.  The barrier
  // of chunk j also tells every thread whether any thread's copy wait ran out, and it frees the
  // slot of chunk j - 1 (every thread has finished it) for the copy of chunk j + kAhead; the
  // warps' escape counts alternate between two arrays, so that no second barrier is needed.
  unsigned long long* table = reinterpret_cast<unsigned long long*>(p.out + kHeaderBytes);
  const unsigned v0 = 32 * tid;
  for (unsigned j = 0; j < mine; ++j) {
    const unsigned s = j % kRing;
    const bool arrived = mbar_wait(&S.mbar[s], (j / kRing) & 1, kCopyWaitLimit);
    const uint64_t c = first + j;
    const unsigned m = chunk_values(n, c);
    const bool full = m == kChunk;
    if (!full) {  // the ragged last chunk: its last partial vector and zeros, by the threads
      if (arrived) {
        const uint64_t vbase = c * kChunk;
        for (unsigned i = tid; i < kChunk / 8; i += kThreads)
          if (16 * i >= ((2 * m) & ~15u)) S.ring[s][i] = tail_vector(p.in, n, vbase + 8 * i);
      }
      bar_cta();
    }
    if (raw_form) {  // the values behind the header (the last vector carries the zero padding)
      if (arrived) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + kHeaderBytes + c * 2 * kChunk);
        const unsigned vecs = (2 * m + 15) / 16;
        for (unsigned i = tid; i < vecs; i += kThreads) dst[i] = S.ring[s][i];
      }
      if (__syncthreads_or(!arrived)) {
        if (tid == 0) set_error(p.status, ZC_ERR_TIMEOUT);
        return abandon(j, j + kAhead);
      }
      if (tid == 0 && j + kAhead < mine) issue_chunk(S, p.in, n, first + j + kAhead, (j + kAhead) % kRing);
      continue;
    }
    // (a thread whose wait ran out codes zeros and stores nothing; the barrier then stops all)
    const unsigned cbytes = full ? kFullCodeBytes : static_cast<unsigned>(code_section_bytes(m));
    const unsigned smbytes = full ? kChunk : static_cast<unsigned>(pad16(m));
    uint4 xv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) xv[q] = arrived ? S.ring[s][4 * tid + q] : make_uint4(0, 0, 0, 0);
    Coded32 kd;
    code32(xv, kadd, v0, m, full, kd);
    if (arrived) store_fixed32(p.out + R0 + c * kFullFixedBytes, cbytes, smbytes, v0, full, kd);
    const unsigned cnt = __popc(kd.e[0]) + __popc(kd.e[1]) + __popc(kd.e[2]) + __popc(kd.e[3]);
    unsigned x = cnt;  // ranks: a warp scan of the counts, then the warps' totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned t = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= static_cast<unsigned>(o)) x += t;
    }
    unsigned* scan = S.scan[j & 1];
    if (lane == 31) scan[warp] = x;
    if (__syncthreads_or(!arrived)) {
      if (tid == 0) set_error(p.status, ZC_ERR_TIMEOUT);
      return abandon(j, j + kAhead);
    }
    if (tid == 0 && j + kAhead < mine) issue_chunk(S, p.in, n, first + j + kAhead, (j + kAhead) % kRing);
    unsigned before = 0, k = 0;
#pragma unroll
    for (int i = 0; i < kResidentWarps; ++i) {
      before += i < static_cast<int>(warp) ? scan[i] : 0u;
      k += scan[i];
    }
    const unsigned esc_bytes = escape_section_bytes(m, k);
    uint8_t* sec = p.out + S.offset[j];
    if (exponent_plane(m, k)) {  // every exponent, in value order (values past m are zero: the padding)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t lo = prmt((xv[q].x >> 7) & 0x00FF00FFu, (xv[q].y >> 7) & 0x00FF00FFu, 0x6420);
        const uint32_t hi = prmt((xv[q].z >> 7) & 0x00FF00FFu, (xv[q].w >> 7) & 0x00FF00FFu, 0x6420);
        if (v0 + 8 * q < esc_bytes) *reinterpret_cast<uint2*>(sec + v0 + 8 * q) = make_uint2(lo, hi);
      }
    } else {  // positions and exponents in rank order; this thread's escapes take consecutive ranks
      unsigned m32 = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) m32 |= compact8(kd.e[q]) << (8 * q);
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(S.ring[s]);
      unsigned rank = before + x;  // one past this thread's last rank
      while (m32) {  // the highest value first
        const unsigned b = msb_index(m32);
        m32 ^= 1u << b;
        --rank;
        *reinterpret_cast<uint16_t*>(sec + 2 * rank) = static_cast<uint16_t>(v0 + b);
        sec[2 * k + rank] = static_cast<uint8_t>(xs[v0 + b] >> 7);
      }
      if (tid < esc_bytes - 3 * k) sec[3 * k + tid] = 0;  // zero padding, < 16 bytes
    }
    if (tid == 0) table[c] = S.offset[j];
  }
  if (r == 0 && tid == 0) {
    unsigned long long* hdr = reinterpret_cast<unsigned long long*>(p.out);
    if (raw_form) {
      hdr[0] = kRawMagicWord | (static_cast<unsigned long long>(e0) << 56);
      hdr[1] = n;
      hdr[2] = 0;
      hdr[3] = raw;
    } else {
      hdr[0] = kMagicWord | (static_cast<unsigned long long>(e0) << 56);
      hdr[1] = n;
      hdr[2] = N;
      hdr[3] = coded;
      table[N] = coded;
      if (kHeaderBytes + 8 * (N + 1) < R0) table[N + 1] = 0;  // zero pad
    }
    ctrl->total = raw_form ? raw : coded;
    if (p.out_bytes) *p.out_bytes = raw_form ? raw : coded;
  }
}

}  // namespace

cudaError_t fused_setup(int* fused_ctas) {
  int dev = 0, sms = 0, per_sm = 0, coop = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (err != cudaSuccess) return err;
  // the ring's 35 KiB per CTA: as much of the SM's memory as shared memory as it takes
  err = cudaFuncSetAttribute(fused_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_kernel, kThreads, 0);
  if (err != cudaSuccess) return err;
  const int grid = coop ? per_sm * sms : 0;
  *fused_ctas = grid < static_cast<int>(kMaxGridCtas) ? grid : static_cast<int>(kMaxGridCtas);
  return cudaSuccess;
}

uint64_t fused_max_values(const DeviceInfo& dev) {
  const uint64_t by_grid = static_cast<uint64_t>(dev.fused_ctas) * kMaxPerCta * kChunk;
  const uint64_t by_l2 = 1ull << ZC_FUSED_MAX_LOG2;  // the passes after the first read from the L2
  return by_grid < by_l2 ? by_grid : by_l2;
}

cudaError_t launch_fused(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                         uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream) {
  // J = ceil(N / gmax) chunks per CTA and G = ceil(N / J) CTAs: every CTA owns at least one
  // chunk, and G <= N / 2 leaves two scan-state slots for each CTA's partial sum
  const uint64_t N = num_chunks(n), gmax = static_cast<uint64_t>(dev.fused_ctas) < N / 2 ? dev.fused_ctas : N / 2;
  const uint64_t J = (N + gmax - 1) / gmax;
  const unsigned G = static_cast<unsigned>((N + J - 1) / J);
  FusedParams p{in, n, base, out, out_bytes, ws, dev.status};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: the grid barriers
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TimingRecord t = timing_begin(ZC_KERNEL_FUSED, stream);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, fused_kernel, p);
  timing_end(t, stream);
  return err;
}

}  // namespace zc
