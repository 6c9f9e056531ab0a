// zc_grid.cuh -- pieces shared by the kernels that run with every CTA resident at once (a
// thread-block cluster or a cooperatively launched grid) in 128-thread CTAs: fixed-order sums over
// a warp or a CTA, and a bounded barrier over the CTAs of a cooperative grid.
#pragma once

#include "zc_common.cuh"
#include "zc_stats_core.cuh"

namespace zc {
namespace {

constexpr int kResidentThreads = 128;  // threads of a CTA: a chunk's coding threads, 32 values each
constexpr int kResidentWarps = kResidentThreads / 32;

__device__ __forceinline__ void bar_cta() { __syncthreads(); }

__device__ __forceinline__ unsigned atom_add_acq_rel_u32(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// A barrier over the CTAs of a cooperative grid (all resident at once), bounded: *arrivals was
// cleared before the launch, and barrier k (k = 1, 2, ..) is passed when it reaches k G.  A wait
// that runs out sets ZC_ERR_TIMEOUT.  Returns, the same in every thread of the CTA, whether the
// barrier was passed with no error recorded; after an error the CTAs stop waiting and the caller
// stops (the call has failed and reports it), so no CTA is left spinning and nothing is written
// from data that may be missing.
__device__ bool grid_barrier(unsigned* arrivals, unsigned target, int* status, unsigned spin_limit) {
  __shared__ int barrier_ok;
  bar_cta();
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's writes, before its arrival
    atomicAdd(arrivals, 1u);
    unsigned spins = 0, backoff = 32;
    bool ok = true;
    while (ld_acquire_u32(arrivals) < target) {
      if (read_status(status) != 0 || ++spins > spin_limit) {
        if (spins > spin_limit) set_error(status, ZC_ERR_TIMEOUT);
        ok = false;
        break;
      }
      __nanosleep(backoff);
      backoff = backoff < 256 ? backoff * 2 : 256;
    }
    __threadfence();  // the other CTAs' writes, from here on
    barrier_ok = ok && read_status(status) == 0;
  }
  bar_cta();
  return barrier_ok != 0;
}

// A barrier over the CTAs of a cooperative grid whose last CTA to arrive does some work before
// the others go on: *arrivals counts as in grid_barrier (target k G for barrier k); the CTA whose
// arrival completes the count runs work() with all its threads, then releases the others by
// setting *release to k.  The others wait, bounded, for that release.  So a result that every CTA
// needs (a reduction, a scan) is computed once, by one CTA, instead of by every CTA from every
// other CTA's data.  Returns, the same in every thread of the CTA, whether the barrier was passed
// with no error recorded.
// The memory ordering rides on the synchronizing operations themselves, with no separate fence:
// the CTA's writes are ordered before thread 0's arrival by the CTA barrier, the arrival is an
// acquire-release add (it publishes them, and the last arrival sees every other CTA's), the
// release is a release store after the work and the waiters' polls are acquire loads.
template <typename Work>
__device__ bool grid_barrier_last(unsigned* arrivals, unsigned target, unsigned* release, unsigned k, int* status,
                                  unsigned spin_limit, Work work) {
  __shared__ int barrier_last, barrier_ok;
  bar_cta();
  if (threadIdx.x == 0) barrier_last = atom_add_acq_rel_u32(arrivals, 1u) == target - 1;
  bar_cta();
  if (barrier_last) {
    work();
    bar_cta();
    if (threadIdx.x == 0) {
      st_release_u32(release, k);
      barrier_ok = read_status(status) == 0;
    }
  } else if (threadIdx.x == 0) {
    unsigned spins = 0, backoff = 32;
    bool ok = true;
    while (ld_acquire_u32(release) < k) {
      if (read_status(status) != 0 || ++spins > spin_limit) {
        if (spins > spin_limit) set_error(status, ZC_ERR_TIMEOUT);
        ok = false;
        break;
      }
      __nanosleep(backoff);
      backoff = backoff < 256 ? backoff * 2 : 256;
    }
    barrier_ok = ok && read_status(status) == 0;
  }
  bar_cta();
  return barrier_ok != 0;
}

// Sum over a warp in a fixed order (a butterfly tree), in every lane.
template <typename T>
__device__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Sum over the CTA's threads in a fixed order (warp tree, then warps in order), in every thread.
template <typename T>
__device__ T cta_sum(T v, T* scratch) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = v;
  bar_cta();
  T t = 0;
#pragma unroll
  for (int i = 0; i < kResidentWarps; ++i) t += scratch[i];
  bar_cta();
  return t;
}

// f(i, a, b) adds term i to the pair (a, b) for i < count; the pairs are summed in a fixed order,
// valid in thread 0: by warp 0 alone (no CTA barrier) when count <= 32 * per_lane, else by the
// whole CTA.
template <typename A, typename B, typename F>
__device__ void fixed_sum2(uint64_t count, unsigned per_lane, A* sa, B* sb, A* a, B* b, F f) {
  const bool wide = count > 32ull * per_lane;
  const unsigned step = wide ? kResidentThreads : 32;
  A va = 0;
  B vb = 0;
  if (wide || threadIdx.x < 32)
    for (uint64_t i = threadIdx.x; i < count; i += step) f(i, va, vb);
  *a = wide ? cta_sum(va, sa) : warp_sum(va);
  *b = wide ? cta_sum(vb, sb) : warp_sum(vb);
}

// Work for the last CTA of a grid barrier (all its threads): the CTAs' statistics partials
// added up in one fixed order (thread t takes CTAs t, t + 128, ..; then a fixed tree), and the
// window rule at both ends of the estimate's error interval, one end per thread (as decide_e0_pair): e0
// is settled when they agree, else the exact sums must decide it.  Writes e0, the exact flag and
// the finite count to the control block.  G <= kMaxGridCtas.
constexpr unsigned kMaxGridCtas = 1024;
constexpr unsigned kGridPerThread = kMaxGridCtas / kResidentThreads;

__device__ void settle_e0_work(const StatsPartial* partials, unsigned G, uint64_t n, Control* ctrl, double* wsum,
                               unsigned long long* wnf) {
  const unsigned tid = threadIdx.x;
  double v[kGridPerThread];
  unsigned long long c[kGridPerThread];
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i) {  // all loads in flight at once
    const unsigned q = tid + kResidentThreads * i;
    v[i] = q < G ? __ldcg(&partials[q].sum) : 0.0;
    c[i] = q < G ? __ldcg(&partials[q].nonfinite) : 0ull;
  }
  double a = 0.0;
  unsigned long long b = 0;
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i) {
    a += v[i];
    b += c[i];
  }
  const double S_all = cta_sum(a, wsum);
  const unsigned long long nf_all = cta_sum(b, wnf);
  if (tid < 2) {
    const unsigned long long n_f = n - nf_all;
    int e = 0;
    const bool settled = decide_e0_pair(S_all, n_f, &e);
    if (tid == 0) {
      ctrl->grid_e0 = e;
      ctrl->grid_exact = settled ? 0u : 1u;
      ctrl->n_finite = n_f;
    }
  }
}

// Work for the last CTA of a grid barrier (all its threads): totals[0 .. G) replaced by their
// exclusive prefix sums in index order -- each thread over a run of consecutive entries, all
// loaded at once, then over the threads -- and the sum of all written to the control block.
// G <= kMaxGridCtas.
__device__ void scan_totals_work(unsigned long long* totals, unsigned G, Control* ctrl, unsigned long long* wtot) {
  const unsigned tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned per = (G + kResidentThreads - 1) / kResidentThreads, lo = min(tid * per, G), hi = min(lo + per, G);
  unsigned long long t[kGridPerThread], run = 0;
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i) t[i] = lo + i < hi ? __ldcg(totals + lo + i) : 0ull;
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i) run += t[i];
  unsigned long long x = run;  // inclusive scan over the threads
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long u = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= static_cast<unsigned>(o)) x += u;
  }
  if (lane == 31) wtot[warp] = x;
  bar_cta();
  unsigned long long at = x - run, all = 0;
#pragma unroll
  for (int w = 0; w < kResidentWarps; ++w) {
    at += w < static_cast<int>(warp) ? wtot[w] : 0ull;
    all += wtot[w];
  }
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i)
    if (lo + i < hi) {
      totals[lo + i] = at;
      at += t[i];
    }
  if (tid == 0) ctrl->grid_escape_bytes = all;
}

// Work for the last CTA of the one barrier that both settles e0 and places the sections (all its
// threads): what settle_e0_work and scan_totals_work do, plus the check of every CTA's own e0
// (guesses[q], the e0 CTA q counted or coded with) against the settled one -- with every load
// (partials, own e0, totals) issued at once, so the work costs one memory round trip, not three.
// Writes e0, the exact flag, the finite count, whether every CTA's own e0 was the settled one,
// the offsets (in place of the totals) and the sections' total to the control block.
// G <= kMaxGridCtas; e_shared: one int of shared memory.
__device__ void settle_scan_work(const StatsPartial* partials, const unsigned char* guesses,
                                 unsigned long long* totals, unsigned G, uint64_t n, Control* ctrl, double* wsum,
                                 unsigned long long* wnf, unsigned long long* wtot, int* e_shared) {
  const unsigned tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned per = (G + kResidentThreads - 1) / kResidentThreads, lo = min(tid * per, G), hi = min(lo + per, G);
  double v[kGridPerThread];
  unsigned long long c[kGridPerThread], t[kGridPerThread];
  unsigned g[kGridPerThread];
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i) {  // all loads in flight at once
    const unsigned q = tid + kResidentThreads * i;
    v[i] = q < G ? __ldcg(&partials[q].sum) : 0.0;
    c[i] = q < G ? __ldcg(&partials[q].nonfinite) : 0ull;
    g[i] = q < G ? __ldcg(guesses + q) : 0u;
    t[i] = lo + i < hi ? __ldcg(totals + lo + i) : 0ull;
  }
  // e0 from the partials, in one fixed order (as settle_e0_work)
  double a = 0.0;
  unsigned long long b = 0;
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i) {
    a += v[i];
    b += c[i];
  }
  const double S_all = cta_sum(a, wsum);
  const unsigned long long nf_all = cta_sum(b, wnf);
  if (tid < 2) {
    const unsigned long long n_f = n - nf_all;
    int e = 0;
    const bool settled = decide_e0_pair(S_all, n_f, &e);
    if (tid == 0) {
      ctrl->grid_e0 = e;
      ctrl->grid_exact = settled ? 0u : 1u;
      ctrl->n_finite = n_f;
      *e_shared = e;
    }
  }
  bar_cta();
  // every CTA's own e0 against the settled one
  const unsigned e = static_cast<unsigned>(*e_shared);
  bool same = true;
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i)
    if (tid + kResidentThreads * i < G) same = same && g[i] == e;
  same = __syncthreads_and(same);
  if (tid == 0) ctrl->grid_guesses_held = same ? 1u : 0u;
  // the totals' exclusive prefix sums (as scan_totals_work)
  unsigned long long run = 0;
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i) run += t[i];
  unsigned long long x = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long u = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= static_cast<unsigned>(o)) x += u;
  }
  if (lane == 31) wtot[warp] = x;
  bar_cta();
  unsigned long long at = x - run, all = 0;
#pragma unroll
  for (int w = 0; w < kResidentWarps; ++w) {
    at += w < static_cast<int>(warp) ? wtot[w] : 0ull;
    all += wtot[w];
  }
#pragma unroll
  for (unsigned i = 0; i < kGridPerThread; ++i)
    if (lo + i < hi) {
      totals[lo + i] = at;
      at += t[i];
    }
  if (tid == 0) ctrl->grid_escape_bytes = all;
}

}  // namespace
}  // namespace zc
