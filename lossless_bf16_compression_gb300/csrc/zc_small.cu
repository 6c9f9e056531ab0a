// zc_small.cu -- compression of a small or medium tensor in one launch, with every CTA resident
// at once: one thread-block cluster for up to 64 chunks of 4096 values, or one cooperative grid
// for up to four chunks per resident CTA.  No tensor map, no second kernel.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution": the window base from the
// tensor's standard deviation, 3-bit codes with the full exponents of the others kept apart
// (first technique), and the native form where coding does not pay (third technique).  The
// overhead of a compressor on small messages is what the page calls its performance cliff
// (general-purpose compressors can be slower than sending the data as it is); here such a
// tensor costs one launch.
//
// GB300 design.  G CTAs of 128 threads; CTA r holds chunks r J .. r J + J - 1 (J = ceil(N / G),
// at most four) in shared memory: 32 KiB of input and their escape sections.  The input arrives
// by bulk async copies.  Each CTA sums its squares in fp32 blocks as the statistics kernel does
// (of 32 values, one per thread and chunk, inside that kernel's error bound for its blocks of
// 64) and publishes its partial; after a barrier the partials are
// combined in one fixed order, so that one e0 is settled for all (and, when the bound straddles a
// switching point, the exact per-exponent sums decide it).  The CTAs code their chunks (escape
// sections into shared memory; fixed parts too in a cluster, so that its barriers wait for no
// global store, or straight to their places in `out` in a grid), publish the sections' sizes,
// and after another barrier each knows its sections' offsets and the stream's length, then
// writes the coded form (fixed parts, sections, offset table, header) or the raw form (the
// values from shared memory, over anything written before the barrier).
//  - Cluster (up to 16 CTAs, 64 chunks): before each barrier every CTA pushes its partial (or its
//    sections' sizes) into every other CTA's shared memory (distributed shared memory), and each
//    combines them itself after it; the barriers are the cluster's, in hardware.
//  - Cooperative grid (as many CTAs as the device holds at once, launched cooperatively so that
//    all are resident): partials, bins, the CTAs' own e0 and per-CTA totals go through the
//    call's workspace (slots each CTA writes before the barrier; the exact path's bins are
//    cleared by CTA 0 before the first barrier).  The barriers count arrivals in the control
//    block, cleared before the launch; the last CTA to arrive does the combining -- the sum of
//    the partials and the window rule, the scan of the CTAs' totals into offsets -- and releases
//    the others, so it is done once instead of by every CTA from every other CTA's slots.  A
//    grid barrier costs microseconds, so in auto mode each CTA codes at once with its own e0
//    (the rule at its own partial) and one barrier settles e0 and places the sections; when some
//    CTA's own e0 was not the settled one, the chunks are coded again and a second barrier
//    places them.  The waits are bounded.
// Every CTA takes part in every barrier (a CTA whose copies did not arrive goes on with zeros
// and sets the error); every wait that polls (the copies' mbarrier, the grid barriers) is
// bounded, and a grid barrier that fails stops the CTAs (the cluster's never fail).
#include <cooperative_groups.h>

#include "zc_code_core.cuh"
#include "zc_common.cuh"
#include "zc_grid.cuh"
#include "zc_stats_core.cuh"

namespace cg = cooperative_groups;

namespace zc {
namespace {

#ifndef ZC_SMALL_CTAS
#define ZC_SMALL_CTAS 16
#endif
// CTAs of the cluster, at most: 16 (a non-portable cluster size, taken when the device can
// schedule such a cluster of this kernel), else 8 (the portable size).
constexpr unsigned kSmallCtas = ZC_SMALL_CTAS;
constexpr unsigned kSmallPortableCtas = 8;
static_assert(kSmallCtas >= kSmallPortableCtas && kSmallCtas <= 16, "a cluster of 8 to 16 CTAs");
constexpr unsigned kPerCta = 4;         // chunks per CTA, at most
constexpr int kSmallThreads = kResidentThreads;
static_assert(32 * kSmallThreads == kChunk, "a thread codes 32 consecutive values of a chunk");
constexpr unsigned kSmallWaitLimit = 1u << 22;
constexpr int kWarpsPerCta = kResidentWarps;

struct __align__(128) ResidentSmem {
  uint4 x[kPerCta][kChunk / 8];                 // inputs, 8 KiB per chunk (zero past m)
  uint4 sec[kPerCta][kMaxEscapeBytes / 16];     // escape sections
  unsigned long long bins[256];                 // exact fallback: this CTA's exponent sums, then all
  uint64_t mbar;
  double wsum[kWarpsPerCta];
  unsigned long long wnf[kWarpsPerCta];
  unsigned long long wbefore[kWarpsPerCta], wtotal[kWarpsPerCta];
  double cta_sum;
  unsigned long long cta_nonfinite;
  unsigned long long offset[kPerCta];          // this CTA's sections' offsets in the stream
  unsigned long long total;
  unsigned long long n_finite;
  unsigned scan[kWarpsPerCta];
  unsigned my_size[kPerCta];
  int e0;
  int need_exact;
  int ok;
  int guess;      // the cooperative grid, auto mode: this CTA's own e0, coded with at once
  int held;       // ... and whether every CTA's was the settled e0
  // last, for cluster launches only (the grid launch does not allocate them): the fixed parts,
  // kept here until the stream's form is known (the grid launch stores them in place at once),
  // and every CTA's partial and sections' sizes, pushed here by their CTAs before the barrier
  // that publishes them, so that they are read locally after it
  uint4 fixed[kPerCta][kFullFixedBytes / 16];
  double all_sum[kSmallCtas];
  unsigned long long all_nf[kSmallCtas];
  unsigned all_size[kSmallCtas * kPerCta];
};
constexpr size_t kGridSmemBytes = offsetof(ResidentSmem, fixed);
static_assert(kMaxGridCtas <= 8 * 256, "a cooperative grid's e0 per CTA fits the exponent-sample region");

// The exchange between the CTAs of a cluster: distributed shared memory, cluster barriers.
struct ClusterExchange {
  cg::cluster_group cl = cg::this_cluster();
  __device__ unsigned ctas() const { return cl.num_blocks(); }
  __device__ unsigned rank() const { return cl.block_rank(); }
  __device__ bool sync() {  // a hardware barrier: always passed
    cl.sync();
    return true;
  }
  __device__ void put_partial(ResidentSmem& S, double s, unsigned long long nf) {
    S.cta_sum = s;
    S.cta_nonfinite = nf;
  }
  // exact path: the CTA's bins are in S.bins; every CTA adds up all of them (after a barrier)
  __device__ void share_bins(ResidentSmem&) {}
  __device__ unsigned long long all_bins(ResidentSmem& S, unsigned e) {
    unsigned long long t = 0;
    for (unsigned q = 0; q < ctas(); ++q) t += cl.map_shared_rank(S.bins, q)[e];
    return t;
  }
  // Thread t pushes this CTA's partial (put_partial, then a CTA barrier) or its sections' sizes
  // (S.my_size, complete: the coding loop ends with a CTA barrier) to CTA t, before the barrier
  // that publishes them; after it each CTA reads them from its own shared memory.
  __device__ void push_partial(ResidentSmem& S) {
    if (threadIdx.x < ctas()) {
      cl.map_shared_rank(S.all_sum, threadIdx.x)[rank()] = S.cta_sum;
      cl.map_shared_rank(S.all_nf, threadIdx.x)[rank()] = S.cta_nonfinite;
    }
  }
  __device__ void push_sizes(ResidentSmem& S, uint64_t first, unsigned mine) {
    if (threadIdx.x < ctas()) {
      unsigned* dst = cl.map_shared_rank(S.all_size, threadIdx.x);
      for (unsigned j = 0; j < mine; ++j) dst[first + j] = S.my_size[j];
    }
  }
  // Every CTA combines the partials in the same fixed order (thread t takes CTAs t, t + 32, ..,
  // then a fixed tree), so every CTA settles the same e0: S.e0, S.need_exact, S.n_finite.
  __device__ void settle_local(ResidentSmem& S, uint64_t n) {
    double s = 0.0;
    unsigned long long nf_all = 0;
    fixed_sum2(ctas(), 1, S.wsum, S.wnf, &s, &nf_all, [&](uint64_t q, double& a, unsigned long long& b) {
      a += S.all_sum[q];
      b += S.all_nf[q];
    });
    if (threadIdx.x < 2) {  // (warp 0's lanes all hold the sums) one end of the rule each
      int e = 0;
      const bool settled = decide_e0_pair(s, n - nf_all, &e);
      if (threadIdx.x == 0) {
        S.need_exact = settled ? 0 : 1;
        S.e0 = e;
        S.n_finite = n - nf_all;  // for the exact path
      }
    }
    bar_cta();
  }
  // The sizes of the chunks before this CTA's and of all, in thread 0.
  __device__ void offsets_local(ResidentSmem& S, uint64_t first, uint64_t N, unsigned long long* bef,
                                unsigned long long* tot) {
    fixed_sum2(N, 2, S.wbefore, S.wtotal, bef, tot, [&](uint64_t c, unsigned long long& a, unsigned long long& b) {
      const unsigned long long sz = S.all_size[c];
      a += c < first ? sz : 0ull;
      b += sz;
    });
  }
  __device__ bool settle(ResidentSmem& S, double s_cta, unsigned long long nf_cta, uint64_t n) {
    if (threadIdx.x == 0) put_partial(S, s_cta, nf_cta);
    bar_cta();
    push_partial(S);
    sync();
    settle_local(S, n);
    return true;
  }
  __device__ bool offsets(ResidentSmem& S, uint64_t first, unsigned mine, unsigned, uint64_t N,
                          unsigned long long* bef, unsigned long long* tot) {
    push_sizes(S, first, mine);
    sync();
    offsets_local(S, first, N, bef, tot);
    return true;
  }
  // Cluster barriers are cheap: e0 is settled before any chunk is coded.
  static constexpr bool kSpeculate = false;
  __device__ bool settle_offsets(ResidentSmem&, double, unsigned long long, uint64_t, uint64_t, unsigned, int,
                                 unsigned long long*, unsigned long long*) {
    return false;
  }
  static constexpr bool kKeepFixed = true;  // no store to global memory before the last barrier
  __device__ void finish() {  // no CTA leaves while another may read its shared memory: order no memory
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
  }
};

// The exchange between the CTAs of a cooperative grid: the call's workspace, bounded barriers.
struct GridExchange {
  StatsPartial* partials;        // one per CTA
  unsigned long long* bins;      // 256, cleared by CTA 0 before the first barrier
  unsigned long long* totals;    // one per CTA (the scan-state slots, G <= N): escape bytes, then offsets
  unsigned char* guesses;        // one per CTA: the e0 it coded with first (auto mode)
  Control* ctrl;                 // the barriers' counter and release word (cleared before the launch)
  unsigned* arrivals;
  int* status;
  unsigned passed = 0;           // barriers passed so far
  __device__ unsigned ctas() const { return gridDim.x; }
  __device__ unsigned rank() const { return blockIdx.x; }
  __device__ bool sync() { return grid_barrier(arrivals, ++passed * gridDim.x, status, kDefaultSpinLimit); }
  __device__ void put_partial(ResidentSmem&, double s, unsigned long long nf) {
    partials[blockIdx.x].sum = s;
    partials[blockIdx.x].nonfinite = nf;
  }
  __device__ void share_bins(ResidentSmem& S) {
    for (unsigned e = threadIdx.x; e < 256; e += kSmallThreads)
      if (S.bins[e]) atomicAdd(bins + e, S.bins[e]);
  }
  __device__ unsigned long long all_bins(ResidentSmem&, unsigned e) { return __ldcg(bins + e); }
  // The last CTA to arrive adds the partials up and settles e0 for all (settle_e0_work).
  __device__ bool settle(ResidentSmem& S, double s_cta, unsigned long long nf_cta, uint64_t n) {
    if (threadIdx.x == 0) put_partial(S, s_cta, nf_cta);
    ++passed;
    if (!grid_barrier_last(arrivals, passed * gridDim.x, &ctrl->grid_release, passed, status, kDefaultSpinLimit,
                           [&] { settle_e0_work(partials, gridDim.x, n, ctrl, S.wsum, S.wnf); }))
      return false;
    if (threadIdx.x == 0) {
      S.e0 = __ldcg(&ctrl->grid_e0);
      S.need_exact = static_cast<int>(__ldcg(&ctrl->grid_exact));
      S.n_finite = __ldcg(&ctrl->n_finite);
    }
    bar_cta();
    return true;
  }
  // Each CTA's escape bytes; the last CTA to arrive turns them into offsets (scan_totals_work).
  __device__ bool offsets(ResidentSmem& S, uint64_t, unsigned mine, unsigned, uint64_t, unsigned long long* bef,
                          unsigned long long* tot) {
    if (threadIdx.x == 0) {
      unsigned long long t = 0;
      for (unsigned j = 0; j < mine; ++j) t += S.my_size[j];
      totals[blockIdx.x] = t;
    }
    ++passed;
    if (!grid_barrier_last(arrivals, passed * gridDim.x, &ctrl->grid_release, passed, status, kDefaultSpinLimit,
                           [&] { scan_totals_work(totals, gridDim.x, ctrl, S.wbefore); }))
      return false;
    if (threadIdx.x == 0) {
      *bef = __ldcg(totals + blockIdx.x);
      *tot = __ldcg(&ctrl->grid_escape_bytes);
    }
    return true;
  }
  // Grid barriers are dear (a few microseconds each): each CTA codes at once with its own e0 (the
  // rule at its own partial), and one barrier settles e0 and turns the sizes into offsets; when
  // every CTA's own e0 was the settled one (S.held), that barrier did for both.
  static constexpr bool kSpeculate = true;
  __device__ bool settle_offsets(ResidentSmem& S, double s_cta, unsigned long long nf_cta, uint64_t n, uint64_t,
                                 unsigned mine, int own_e0, unsigned long long* bef, unsigned long long* tot) {
    if (threadIdx.x == 0) {
      put_partial(S, s_cta, nf_cta);
      guesses[blockIdx.x] = static_cast<unsigned char>(own_e0);
      unsigned long long t = 0;
      for (unsigned j = 0; j < mine; ++j) t += S.my_size[j];
      totals[blockIdx.x] = t;
    }
    ++passed;
    if (!grid_barrier_last(arrivals, passed * gridDim.x, &ctrl->grid_release, passed, status, kDefaultSpinLimit,
                           [&] {
                             settle_scan_work(partials, guesses, totals, gridDim.x, n, ctrl, S.wsum, S.wnf,
                                              S.wbefore, &S.guess);
                           }))
      return false;
    if (threadIdx.x == 0) {
      S.e0 = __ldcg(&ctrl->grid_e0);
      S.need_exact = static_cast<int>(__ldcg(&ctrl->grid_exact));
      S.n_finite = __ldcg(&ctrl->n_finite);
      S.held = !S.need_exact && __ldcg(&ctrl->grid_guesses_held) != 0;
      *bef = __ldcg(totals + blockIdx.x);
      *tot = __ldcg(&ctrl->grid_escape_bytes);
    }
    bar_cta();
    return true;
  }
  static constexpr bool kKeepFixed = false;  // fixed parts stored in place while coding
  __device__ void finish() {}
};

template <typename Exchange>
__device__ void compress_resident(Exchange& X, ResidentSmem& S, const uint16_t* in, uint64_t n, int base,
                                  uint8_t* out, unsigned long long* out_bytes, Control* ctrl, int* status) {
  const unsigned G = X.ctas(), r = X.rank();
  const unsigned tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint64_t N = num_chunks(n);
  const unsigned J = static_cast<unsigned>((N + G - 1) / G);  // chunks per CTA
  const uint64_t first = static_cast<uint64_t>(r) * J;        // this CTA's chunks: first .. first + mine - 1
  const unsigned mine = first < N ? static_cast<unsigned>(N - first < J ? N - first : J) : 0u;
  const uint64_t R0 = records_base(n), E0 = escape_base(n);

  // ---- the input: whole 16-byte vectors by bulk async copies, the ragged tail and zeros by threads
  if (tid == 0) {
    mbar_init(&S.mbar, 1);
    fence_mbar_init();
    unsigned bytes = 0;
    for (unsigned j = 0; j < mine; ++j) bytes += (2 * chunk_values(n, first + j)) & ~15u;
    mbar_arrive_expect_tx(&S.mbar, bytes);
    for (unsigned j = 0; j < mine; ++j) {
      const unsigned vb = (2 * chunk_values(n, first + j)) & ~15u;
      if (vb) bulk_load(S.x[j], in + (first + j) * kChunk, vb, &S.mbar);
    }
  }
  for (unsigned j = 0; j < mine; ++j) {
    const uint64_t c = first + j;
    const unsigned m = chunk_values(n, c);
    if (m == kChunk) continue;
    for (unsigned i = tid; i < kChunk / 8; i += kSmallThreads) {
      if (16 * i < ((2 * m) & ~15u)) continue;  // that vector comes by the copy
      uint32_t w[4] = {0, 0, 0, 0};
      for (unsigned t = 0; t < 8; ++t) {
        const unsigned v = 8 * i + t;
        if (v < m) w[t >> 1] |= static_cast<uint32_t>(in[c * kChunk + v]) << (16 * (t & 1));
      }
      S.x[j][i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  const bool arrived = mbar_wait(&S.mbar, 0, kSmallWaitLimit);
  if (tid == 0) S.ok = 1;
  bar_cta();
  if (!arrived) {
    S.ok = 0;
    set_error(status, ZC_ERR_TIMEOUT);
  }
  bar_cta();
  if (!S.ok && tid == 0) mbar_wait(&S.mbar, 0, kSmallWaitLimit);  // never leave a copy in flight
  // (a CTA whose copies did not arrive still takes part in every barrier below, with zeros)

  // ---- the window base.  Auto mode: this CTA's partial sum of squares.  In a cooperative grid
  // (Exchange::kSpeculate) the CTA codes at once with its own e0 -- the rule at its own partial --
  // and the barrier that publishes the sections' sizes publishes the partials and those e0 too:
  // when every CTA's was the settled e0, one barrier did for both; otherwise the chunks are coded
  // again with the settled (or exact) e0.
  int e0 = base;
  int guess = -1;
  double s_cta = 0.0;  // (thread 0)
  unsigned long long nf_cta = 0;
  if (base < 0) {
    double acc = 0.0;
    unsigned nonfinite = 0;
    const unsigned B = 128 * mine;  // blocks of 32 values of this CTA's chunks (zeros past m add nothing)
    for (unsigned b0 = 0; b0 < B; b0 += kSmallThreads) {
      const unsigned b = b0 + tid;
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 v = b < B && S.ok ? S.x[b / 128][4 * (b % 128) + k] : make_uint4(0, 0, 0, 0);
        w[4 * k] = v.x;
        w[4 * k + 1] = v.y;
        w[4 * k + 2] = v.z;
        w[4 * k + 3] = v.w;
      }
      block_sum(w, &acc, &nonfinite);
    }
    unsigned long long nf = nonfinite;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc += __shfl_down_sync(0xFFFFFFFFu, acc, o);
      nf += __shfl_down_sync(0xFFFFFFFFu, nf, o);
    }
    if (lane == 0) {
      S.wsum[warp] = acc;
      S.wnf[warp] = nf;
    }
    bar_cta();
    if (tid == 0)
      for (int i = 0; i < kWarpsPerCta; ++i) {
        s_cta += S.wsum[i];
        nf_cta += S.wnf[i];
      }
    if (Exchange::kSpeculate) {
      if (tid == 0) {
        unsigned long long values = 0;
        for (unsigned j = 0; j < mine; ++j) values += chunk_values(n, first + j);
        S.guess = rough_e0(s_cta, values - nf_cta);
      }
      bar_cta();
      guess = S.guess;
    }
  }

  // The exact per-exponent sums over all CTAs, when the estimate cannot settle e0 (the same in
  // every CTA): S.e0 from S.bins.
  auto exact_e0 = [&]() -> bool {
    for (unsigned e = tid; e < 256; e += kSmallThreads) S.bins[e] = 0;
    bar_cta();
    for (unsigned j = 0; j < mine; ++j)
      add_exponent_sums(reinterpret_cast<const uint16_t*>(S.x[j]), chunk_values(n, first + j), tid, kSmallThreads,
                        S.bins, S.e0);
    bar_cta();
    X.share_bins(S);
    if (!X.sync()) return false;
    unsigned long long t[2] = {0, 0};
    for (unsigned e = tid, i = 0; e < 256; e += kSmallThreads, ++i) t[i] = X.all_bins(S, e);
    if (!X.sync()) return false;  // every CTA has read the others' bins before any overwrites its own
    for (unsigned e = tid, i = 0; e < 256; e += kSmallThreads, ++i) S.bins[e] = t[i];
    bar_cta();
    if (tid == 0) S.e0 = select_e0(exact_from_bins(S.bins), S.n_finite);
    bar_cta();
    return true;
  };

  // ---- code this CTA's chunks with e: fixed parts to their places, escape sections into shared
  // memory, their sizes to S.my_size
  auto code_chunks = [&](int e) {
    const uint32_t kadd = ((256u - static_cast<unsigned>(e)) << 7) * 0x00010001u;
    const unsigned v0 = 32 * tid;
    for (unsigned j = 0; j < mine; ++j) {
      const uint64_t c = first + j;
      const unsigned m = chunk_values(n, c);
      const bool full = m == kChunk;
      const unsigned cbytes = full ? kFullCodeBytes : static_cast<unsigned>(code_section_bytes(m));
      const unsigned smbytes = full ? kChunk : static_cast<unsigned>(pad16(m));
      uint4 xv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) xv[q] = S.x[j][4 * tid + q];
      Coded32 kd;
      code32(xv, kadd, v0, m, full, kd);
      // (a ragged chunk's threads past m store zero codes and bytes: the sections' padding)
      store_fixed32(Exchange::kKeepFixed ? reinterpret_cast<uint8_t*>(S.fixed[j]) : out + R0 + c * kFullFixedBytes,
                    cbytes, smbytes, v0, full, kd);
      const unsigned cnt = __popc(kd.e[0]) + __popc(kd.e[1]) + __popc(kd.e[2]) + __popc(kd.e[3]);
      // ranks: a warp scan of the counts, then the warps' totals
      unsigned x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= static_cast<unsigned>(o)) x += t;
      }
      if (lane == 31) S.scan[warp] = x;
      bar_cta();
      unsigned before = 0, k = 0;
#pragma unroll
      for (int i = 0; i < kWarpsPerCta; ++i) {
        before += i < static_cast<int>(warp) ? S.scan[i] : 0u;
        k += S.scan[i];
      }
      const unsigned base_rank = before + x - cnt;
      const bool plane = exponent_plane(m, k);
      const unsigned esc_bytes = escape_section_bytes(m, k);
      const uint32_t sec = smem_u32(S.sec[j]), xs = smem_u32(S.x[j]);
      if (plane) {  // every exponent, in value order (values past m are zero: the padding)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t lo = prmt((xv[q].x >> 7) & 0x00FF00FFu, (xv[q].y >> 7) & 0x00FF00FFu, 0x6420);
          const uint32_t hi = prmt((xv[q].z >> 7) & 0x00FF00FFu, (xv[q].w >> 7) & 0x00FF00FFu, 0x6420);
          if (v0 + 8 * q < esc_bytes) sts_v2(sec + v0 + 8 * q, lo, hi);
        }
      } else {
        unsigned m32 = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) m32 |= compact8(kd.e[q]) << (8 * q);
        write_list32(m32, cnt, v0, base_rank, k, sec, false,
                     [&](unsigned b) { return lds_u16(xs + 2 * (v0 + b)) >> 7; });
        if (tid < esc_bytes - 3 * k) sts_u8(sec + 3 * k + tid, 0);  // zero padding, < 16 bytes
      }
      if (tid == 0) S.my_size[j] = esc_bytes;
      bar_cta();  // S.scan is free for the next chunk
    }
  };

  // ---- e0, the coding, and the sections' offsets: the sizes of the chunks before this CTA's,
  // and the stream's length (thread 0)
  unsigned long long bef = 0, tot = 0;
  bool coded_with_e0 = false;
  if (guess >= 0) {
    code_chunks(guess);
    if (!X.settle_offsets(S, s_cta, nf_cta, n, first, mine, guess, &bef, &tot)) return;
    coded_with_e0 = S.held != 0;  // the same in every CTA
  } else if (base < 0) {
    if (!X.settle(S, s_cta, nf_cta, n)) return;  // S.e0, S.need_exact, S.n_finite
  }
  if (base < 0) {
    if (!coded_with_e0 && S.need_exact && !exact_e0()) return;
    e0 = S.e0;
    if (r == 0 && tid == 0) {
      ctrl->e0 = e0;
      ctrl->exact_path = S.need_exact;
    }
  }
  if (!coded_with_e0) {
    code_chunks(e0);
    if (!X.offsets(S, first, mine, J, N, &bef, &tot)) return;
  }
  if (tid == 0) {
    unsigned long long at = E0 + bef;
    for (unsigned j = 0; j < mine; ++j) {
      S.offset[j] = at;
      at += S.my_size[j];
    }
    S.total = E0 + tot;
  }
  bar_cta();
  const unsigned long long coded = S.total, raw = raw_stream_bytes(n);
  if (coded > raw) {  // the raw form: the header, the values as they are, zero padding
    for (unsigned j = 0; j < mine; ++j) {
      const uint64_t c = first + j;
      const unsigned vecs = (2 * chunk_values(n, c) + 15) / 16;  // the last one carries the padding
      uint4* dst = reinterpret_cast<uint4*>(out + kHeaderBytes + c * 2 * kChunk);
      for (unsigned i = tid; i < vecs; i += kSmallThreads) dst[i] = S.x[j][i];
    }
    if (r == 0 && tid == 0) {
      unsigned long long* hdr = reinterpret_cast<unsigned long long*>(out);
      hdr[0] = kRawMagicWord | (static_cast<unsigned long long>(e0) << 56);
      hdr[1] = n;
      hdr[2] = 0;
      hdr[3] = raw;
      ctrl->total = raw;
      if (out_bytes) *out_bytes = raw;
    }
  } else {  // the coded form: (fixed parts,) escape sections, offset table, header
    unsigned long long* table = reinterpret_cast<unsigned long long*>(out + kHeaderBytes);
    for (unsigned j = 0; j < mine; ++j) {
      if (Exchange::kKeepFixed) {
        const unsigned fb = static_cast<unsigned>(fixed_bytes(chunk_values(n, first + j))) / 16;
        uint4* df = reinterpret_cast<uint4*>(out + R0 + (first + j) * kFullFixedBytes);
        for (unsigned i = tid; i < fb; i += kSmallThreads) df[i] = S.fixed[j][i];
      }
      uint4* ds = reinterpret_cast<uint4*>(out + S.offset[j]);
      for (unsigned i = tid; i < S.my_size[j] / 16; i += kSmallThreads) ds[i] = S.sec[j][i];
      if (tid == 0) table[first + j] = S.offset[j];
    }
    if (r == 0 && tid == 0) {
      unsigned long long* hdr = reinterpret_cast<unsigned long long*>(out);
      hdr[0] = kMagicWord | (static_cast<unsigned long long>(e0) << 56);
      hdr[1] = n;
      hdr[2] = N;
      hdr[3] = coded;
      table[N] = coded;
      if (kHeaderBytes + 8 * (N + 1) < R0) table[N + 1] = 0;  // zero pad
      ctrl->total = coded;
      if (out_bytes) *out_bytes = coded;
    }
  }
  X.finish();
}

__global__ void __launch_bounds__(kSmallThreads) small_kernel(const uint16_t* in, uint64_t n, int base,
                                                               uint8_t* out, unsigned long long* out_bytes,
                                                               Control* ctrl, int* status) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ClusterExchange X;
  compress_resident(X, *reinterpret_cast<ResidentSmem*>(smem_raw), in, n, base, out, out_bytes, ctrl, status);
}

__global__ void __launch_bounds__(kSmallThreads) medium_kernel(const uint16_t* in, uint64_t n, int base,
                                                                uint8_t* out, unsigned long long* out_bytes,
                                                                uint8_t* ws, int* status) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  GridExchange X;
  X.partials = reinterpret_cast<StatsPartial*>(ws + kWsControlBytes);
  X.bins = reinterpret_cast<unsigned long long*>(ws + kWsExactBinsOffset);
  X.totals = reinterpret_cast<unsigned long long*>(ws + kWsControlBytes + kWsPartialsBytes);
  X.guesses = ws + kWsSampleOffset;  // (the statistics kernel's exponent sample; unused here)
  X.ctrl = reinterpret_cast<Control*>(ws);
  X.arrivals = &X.ctrl->grid_arrivals;
  X.status = status;
  if (blockIdx.x == 0)  // before the first barrier; only the exact path adds to them, after it
    for (unsigned e = threadIdx.x; e < 256; e += kSmallThreads) X.bins[e] = 0;
  compress_resident(X, *reinterpret_cast<ResidentSmem*>(smem_raw), in, n, base, out, out_bytes,
                    reinterpret_cast<Control*>(ws), status);
}

}  // namespace

cudaError_t small_setup(int* small_ctas, int* medium_ctas) {
  const int smem = static_cast<int>(sizeof(ResidentSmem));
  cudaError_t err = cudaFuncSetAttribute(small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(medium_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGridSmemBytes));
  if (err != cudaSuccess) return err;
  // the cooperative grid: every CTA resident at once, and one statistics partial slot each
  int dev = 0, sms = 0, per_sm = 0, coop = 0;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (err != cudaSuccess) return err;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, medium_kernel, kSmallThreads, kGridSmemBytes);
  if (err != cudaSuccess) return err;
  const int grid = coop ? per_sm * sms : 0;
  *medium_ctas = grid < kStatsMaxCtas ? grid : kStatsMaxCtas;

  *small_ctas = static_cast<int>(kSmallPortableCtas);
  if (kSmallCtas > kSmallPortableCtas) {
    err = cudaFuncSetAttribute(small_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) {
      cudaGetLastError();
      return cudaSuccess;  // the portable size then
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kSmallCtas);
    cfg.blockDim = dim3(kSmallThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSmallCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, small_kernel, &cfg) == cudaSuccess && clusters > 0)
      *small_ctas = static_cast<int>(kSmallCtas);
    cudaGetLastError();
  }
  return cudaSuccess;
}

uint64_t small_max_values(const DeviceInfo& dev) {
  return static_cast<uint64_t>(dev.small_ctas) * kPerCta * kChunk;
}

uint64_t medium_max_values(const DeviceInfo& dev) {
  return static_cast<uint64_t>(dev.medium_ctas) * kPerCta * kChunk;
}

cudaError_t launch_small(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                         uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream) {
  const uint64_t N = num_chunks(n);
  const unsigned cmax = static_cast<unsigned>(dev.small_ctas);
  const unsigned C = static_cast<unsigned>(N < cmax ? N : cmax);  // then J = ceil(N / C) <= 4
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = sizeof(ResidentSmem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TimingRecord t = timing_begin(ZC_KERNEL_SMALL, stream);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, small_kernel, in, n, base, out, out_bytes,
                                             reinterpret_cast<Control*>(ws), dev.status);
  timing_end(t, stream);
  return err;
}

cudaError_t launch_medium(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                          uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream) {
  // one chunk per CTA while the device holds that many CTAs, else up to four
  const uint64_t N = num_chunks(n), gmax = static_cast<uint64_t>(dev.medium_ctas);
  const uint64_t J = (N + gmax - 1) / gmax;
  const unsigned G = static_cast<unsigned>((N + J - 1) / J);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = kGridSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: the grid barriers
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TimingRecord t = timing_begin(ZC_KERNEL_MEDIUM, stream);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, medium_kernel, in, n, base, out, out_bytes, ws, dev.status);
  timing_end(t, stream);
  return err;
}

}  // namespace zc
