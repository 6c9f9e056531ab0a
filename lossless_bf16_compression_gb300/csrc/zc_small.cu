// zc_small.cu -- compression of a small tensor (up to 64 chunks of 4096 values) in one launch of
// one thread-block cluster: no workspace, no memset, no tensor map, no second kernel.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution": the window base from the
// tensor's standard deviation, 3-bit codes with the full exponents of the others kept apart
// (first technique), and the native form where coding does not pay (third technique).  The
// overhead of a compressor on small messages is what the page calls its performance cliff
// (general-purpose compressors can be slower than sending the data as it is); here a small
// tensor costs one launch.
//
// GB300 design.  C = min(N, 16) CTAs of 128 threads form one cluster; CTA r holds chunks r, r + C,
// ... in shared memory (up to four: 32 KiB of input, their fixed parts and escape sections, about
// 70 KB).  The input arrives by bulk async copies.  Each CTA sums its squares in the same fp32
// blocks with the same error bound as the statistics kernel; after a cluster barrier every CTA
// reads all partials through distributed shared memory, in rank order, so all settle the same e0
// (and, when the bound straddles a switching point, the same exact per-exponent sums).  The CTAs
// code their chunks into shared memory, exchange the sections' sizes the same way, and write
// either the coded stream (fixed parts, sections at their scanned offsets, table, header) or the
// raw form.  Every cluster barrier is the hardware's; the one wait that polls (the copies'
// mbarrier) is bounded.
#include <cooperative_groups.h>

#include "zc_code_core.cuh"
#include "zc_common.cuh"
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
constexpr unsigned kSmallPerCta = 4;    // chunks per CTA, at most (more are faster on the big path)
constexpr int kSmallThreads = 128;      // a chunk's coding threads, 32 values each
static_assert(32 * kSmallThreads == kChunk, "a thread codes 32 consecutive values of a chunk");
constexpr unsigned kSmallWaitLimit = 1u << 22;

struct __align__(128) SmallSmem {
  uint4 x[kSmallPerCta][kChunk / 8];                 // inputs, 8 KiB per chunk (zero past m)
  uint4 fixed[kSmallPerCta][kFullFixedBytes / 16];   // fixed parts: codes, then sign|mantissa
  uint4 sec[kSmallPerCta][kMaxEscapeBytes / 16];     // escape sections
  unsigned long long bins[256];                      // exact fallback: this CTA's exponent sums
  unsigned long long allbins[256];                   // ... and the cluster's
  unsigned long long offset[kSmallCtas * kSmallPerCta];  // every chunk's section offset (stream)
  unsigned size[kSmallCtas * kSmallPerCta];          // every chunk's section bytes
  uint64_t mbar;
  double wsum[kSmallThreads / 32];
  unsigned long long wnf[kSmallThreads / 32];
  double cta_sum;
  unsigned long long cta_nonfinite;
  unsigned long long total;
  unsigned scan[kSmallThreads / 32];
  unsigned my_size[kSmallPerCta];
  int e0;
  int need_exact;
  int ok;
};

__device__ __forceinline__ void bar_cta() { __syncthreads(); }

__global__ void __launch_bounds__(kSmallThreads) small_kernel(const uint16_t* in, uint64_t n, int base,
                                                               uint8_t* out, unsigned long long* out_bytes,
                                                               Control* ctrl, int* status) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SmallSmem& S = *reinterpret_cast<SmallSmem*>(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned C = cluster.num_blocks(), r = cluster.block_rank();
  const unsigned tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint64_t N = num_chunks(n);
  const unsigned J = N > r ? static_cast<unsigned>((N - r + C - 1) / C) : 0u;  // chunks r + C j, j < J

  // ---- the input: whole 16-byte vectors by bulk async copies, the ragged tail and zeros by threads
  if (tid == 0) {
    mbar_init(&S.mbar, 1);
    fence_mbar_init();
    unsigned bytes = 0;
    for (unsigned j = 0; j < J; ++j) bytes += (2 * chunk_values(n, r + C * j)) & ~15u;
    mbar_arrive_expect_tx(&S.mbar, bytes);
    for (unsigned j = 0; j < J; ++j) {
      const uint64_t c = r + C * j;
      const unsigned vb = (2 * chunk_values(n, c)) & ~15u;
      if (vb) bulk_load(S.x[j], in + c * kChunk, vb, &S.mbar);
    }
  }
  for (unsigned j = 0; j < J; ++j) {
    const uint64_t c = r + C * j;
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
  // (a CTA whose copies did not arrive still takes part in every cluster barrier below, with zeros)

  // ---- the window base
  int e0 = base;
  if (base < 0) {
    double acc = 0.0;
    unsigned nonfinite = 0;
    const unsigned B = 64 * J;  // blocks of 64 values of this CTA's chunks (zeros past m add nothing)
    for (unsigned b0 = 0; b0 < B; b0 += kSmallThreads) {
      const unsigned b = b0 + tid;
      uint32_t w[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 v = b < B && S.ok ? S.x[b / 64][8 * (b % 64) + k] : make_uint4(0, 0, 0, 0);
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
    if (tid == 0) {
      double s = 0.0;
      unsigned long long c = 0;
      for (int i = 0; i < kSmallThreads / 32; ++i) {
        s += S.wsum[i];
        c += S.wnf[i];
      }
      S.cta_sum = s;
      S.cta_nonfinite = c;
    }
    cluster.sync();
    if (tid == 0) {  // every CTA combines the partials in rank order: the same e0 everywhere
      double s = 0.0;
      unsigned long long nf_all = 0;
      for (unsigned q = 0; q < C; ++q) {
        s += *cluster.map_shared_rank(&S.cta_sum, q);
        nf_all += *cluster.map_shared_rank(&S.cta_nonfinite, q);
      }
      int e = 0;
      S.need_exact = decide_e0(s, n - nf_all, &e) ? 0 : 1;
      S.e0 = e;
      S.total = n - nf_all;  // the finite count, kept for the exact path
    }
    bar_cta();
    if (S.need_exact) {  // the same in every CTA: exact per-exponent sums over the cluster
      for (unsigned e = tid; e < 256; e += kSmallThreads) S.bins[e] = 0;
      bar_cta();
      for (unsigned j = 0; j < J; ++j)
        add_exponent_sums(reinterpret_cast<const uint16_t*>(S.x[j]), chunk_values(n, r + C * j), tid, kSmallThreads,
                          S.bins);
      cluster.sync();
      for (unsigned e = tid; e < 256; e += kSmallThreads) {
        unsigned long long t = 0;
        for (unsigned q = 0; q < C; ++q) t += cluster.map_shared_rank(S.bins, q)[e];
        S.allbins[e] = t;
      }
      bar_cta();
      if (tid == 0) S.e0 = select_e0(exact_from_bins(S.allbins), S.total);
      cluster.sync();  // no CTA overwrites its bins while another one reads them
    }
    e0 = S.e0;
    if (r == 0 && tid == 0 && ctrl) {
      ctrl->e0 = e0;
      ctrl->exact_path = S.need_exact;
    }
  }

  // ---- code this CTA's chunks into shared memory
  const uint32_t kadd = ((256u - static_cast<unsigned>(e0)) << 7) * 0x00010001u;
  const unsigned v0 = 32 * tid;
  for (unsigned j = 0; j < J; ++j) {
    const unsigned m = chunk_values(n, r + C * j);
    const bool full = m == kChunk;
    const unsigned cbytes = full ? kFullCodeBytes : static_cast<unsigned>(code_section_bytes(m));
    const unsigned smbytes = full ? kChunk : static_cast<unsigned>(pad16(m));
    uint4 xv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) xv[q] = S.x[j][4 * tid + q];
    Coded32 kd;
    code32(xv, kadd, v0, m, full, kd);
    // (a ragged chunk's threads past m store zero codes and bytes: the sections' padding)
    store_fixed32(reinterpret_cast<uint8_t*>(S.fixed[j]), cbytes, smbytes, v0, full, kd);
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
    for (int i = 0; i < kSmallThreads / 32; ++i) {
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

  // ---- the sections' offsets: every chunk's size from its CTA, in chunk order
  cluster.sync();
  const uint64_t E0 = escape_base(n), R0 = records_base(n);
  for (unsigned c = tid; c < N; c += kSmallThreads) S.size[c] = cluster.map_shared_rank(S.my_size, c % C)[c / C];
  bar_cta();
  if (tid == 0) {
    unsigned long long at = E0;
    for (unsigned c = 0; c < N; ++c) {
      S.offset[c] = at;
      at += S.size[c];
    }
    S.total = at;
  }
  bar_cta();
  const unsigned long long coded = S.total, raw = raw_stream_bytes(n);
  if (coded > raw) {  // the raw form: the header, the values as they are, zero padding
    for (unsigned j = 0; j < J; ++j) {
      const uint64_t c = r + C * j;
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
      if (ctrl) ctrl->total = raw;
      if (out_bytes) *out_bytes = raw;
    }
  } else {  // the coded form: fixed parts, escape sections, offset table, header
    unsigned long long* table = reinterpret_cast<unsigned long long*>(out + kHeaderBytes);
    for (unsigned j = 0; j < J; ++j) {
      const uint64_t c = r + C * j;
      const unsigned fb = static_cast<unsigned>(fixed_bytes(chunk_values(n, c))) / 16;
      uint4* df = reinterpret_cast<uint4*>(out + R0 + c * kFullFixedBytes);
      for (unsigned i = tid; i < fb; i += kSmallThreads) df[i] = S.fixed[j][i];
      uint4* ds = reinterpret_cast<uint4*>(out + S.offset[c]);
      for (unsigned i = tid; i < S.size[c] / 16; i += kSmallThreads) ds[i] = S.sec[j][i];
      if (tid == 0) table[c] = S.offset[c];
    }
    if (r == 0 && tid == 0) {
      unsigned long long* hdr = reinterpret_cast<unsigned long long*>(out);
      hdr[0] = kMagicWord | (static_cast<unsigned long long>(e0) << 56);
      hdr[1] = n;
      hdr[2] = N;
      hdr[3] = coded;
      table[N] = coded;
      if (kHeaderBytes + 8 * (N + 1) < R0) table[N + 1] = 0;  // zero pad
      if (ctrl) ctrl->total = coded;
      if (out_bytes) *out_bytes = coded;
    }
  }
  cluster.sync();  // no CTA leaves while another one may still read its shared memory
}

}  // namespace

cudaError_t small_setup(int* max_ctas) {
  cudaError_t err = cudaFuncSetAttribute(small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sizeof(SmallSmem)));
  if (err != cudaSuccess) return err;
  *max_ctas = static_cast<int>(kSmallPortableCtas);
  if (kSmallCtas > kSmallPortableCtas) {
    err = cudaFuncSetAttribute(small_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) {
      cudaGetLastError();
      return cudaSuccess;  // the portable size then
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kSmallCtas);
    cfg.blockDim = dim3(kSmallThreads);
    cfg.dynamicSmemBytes = sizeof(SmallSmem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSmallCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, small_kernel, &cfg) == cudaSuccess && clusters > 0)
      *max_ctas = static_cast<int>(kSmallCtas);
    cudaGetLastError();
  }
  return cudaSuccess;
}

uint64_t small_max_values(const DeviceInfo& dev) {
  return static_cast<uint64_t>(dev.small_ctas) * kSmallPerCta * kChunk;
}

cudaError_t launch_small(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                         uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream) {
  const uint64_t N = num_chunks(n);
  const unsigned cmax = static_cast<unsigned>(dev.small_ctas);
  const unsigned C = static_cast<unsigned>(N < cmax ? N : cmax);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = sizeof(SmallSmem);
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

}  // namespace zc
