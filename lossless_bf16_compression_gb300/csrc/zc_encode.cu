// zc_encode.cu -- chunked encoder: 3-bit exponent codes, sign|mantissa byte plane, escape
// compaction, and a single-pass device-wide scan that places every chunk record in one
// contiguous stream behind a chunk-offset table.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution": in-window exponents are
// coded in 3 bits, out-of-window exponents are kept whole "separately" (first technique); the
// kernels use a communication-aware layout, aligned global/shared memory access and pipeline
// data movement with compression compute (second technique).
//
// GB300 design.  A persistent grid of 128-thread CTAs, several per SM.  Each CTA takes chunks
// from an atomic ticket, so chunk order follows execution order and every predecessor of a
// chunk belongs to a running CTA.  Input chunks (8 KiB) arrive by bulk async copy (TMA engine,
// mbarrier completion) two stages ahead; a thread holds 4 slices of 8 values, codes two values
// per 32-bit word with packed 16-bit arithmetic, and writes the record into shared memory.
// The record's stream offset comes from a decoupled look-back over per-chunk state words read
// 32 at a time by one warp (Merrill & Garland, single-pass parallel prefix scan); every wait
// is bounded.  The finished record leaves shared memory in one bulk async store, so the
// compaction costs no extra pass over HBM.
#include "zc_common.cuh"

namespace zc {
namespace {

constexpr int kThreads = kChunkThreads;  // 128
constexpr int kStages = 2;
constexpr unsigned kInBytes = 2 * kChunk;
constexpr unsigned kWaitLimit = 1u << 22;  // mbarrier polls before giving up

struct EncodeParams {
  const uint16_t* in;
  uint64_t n;
  uint64_t N;
  uint8_t* out;
  Control* ctrl;
  unsigned long long* flags;
  unsigned long long* out_bytes;
  int base;  // -1: read e0 from the control block
  int* status;
  uint64_t stall_chunk;
  unsigned spin_limit;
};

struct __align__(128) EncodeSmem {
  uint4 xin[kStages][kInBytes / 16];
  uint4 rec[kStages][kMaxRecordBytes / 16];
  uint64_t mbar[kStages];
  unsigned ticket[kStages];
  unsigned scan[8];
  unsigned long long rec_off;
  int publish;  // look-back succeeded: store the record
  int abort;
  int e0;
};

__device__ void issue_load(EncodeSmem& S, int s, unsigned c, const EncodeParams& p) {
  const uint64_t first = static_cast<uint64_t>(c) * kChunk;
  const unsigned m = chunk_values(p.n, c);
  const unsigned bytes = 2 * m, bulk = bytes & ~15u;
  uint8_t* dst = reinterpret_cast<uint8_t*>(S.xin[s]);
  for (unsigned b = bulk; b < bytes; b += 2)  // ragged tail of the last chunk: < 16 bytes
    *reinterpret_cast<uint16_t*>(dst + b) = p.in[first + b / 2];
  if (bulk) {
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&S.mbar[s], bulk);
    bulk_load(dst, p.in + first, bulk, &S.mbar[s]);
  } else {
    mbar_arrive(&S.mbar[s]);
  }
}

// Warp 0: publish this chunk's size and find the sum of all earlier record sizes.
__device__ bool look_back(const EncodeParams& p, unsigned c, unsigned long long size,
                          unsigned long long* exclusive) {
  const unsigned lane = threadIdx.x & 31;
  if (lane == 0) st_relaxed_u64(&p.flags[c], (c == 0 ? kFlagInclusive : kFlagAggregate) | size);
  unsigned long long excl = 0;
  if (c > 0) {
    long long hi = static_cast<long long>(c) - 1;
    unsigned spins = 0, backoff = 32;
    for (;;) {
      const long long idx = hi - static_cast<long long>(lane);
      const unsigned long long f = idx >= 0 ? ld_relaxed_u64(&p.flags[idx]) : kFlagInclusive;
      const unsigned st = static_cast<unsigned>(f >> 62);
      const unsigned incl = __ballot_sync(0xFFFFFFFFu, st == 2);
      const unsigned zero = __ballot_sync(0xFFFFFFFFu, st == 0);
      const int first = incl ? __ffs(incl) - 1 : 31;
      const unsigned window = first == 31 ? 0xFFFFFFFFu : ((2u << first) - 1u);
      if (zero & window) {  // a predecessor in the window has not published yet
        int bad = lane == 0 ? read_status(p.status) : 0;
        bad = __shfl_sync(0xFFFFFFFFu, bad, 0);
        if (++spins > p.spin_limit || bad != 0) return false;
        __nanosleep(backoff);
        backoff = backoff < 1024 ? backoff * 2 : 1024;
        continue;
      }
      unsigned long long v = static_cast<int>(lane) <= first ? (f & kFlagValueMask) : 0ull;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      excl += v;
      if (incl) break;
      hi -= 32;
      spins = 0;
      backoff = 32;
    }
    if (lane == 0) st_relaxed_u64(&p.flags[c], kFlagInclusive | (excl + size));
  }
  *exclusive = excl;
  return true;
}

__global__ void __launch_bounds__(kThreads) encode_kernel(EncodeParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  EncodeSmem& S = *reinterpret_cast<EncodeSmem*>(smem_raw);
  const unsigned tid = threadIdx.x, warp = tid >> 5;
  // Thread 0's bookkeeping, bit s for stage s: a load is in flight; parity of its next wait.
  unsigned pending = 0, parity = 0;

  if (tid == 0) {
    S.abort = 0;
    S.e0 = p.base >= 0 ? p.base : __ldcg(&p.ctrl->e0);
    for (int s = 0; s < kStages; ++s) mbar_init(&S.mbar[s], 1);
    fence_mbar_init();
    for (int s = 0; s < kStages; ++s) {
      const unsigned c = atomicAdd(&p.ctrl->encode_ticket, 1u);
      S.ticket[s] = c;
      if (c < p.N) {
        issue_load(S, s, c, p);
        pending |= 1u << s;
      }
    }
  }
  __syncthreads();
  const int e0 = S.e0;
  const uint32_t neg_e0x2 = ((0x10000u - static_cast<unsigned>(e0)) & 0xFFFFu) * 0x00010001u;

  for (unsigned it = 0;; ++it) {
    const int s = it & 1;
    if (tid == 0 && it >= 2) bulk_wait_read<1>();  // the store that last used rec[s] has read it
    __syncthreads();                                 // [A]
    const unsigned c = S.ticket[s];
    if (c >= p.N || S.abort) break;

    if (!mbar_wait(&S.mbar[s], (it >> 1) & 1, kWaitLimit)) {
      set_error(p.status, ZC_ERR_TIMEOUT);
      S.abort = 1;
    }
    if (tid == 0) {
      pending &= ~(1u << s);
      parity ^= 1u << s;
    }
    uint4 xq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) xq[q] = S.xin[s][128 * q + tid];
    __syncthreads();  // [B] xin[s] is free again
    if (S.abort) break;
    if (tid == 0) {
      const unsigned nc = atomicAdd(&p.ctrl->encode_ticket, 1u);
      S.ticket[s] = nc;
      if (nc < p.N) {
        issue_load(S, s, nc, p);
        pending |= 1u << s;
      }
    }

    // ---- code the chunk into rec[s]
    const unsigned m = chunk_values(p.n, c);
    const bool full = m == kChunk;
    const unsigned cbytes = full ? kFullCodeBytes : static_cast<unsigned>(code_section_bytes(m));
    const unsigned smbytes = full ? kChunk : static_cast<unsigned>(pad16(m));
    uint8_t* rec = reinterpret_cast<uint8_t*>(S.rec[s]);
    uint8_t* codes = rec + kRecordHeaderBytes;
    uint8_t* smp = codes + cbytes;

    unsigned cnt[4], msk[4];
    uint32_t words[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4] = {xq[q].x, xq[q].y, xq[q].z, xq[q].w};
      const unsigned v0 = 1024 * q + 8 * tid;
      uint32_t c2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) c2[i] = codes_x2(w[i], neg_e0x2);
      if (!full) {  // values past m: code 0, byte 0, no escape
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t keep = (v0 + 2 * i < m ? 0x0000FFFFu : 0u) | (v0 + 2 * i + 1 < m ? 0xFFFF0000u : 0u);
          c2[i] &= keep;
          w[i] &= keep;
        }
      }
      const uint2 smv = make_uint2(sign_mantissa_x4(w[0], w[1]), sign_mantissa_x4(w[2], w[3]));
      if (full || v0 < smbytes) *reinterpret_cast<uint2*>(smp + v0) = smv;
      const uint32_t bits = pack_codes8(c2);
      const unsigned b0 = 3 * (128 * q + tid);
#pragma unroll
      for (int b = 0; b < 3; ++b)
        if (full || b0 + b < cbytes) codes[b0 + b] = static_cast<uint8_t>(bits >> (8 * b));
      msk[q] = escape_mask8(c2);
      cnt[q] = __popc(msk[q]);
#pragma unroll
      for (int i = 0; i < 4; ++i) words[q][i] = w[i];
    }

    unsigned base[4];
    const unsigned k = chunk_ranks(cnt, base, S.scan);  // contains [C]
    const unsigned long long size = kRecordHeaderBytes + cbytes + smbytes + pad16(3ull * k);
    uint8_t* esc = smp + smbytes;

    if (warp == 0) {
      unsigned long long excl = 0;
      bool ok = false;
      if (c != p.stall_chunk) {
        ok = look_back(p, c, size, &excl);
        if (!ok && tid == 0) set_error(p.status, ZC_ERR_TIMEOUT);
      }
      if (tid == 0) {
        S.rec_off = records_base(p.n) + excl;
        S.publish = ok;
        if (!ok) S.abort = 1;
      }
    }
    if (tid == kThreads - 1) {
      *reinterpret_cast<uint4*>(rec) = make_uint4(k, m, 0u, 0u);
      for (unsigned b = 3 * k; b < pad16(3ull * k); ++b) esc[b] = 0;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      unsigned r = base[q];
      unsigned mk = msk[q];
      while (mk) {
        const int j = __ffs(mk) - 1;
        mk &= mk - 1;
        const unsigned E = (pick4(words[q], j >> 1) >> (16 * (j & 1) + 7)) & 0xFFu;
        *reinterpret_cast<uint16_t*>(esc + 2 * r) = static_cast<uint16_t>(1024 * q + 8 * tid + j);
        esc[2 * k + r] = static_cast<uint8_t>(E);
        ++r;
      }
    }
    fence_proxy_async_smem();
    __syncthreads();  // [D] record complete, offset known

    if (tid == 0 && S.publish) {
      const unsigned long long off = S.rec_off;
      bulk_store(p.out + off, rec, static_cast<unsigned>(size));
      unsigned long long* table = reinterpret_cast<unsigned long long*>(p.out + kHeaderBytes);
      table[c] = off;
      if (c == 0) {
        unsigned long long* hdr = reinterpret_cast<unsigned long long*>(p.out);
        hdr[0] = kMagicWord | (static_cast<unsigned long long>(e0) << 56);
        hdr[1] = p.n;
        hdr[2] = p.N;
        if (kHeaderBytes + 8 * (p.N + 1) < records_base(p.n)) table[p.N + 1] = 0;  // zero pad
      }
      if (c == p.N - 1) {
        const unsigned long long total = off + size;
        table[p.N] = total;
        reinterpret_cast<unsigned long long*>(p.out)[3] = total;
        p.ctrl->total = total;
        if (p.out_bytes) *p.out_bytes = total;
      }
    }
    if (tid == 0) bulk_commit();  // one group per iteration, possibly empty
  }

  if (tid == 0) {
    bulk_wait_all<0>();
    // After an abort, loads may still be in flight into this CTA's shared memory.
    for (int s = 0; s < kStages; ++s)
      if (pending & (1u << s)) mbar_wait(&S.mbar[s], (parity >> s) & 1u, kWaitLimit);
  }
}

// n = 0: the stream is the header, offsets[0] = 48 and 8 bytes of padding.
__global__ void empty_stream_kernel(uint8_t* out, int base, Control* ctrl, unsigned long long* out_bytes) {
  unsigned long long* w = reinterpret_cast<unsigned long long*>(out);
  const int e0 = base >= 0 ? base : 0;  // no finite value: e0 = 0
  w[0] = kMagicWord | (static_cast<unsigned long long>(e0) << 56);
  w[1] = 0;
  w[2] = 0;
  w[3] = 48;
  w[4] = 48;
  w[5] = 0;
  ctrl->total = 48;
  if (out_bytes) *out_bytes = 48;
}

}  // namespace

cudaError_t launch_encode(const uint16_t* in, uint64_t n, int base, uint8_t* out,
                          unsigned long long* out_bytes, const DeviceInfo& dev, cudaStream_t stream,
                          uint64_t stall_chunk, unsigned spin_limit) {
  uint8_t* ws = out + workspace_offset(n);
  Control* ctrl = reinterpret_cast<Control*>(ws);
  if (n == 0) {
    empty_stream_kernel<<<1, 1, 0, stream>>>(out, base, ctrl, out_bytes);
    return cudaGetLastError();
  }
  static_assert(sizeof(EncodeSmem) <= 227 * 1024, "shared memory");
  EncodeParams p;
  p.in = in;
  p.n = n;
  p.N = num_chunks(n);
  p.out = out;
  p.ctrl = ctrl;
  p.flags = reinterpret_cast<unsigned long long*>(ws + kWsControlBytes + kWsPartialsBytes);
  p.out_bytes = out_bytes;
  p.base = base;
  p.status = dev.status;
  p.stall_chunk = stall_chunk;
  p.spin_limit = spin_limit;

  const int smem = static_cast<int>(sizeof(EncodeSmem));
  cudaError_t err = cudaFuncSetAttribute(encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, encode_kernel, kThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  uint64_t grid = static_cast<uint64_t>(per_sm) * dev.sm_count;
  if (grid > p.N) grid = p.N;
  timing_begin(ZC_KERNEL_ENCODE, stream);
  encode_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(p);
  timing_end(stream);
  return cudaGetLastError();
}

}  // namespace zc
