// zc_decode.cu -- decoder: unpack 3-bit codes, add the window base, scatter the escaped
// exponents, rebuild the BF16 bit patterns, and validate the stream as it goes.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution": in-window exponents are
// e0 + code, out-of-window exponents come from the separate full-exponent list, so the
// reconstruction is exact (first technique); decompression kernels with aligned global and
// shared memory access (second technique).
//
// GB300 design.  One 128-thread CTA per chunk, many CTAs per SM: the chunk-offset table makes
// every record independently addressable, so there is no inter-CTA dependency.  A thread holds
// 4 slices of 8 values; per slice it reads its 24 code bits (two aligned 32-bit loads and a
// funnel shift) and 8 sign|mantissa bytes, builds two values per 32-bit word, and writes one
// coalesced 16-byte store.  Escapes get their rank from the same block scan the encoder uses,
// which also checks every stored position and exponent.  Every offset and size is checked
// against the header and the record's own header before it is used, so a corrupt stream sets
// an error instead of steering a read outside [0, total_bytes).
#include "zc_common.cuh"

namespace zc {
namespace {

constexpr int kThreads = kChunkThreads;  // 128

struct DecodeParams {
  const uint8_t* in;
  uint16_t* out;
  uint64_t n;
  uint64_t N;
  int* status;
};

__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeParams p) {
  __shared__ unsigned scan[8];
  __shared__ int hdr_ok;
  __shared__ int e0_s;
  __shared__ unsigned k_s;
  __shared__ unsigned long long off_s;

  const unsigned tid = threadIdx.x;
  const uint64_t c = blockIdx.x;
  const uint64_t first = c * kChunk;
  const unsigned m = c < p.N ? chunk_values(p.n, c) : 0;

  if (tid == 0) {
    const unsigned long long* w = reinterpret_cast<const unsigned long long*>(p.in);
    const unsigned long long h0 = w[0], h1 = w[1], h2 = w[2], total = w[3];
    const unsigned long long off0 = w[4 + c];
    const unsigned long long off1 = c < p.N ? w[5 + c] : 0;
    const uint64_t R0 = records_base(p.n);
    int bad = 0;
    const int e0 = static_cast<int>(h0 >> 56);
    if ((h0 & 0x00FFFFFFFFFFFFFFull) != kMagicWord || e0 > kE0Max) bad = ZC_ERR_CORRUPT;
    else if (h1 != p.n) bad = ZC_ERR_SIZE_MISMATCH;
    else if (h2 != p.N || total < R0 || total > max_stream_bytes(p.n)) bad = ZC_ERR_CORRUPT;
    if (!bad && (c == 0 || c == p.N - 1 || p.N == 0)) {
      // the table's zero pad, and the ends of the table
      if (kHeaderBytes + 8 * (p.N + 1) < R0 && w[5 + p.N] != 0) bad = ZC_ERR_CORRUPT;
      if (c == 0 && off0 != R0) bad = ZC_ERR_CORRUPT;
      if (p.N == 0 && total != R0) bad = ZC_ERR_CORRUPT;
      if (p.N > 0 && c == p.N - 1 && off1 != total) bad = ZC_ERR_CORRUPT;
    }
    unsigned k = 0;
    if (!bad && c < p.N) {
      if (off0 < R0 || off1 > total || off1 <= off0 || ((off0 | off1) & 15) ||
          off1 - off0 > static_cast<unsigned long long>(kMaxRecordBytes)) {
        bad = ZC_ERR_CORRUPT;
      } else {
        const uint4 rh = *reinterpret_cast<const uint4*>(p.in + off0);
        k = rh.x;
        if (rh.y != m || k > m || rh.z != 0 || rh.w != 0 || off1 - off0 != record_bytes(m, k))
          bad = ZC_ERR_CORRUPT;
      }
    }
    if (bad) set_error(p.status, bad);
    hdr_ok = !bad;
    e0_s = e0;
    k_s = k;
    off_s = off0;
  }
  __syncthreads();
  if (!hdr_ok || c >= p.N) return;

  const int e0 = e0_s;
  const unsigned k = k_s;
  const bool full = m == kChunk;
  const unsigned cbytes = full ? kFullCodeBytes : static_cast<unsigned>(code_section_bytes(m));
  const unsigned smbytes = full ? kChunk : static_cast<unsigned>(pad16(m));
  const uint8_t* rec = p.in + off_s;
  const uint8_t* codes = rec + kRecordHeaderBytes;
  const uint8_t* smp = codes + cbytes;
  const uint8_t* esc = smp + smbytes;
  const uint32_t e0x2 = static_cast<uint32_t>(e0) * 0x00010001u;

  uint32_t x[4][4];
  unsigned cnt[4], msk[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const unsigned g = 128 * q + tid, v0 = 8 * g;
    cnt[q] = 0;
    msk[q] = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) x[q][i] = 0;
    if (!full && v0 >= m) continue;
    const unsigned b = 3 * g;
    const uint32_t* cw = reinterpret_cast<const uint32_t*>(codes + (b & ~3u));
    const uint32_t bits = __funnelshift_r(__ldg(cw), __ldg(cw + 1), 8 * (b & 3));
    const uint2 sm = __ldg(reinterpret_cast<const uint2*>(smp + v0));
    uint32_t c2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      c2[i] = ((bits >> (6 * i)) & 7u) | (((bits >> (6 * i + 3)) & 7u) << 16);
      const uint32_t sw = i < 2 ? sm.x : sm.y;
      const unsigned lo = (2 * i) & 3;
      const uint32_t s2 = prmt(sw, 0u, lo | (4u << 4) | ((lo + 1) << 8) | (4u << 12));  // two bytes -> halves
      const uint32_t sign_mant = ((s2 << 8) & 0x80008000u) | (s2 & 0x007F007Fu);
      x[q][i] = sign_mant | (((c2[i] + e0x2) & 0x00FF00FFu) << 7);
    }
    msk[q] = escape_mask8(c2);
    if (!full && v0 + 8 > m) msk[q] &= (1u << (m - v0)) - 1u;  // padding codes are checked below
    cnt[q] = __popc(msk[q]);
  }

  unsigned base[4];
  const unsigned total = chunk_ranks(cnt, base, scan);
  bool corrupt = total != k;

#pragma unroll
  for (int q = 0; q < 4; ++q) {
    unsigned mk = msk[q], r = base[q];
    const unsigned v0 = 1024 * q + 8 * tid;
    while (mk) {
      const int j = __ffs(mk) - 1;
      mk &= mk - 1;
      if (r >= k) {
        corrupt = true;
        break;
      }
      const unsigned pos = __ldg(reinterpret_cast<const uint16_t*>(esc) + r);
      const unsigned E = __ldg(esc + 2 * k + r);
      if (pos != v0 + j || (E >= static_cast<unsigned>(e0) && E <= static_cast<unsigned>(e0) + 6)) corrupt = true;
      const unsigned sh = 16 * (j & 1);
      const uint32_t clear = ~(0xFFu << (sh + 7));
      const uint32_t v = (pick4(x[q], j >> 1) & clear) | (E << (sh + 7));
      const unsigned wi = j >> 1;
      x[q][0] = wi == 0 ? v : x[q][0];
      x[q][1] = wi == 1 ? v : x[q][1];
      x[q][2] = wi == 2 ? v : x[q][2];
      x[q][3] = wi == 3 ? v : x[q][3];
      ++r;
    }
  }

#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const unsigned v0 = 1024 * q + 8 * tid;
    if (full || v0 + 8 <= m) {
      *reinterpret_cast<uint4*>(p.out + first + v0) = make_uint4(x[q][0], x[q][1], x[q][2], x[q][3]);
    } else if (v0 < m) {
      for (unsigned j = 0; v0 + j < m; ++j)
        p.out[first + v0 + j] = static_cast<uint16_t>(pick4(x[q], j >> 1) >> (16 * (j & 1)));
    }
  }

  if (tid == 0) {  // zero padding: escapes always, codes and bytes of a partial chunk
    for (unsigned b = 3 * k; b < pad16(3ull * k); ++b) corrupt |= esc[b] != 0;
    if (!full) {
      for (unsigned b = m; b < smbytes; ++b) corrupt |= smp[b] != 0;
      for (unsigned bit = 3 * m; bit < 8 * cbytes; ++bit) corrupt |= ((codes[bit >> 3] >> (bit & 7)) & 1u) != 0;
    }
  }
  if (corrupt) set_error(p.status, ZC_ERR_CORRUPT);
}

}  // namespace

cudaError_t launch_decode(const uint8_t* in, uint16_t* out, uint64_t n, const DeviceInfo& dev,
                          cudaStream_t stream) {
  DecodeParams p;
  p.in = in;
  p.out = out;
  p.n = n;
  p.N = num_chunks(n);
  p.status = dev.status;
  const uint64_t grid = p.N ? p.N : 1;  // n = 0: one CTA checks the header
  timing_begin(ZC_KERNEL_DECODE, stream);
  decode_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
  timing_end(stream);
  return cudaGetLastError();
}

}  // namespace zc
