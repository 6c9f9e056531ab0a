// zc_decode.cu -- decoder: unpack 3-bit codes, add the window base, scatter the escaped
// exponents, rebuild the BF16 bit patterns, and validate the stream as it goes.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution": in-window exponents are
// e0 + code, out-of-window exponents come from the separate store of full exponents (a list of
// (position, exponent) pairs, or a plane of every exponent when more than a third of the chunk
// escapes), so the reconstruction is exact (first technique); decompression kernels with
// aligned global and shared memory access (second technique).
//
// GB300 design.  One 128-thread CTA per chunk, sixteen CTAs per SM (32 registers, under 10 KB of
// shared memory each): fixed parts sit at places that follow from n and the offset table
// locates every escape section, so there is no inter-CTA dependency.  Warp 0 reads and checks
// the header, then reads and checks the chunk's two escape offsets; the fixed part (5,632 B)
// and the escape section (at most 4 KB, the size of a plane) then arrive in shared memory by
// bulk async copies (TMA engine, one mbarrier).  A thread holds 4 slices of 8 values; per slice
// it takes its 24 code bits and 8 sign|mantissa bytes from shared memory, builds two values per
// 32-bit word with a few integer ops, and writes one coalesced 16-byte store, escaped values
// with a placeholder exponent.  Then the threads walk a list together, one entry each, check it
// against the codes and patch the value, so escape work is proportional to the number of
// escapes rather than to the busiest lane.  A section of a plane's size is built from instead
// in the same single pass (sign|mantissa bytes plus the plane's exponents, each checked against
// its code), and again from the codes in the rare case that the count shows a list of that size.
// A raw stream (the values after the header, when coding did not pay: third technique) is
// copied with 16-byte loads and stores, one chunk's worth per CTA.  Every offset and size is
// checked before it is used, so a corrupt stream sets an error instead of steering a read
// outside [0, total_bytes).
#include "zc_common.cuh"
#include "zc_decode_core.cuh"

namespace zc {
namespace {

constexpr int kThreads = kChunkThreads;  // 128
constexpr int kCtasPerSm = 16;           // 2048 threads per SM: 32 registers and < 14 KB each
constexpr unsigned kEscSmemBytes = 4096; // a chunk's escape section, staged in shared memory
static_assert(kEscSmemBytes >= kMaxEscapeBytes, "every escape section fits the staging buffer");
constexpr unsigned kWaitLimit = 1u << 22;   // mbarrier polls before giving up

struct DecodeParams {
  const uint8_t* in;
  uint16_t* out;
  uint64_t n;
  uint64_t N;
  int* status;
};

struct __align__(128) DecodeSmem {
  uint4 fixed[kFullFixedBytes / 16];
  uint4 esc[kEscSmemBytes / 16];
  uint64_t mbar;
  unsigned escapes;  // code-7 count of the chunk, summed by the warps
  int ok;
  int raw;  // the stream is in the raw form
  int e0;
  unsigned esc_bytes;
};

// A raw stream: chunk c's values are bytes [32 + 8192 c, 32 + 8192 c + 2m) of the stream, copied
// with 16-byte loads and stores.  The last vector of the stream also holds its zero padding,
// which is checked.  Every read lies inside [0, 32 + pad16(2n)) = [0, total_bytes).
__device__ __noinline__ void raw_chunk(const uint8_t* in, uint16_t* out, int* status, uint64_t c, unsigned m) {
  const uint4* src = reinterpret_cast<const uint4*>(in + kHeaderBytes) + c * (kChunk / 8);
  uint4* dst = reinterpret_cast<uint4*>(out + c * kChunk);
  const unsigned whole = m / 8;  // whole vectors of this chunk
  for (unsigned i = threadIdx.x; i < whole; i += kChunkThreads) dst[i] = __ldcs(src + i);
  if (m % 8 && threadIdx.x == 0) {  // the stream's last vector: m % 8 values, then zero padding
    const uint4 v = src[whole];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint16_t* tail = out + c * kChunk + 8 * whole;
    bool bad = false;
    for (unsigned i = 0; i < 8; ++i) {
      const uint16_t x = static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1)));
      if (i < m % 8) tail[i] = x;
      else bad |= x != 0;
    }
    if (bad) set_error(status, ZC_ERR_CORRUPT);
  }
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_kernel(DecodeParams p) {
  __shared__ DecodeSmem S;
  const unsigned tid = threadIdx.x, lane = tid & 31;
  const uint64_t c = blockIdx.x;
  const uint64_t first = c * kChunk;
  const unsigned m = c < p.N ? chunk_values(p.n, c) : 0;

  if (tid < 32) {
    // Lanes 0..3 fetch the 32-byte header, and every lane checks it against the caller's n:
    // magic, version, form, base, n, N, and total_bytes -- for the coded form between the start
    // of the escape region and the raw form's length, for the raw form exactly that length.  Only
    // then, and only for the coded form, do lanes 4..6 fetch the chunk's two escape offsets and
    // the table's zero pad; they lie below records_base(n) <= escape_base(n) <= total_bytes, so a
    // wrong n or a short total_bytes never steers a read past the stream.
    const unsigned long long* w = reinterpret_cast<const unsigned long long*>(p.in);
    const uint64_t R0 = records_base(p.n), E0 = escape_base(p.n), RAW = raw_stream_bytes(p.n);
    const bool has_pad = kHeaderBytes + 8 * (p.N + 1) < R0;
    const unsigned long long hv = lane < 4 ? w[lane] : 0ull;
    const unsigned long long h0 = __shfl_sync(0xFFFFFFFFu, hv, 0), h1 = __shfl_sync(0xFFFFFFFFu, hv, 1);
    const unsigned long long h2 = __shfl_sync(0xFFFFFFFFu, hv, 2), total = __shfl_sync(0xFFFFFFFFu, hv, 3);
    const int e0 = static_cast<int>(h0 >> 56);
    const unsigned long long head = h0 & 0x00FFFFFFFFFFFFFFull;  // bytes 0..6
    const bool raw = head == kRawMagicWord;
    int bad = 0;
    if ((head != kMagicWord && !raw) || e0 > kE0Max) bad = ZC_ERR_CORRUPT;
    else if (h1 != p.n) bad = ZC_ERR_SIZE_MISMATCH;
    else if (raw ? (h2 != 0 || total != RAW) : (h2 != p.N || total < E0 || total > RAW)) bad = ZC_ERR_CORRUPT;
    unsigned long long v = 0;
    if (!bad && !raw) {  // the same in every lane
      if (lane == 4) v = w[4 + c];
      else if (lane == 5 && c < p.N) v = w[5 + c];
      else if (lane == 6 && has_pad && (c == 0 || c + 1 >= p.N)) v = w[5 + p.N];
    }
    const unsigned long long off0 = __shfl_sync(0xFFFFFFFFu, v, 4), off1 = __shfl_sync(0xFFFFFFFFu, v, 5);
    const unsigned long long pad = __shfl_sync(0xFFFFFFFFu, v, 6);
    if (lane == 0) {
      if (bad == 0 && !raw &&
          (pad != 0 || (c == 0 && off0 != E0) || (p.N == 0 && total != E0) ||
           (p.N > 0 && c == p.N - 1 && off1 != total) ||
           (c < p.N && (off0 < E0 || off1 > total || off1 < off0 || ((off0 | off1) & 15) ||
                        off1 - off0 > pad16(m)))))  // an escape section is at most a plane
        bad = ZC_ERR_CORRUPT;
      if (bad) set_error(p.status, bad);
      S.ok = !bad && c < p.N;
      S.raw = raw;
      S.e0 = e0;
      S.escapes = 0;
      S.esc_bytes = static_cast<unsigned>(off1 - off0);
      if (S.ok && !raw) {
        const unsigned fbytes = static_cast<unsigned>(fixed_bytes(m));
        mbar_init(&S.mbar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&S.mbar, fbytes + S.esc_bytes);
        bulk_load(S.fixed, p.in + fixed_offset(p.n, c), fbytes, &S.mbar);
        if (S.esc_bytes) bulk_load(S.esc, p.in + off0, S.esc_bytes, &S.mbar);
      }
    }
  }
  __syncthreads();
  if (!S.ok) return;
  if (S.raw) {  // the values follow the header as they are
    raw_chunk(p.in, p.out, p.status, c, m);
    return;
  }
  // every thread polls; the CTA acts on one shared answer
  if (__syncthreads_or(!mbar_wait(&S.mbar, 0, kWaitLimit))) {
    if (tid == 0) {
      set_error(p.status, ZC_ERR_TIMEOUT);
      mbar_wait(&S.mbar, 0, kWaitLimit);  // never leave a copy in flight
    }
    return;
  }

  decode_chunk(S.fixed, S.esc, &S.escapes, p.out + first, m, S.e0, S.esc_bytes, p.status, tid,
               [] { __syncthreads(); });
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
  TimingRecord t = timing_begin(ZC_KERNEL_DECODE, stream);
  decode_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
  timing_end(t, stream);
  return cudaGetLastError();
}

}  // namespace zc
