// zc_common.cuh -- layout arithmetic, workspace, PTX wrappers and value-level helpers shared by
// the sm_103a kernels of the lossless BF16 exponent codec.
//
// Method: ZipCCL (SIGCOMM scribe notes), "Key idea and contribution": exponent coding with a
// window taken from the standard deviation (first technique) and GPU kernels with a
// layout shaped by the communication, aligned global/shared memory access and data movement pipelined
// with compute (second technique).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "zc.h"

namespace zc {

// ------------------------------------------------------------------ stream layout ("ZCB1" v4)
//
// Coded form (header byte 6 = 12):
// header (32 B) | u64 escape offsets [N+1] | zero pad to 16 | fixed parts | escape sections
// The fixed part of chunk c (3-bit codes, then the sign|mantissa plane) starts at
// records_base(n) + c * kFullFixedBytes, so its place follows from n alone; only the escape
// sections are placed by the scan.  A chunk of m values with k escapes keeps them as a list (u16
// positions, u8 exponents, zero pad) when 3k <= m, else as a plane of all m exponents (zero
// pad): whichever is smaller, chosen from k, which the codes give.
// Raw form (header byte 6 = 0, N = 0): header (32 B) | the n values | zero pad to 16.  A tensor
// whose coded form would be longer than its raw form is stored raw (ties keep the coded form).
constexpr int kChunk = 4096;                       // values per chunk
constexpr int kHeaderBytes = 32;                   // stream header
constexpr int kFullCodeBytes = 3 * kChunk / 8;     // 1536: 3-bit codes of a full chunk
constexpr int kFullFixedBytes = kFullCodeBytes + kChunk;  // 5632: fixed part of a full chunk
constexpr int kMaxEscapeBytes = kChunk;            // 4096: an exponent plane, the largest section
constexpr int kE0Max = 249;
constexpr unsigned long long kRawMagicWord =       // bytes 0..6 of a raw header: "ZCB1", v4, 0
    0x5Aull | (0x43ull << 8) | (0x42ull << 16) | (0x31ull << 24) | (4ull << 32);
constexpr unsigned long long kMagicWord =          // bytes 0..6 of a coded header: "ZCB1", v4, 12
    kRawMagicWord | (12ull << 48);

__host__ __device__ constexpr uint64_t pad16(uint64_t v) { return (v + 15u) & ~uint64_t(15); }
__host__ __device__ constexpr uint64_t num_chunks(uint64_t n) { return (n + kChunk - 1) / kChunk; }
// Values in chunk c of an n-value tensor (c < num_chunks(n)).
__host__ __device__ inline unsigned chunk_values(uint64_t n, uint64_t c) {
  const uint64_t left = n - c * kChunk;
  return left < static_cast<uint64_t>(kChunk) ? static_cast<unsigned>(left) : static_cast<unsigned>(kChunk);
}
// Start of the fixed region.
__host__ __device__ inline uint64_t records_base(uint64_t n) {
  return pad16(kHeaderBytes + 8 * (num_chunks(n) + 1));
}
__host__ __device__ inline uint64_t code_section_bytes(uint64_t m) { return pad16((3 * m + 7) / 8); }
__host__ __device__ inline uint64_t fixed_bytes(uint64_t m) { return code_section_bytes(m) + pad16(m); }
__host__ __device__ inline uint64_t fixed_offset(uint64_t n, uint64_t c) {
  return records_base(n) + c * static_cast<uint64_t>(kFullFixedBytes);
}
// Start of the escape region, right after the last fixed part.
__host__ __device__ inline uint64_t escape_base(uint64_t n) {
  const uint64_t N = num_chunks(n);
  return N ? fixed_offset(n, N - 1) + fixed_bytes(chunk_values(n, N - 1)) : records_base(n);
}
// Escape section of a chunk of m values with k escapes: a list when 3k <= m, else a plane.
__host__ __device__ inline bool exponent_plane(unsigned m, unsigned k) { return 3 * k > m; }
__host__ __device__ inline unsigned escape_section_bytes(unsigned m, unsigned k) {
  return static_cast<unsigned>(exponent_plane(m, k) ? pad16(m) : pad16(3ull * k));
}
// Length of the raw form: the header, the n values, zero padding.
__host__ __device__ constexpr uint64_t raw_stream_bytes(uint64_t n) { return kHeaderBytes + pad16(2 * n); }
// Bytes of `out` that a call may write: the stream is at most raw_stream_bytes(n) long, and the
// coded fixed parts, written before the form is known, end at escape_base(n).  (Escape sections
// that would end past raw_stream_bytes(n) are never written: the stream is then raw.)
__host__ __device__ inline uint64_t max_stream_bytes(uint64_t n) {
  const uint64_t e = escape_base(n), r = raw_stream_bytes(n);
  return e > r ? e : r;
}
// The longest coded form (every chunk keeps a plane of exponents): the room the loopback needs,
// since it writes every escape section before the form is chosen.
__host__ __device__ inline uint64_t max_coded_bytes(uint64_t n) {
  return escape_base(n) + (n / kChunk) * kMaxEscapeBytes + pad16(n % kChunk);
}

// ------------------------------------------------------------------ workspace (tail of `out`)
//
// [ws + 0,    ws + 256)            Control block
// [ws + 256,  ws + 256 + 12 KiB)   per-CTA partials of the statistics pass
// [.., ws + 256 + 14 KiB)          exact fallback: per-exponent sums of sig^2, 256 x u64
// [.., ws + 256 + 16 KiB)          exponent sample of the statistics pass, 256 x u64 counts
// [ws + 16640, ...)                scan state, one u64 per chunk
constexpr int kStatsMaxCtas = 768;
constexpr uint64_t kWsControlBytes = 256;
constexpr uint64_t kWsExactBinsOffset = kWsControlBytes + 16ull * kStatsMaxCtas;
constexpr uint64_t kWsSampleOffset = kWsExactBinsOffset + 8 * 256;
constexpr uint64_t kWsPartialsBytes = 16ull * kStatsMaxCtas + 8 * 256 + 8 * 256;  // partials, bins, sample
static_assert(kWsPartialsBytes == 16384, "the workspace is 16,640 bytes plus 8 per chunk");

struct Control {
  unsigned encode_ticket;   // next chunk to hand out (encoder)
  unsigned stats_done;      // CTAs of the statistics pass that have finished
  int e0;                   // window base chosen by the statistics pass
  unsigned exact_path;      // 1 when the statistics pass needed its exact fallback
  unsigned long long total; // stream length, for the pageable out_bytes path
  unsigned role_ticket;     // encoder CTAs in start order: the first one to start scans
  unsigned decode_ticket;   // loopback: next chunk to decode
  unsigned first_ticket;    // the encoder's first phase: next chunk to take
  unsigned long long n_finite;  // finite values, for the exact fallback
  unsigned long long exact_pieces[4];  // exact fallback: 32-bit pieces of the window sums
  unsigned raw_predicted;   // 1: the statistics pass's exponent sample predicts a raw stream
  unsigned raw_done;        // 1: the raw pass found the coded form longer and wrote the raw form
  unsigned first_done;      // the encoder's first phase: chunks finished
  unsigned first_ready;     // the encoder's first phase: e0 and the stream form are final
  unsigned long long raw_escape_bytes;  // raw pass: the escape sections' bytes, summed
  unsigned grid_arrivals;   // the grid kernels' barriers: CTAs arrived so far
  unsigned grid_release;    // the L2-resident kernel: the last barrier its last CTA released
  int grid_e0;              // ... the window base, and 1 when the exact sums must decide it
  unsigned grid_exact;
  unsigned long long grid_escape_bytes;  // ... the escape sections' bytes, all chunks
  // The speculative encode kernel: its sums of squares and Inf/NaN counts (added by each CTA
  // as it leaves), the chunks they cover, and a CTA's report that too few of its values were
  // inside the window for its fast sums to be trusted.
  double spec_sum;
  unsigned long long spec_nonfinite;
  unsigned spec_chunks;
  unsigned spec_untrusted;
  unsigned grid_guesses_held;  // the cooperative grid: 1 when every CTA coded with the settled e0
  unsigned reserved[21];
  // 1: the speculative encode kernel did not speculate (its sample was not confident) or found
  // its guess wrong: the statistics and encode kernels after it do the job.
  unsigned fallback;
  unsigned fallback_pad[3];
};
static_assert(sizeof(Control) == kWsControlBytes, "the control block fills its place");
static_assert(offsetof(Control, fallback) == kWsControlBytes - 16,
              "the fallback word sits alone in the control block's last 16 bytes");
static_assert(offsetof(Control, exact_path) == 12 && offsetof(Control, raw_predicted) == 80 &&
                  offsetof(Control, raw_done) == 84,
              "the tests read these words of the control block at these offsets");

struct StatsPartial {
  double sum;               // fp64 sum of block sums of squares
  unsigned long long nonfinite;
};

__host__ __device__ inline uint64_t workspace_offset(uint64_t n) {
  return (max_stream_bytes(n) + 255) & ~uint64_t(255);
}
__host__ __device__ constexpr uint64_t workspace_bytes(uint64_t n) {
  return kWsControlBytes + kWsPartialsBytes + 8 * num_chunks(n);
}

// Scan state word of a chunk: bits 62..63 status, bits 0..61 value.
constexpr unsigned long long kFlagAggregate = 1ull << 62;   // value = this chunk's record size
constexpr unsigned long long kFlagInclusive = 2ull << 62;   // value = sizes up to and including it
constexpr unsigned long long kFlagCopied = 3ull << 62;      // inclusive, and the section is written (loopback)
constexpr unsigned long long kFlagValueMask = (1ull << 62) - 1;

// ------------------------------------------------------------------ errors

__device__ __forceinline__ void set_error(int* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ int read_status(const int* status) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(status) : "memory");
  return v;
}

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, unsigned limit) {
  for (unsigned i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Bulk (non-tensor) async copies: 16-byte aligned addresses, size a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Packed 16-bit lane arithmetic (two BF16 values per 32-bit word).
__device__ __forceinline__ uint32_t add_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Shared-memory accesses by 32-bit shared-window address.
__device__ __forceinline__ void sts_u8(uint32_t a, unsigned v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "h"(static_cast<unsigned short>(v)) : "memory");
}
__device__ __forceinline__ void sts_u16(uint32_t a, unsigned v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(static_cast<unsigned short>(v)) : "memory");
}
__device__ __forceinline__ unsigned lds_u8(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ unsigned lds_u16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ unsigned lds_u32(uint32_t a) {
  unsigned v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_v2(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}

// ------------------------------------------------------------------ value-level helpers

// a[i] for a runtime i without local-memory indexing.
__device__ __forceinline__ uint32_t pick4(const uint32_t (&a)[4], unsigned i) {
  return i < 2 ? (i == 0 ? a[0] : a[1]) : (i == 2 ? a[2] : a[3]);
}

// Codes of two BF16 values (halves of w), each shifted left by 7: e - e0 when 0 <= e - e0 <= 6,
// else 7.  kadd holds (256 - e0) << 7 in both halves: the masked exponent field plus it stays
// below 2^16, and bits 7..14 of the sum are (e - e0) mod 256, which is at least 7 whenever
// e < e0 because e0 <= 249.  Three logic/add operations and one packed 16-bit minimum.
__device__ __forceinline__ uint32_t codes7_x2(uint32_t w, uint32_t kadd) {
  return min_u16x2(((w & 0x7F807F80u) + kadd) & 0x7F807F80u, 0x03800380u);
}

// Sign|mantissa bytes of the four values in (w0, w1): (x >> 8 & 0x80) | (x & 0x7F).
__device__ __forceinline__ uint32_t sign_mantissa_x4(uint32_t w0, uint32_t w1) {
  const uint32_t lo = prmt(w0, w1, 0x6420);  // low byte of each value
  const uint32_t hi = prmt(w0, w1, 0x7531);  // high byte of each value
  return (hi & 0x80808080u) | (lo & 0x7F7F7F7Fu);
}

// 24-bit little-endian bitstream of the 8 codes in four words of codes7_x2: code j at bits
// [3j, 3j+3).  In t = w0 + (w1 << 6) the codes of values 0, 2 sit at bits 7, 13 and those of
// values 1, 3 at bits 23, 29, so two shifts and a masked merge put all four in place.
__device__ __forceinline__ uint32_t pack_codes8(const uint32_t (&c7)[4]) {
  const uint32_t t01 = c7[0] + (c7[1] << 6), t23 = c7[2] + (c7[3] << 6);
  const uint32_t g01 = ((t01 >> 7) & 0x1C7u) | (t01 >> 20);
  const uint32_t g23 = ((t23 >> 7) & 0x1C7u) | (t23 >> 20);
  return g01 + (g23 << 12);
}

constexpr int kChunkThreads = 128;  // threads of a decode CTA, one chunk each

// ------------------------------------------------------------------ launchers (host side)

struct DeviceInfo {
  int sm_count;
  int* status;        // device address of the library's status word on this device
  int stats_per_sm;   // resident CTAs per SM of the statistics and encode kernels, found once
  int encode_per_sm;  // per device (host-side launch work stays small for small tensors)
  int small_ctas;     // the small-tensor kernel's largest cluster on this device (16, else 8)
  int medium_ctas;    // CTAs of the medium-tensor kernel's cooperative grid (0: none)
  int fused_ctas;     // CTAs of the L2-resident kernel's cooperative grid (0: none)
};

cudaError_t device_info(DeviceInfo* info);  // defined in zc_api.cu
cudaError_t stats_occupancy(int* per_sm);   // defined in zc_stats.cu
cudaError_t encode_occupancy(int* per_sm);  // defined in zc_encode.cu; also sets the kernel's
                                            // dynamic shared memory size, for the current device

// CUDA events around one library kernel on its stream; inert unless timing is enabled.  The
// open record lives with the caller, so concurrent host threads never pair each other's events.
struct TimingRecord {
  int kernel = 0;
  cudaEvent_t start = nullptr, stop = nullptr;
};
TimingRecord timing_begin(int kernel_id, cudaStream_t stream);
void timing_end(TimingRecord& rec, cudaStream_t stream);

// The speculative encode kernel samples one 16-byte vector from each of 512 full chunks spread
// over the tensor: it runs only on tensors with at least that many full chunks.
constexpr uint64_t kSpecSampleChunks = 512;
// The launches.  `ws` is the call's workspace (workspace_bytes(n) bytes, cleared): the tail of
// `out` for zc_compress, the library's static array for zc_compress_static_scratch.
// predict_raw: also sample the exponents and, when the sample predicts that the coded stream
// will be longer than the raw form, have the encode kernel take the raw pass first.
// gated: after the speculative encode kernel (below), run only when it fell back.
cudaError_t launch_stats(const uint16_t* in, uint64_t n, uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream,
                         bool predict_raw, bool gated = false);
// mode: 0 plain, 1 speculative unless the sample was not confident, 2 only when the speculation
// fell back (the encode kernel's kPlain, kSpeculative, kGated).
cudaError_t launch_encode(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                          uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream, uint64_t stall_chunk,
                          unsigned spin_limit, uint16_t* loopback_values = nullptr, int mode = 0);
// The speculative path (auto mode, tensors above the single-launch sizes): the encode kernel
// guesses e0 from a sample (every CTA the same guess), codes with it and checks it against the
// whole tensor's sum of squares, which it takes as it codes; when the sample was not confident or
// the guess did not hold, the statistics and encode kernels after it, gated on the fallback
// word, do the job as they do without the speculation.  loopback_values: the loopback's decoded
// values (both encode launches decode what they code), or null.
cudaError_t launch_speculative(const uint16_t* in, uint64_t n, uint8_t* out, unsigned long long* out_bytes,
                               uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream,
                               uint16_t* loopback_values = nullptr);
cudaError_t launch_decode(const uint8_t* in, uint16_t* out, uint64_t n, const DeviceInfo& dev,
                          cudaStream_t stream);
// After the encode kernel: when the coded stream came out longer than the raw form, rewrite the
// stream in the raw form (header, the n values, zero padding); otherwise return at once.
cudaError_t launch_raw_form(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                            uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream);

// Small and medium tensors: the whole compression in one launch with every CTA resident, up to
// four chunks per CTA -- one thread-block cluster up to small_max_values(dev) (262,144 values, or
// 131,072 where 16-CTA clusters cannot be scheduled), one cooperative grid up to
// medium_max_values(dev).  The small path uses no workspace beyond the control block's e0,
// exact-path flag and length; the medium path needs only its control block cleared (its
// barriers' counter): its other workspace slots are each written before they are read.
cudaError_t small_setup(int* small_ctas, int* medium_ctas);  // per device
uint64_t small_max_values(const DeviceInfo& dev);
uint64_t medium_max_values(const DeviceInfo& dev);
cudaError_t launch_medium(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                          uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_small(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                         uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream);

// Tensors above the medium size that the L2 nearly holds: one cooperative launch that reads the
// input three times (statistics from HBM; an exact escape count per chunk and the coding, mostly
// from the L2) and writes every part of the stream straight to its place.  Needs the control block
// cleared; its other workspace slots are each written before they are read.
cudaError_t fused_setup(int* fused_ctas);  // per device
uint64_t fused_max_values(const DeviceInfo& dev);
cudaError_t launch_fused(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                         uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream);

// Whether a tensor of n values (n > 0) compresses in one launch, and that launch (the small,
// medium or L2-resident kernel, with the control block cleared for the grid kernels).
bool single_launch(uint64_t n, const DeviceInfo& dev);
cudaError_t launch_one(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                       uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream);

// After the launches of a compression: when the caller's length is pageable host memory, copy
// it back from the control block and synchronize the stream.  Returns a ZC_ status.
int finish_length(bool pageable, uint8_t* ws, size_t* out_bytes, cudaStream_t stream);

constexpr unsigned kDefaultSpinLimit = 1u << 20;  // polls of a bounded wait in the encoder

}  // namespace zc
