// zc_api.cu -- the C ABI: argument checks, workspace set-up, launches, status and timing.
//
// Call sequence of zc_compress (ZipCCL SIGCOMM scribe notes, "Key idea and contribution":
// window from the standard deviation, 3-bit codes, separate full exponents):
//   1. clear the workspace in the tail of `out` (one memset on `stream`);
//   2. statistics kernel (auto mode only): sum of squares, non-finite count, e0;
//   3. encode kernel: codes, sign|mantissa plane, escape sections, the single-pass chunk scan,
//      the offset table and the lists compacted behind it;
//   4. raw-form step (third technique: the native path where compressing does not pay): when
//      the coded stream came out longer than the header plus the values, the stream is
//      rewritten in that raw form; otherwise the kernel returns at once.
// zc_decompress is one decode kernel.  No call synchronizes except zc_status, and
// zc_compress when `out_bytes` is pageable host memory.
#include <cstring>
#include <mutex>
#include <vector>

#include "zc_common.cuh"

namespace zc {
namespace {

__device__ int g_status;  // first device-side error since the last reset, per device

constexpr int kMaxDevices = 64;

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
bool g_device_ready[kMaxDevices];

bool g_timing = false;
std::vector<TimingRecord> g_records;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

}  // namespace

cudaError_t device_info(DeviceInfo* info) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_device_ready[dev]) {
    DeviceInfo d{};
    err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status);
    if (err != cudaSuccess) return err;
    err = stats_occupancy(&d.stats_per_sm);
    if (err != cudaSuccess) return err;
    err = encode_occupancy(&d.encode_per_sm);
    if (err != cudaSuccess) return err;
    err = small_setup(&d.small_ctas, &d.medium_ctas);
    if (err != cudaSuccess) return err;
    err = fused_setup(&d.fused_ctas);
    if (err != cudaSuccess) return err;
    g_devices[dev] = d;
    g_device_ready[dev] = true;
  }
  *info = g_devices[dev];
  return cudaSuccess;
}

TimingRecord timing_begin(int kernel_id, cudaStream_t stream) {
  TimingRecord rec;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_timing) return rec;
  rec.kernel = kernel_id;
  rec.start = take_event();
  rec.stop = take_event();
  if (rec.start && rec.stop) {
    cudaEventRecord(rec.start, stream);
  } else {  // no events: record nothing for this kernel
    if (rec.start) g_event_pool.push_back(rec.start);
    if (rec.stop) g_event_pool.push_back(rec.stop);
    rec.start = rec.stop = nullptr;
  }
  return rec;
}

void timing_end(TimingRecord& rec, cudaStream_t stream) {
  if (rec.start == nullptr) return;
  std::lock_guard<std::mutex> lock(g_mutex);
  cudaEventRecord(rec.stop, stream);
  g_records.push_back(rec);
  rec.start = rec.stop = nullptr;
}

}  // namespace zc

using namespace zc;

namespace {

// The workspace's place in `out`: after the longest stream the call may write (the loopback
// writes every escape section of the coded form before the form is chosen).
uint64_t workspace_at(uint64_t n, bool loopback) {
  return loopback ? (max_coded_bytes(n) + 255) & ~uint64_t(255) : workspace_offset(n);
}

}  // namespace

namespace zc {

// A pageable length: copy it back from the control block and wait for it.
bool single_launch(uint64_t n, const DeviceInfo& dev) {
  return n <= medium_max_values(dev) || n <= fused_max_values(dev);
}

cudaError_t launch_one(const uint16_t* in, uint64_t n, int base, uint8_t* out, unsigned long long* out_bytes,
                       uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream) {
  if (n <= small_max_values(dev)) return launch_small(in, n, base, out, out_bytes, ws, dev, stream);
  // the grid kernels' barrier counter is in the control block: cleared first
  const cudaError_t err = cudaMemsetAsync(ws, 0, kWsControlBytes, stream);
  if (err != cudaSuccess) return err;
  if (n <= medium_max_values(dev)) return launch_medium(in, n, base, out, out_bytes, ws, dev, stream);
  return launch_fused(in, n, base, out, out_bytes, ws, dev, stream);
}

int finish_length(bool pageable, uint8_t* ws, size_t* out_bytes, cudaStream_t stream) {
  if (!pageable) return ZC_OK;
  unsigned long long total = 0;
  const Control* ctrl = reinterpret_cast<const Control*>(ws);
  if (cudaMemcpyAsync(&total, &ctrl->total, sizeof total, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return ZC_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ZC_ERR_CUDA;
  *out_bytes = static_cast<size_t>(total);
  return ZC_OK;
}

}  // namespace zc

namespace {

int compress_impl(const void* in, size_t n, int base, void* out, size_t* out_bytes, cudaStream_t stream,
                  uint64_t stall_chunk, unsigned spin_limit, void* values = nullptr) {
  if (n > ZC_MAX_N || base < ZC_BASE_AUTO || base > kE0Max) return ZC_ERR_INVALID_ARG;
  if (out == nullptr || out_bytes == nullptr || (n > 0 && in == nullptr)) return ZC_ERR_INVALID_ARG;
  if (!aligned(in, 16) || !aligned(out, 16) || !aligned(out_bytes, 8)) return ZC_ERR_MISALIGNED;
  const bool loopback = values != nullptr;
  if (loopback && !aligned(values, 16)) return ZC_ERR_MISALIGNED;
  const size_t cap = loopback ? zc_loopback_bytes(n) : zc_max_compressed_bytes(n);
  if (overlap(in, 2 * n, out, cap)) return ZC_ERR_INVALID_ARG;
  if (loopback && (overlap(values, 2 * n, out, cap) || overlap(values, 2 * n, in, 2 * n))) return ZC_ERR_INVALID_ARG;

  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;

  // Where the kernel writes the length: any device-visible address, else the control block.
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, out_bytes) != cudaSuccess) {
    cudaGetLastError();
    return ZC_ERR_CUDA;
  }
  unsigned long long* len_ptr = nullptr;
  const bool pageable = attr.type == cudaMemoryTypeUnregistered || attr.devicePointer == nullptr;
  if (!pageable) len_ptr = static_cast<unsigned long long*>(attr.devicePointer);

  uint8_t* o = static_cast<uint8_t*>(out);
  uint8_t* ws = o + workspace_at(n, loopback);
  const uint16_t* x = static_cast<const uint16_t*>(in);
  if (n > 0 && !loopback && stall_chunk == ~uint64_t(0) && single_launch(n, dev)) {
    if (launch_one(x, n, base, o, len_ptr, ws, dev, stream) != cudaSuccess) return ZC_ERR_CUDA;
    return finish_length(pageable, ws, out_bytes, stream);
  }
  if (cudaMemsetAsync(ws, 0, workspace_bytes(n), stream) != cudaSuccess) return ZC_ERR_CUDA;
  if (base == ZC_BASE_AUTO && stall_chunk == ~uint64_t(0) && n / kChunk >= kSpecSampleChunks) {
    // auto mode: code with the e0 of a sample and check it (the statistics pass runs only when
    // the check fails or the sample is not confident); the loopback decodes on either pass
    if (launch_speculative(x, n, o, len_ptr, ws, dev, stream, static_cast<uint16_t*>(values)) != cudaSuccess)
      return ZC_ERR_CUDA;
    return finish_length(pageable, ws, out_bytes, stream);
  }
  if (n > 0 && base == ZC_BASE_AUTO) {
    // The loopback decodes the coded form and the stall test needs the encoder: neither takes
    // the raw pass.
    const bool predict_raw = !loopback && stall_chunk == ~uint64_t(0);
    if (launch_stats(x, n, ws, dev, stream, predict_raw) != cudaSuccess) return ZC_ERR_CUDA;
  }
  if (launch_encode(x, n, base, o, len_ptr, ws, dev, stream, stall_chunk, spin_limit,
                    static_cast<uint16_t*>(values)) != cudaSuccess)
    return ZC_ERR_CUDA;
  if (launch_raw_form(x, n, base, o, len_ptr, ws, dev, stream) != cudaSuccess) return ZC_ERR_CUDA;
  return finish_length(pageable, ws, out_bytes, stream);
}

}  // namespace

extern "C" {

size_t zc_max_stream_bytes(size_t n) {
  if (n > ZC_MAX_N) return 0;
  return static_cast<size_t>(max_stream_bytes(n));
}

size_t zc_max_compressed_bytes(size_t n) {
  if (n > ZC_MAX_N) return 0;
  return static_cast<size_t>(workspace_offset(n) + workspace_bytes(n));
}

int zc_compress(const void* in, size_t n, int base_or_auto, void* out, size_t* out_bytes, cudaStream_t stream) {
  return compress_impl(in, n, base_or_auto, out, out_bytes, stream, ~uint64_t(0), kDefaultSpinLimit);
}

int zc_compress_stall_test(const void* in, size_t n, int base_or_auto, void* out, size_t* out_bytes,
                           cudaStream_t stream, size_t stalled_chunk, unsigned spin_limit) {
  return compress_impl(in, n, base_or_auto, out, out_bytes, stream, stalled_chunk, spin_limit);
}

size_t zc_loopback_bytes(size_t n) {
  if (n > ZC_MAX_N) return 0;
  return static_cast<size_t>(workspace_at(n, true) + workspace_bytes(n));
}

int zc_loopback(const void* in, size_t n, int base_or_auto, void* out, size_t* out_bytes, void* values,
                cudaStream_t stream) {
  if (values == nullptr && n > 0) return ZC_ERR_INVALID_ARG;
  return compress_impl(in, n, base_or_auto, out, out_bytes, stream, ~uint64_t(0), kDefaultSpinLimit,
                       n > 0 ? values : nullptr);
}

int zc_loopback_stall_test(const void* in, size_t n, int base_or_auto, void* out, size_t* out_bytes, void* values,
                           cudaStream_t stream, size_t stalled_chunk, unsigned spin_limit) {
  if (values == nullptr || n == 0) return ZC_ERR_INVALID_ARG;
  return compress_impl(in, n, base_or_auto, out, out_bytes, stream, stalled_chunk, spin_limit, values);
}

int zc_decompress(const void* in, void* out, size_t n, cudaStream_t stream) {
  if (n > ZC_MAX_N || in == nullptr || (n > 0 && out == nullptr)) return ZC_ERR_INVALID_ARG;
  if (!aligned(in, 16) || !aligned(out, 16)) return ZC_ERR_MISALIGNED;
  if (overlap(in, kHeaderBytes, out, 2 * n)) return ZC_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  if (launch_decode(static_cast<const uint8_t*>(in), static_cast<uint16_t*>(out), n, dev, stream) != cudaSuccess)
    return ZC_ERR_CUDA;
  return ZC_OK;
}

int zc_status(cudaStream_t stream, int reset) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ZC_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) return ZC_ERR_CUDA;
  if (reset) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof zero) != cudaSuccess) return ZC_ERR_CUDA;
  }
  return v;
}

int zc_timing_enable(int enable) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_timing = enable != 0;
  return ZC_OK;
}

int zc_timing_collect(int* kernel_ids, float* ms, int max) {
  std::vector<TimingRecord> recs;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    recs.swap(g_records);
  }
  int written = 0;
  int result = 0;
  for (const TimingRecord& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
      result = -ZC_ERR_CUDA;
    if (written < max && kernel_ids && ms) {
      kernel_ids[written] = r.kernel;
      ms[written] = t;
      ++written;
    }
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  for (const TimingRecord& r : recs) {
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  return result < 0 ? result : written;
}

}  // extern "C"
