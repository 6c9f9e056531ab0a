// zc_static.cu -- zc_compress for callers that cannot allocate device memory.
//
// zc_compress keeps its per-call workspace (the scan state, 8 bytes per chunk, and a 16.25 KiB
// control block) in the tail of `out`, so its caller must provide zc_max_compressed_bytes(n)
// bytes there.  Some callers cannot: a communication layer whose send buffers are registered
// once, at exactly the worst-case stream size, and that may not call cudaMalloc on its progress
// path (cudaMalloc can synchronize the device and is not allowed while a stream is being
// captured).  zc_compress_static_scratch compresses into an `out` of zc_max_stream_bytes(n)
// bytes and takes its workspace from the file-scope array below instead, allocating nothing.
//
// The array is 2 MiB on every device that loads this library, for the life of the process.  All
// calls on a device share it, so two calls whose work overlaps on that GPU (different streams
// running at the same time) corrupt each other; calls in one stream, or otherwise ordered, are
// fine.  Each call clears the part of it that must start at zero.
#include <mutex>

#include "zc_common.cuh"

namespace zc {
namespace {

constexpr uint64_t kStaticScratchBytes = 2ull << 20;
static_assert(workspace_bytes(ZC_STATIC_SCRATCH_MAX_N) <= kStaticScratchBytes, "the limit fits the array");
static_assert(workspace_bytes(ZC_STATIC_SCRATCH_MAX_N + kChunk) > kStaticScratchBytes, "the limit is the largest");

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
unsigned char* g_scratch_ptr[kMaxDevices];  // device address of g_static_scratch, per device

// The array's device address on the current device.  In host code its name is only a host-side
// stand-in, so the address comes from the runtime, once per device, with that device current.
cudaError_t static_scratch(unsigned char** ptr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_static_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *ptr = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace zc

using namespace zc;

extern "C" int zc_compress_static_scratch(const void* in, size_t n, int base_or_auto, void* out, size_t* out_bytes,
                                          cudaStream_t stream) {
  if (n > ZC_STATIC_SCRATCH_MAX_N || base_or_auto < ZC_BASE_AUTO || base_or_auto > kE0Max) return ZC_ERR_INVALID_ARG;
  if (out == nullptr || out_bytes == nullptr || (n > 0 && in == nullptr)) return ZC_ERR_INVALID_ARG;
  if (!aligned_to(in, 16) || !aligned_to(out, 16) || !aligned_to(out_bytes, 8)) return ZC_ERR_MISALIGNED;
  const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
  const uint64_t cap = max_stream_bytes(n);
  if (n > 0 && a < b + cap && b < a + 2 * n) return ZC_ERR_INVALID_ARG;  // overlapping buffers

  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return ZC_ERR_CUDA;
  unsigned char* ws = nullptr;
  if (static_scratch(&ws) != cudaSuccess) return ZC_ERR_CUDA;

  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, out_bytes) != cudaSuccess) {
    cudaGetLastError();
    return ZC_ERR_CUDA;
  }
  const bool pageable = attr.type == cudaMemoryTypeUnregistered || attr.devicePointer == nullptr;
  unsigned long long* len_ptr = pageable ? nullptr : static_cast<unsigned long long*>(attr.devicePointer);

  const uint16_t* x = static_cast<const uint16_t*>(in);
  uint8_t* o = static_cast<uint8_t*>(out);
  if (n > 0 && single_launch(n, dev)) {
    if (launch_one(x, n, base_or_auto, o, len_ptr, ws, dev, stream) != cudaSuccess) return ZC_ERR_CUDA;
    return finish_length(pageable, ws, out_bytes, stream);
  }
  if (cudaMemsetAsync(ws, 0, workspace_bytes(n), stream) != cudaSuccess) return ZC_ERR_CUDA;
  if (base_or_auto == ZC_BASE_AUTO && n / kChunk >= kSpecSampleChunks) {  // as zc_compress: speculative
    if (launch_speculative(x, n, o, len_ptr, ws, dev, stream) != cudaSuccess) return ZC_ERR_CUDA;
    return finish_length(pageable, ws, out_bytes, stream);
  }
  if (n > 0 && base_or_auto == ZC_BASE_AUTO && launch_stats(x, n, ws, dev, stream, true) != cudaSuccess)
    return ZC_ERR_CUDA;
  if (launch_encode(x, n, base_or_auto, o, len_ptr, ws, dev, stream, ~uint64_t(0), kDefaultSpinLimit) != cudaSuccess)
    return ZC_ERR_CUDA;
  if (launch_raw_form(x, n, base_or_auto, o, len_ptr, ws, dev, stream) != cudaSuccess) return ZC_ERR_CUDA;
  return finish_length(pageable, ws, out_bytes, stream);
}
