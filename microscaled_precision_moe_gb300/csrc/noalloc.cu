// Allocation-free variant of the NVFP4 joint-weight quantiser.
//
// mpm_nvfp4_quantize_weight needs a small device workspace (one 32-bit amax
// per expert) that its caller allocates.  Some callers cannot allocate device
// memory at the point where they quantise weights: for example code whose
// device memory is owned entirely by a pooling allocator it cannot reach from
// there, or a latency-critical loop where a cudaMalloc, which may synchronise
// the device, is not allowed.  This entry point takes the same inputs and
// outputs but keeps that workspace in a fixed array in device memory that the
// library itself declares, so nothing is allocated per call.
#include "quant.cuh"

#include <mutex>

namespace {

// Maximum number of experts one call may quantise: the scratch holds one
// 32-bit amax per expert (16 KiB).  Every GPU that loads the library holds
// this array until the process exits.
constexpr long long kNoAllocMaxExperts = 4096;

static __device__ __align__(256) unsigned g_weight_amax_scratch[kNoAllocMaxExperts];

constexpr int kMaxDevices = 64;

// Device address of the scratch array for the current device.  In host code
// the array's name only stands in for the device symbol, so the address must
// be looked up on each device (with that device current) before a kernel can
// use it.  A call made outside stream capture looks it up again every time,
// so a device reset or a new context on the device (which reloads the module
// at another address) is picked up; a call made while `stream` is capturing
// uses the address the last uncaptured call on that device found (the first
// call on a device must therefore come before any capture).
unsigned* scratch_on_current_device(cudaStream_t stream, cudaError_t* err) {
  static unsigned* ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  *err = cudaStreamIsCapturing(stream, &cap);
  if (*err != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_weight_amax_scratch);
    if (*err != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned*>(p);
  } else if (!ptrs[dev]) {
    *err = cudaErrorStreamCaptureUnsupported;
    return nullptr;
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

}  // namespace

extern "C" mpm_status mpm_nvfp4_quantize_weight_noalloc(const void* const* parts,
                                                        const int64_t* part_rows, int nparts,
                                                        int64_t K, int64_t E, uint8_t* q,
                                                        uint8_t* s, float* ts,
                                                        cudaStream_t stream) {
  if (!parts || !part_rows || !q || !s || !ts) return MPM_ERR_NULL;
  if (nparts < 1 || nparts > 4 || E < 1 || K < 64 || K % 64 != 0 || K > 8192) return MPM_ERR_SHAPE;
  if (E > kNoAllocMaxExperts) return MPM_ERR_SHAPE;   // beyond the fixed scratch
  long long R = 0;
  long long rows[4];
  for (int i = 0; i < nparts; ++i) {
    if (!parts[i]) return MPM_ERR_NULL;
    if (part_rows[i] < 1) return MPM_ERR_SHAPE;
    if (!aligned16(parts[i])) return MPM_ERR_ALIGN;
    rows[i] = part_rows[i];
    R += part_rows[i];
  }
  if (R % 128 != 0 || E * R > (1ll << 31) - 256) return MPM_ERR_SHAPE;
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(ts) % 4) != 0) return MPM_ERR_ALIGN;
  cudaError_t err = cudaSuccess;
  unsigned* scratch = scratch_on_current_device(stream, &err);
  if (!scratch) return MPM_ERR_CUDA;
  // The launcher clears the E amax slots it uses (an async memset on
  // `stream`) before the reduction, so the previous call's contents do not
  // leak into this one.
  err = mpm::launch_nvfp4_weight(parts, rows, nparts, (int)K, E, q, s, ts, scratch, stream);
  return err == cudaSuccess ? MPM_OK : MPM_ERR_CUDA;
}
