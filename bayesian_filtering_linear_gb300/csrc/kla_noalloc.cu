// kla_forward_chunked_noalloc: the chunk-parallel forward scan for callers
// that cannot allocate device memory.
//
// Who needs this: code that runs where a cudaMalloc is not allowed or not
// wanted — inside a custom allocator or memory-pool callback, in a real-time
// loop that must never take the driver's allocation lock, or under a host
// framework that owns every device allocation and hands kernels only their
// inputs and outputs. The chunk-parallel path needs scratch (per-chunk maps
// and chunk-start states); kla_forward takes it from the caller, this entry
// point takes it from a buffer the library owns.
//
// The scratch is a fixed array in device memory, sized kScratchBytes (32 MiB).
// It exists on every GPU that loads this library, for as long as the process
// runs. All calls on a device share it and it keeps the last call's contents;
// nothing in it needs to start at zero, because within one call every scratch
// value is written (chunk maps by the composition kernel, chunk starts by the
// carry kernel) before it is read. Two calls whose work overlaps on the GPU —
// on different streams, or from different host threads without ordering —
// race on the scratch and produce wrong results; issue them on one stream or
// order them.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "kla.h"

namespace {

constexpr size_t kScratchBytes = 32u << 20;  // 32 MiB

// Device-side scratch. In host code this name is only a stand-in for the
// symbol, not a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Look up (once per device, with that device current) the device address of
// the scratch array.
kla_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return KLA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return KLA_OK;
}

}  // namespace

extern "C" {

kla_status kla_forward_chunked_noalloc(const void* q, const void* k, const void* v, const void* lam_v,
                                       const void* a, const void* pbar, const float* lam0, const float* eta0,
                                       void* y, float* lamT, float* etaT, int B, int H, int T, int dk, int dv,
                                       kla_dtype io, int chunk_len, void* stream) {
  const kla_options opt{KLA_CHUNKED, chunk_len};
  // Shape and option checks first, without any CUDA call.
  kla_plan_info info{};
  kla_status st = kla_plan_for_sms(B, H, T, dk, dv, io, &opt, 1, &info);
  if (st != KLA_OK) return st;
  if ((long long)B * H == 0)
    return kla_forward(q, k, v, lam_v, a, pbar, lam0, eta0, y, lamT, etaT, B, H, T, dk, dv, io, nullptr, 0, &opt,
                       stream);
  if ((st = kla_plan(B, H, T, dk, dv, io, &opt, &info)) != KLA_OK) return st;
  if (info.workspace_bytes > kScratchBytes) return KLA_ERR_WORKSPACE;  // larger than the fixed scratch
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != KLA_OK) return st;
  return kla_forward(q, k, v, lam_v, a, pbar, lam0, eta0, y, lamT, etaT, B, H, T, dk, dv, io, scratch,
                     kScratchBytes, &opt, stream);
}

}  // extern "C"
