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

#include <cuda.h>
#include <cuda_runtime.h>

#include "kla.h"
#include "kla_ctx_cache.h"

namespace {

constexpr size_t kScratchBytes = 32u << 20;  // 32 MiB

// Device-side scratch. In host code this name is only a stand-in for the
// symbol, not a device address: the address comes from cudaGetSymbolAddress,
// once per CUDA context (each context that loads the module has its own copy).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Driver calls that identify the current context, taken through the runtime's
// entry-point query so that the library does not link the driver library.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_mutex;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
kla::ContextAddressCache<64> g_cache;  // context ID -> scratch address

bool driver_entry_points() {
  if (g_ctx_current && g_ctx_id) return true;
  void* f1 = nullptr;
  void* f2 = nullptr;
  cudaDriverEntryPointQueryResult q1{}, q2{};
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
      cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
      q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
    return false;
  g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f1);
  g_ctx_id = reinterpret_cast<CtxGetIdFn>(f2);
  return true;
}

// The device address of the scratch array in the calling thread's current
// context: looked up with cudaGetSymbolAddress on the first call in each
// context (which, with no context current yet, also creates the device's
// primary context), then taken from the cache.
kla_status scratch_address(void** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!driver_entry_points()) return KLA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return KLA_ERR_CUDA;
  void* ptr = nullptr;
  if (!ctx) {  // nothing current yet: the lookup makes the primary context current
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return KLA_ERR_CUDA;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return KLA_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return KLA_ERR_CUDA;
  if (!ptr) ptr = g_cache.find(id);
  if (!ptr) {
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return KLA_ERR_CUDA;
  }
  g_cache.insert(id, ptr);
  *out = ptr;
  return KLA_OK;
}

}  // namespace

extern "C" {

kla_status kla_forward_chunked_noalloc(const void* q, const void* k, const void* v, const void* lam_v,
                                       const void* a, const void* pbar, const float* lam0, const float* eta0,
                                       void* y, float* lamT, float* etaT, int B, int H, int T, int dk, int dv,
                                       kla_dtype io, int chunk_len, void* stream) {
  // no coefficient pass: a short sequence falls back to the sequential plan,
  // which must then need no workspace either
  const kla_options opt{KLA_CHUNKED, chunk_len, 0, 0, KLA_COEF_OFF};
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
