// Pieces shared by the sequence kernels (scan and chunk composition): launch
// parameters, the lane geometry and the asynchronous staging of input tiles.
#pragma once

#include "kla_device.cuh"
#include "kla_launch.h"

namespace kla {

// Build-time geometry knobs (defaults are the measured best on GB300):
// columns per lane, scanning threads per block, rows per lane of the
// composition kernel at d_k = 64, and lane-exchange rounds of the readout
// (-1: one round per halving of the columns a lane holds).
#ifndef KLA_CL
#define KLA_CL 2
#endif
#ifndef KLA_MAXT
#define KLA_MAXT 256
#endif
#ifndef KLA_RL64
#define KLA_RL64 8
#endif
#ifndef KLA_XR
#define KLA_XR -1
#endif

constexpr int CL = KLA_CL;             // d_v columns per lane (2 or 4)
constexpr int kMaxThreads = KLA_MAXT;  // scanning threads per block (256 leaves up to 168 registers each)
constexpr int kProducerWarps = 4;      // scan: warps that stage tiles, build coefficients and store y

// Named barriers (ids 1..15; 0 is __syncthreads). bar.arrive counts this
// warp in without waiting; bar.sync counts it in and waits for `count`
// threads in total.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Rows per lane for a head size (compile-time twin of rows_per_lane_for()).
template <int DK>
struct RowsPerLane {
  static constexpr int value = DK <= 32 ? 4 : (DK == 64 ? KLA_RL64 : 8);
};

// A lane owns RL rows × CL columns of one head; rows are paired so that one
// packed fp32x2 instruction serves two rows. Rows vary slowest across lanes,
// so the eight lanes of a quarter-warp share rows and per-row coefficient
// loads from shared memory are broadcasts.
template <int DK, int RL>
struct Geo {
  static constexpr int LANES_I = DK / RL;       // lanes along rows
  static constexpr int LANES_J = 32 / LANES_I;  // lanes along columns
  static constexpr int WC = LANES_J * CL;       // columns per warp
  // Lane-exchange rounds of the readout reduction (each halves the partial
  // sums a lane holds) and the partial sums per output left for shared memory.
  static constexpr int XR = KLA_XR >= 0 ? KLA_XR : (CL == 4 ? 2 : 1);
  static constexpr int NP = LANES_I >> XR;
  static constexpr int VALS = CL >> XR;          // partial sums a lane stores per token
  static_assert(LANES_I >= (1 << XR) && LANES_I <= 32 && RL % 4 == 0 && (CL == 2 || CL == 4) && VALS >= 1,
                "unsupported geometry");
};

struct KernelParams {
  const void *q, *k, *v, *lam_v, *a, *pbar;
  const float *lam0, *eta0;
  const float* starts;  // [S][2][elems] chunk-start (P, μ), or nullptr
  float* maps;          // compose output [S-1][7][elems]
  void* y;              // nullptr: y is not stored (checkpoint pass of the backward)
  void* y_var;          // the variance readout when the scan computes both readouts
  float *lamT, *etaT;
  float* ckpt;          // scan MODE 3 only: [T/16 + 1][2][elems] scaled states (P̃, μ)
                        // at every 16-token tile start and at the end
  const float* coefs;   // scan MODE 4 only: per-row coefficients [B·H][T][5][d_k] of the
                        // coefficient pass (A, B, 1/a, k/K, q per token and row)
  int T, dv, chunk_len, cc, log2cc;
  int gates;        // kla_gate bits
  long long elems;  // B·H·dk·dv
};

// One staged tile of raw inputs: the four per-row arrays q, k, a, p̄
// ([TC][DK] each, contiguous in global memory) followed by the two per-column
// arrays v, Λ^v ([TC][cc], rows dv apart in global memory).
template <typename IO, int DK, int TC>
struct RawTile {
  __host__ __device__ static constexpr size_t row_bytes() { return (size_t)TC * DK * sizeof(IO); }
  __host__ __device__ static size_t col_bytes(int cc) { return (size_t)TC * cc * sizeof(IO); }
  __host__ __device__ static size_t bytes(int cc) { return 4 * row_bytes() + 2 * col_bytes(cc); }
};

// Queue 16-byte asynchronous copies of tokens [t0, t0 + tl) of this block's
// per-column inputs (v, Λ^v) into the raw tile at `dst`.
// (tid, nthr): this thread's index among the nthr threads sharing the work.
template <typename IO, int DK, int TC>
__device__ __forceinline__ void stage_cols(const KernelParams& p, unsigned char* dst, long long bh, int jb, int t0,
                                           int tl, int tid, int nthr) {
  using R = RawTile<IO, DK, TC>;
  // 16-byte chunks per staged row: cc·sizeof(IO)/16, a power of two (cc is)
  const int lcpr = p.log2cc + (sizeof(IO) == 4 ? 2 : 1) - 4;
  const int chunks_j = tl << lcpr;
  const size_t row_j = (size_t)p.dv * sizeof(IO);
  const size_t base_j = ((size_t)bh * p.T + t0) * row_j + (size_t)jb * sizeof(IO);
#pragma unroll
  for (int arr = 0; arr < 2; ++arr) {
    const char* src = (const char*)(arr == 0 ? p.v : p.lam_v) + base_j;
    unsigned char* d = dst + 4 * R::row_bytes() + arr * R::col_bytes(p.cc);
    for (int c = tid; c < chunks_j; c += nthr) {
      const int row = c >> lcpr, col = c & ((1 << lcpr) - 1);
      cp_async16(d + (size_t)c * 16, src + (size_t)row * row_j + (size_t)col * 16);
    }
  }
}

// The same for all of the tile's inputs: the per-row arrays q, k, a, p̄, then
// the per-column ones.
template <typename IO, int DK, int TC>
__device__ __forceinline__ void stage_raw(const KernelParams& p, unsigned char* dst, long long bh, int jb, int t0,
                                          int tl, int tid, int nthr) {
  using R = RawTile<IO, DK, TC>;
  const size_t row_i = (size_t)DK * sizeof(IO);
  const int chunks_i = (int)(tl * row_i / 16);
  const size_t base_i = ((size_t)bh * p.T + t0) * row_i;
#pragma unroll
  for (int arr = 0; arr < 4; ++arr) {
    const char* src = (const char*)(arr == 0 ? p.q : arr == 1 ? p.k : arr == 2 ? p.a : p.pbar) + base_i;
    unsigned char* d = dst + arr * R::row_bytes();
    for (int c = tid; c < chunks_i; c += nthr) cp_async16(d + (size_t)c * 16, src + (size_t)c * 16);
  }
  stage_cols<IO, DK, TC>(p, dst, bh, jb, t0, tl, tid, nthr);
}

// Four consecutive I/O values from shared memory, widened to fp32.
template <typename IO>
__device__ __forceinline__ float4 load4(const IO* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xffff0000u));
}

// Per-(t, j) column terms (Λ^v, Λ^v, Λ^v·v, Λ^v·v) of a staged tile, one
// (t, j) per thread so that consecutive threads store consecutive 16-byte
// entries (no bank conflicts); the duplicated pairs let one packed
// instruction serve two rows.
template <typename IO, int DK, int TC, bool GATED = true>
__device__ __forceinline__ void column_terms(const unsigned char* raw, float4* pj, int cc, int tl, int tid, int nthr,
                                             int gates) {
  using R = RawTile<IO, DK, TC>;
  const IO* rv = reinterpret_cast<const IO*>(raw + 4 * R::row_bytes());
  const IO* rL = reinterpret_cast<const IO*>(raw + 4 * R::row_bytes() + R::col_bytes(cc));
  for (int g = tid; g < tl * cc; g += nthr) {
    const float L = GATED ? gate_lamv(to_f32<IO>(rL[g]), gates) : to_f32<IO>(rL[g]);
    const float Lv = L * to_f32<IO>(rv[g]);
    pj[g] = make_float4(L, L, Lv, Lv);
  }
}

// ---- host helpers -------------------------------------------------------------
inline KernelParams make_params(const ForwardArgs& f, const Plan& p) {
  KernelParams kp{};
  kp.q = f.q; kp.k = f.k; kp.v = f.v; kp.lam_v = f.lam_v; kp.a = f.a; kp.pbar = f.pbar;
  kp.lam0 = f.lam0; kp.eta0 = f.eta0;
  kp.y = f.y; kp.y_var = f.y_var; kp.lamT = f.lamT; kp.etaT = f.etaT;
  kp.T = f.T; kp.dv = f.dv; kp.chunk_len = p.chunk_len; kp.cc = p.cols_per_block;
  int l2 = 0;
  while ((1 << l2) < p.cols_per_block) ++l2;
  kp.log2cc = l2;
  kp.elems = (long long)f.B * f.H * f.dk * f.dv;
  kp.gates = f.gates;
  return kp;
}

// Launch with the dynamic shared memory a kernel needs (opting in above 48 KB).
template <typename Kern>
inline cudaError_t launch_kernel(Kern fn, dim3 grid, int threads, size_t smem, cudaStream_t s,
                                 const KernelParams& kp) {
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  fn<<<grid, threads, smem, s>>>(kp);
  return cudaGetLastError();
}

}  // namespace kla
