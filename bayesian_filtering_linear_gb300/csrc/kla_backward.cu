// Backward pass of the KLA scan: gradients of a scalar loss with respect to
// every input, given dL/dy and (optionally) dL/dλ_T, dL/dη_T.
//
// The forward is the per-element filter of "Technische Samenvatting: Kalman
// Linear Attention (KLA)", Methodologie §1–§2 (every state element (i, j) of
// a head is a scalar Kalman filter; y_t = Σ_i q_{t,i} μ_{t,i,j}). Written in
// variance form with
//     P⁻ = a²P + p̄,  c = k²Λ^v,  b = kΛ^v v,  w = 1/(1 + cP⁻),
//     P' = wP⁻,      u = aμ + P⁻b,  μ' = wu,
// its reverse-mode derivative carries the adjoints (P̄, μ̄) of one element
// backwards through the tokens:
//     μ̄ += q·dy_j                                   (readout)
//     ū = μ̄w,  w̄ = μ̄u + P̄P⁻
//     P̄⁻ = P̄w + ūb − w̄cw²,  c̄ = −w̄P⁻w²,  b̄ = ūP⁻
//     dq += dy_j μ',  da += ūμ + 2aP·P̄⁻,  dp̄ += P̄⁻,
//     dk += 2kΛ^v c̄ + Λ^v v b̄,  dΛ^v += k²c̄ + kv b̄,  dv += kΛ^v b̄
//     (P̄, μ̄) ← (a²P̄⁻, aū)
// starting from (P̄, μ̄) = (−(dλ_T + dη_T μ_T)/P_T², dη_T/P_T) and ending with
// dλ0 = −(P̄ + μ̄η0)/λ0², dη0 = μ̄/λ0 (P0 = 1/λ0, μ0 = η0/λ0).
//
// GPU plan (three kernels, all on the caller's stream):
//  1. kla_bwd_checkpoint_kernel runs the forward once and stores the state
//     (P, μ) of every element at the start of every chunk of kChunk tokens,
//     and at the end, into the workspace.
//  2. kla_bwd_kernel walks the chunks from last to first. For each chunk it
//     re-runs the forward from the checkpoint, keeping the state before each
//     token in thread-local memory (each thread reads back only what it
//     wrote), then runs the adjoint recursion backwards over the chunk.
//  3. kla_bwd_finish_kernel (only when a head's columns are split over
//     several blocks) adds the per-row partial sums of the blocks.
//
// Layout of a block: (head, column block of cc columns, all d_k rows). A lane
// owns one row and CPL consecutive columns, so every per-row sum (dq, dk, da,
// dp̄) is first a sum inside the lane; a warp covers RW = min(32, d_k) rows
// and 32/RW column groups; per-column sums (dv, dΛ^v) over the warp's rows
// are a butterfly reduce-scatter across its lanes. Sums across warps go
// through shared-memory atomics (their order is not fixed, so the last bits
// of those sums can differ from run to run).
#include <algorithm>

#include <cuda_runtime.h>

#include "kla_device.cuh"
#include "kla_launch.h"

namespace kla {
namespace {

constexpr int kChunk = 16;  // tokens per checkpoint interval and per staged tile

struct BwdParams {
  const void *q, *k, *v, *lam_v, *a, *pbar;
  const float *lam0, *eta0;
  const void* dy;
  const float *dlamT, *detaT;
  void *gq, *gk, *gv, *glam_v, *ga, *gpbar;  // per-token gradients (io dtype)
  float *dlam0, *deta0;
  float* ckpt;     // [nchunks + 1][2][elems]: (P, μ) at each chunk start, then at T
  float* rowpart;  // [ncb][4][B·H·T·d_k] per-row partial sums when ncb > 1, else null
  int T, dk, dv, cc, ncb, nchunks;
  long long elems;  // B·H·d_k·d_v
};

template <int DK, int CPL>
struct BwdGeo {
  static constexpr int RW = DK < 32 ? DK : 32;  // rows per warp
  static constexpr int CG = 32 / RW;            // column groups per warp
  static constexpr int WCOLS = CG * CPL;        // columns per warp
  static constexpr int NWR = DK / RW;           // warps along rows
  static constexpr int NV = 2 * CPL;            // per-column values a lane reduces per token
};

// Shared memory of one block (fp32): staged per-row inputs q, k, a, p̄
// [kChunk][DK] and per-column inputs v, Λ^v, dy [kChunk][cc], and the
// per-token accumulators of the row sums [kChunk][4][DK] and column sums
// [kChunk][2][cc].
struct BwdSmem {
  float *q, *k, *a, *p, *v, *L, *dy, *racc, *cacc;
  __device__ BwdSmem(float* base, int dk, int cc) {
    q = base;
    k = q + kChunk * dk;
    a = k + kChunk * dk;
    p = a + kChunk * dk;
    v = p + kChunk * dk;
    L = v + kChunk * cc;
    dy = L + kChunk * cc;
    racc = dy + kChunk * cc;
    cacc = racc + kChunk * 4 * dk;
  }
  __host__ __device__ static size_t bytes(int dk, int cc) {
    return sizeof(float) * ((size_t)kChunk * (4 * dk + 3 * cc) + (size_t)kChunk * 4 * dk + (size_t)kChunk * 2 * cc);
  }
};

template <typename IO>
__device__ __forceinline__ float ld(const void* base, size_t idx) {
  return to_f32<IO>(reinterpret_cast<const IO*>(base)[idx]);
}

// Stage tokens [t0, t0 + tl) of the block's inputs as fp32 (rows padded with
// zeros past tl are never read).
template <typename IO>
__device__ void stage_chunk(const BwdParams& p, const BwdSmem& s, long long bh, int jb, int t0, int tl,
                            bool with_dy) {
  const int nthr = blockDim.x;
  const size_t rbase = ((size_t)bh * p.T + t0) * p.dk;
  for (int x = threadIdx.x; x < tl * p.dk; x += nthr) {
    s.q[x] = ld<IO>(p.q, rbase + x);
    s.k[x] = ld<IO>(p.k, rbase + x);
    s.a[x] = ld<IO>(p.a, rbase + x);
    s.p[x] = ld<IO>(p.pbar, rbase + x);
  }
  for (int x = threadIdx.x; x < tl * p.cc; x += nthr) {
    const int t = x / p.cc, j = x - t * p.cc;
    const size_t g = ((size_t)bh * p.T + t0 + t) * p.dv + jb + j;
    s.v[x] = ld<IO>(p.v, g);
    s.L[x] = ld<IO>(p.lam_v, g);
    s.dy[x] = (with_dy && p.dy) ? ld<IO>(p.dy, g) : 0.0f;
  }
}

// One forward token for a lane's CPL elements of row i (staged token t).
template <int DK, int CPL>
__device__ __forceinline__ void forward_token(const BwdSmem& s, int cc, int t, int i, int jl, float (&P)[CPL],
                                              float (&M)[CPL]) {
  const float at = s.a[t * DK + i], pt = s.p[t * DK + i], kt = s.k[t * DK + i];
  const float a2 = at * at, k2 = kt * kt;
#pragma unroll
  for (int u4 = 0; u4 < CPL; u4 += 4) {
    const float4 L4 = *reinterpret_cast<const float4*>(s.L + t * cc + jl + u4);
    const float4 v4 = *reinterpret_cast<const float4*>(s.v + t * cc + jl + u4);
    const float Ls[4] = {L4.x, L4.y, L4.z, L4.w}, vs[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int u = u4 + x;
      const float Pp = fmaf(a2, P[u], pt);
      const float w = rcp_approx(fmaf(k2 * Ls[x], Pp, 1.0f));
      const float b = kt * (Ls[x] * vs[x]);
      const float uu = fmaf(Pp, b, at * M[u]);
      P[u] = w * Pp;
      M[u] = w * uu;
    }
  }
}

// Lane geometry shared by the two sequence kernels.
template <int DK, int CPL>
struct BwdLane {
  int lane, i, jl;
  size_t e0;  // element index of the lane's first (row i, column jb + jl)
  __device__ BwdLane(const BwdParams& p, long long bh, int jb) {
    using G = BwdGeo<DK, CPL>;
    lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int wr = warp % G::NWR, wc = warp / G::NWR;
    i = wr * G::RW + lane % G::RW;
    jl = wc * G::WCOLS + (lane / G::RW) * CPL;
    e0 = (size_t)bh * DK * p.dv + (size_t)i * p.dv + jb + jl;
  }
};

template <int CPL>
__device__ __forceinline__ void store_state(float* dst, size_t e0, long long elems, const float (&P)[CPL],
                                            const float (&M)[CPL]) {
#pragma unroll
  for (int u = 0; u < CPL; u += 4) {
    *reinterpret_cast<float4*>(dst + e0 + u) = make_float4(P[u], P[u + 1], P[u + 2], P[u + 3]);
    *reinterpret_cast<float4*>(dst + elems + e0 + u) = make_float4(M[u], M[u + 1], M[u + 2], M[u + 3]);
  }
}

template <int CPL>
__device__ __forceinline__ void load_state(const float* src, size_t e0, long long elems, float (&P)[CPL],
                                           float (&M)[CPL]) {
#pragma unroll
  for (int u = 0; u < CPL; u += 4) {
    const float4 p4 = *reinterpret_cast<const float4*>(src + e0 + u);
    const float4 m4 = *reinterpret_cast<const float4*>(src + elems + e0 + u);
    P[u] = p4.x; P[u + 1] = p4.y; P[u + 2] = p4.z; P[u + 3] = p4.w;
    M[u] = m4.x; M[u + 1] = m4.y; M[u + 2] = m4.z; M[u + 3] = m4.w;
  }
}

// Pass 1: the forward, storing (P, μ) at every chunk start and at the end.
template <typename IO, int DK, int CPL>
__global__ void __launch_bounds__(512) kla_bwd_checkpoint_kernel(const BwdParams p) {
  extern __shared__ __align__(16) float bwd_smem[];
  const BwdSmem s(bwd_smem, DK, p.cc);
  const long long bh = blockIdx.x;
  const int jb = blockIdx.y * p.cc;
  const BwdLane<DK, CPL> ln(p, bh, jb);
  float P[CPL], M[CPL];
#pragma unroll
  for (int u = 0; u < CPL; ++u) {
    if (p.lam0) {
      P[u] = 1.0f / p.lam0[ln.e0 + u];
      M[u] = p.eta0[ln.e0 + u] * P[u];
    } else {
      P[u] = 1.0f;
      M[u] = 0.0f;
    }
  }
  for (int c = 0; c < p.nchunks; ++c) {
    store_state<CPL>(p.ckpt + (size_t)c * 2 * p.elems, ln.e0, p.elems, P, M);
    const int t0 = c * kChunk, tl = min(kChunk, p.T - t0);
    __syncthreads();  // the previous chunk's staged inputs are no longer read
    stage_chunk<IO>(p, s, bh, jb, t0, tl, false);
    __syncthreads();
#pragma unroll 1
    for (int t = 0; t < tl; ++t) forward_token<DK, CPL>(s, p.cc, t, ln.i, ln.jl, P, M);
  }
  store_state<CPL>(p.ckpt + (size_t)p.nchunks * 2 * p.elems, ln.e0, p.elems, P, M);
}

// Butterfly reduce-scatter of NV per-lane values over the RW lanes of a
// column group (lanes differing in their low log2(RW) bits): afterwards lane
// holds, in v[0 .. NV/RW), the group sums of the values whose indices it
// returns through `first` (consecutive from there).
template <int RW, int NV>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int lane, int& first) {
  static_assert(NV >= RW, "each lane keeps at least one value");
  first = 0;
#pragma unroll
  for (int m = RW / 2, half = NV / 2; m >= 1; m >>= 1, half >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int u = 0; u < half; ++u) {
      const float send = upper ? v[u] : v[u + half];
      const float keep = upper ? v[u + half] : v[u];
      v[u] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
    if (upper) first += half;
  }
}

// Pass 2: chunks from last to first; recompute, then the adjoint recursion.
template <typename IO, int DK, int CPL>
__global__ void __launch_bounds__(512) kla_bwd_kernel(const BwdParams p) {
  using G = BwdGeo<DK, CPL>;
  extern __shared__ __align__(16) float bwd_smem[];
  const BwdSmem s(bwd_smem, DK, p.cc);
  const long long bh = blockIdx.x;
  const int jb = blockIdx.y * p.cc;
  const BwdLane<DK, CPL> ln(p, bh, jb);
  const int i = ln.i, jl = ln.jl;
  const size_t BHTdk = (size_t)gridDim.x * p.T * DK;

  // terminal adjoints from dλ_T, dη_T through λ_T = 1/P_T, η_T = μ_T/P_T
  float Pb[CPL], Mb[CPL];
  {
    float PT[CPL], MT[CPL];
    load_state<CPL>(p.ckpt + (size_t)p.nchunks * 2 * p.elems, ln.e0, p.elems, PT, MT);
#pragma unroll
    for (int u = 0; u < CPL; ++u) {
      const float dl = p.dlamT ? p.dlamT[ln.e0 + u] : 0.0f;
      const float de = p.detaT ? p.detaT[ln.e0 + u] : 0.0f;
      const float r = 1.0f / PT[u];
      Pb[u] = -(dl + de * MT[u]) * r * r;
      Mb[u] = de * r;
    }
  }
  float Ps[kChunk][CPL], Ms[kChunk][CPL];  // states before each token of the chunk (thread-local)
  for (int c = p.nchunks - 1; c >= 0; --c) {
    const int t0 = c * kChunk, tl = min(kChunk, p.T - t0);
    __syncthreads();  // the previous chunk's staged inputs and sums are no longer read
    stage_chunk<IO>(p, s, bh, jb, t0, tl, true);
    for (int x = threadIdx.x; x < kChunk * (4 * DK + 2 * p.cc); x += blockDim.x) s.racc[x] = 0.0f;
    __syncthreads();
    {  // recompute the chunk's states from its checkpoint
      float P[CPL], M[CPL];
      load_state<CPL>(p.ckpt + (size_t)c * 2 * p.elems, ln.e0, p.elems, P, M);
#pragma unroll 1
      for (int t = 0; t < tl; ++t) {
#pragma unroll
        for (int u = 0; u < CPL; ++u) {
          Ps[t][u] = P[u];
          Ms[t][u] = M[u];
        }
        forward_token<DK, CPL>(s, p.cc, t, i, jl, P, M);
      }
    }
#pragma unroll 1
    for (int t = tl - 1; t >= 0; --t) {
      const float at = s.a[t * DK + i], pt = s.p[t * DK + i], kt = s.k[t * DK + i], qt = s.q[t * DK + i];
      const float a2 = at * at, k2 = kt * kt;
      float rq = 0.f, rda1 = 0.f, rda2 = 0.f, rdp = 0.f, rdk1 = 0.f, rdk2 = 0.f;
      float cv[G::NV];  // per column: k²c̄ + kv·b̄ (dΛ^v), then k·b̄ (dv / Λ^v)
#pragma unroll
      for (int u4 = 0; u4 < CPL; u4 += 4) {
        const float4 L4 = *reinterpret_cast<const float4*>(s.L + t * p.cc + jl + u4);
        const float4 v4 = *reinterpret_cast<const float4*>(s.v + t * p.cc + jl + u4);
        const float4 g4 = *reinterpret_cast<const float4*>(s.dy + t * p.cc + jl + u4);
        const float Ls[4] = {L4.x, L4.y, L4.z, L4.w}, vs[4] = {v4.x, v4.y, v4.z, v4.w};
        const float gs[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int u = u4 + x;
          const float P = Ps[t][u], M = Ms[t][u];
          const float Pp = fmaf(a2, P, pt);
          const float cobs = k2 * Ls[x];
          const float w = rcp_approx(fmaf(cobs, Pp, 1.0f));
          const float Lv = Ls[x] * vs[x];
          const float b = kt * Lv;
          const float uu = fmaf(Pp, b, at * M);
          const float mu_t = w * uu;
          const float mb = fmaf(qt, gs[x], Mb[u]);
          rq = fmaf(gs[x], mu_t, rq);
          const float ub = mb * w;
          const float wb = fmaf(mb, uu, Pb[u] * Pp);
          const float w2 = w * w;
          const float Ppb = fmaf(Pb[u], w, fmaf(ub, b, -wb * cobs * w2));
          const float cb = -wb * Pp * w2;
          const float bb = ub * Pp;
          rda1 = fmaf(ub, M, rda1);
          rda2 = fmaf(P, Ppb, rda2);
          rdp += Ppb;
          rdk1 = fmaf(Ls[x], cb, rdk1);
          rdk2 = fmaf(Lv, bb, rdk2);
          cv[u] = fmaf(kt * vs[x], bb, k2 * cb);
          cv[CPL + u] = kt * bb;
          Pb[u] = a2 * Ppb;
          Mb[u] = at * ub;
        }
      }
      float* racc = s.racc + t * 4 * DK + i;
      atomicAdd(racc + 0 * DK, rq);
      atomicAdd(racc + 1 * DK, fmaf(2.0f * kt, rdk1, rdk2));
      atomicAdd(racc + 2 * DK, fmaf(2.0f * at, rda2, rda1));
      atomicAdd(racc + 3 * DK, rdp);
      int first;
      reduce_scatter<G::RW, G::NV>(cv, ln.lane, first);
#pragma unroll
      for (int r = 0; r < G::NV / G::RW; ++r) {
        const int idx = first + r;
        const int kind = idx / CPL, col = jl + idx % CPL;
        atomicAdd(s.cacc + (t * 2 + kind) * p.cc + col, cv[r]);
      }
    }
    __syncthreads();
    // this chunk's gradients
    for (int x = threadIdx.x; x < tl * DK; x += blockDim.x) {
      const int t = x / DK, r = x - t * DK;
      const size_t g = ((size_t)bh * p.T + t0 + t) * DK + r;
      const float* acc = s.racc + t * 4 * DK + r;
      if (p.ncb == 1) {
        reinterpret_cast<IO*>(p.gq)[g] = from_f32<IO>(acc[0]);
        reinterpret_cast<IO*>(p.gk)[g] = from_f32<IO>(acc[DK]);
        reinterpret_cast<IO*>(p.ga)[g] = from_f32<IO>(acc[2 * DK]);
        reinterpret_cast<IO*>(p.gpbar)[g] = from_f32<IO>(acc[3 * DK]);
      } else {
        float* part = p.rowpart + (size_t)blockIdx.y * 4 * BHTdk + g;
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) part[kq * BHTdk] = acc[kq * DK];
      }
    }
    for (int x = threadIdx.x; x < tl * p.cc; x += blockDim.x) {
      const int t = x / p.cc, j = x - t * p.cc;
      const size_t g = ((size_t)bh * p.T + t0 + t) * p.dv + jb + j;
      reinterpret_cast<IO*>(p.glam_v)[g] = from_f32<IO>(s.cacc[(t * 2) * p.cc + j]);
      reinterpret_cast<IO*>(p.gv)[g] = from_f32<IO>(s.L[t * p.cc + j] * s.cacc[(t * 2 + 1) * p.cc + j]);
    }
  }
  // initial-state gradients through P0 = 1/λ0, μ0 = η0/λ0
  if (p.dlam0) {
#pragma unroll
    for (int u = 0; u < CPL; ++u) {
      const float l0 = p.lam0 ? p.lam0[ln.e0 + u] : 1.0f;
      const float n0 = p.eta0 ? p.eta0[ln.e0 + u] : 0.0f;
      const float r = 1.0f / l0;
      p.dlam0[ln.e0 + u] = -(Pb[u] + Mb[u] * n0) * r * r;
      p.deta0[ln.e0 + u] = Mb[u] * r;
    }
  }
}

// Pass 3 (ncb > 1): add the column blocks' per-row partial sums.
template <typename IO>
__global__ void kla_bwd_finish_kernel(const BwdParams p, size_t BHTdk) {
  for (size_t g = blockIdx.x * (size_t)blockDim.x + threadIdx.x; g < BHTdk; g += (size_t)gridDim.x * blockDim.x) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int cb = 0; cb < p.ncb; ++cb)
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) acc[kq] += p.rowpart[((size_t)cb * 4 + kq) * BHTdk + g];
    reinterpret_cast<IO*>(p.gq)[g] = from_f32<IO>(acc[0]);
    reinterpret_cast<IO*>(p.gk)[g] = from_f32<IO>(acc[1]);
    reinterpret_cast<IO*>(p.ga)[g] = from_f32<IO>(acc[2]);
    reinterpret_cast<IO*>(p.gpbar)[g] = from_f32<IO>(acc[3]);
  }
}

template <typename IO, int DK, int CPL>
cudaError_t launch_bwd_typed(const BwdParams& bp, dim3 grid, int threads, size_t smem, cudaStream_t s) {
  auto ck = kla_bwd_checkpoint_kernel<IO, DK, CPL>;
  auto bw = kla_bwd_kernel<IO, DK, CPL>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(bw, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  ck<<<grid, threads, smem, s>>>(bp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bw<<<grid, threads, smem, s>>>(bp);
  e = cudaGetLastError();
  if (e != cudaSuccess || bp.ncb == 1) return e;
  const size_t BHTdk = (size_t)grid.x * bp.T * DK;
  if (BHTdk == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)std::min<size_t>((BHTdk + 255) / 256, 4096);
  kla_bwd_finish_kernel<IO><<<blocks, 256, 0, s>>>(bp, BHTdk);
  return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_bwd_io(int dk, int cpl, const BwdParams& bp, dim3 grid, int threads, size_t smem,
                          cudaStream_t s) {
  switch (dk * 100 + cpl) {
    case 1608: return launch_bwd_typed<IO, 16, 8>(bp, grid, threads, smem, s);
    case 1616: return launch_bwd_typed<IO, 16, 16>(bp, grid, threads, smem, s);
    case 3216: return launch_bwd_typed<IO, 32, 16>(bp, grid, threads, smem, s);
    case 6416: return launch_bwd_typed<IO, 64, 16>(bp, grid, threads, smem, s);
    case 12816: return launch_bwd_typed<IO, 128, 16>(bp, grid, threads, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

BwdPlan backward_plan(long long bh, int T, int dk, int dv, int num_sms) {
  BwdPlan b{};
  b.cpl = (dk == 16 && dv == 16) ? 8 : 16;
  const int rw = dk < 32 ? dk : 32, wcols = (32 / rw) * b.cpl, nwr = dk / rw;
  int cc = dv;
  while (cc > wcols && (nwr * (cc / wcols) > 16 || BwdSmem::bytes(dk, cc) > 200 * 1024)) cc /= 2;
  // Few heads: narrower column blocks, so that there are blocks for every SM.
  while (cc > wcols && bh * (dv / cc) < num_sms) cc /= 2;
  b.cc = cc;
  b.threads = 32 * nwr * (cc / wcols);
  b.ncb = dv / cc;
  b.nchunks = (T + kChunk - 1) / kChunk;
  const long long elems = bh * dk * dv;
  b.ckpt_bytes = (size_t)(b.nchunks + 1) * 2 * (size_t)elems * sizeof(float);
  b.rowpart_bytes = b.ncb > 1 ? (size_t)b.ncb * 4 * (size_t)bh * T * dk * sizeof(float) : 0;
  b.smem = BwdSmem::bytes(dk, cc);
  return b;
}

cudaError_t launch_backward(const BackwardArgs& f, const BwdPlan& b, void* workspace, cudaStream_t s) {
  const long long bh = (long long)f.B * f.H;
  if (bh == 0) return cudaSuccess;
  BwdParams bp{};
  bp.q = f.q; bp.k = f.k; bp.v = f.v; bp.lam_v = f.lam_v; bp.a = f.a; bp.pbar = f.pbar;
  bp.lam0 = f.lam0; bp.eta0 = f.eta0;
  bp.dy = f.dy; bp.dlamT = f.dlamT; bp.detaT = f.detaT;
  bp.gq = f.dq; bp.gk = f.dk_; bp.gv = f.dv_; bp.glam_v = f.dlam_v; bp.ga = f.da; bp.gpbar = f.dpbar;
  bp.dlam0 = f.dlam0; bp.deta0 = f.deta0;
  bp.ckpt = reinterpret_cast<float*>(workspace);
  bp.rowpart = b.ncb > 1 ? reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + b.ckpt_bytes) : nullptr;
  bp.T = f.T; bp.dk = f.dk; bp.dv = f.dv; bp.cc = b.cc; bp.ncb = b.ncb; bp.nchunks = b.nchunks;
  bp.elems = bh * f.dk * f.dv;
  const dim3 grid((unsigned)bh, (unsigned)b.ncb);
  return f.io == IO_BF16 ? launch_bwd_io<__nv_bfloat16>(f.dk, b.cpl, bp, grid, b.threads, b.smem, s)
                         : launch_bwd_io<float>(f.dk, b.cpl, bp, grid, b.threads, b.smem, s);
}

}  // namespace kla
