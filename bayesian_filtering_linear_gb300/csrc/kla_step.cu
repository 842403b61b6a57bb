// One recurrent decode step of the KLA filter (sm_103a), in information form
// on the persisted state, for every element of every head:
//
//   r    = 1 / (a² + p̄ λ)                 (OU predict: λ_pred = λ r)
//   λ'   = λ r + c                        c = k² Λ^v   (observation precision)
//   η'   = (a r) η + b                    b = k Λ^v v  (forget gate a λ_pred/λ = a r)
//   y_j  = Σ_i q_i η'_ij / λ'_ij
//
// This is the Möbius step λ' = (αλ + β)/(γλ + δ) with α = 1 + c p̄, β = c a²,
// γ = p̄, δ = a², and the affine information-mean step, of
// "Technische Samenvatting: Kalman Linear Attention (KLA)"
// (gist.science/nl/paper/2602.10743), Methodologie §2. As in the sequence
// kernel, a is floored at 2^-40 and k² is raised by 2^-40.
//
// Work layout: one thread block per head; a thread owns 4 consecutive columns
// (one 16-byte load of λ and of η per row) of 4 rows. The step is bound by
// HBM traffic of the state (16 bytes per element: read and write λ, η).
#include "kla_device.cuh"
#include "kla_launch.h"

namespace kla {

namespace {

constexpr int kRowsPerThread = 4;

template <typename IO, bool GATED>
__global__ void __launch_bounds__(1024) kla_step_kernel(const StepArgs a) {
  extern __shared__ __align__(16) float ysm[];  // [row groups][dv] partial sums
  const int dk = a.dk, dv = a.dv;
  const int col_groups = dv / 4;
  const int tid = threadIdx.x;
  const int cg = tid % col_groups, rg = tid / col_groups;
  const long long bh = blockIdx.x;
  const int j0 = cg * 4, r0 = rg * kRowsPerThread;

  const IO* qv = reinterpret_cast<const IO*>(a.q) + bh * dk;
  const IO* kv = reinterpret_cast<const IO*>(a.k) + bh * dk;
  const IO* av = reinterpret_cast<const IO*>(a.a) + bh * dk;
  const IO* pv = reinterpret_cast<const IO*>(a.pbar) + bh * dk;
  const IO* vv = reinterpret_cast<const IO*>(a.v) + bh * dv;
  const IO* lv = reinterpret_cast<const IO*>(a.lam_v) + bh * dv;

  float Lc[4], Bv[4], y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    Lc[c] = GATED ? gate_lamv(to_f32<IO>(lv[j0 + c]), a.gates) : to_f32<IO>(lv[j0 + c]);
    Bv[c] = Lc[c] * to_f32<IO>(vv[j0 + c]);
  }
  float* lam = a.lam + (size_t)bh * dk * dv;
  float* eta = a.eta + (size_t)bh * dk * dv;
#pragma unroll
  for (int rr = 0; rr < kRowsPerThread; ++rr) {
    const int i = r0 + rr;
    const float ki = to_f32<IO>(kv[i]);
    const float xa = to_f32<IO>(av[i]);
    const float ai = fmaxf(GATED ? gate_a(xa, a.gates) : xa, kAMin);
    const float pi = GATED ? gate_pbar(to_f32<IO>(pv[i]), xa, a.gates) : to_f32<IO>(pv[i]);
    const float qi = to_f32<IO>(qv[i]);
    const float K = fmaf(ki, ki, kK2Floor);
    const float a2 = ai * ai;
    float4 l4 = *reinterpret_cast<const float4*>(lam + (size_t)i * dv + j0);
    float4 e4 = *reinterpret_cast<const float4*>(eta + (size_t)i * dv + j0);
    float* lp = &l4.x;
    float* ep = &e4.x;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float r = rcp_approx(fmaf(pi, lp[c], a2));
      const float ln = fmaf(lp[c], r, K * Lc[c]);
      const float en = fmaf(ai * r, ep[c], ki * Bv[c]);
      y[c] = fmaf(qi, en * rcp_approx(ln), y[c]);
      lp[c] = ln;
      ep[c] = en;
    }
    *reinterpret_cast<float4*>(lam + (size_t)i * dv + j0) = l4;
    *reinterpret_cast<float4*>(eta + (size_t)i * dv + j0) = e4;
  }
  *reinterpret_cast<float4*>(ysm + rg * dv + j0) = make_float4(y[0], y[1], y[2], y[3]);
  __syncthreads();
  const int row_groups = dk / kRowsPerThread;
  IO* yo = reinterpret_cast<IO*>(a.y) + bh * dv;
  for (int j = tid; j < dv; j += blockDim.x) {
    float s = 0.f;
    for (int g = 0; g < row_groups; ++g) s += ysm[g * dv + j];
    yo[j] = from_f32<IO>(s);
  }
}

}  // namespace

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
  const long long heads = (long long)a.B * a.H;
  if (heads == 0) return cudaSuccess;
  const int threads = (a.dv / 4) * (a.dk / kRowsPerThread);
  const size_t smem = (size_t)(a.dk / kRowsPerThread) * a.dv * sizeof(float);
  // gate activations are a separate instantiation (no extra work without them)
  if (a.io == IO_BF16) {
    if (a.gates) kla_step_kernel<__nv_bfloat16, true><<<(unsigned)heads, threads, smem, s>>>(a);
    else kla_step_kernel<__nv_bfloat16, false><<<(unsigned)heads, threads, smem, s>>>(a);
  } else {
    if (a.gates) kla_step_kernel<float, true><<<(unsigned)heads, threads, smem, s>>>(a);
    else kla_step_kernel<float, false><<<(unsigned)heads, threads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kla
