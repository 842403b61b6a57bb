// Device-side helpers shared by the KLA kernels (sm_103a): packed fp32x2
// arithmetic, the hardware reciprocal, I/O dtype conversion and 16-byte
// asynchronous global→shared copies.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace kla {

// k² is raised by 2^-40 before it is used as a scale, and a is floored at
// 2^-40, so every scaled quantity in the forward recursion stays a normal
// fp32 number (see kla_scan_kernel.cuh). For |k| ≥ 2^-8 the raised k² rounds back
// to k² exactly; below that it adds 2^-40·Λ^v to the observation precision.
constexpr float kK2Floor = 0x1p-40f;
constexpr float kAMin = 0x1p-40f;

// ---- packed fp32x2 (one instruction issues two fp32 lanes) -------------------
typedef unsigned long long f2;

__device__ __forceinline__ f2 f2_make(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(f2 v) {
  float lo;
  asm("{\n\t.reg .f32 t;\n\tmov.b64 {%0, t}, %1;\n\t}" : "=f"(lo) : "l"(v));
  return lo;
}
__device__ __forceinline__ float f2_hi(f2 v) {
  float hi;
  asm("{\n\t.reg .f32 t;\n\tmov.b64 {t, %0}, %1;\n\t}" : "=f"(hi) : "l"(v));
  return hi;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Hardware approximate reciprocal (one MUFU op, ≤ 1 ulp off for normal input).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
#ifndef KLA_RCP_ASM
#define KLA_RCP_ASM 1
#endif
// Reciprocal of both halves of a pair, written so that the two results land
// in the halves of one 64-bit register without extra moves.
__device__ __forceinline__ f2 f2_rcp(f2 d) {
#if KLA_RCP_ASM
  f2 r;
  asm("{\n\t.reg .f32 lo, hi;\n\tmov.b64 {lo, hi}, %1;\n\trcp.approx.ftz.f32 lo, lo;\n\t"
      "rcp.approx.ftz.f32 hi, hi;\n\tmov.b64 %0, {lo, hi};\n\t}"
      : "=l"(r) : "l"(d));
  return r;
#else
  return f2_make(rcp_approx(f2_lo(d)), rcp_approx(f2_hi(d)));
#endif
}

// ---- I/O dtypes ------------------------------------------------------------
template <typename IO>
__device__ __forceinline__ float to_f32(IO x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename IO>
__device__ __forceinline__ IO from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ---- 16-byte asynchronous copies (global → shared, L2-only caching) ---------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(smem_dst)), "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}


// ---- gate activations (kla_options.gates) -----------------------------------
// With a gate bit set the corresponding input holds a pre-activation:
//   Λ^v = softplus(x), a = sigmoid(x), p̄ = softplus(x), or the OU-tied
//   p̄ = softplus(x)·(1 − a²) (an exactly discretised OU process with
//   stationary variance softplus(x) and decay a).
constexpr int kGateLamV = 1, kGateA = 2, kGatePbarSoftplus = 4, kGatePbarOU = 8;

__device__ __forceinline__ float softplus_f(float x) { return x > 20.0f ? x : log1pf(expf(x)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

__device__ __forceinline__ float gate_lamv(float x, int gates) { return (gates & kGateLamV) ? softplus_f(x) : x; }
__device__ __forceinline__ float gate_a(float x, int gates) { return (gates & kGateA) ? sigmoid_f(x) : x; }
// p̄ from its input xp and the decay's input xa (both as given to the kernel).
__device__ __forceinline__ float gate_pbar(float xp, float xa, int gates) {
  if (gates & kGatePbarOU) {
    // 1 − a² = (1 − a)(1 + a), with 1 − a = sigmoid(−x) when a = sigmoid(x)
    const float one_minus_a = (gates & kGateA) ? sigmoid_f(-xa) : 1.0f - xa;
    const float a = (gates & kGateA) ? sigmoid_f(xa) : xa;
    return softplus_f(xp) * (one_minus_a * (1.0f + a));
  }
  return (gates & kGatePbarSoftplus) ? softplus_f(xp) : xp;
}


// Gradients with respect to the pre-activations, from the gradients ga, gp
// with respect to a and p̄ (per row) ...
__device__ __forceinline__ void gate_chain_row(float ga, float gp, float xa, float xp, int gates, float& gxa,
                                               float& gxp) {
  const float a = (gates & kGateA) ? sigmoid_f(xa) : xa;
  if (gates & kGatePbarOU) {  // p̄ = S(1 − a²), S = softplus(xp)
    const float one_minus_a = (gates & kGateA) ? sigmoid_f(-xa) : 1.0f - xa;
    gxp = gp * (one_minus_a * (1.0f + a)) * sigmoid_f(xp);
    ga = fmaf(gp * softplus_f(xp), -2.0f * a, ga);
  } else {
    gxp = (gates & kGatePbarSoftplus) ? gp * sigmoid_f(xp) : gp;
  }
  gxa = (gates & kGateA) ? ga * (a * sigmoid_f(-xa)) : ga;  // σ' = σ(x)σ(−x)
}
// ... and from the gradient with respect to Λ^v (per column).
__device__ __forceinline__ float gate_chain_lamv(float gL, float xL, int gates) {
  return (gates & kGateLamV) ? gL * sigmoid_f(xL) : gL;
}

}  // namespace kla
