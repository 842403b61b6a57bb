// Causal depthwise 1-D convolution with an optional SiLU, forward and
// backward (sm_103a): the short convolution of the Mamba-like block that the
// KLA layer sits in ("Technische Samenvatting: Kalman Linear Attention
// (KLA)", gist.science/nl/paper/2602.10743, Methodologie §4: 1-D causal
// convolutions and SiLU activations around the scan).
//
// Per channel (h, d) of a [B, H, T, D] stream, with W taps w[h, d, 0..W-1]:
//   u[t] = bias[h, d] + Σ_k w[k] · x[t − (W−1) + k]        (tap W−1: token t)
//   y[t] = SiLU(u[t]) = u·σ(u)   (or u without the activation)
// x before token 0 comes from the carried window of the W−1 previous inputs
// (zeros when none is given); the window after the last token is returned.
//
// Backward, with gu = gy·SiLU'(u) and SiLU'(u) = σ(u)(1 + u(1 − σ(u))):
//   gx[t]      = Σ_k w[k] · gu[t + (W−1) − k]   (+ the gradient of the window
//                out for the last W−1 inputs; tokens before 0 go to gwindow)
//   gw[h,d,k]  = Σ_{b,t} gu[t] · x[t − (W−1) + k],   gbias[h,d] = Σ_{b,t} gu[t]
//
// Work layout: a block owns a token range of one stream (b, h) and streams
// it through shared-memory stages with cp.async; a thread computes four
// consecutive tokens × four channels of a stage, the channels as two packed
// fp32 pairs (fma/mul/add.rn.f32x2), with the exponential and reciprocal of
// SiLU on the MUFU unit. Their roofline is HBM — the bytes of x and y (and
// gy, gx) — and they run below it limited by instruction issue.
//
// The backward's sums over (b, t) are deterministic: each thread sums its own
// chunk in token order, a block sums its threads in chunk order through
// shared memory, and a second kernel sums the blocks' partials in a fixed
// order. No atomics.
#pragma once

#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>

#include "kla_device.cuh"
#include "kla_launch.h"

namespace kla {

// Internal linkage on purpose: every translation unit that includes this
// header compiles only the kernels of the row widths it instantiates.
namespace {

constexpr int kConvThreads = 256;
constexpr int kMaxDevices = 256;
// Consecutive tokens per thread and stage. With D ≤ 512 a stage holds at
// least two threads' rows, eight tokens, so it always covers the W − 1 ≤ 7
// rows that the next stage reads before its start.
constexpr int kConvRows = 4;
// Shared-memory stages (a stage is TT·D ≈ 4096 elements; stages − 2 are in
// flight while one is computed). Forward: six, 48 KB (bf16) or 96 KB (fp32)
// per block — in bf16 that leaves four blocks per SM, which measured faster
// than eight stages at three blocks (27.3 against 28.9 µs for a B8 H16 T4096
// stream of 64 bf16 channels) or ten at two (32.7 µs). Backward: five stages of x and
// gy plus 32 KB of gu, 112 KB (bf16) or 192 KB (fp32).
template <typename IO>
__host__ __device__ constexpr int conv_stages() { return 6; }
constexpr int kConvBwdStages = 5;
constexpr int kConvFwdMinStages = 8, kConvBwdMinStages = 32;  // stages per block range at least
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): e^x = 2^(x·log2 e)

// ---- four channels as two packed fp32 pairs (channels 0, 1 and 2, 3) --------
struct V4 {
  f2 a, b;
};
__device__ __forceinline__ V4 v4_zero() { return {f2_make(0.f, 0.f), f2_make(0.f, 0.f)}; }
__device__ __forceinline__ V4 v4_from(float4 v) { return {f2_make(v.x, v.y), f2_make(v.z, v.w)}; }
// a bf16 pair (one 32-bit word) as fp32: the bf16 bits are the top half of the fp32 word
__device__ __forceinline__ f2 bf2_to_f2(uint32_t v) {
  return f2_make(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(f2 v) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(f2_lo(v), f2_hi(v));  // round to nearest even
  return *reinterpret_cast<const uint32_t*>(&h);
}
// global, read-only path
__device__ __forceinline__ V4 ldg4(const float* p) { return v4_from(__ldg(reinterpret_cast<const float4*>(p))); }
__device__ __forceinline__ V4 ldg4(const __nv_bfloat16* p) {
  const uint2 r = __ldg(reinterpret_cast<const uint2*>(p));
  return {bf2_to_f2(r.x), bf2_to_f2(r.y)};
}
// shared memory
__device__ __forceinline__ V4 lds4(const float* p) {
  const ulonglong2 r = *reinterpret_cast<const ulonglong2*>(p);
  return {r.x, r.y};
}
__device__ __forceinline__ V4 lds4(const __nv_bfloat16* p) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  return {bf2_to_f2(r.x), bf2_to_f2(r.y)};
}
__device__ __forceinline__ void sts4(float* p, V4 v) { *reinterpret_cast<ulonglong2*>(p) = make_ulonglong2(v.a, v.b); }
// global stores
__device__ __forceinline__ void stg4(float* p, V4 v) { *reinterpret_cast<ulonglong2*>(p) = make_ulonglong2(v.a, v.b); }
__device__ __forceinline__ void stg4(__nv_bfloat16* p, V4 v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(f2_to_bf2(v.a), f2_to_bf2(v.b));
}
__device__ __forceinline__ V4 fma4(V4 w, V4 x, V4 acc) { return {f2_fma(w.a, x.a, acc.a), f2_fma(w.b, x.b, acc.b)}; }

// Base-2 exponential on the MUFU unit (PTX ex2.approx; 0 for large negative input).
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// σ(u) = 1 / (1 + 2^(−u·log2 e)) of a pair; 0 once 2^(…) overflows (u below about −88).
__device__ __forceinline__ f2 sigmoid2(f2 u) {
  const f2 t = f2_mul(u, f2_make(-kLog2e, -kLog2e));
  const f2 e = f2_make(ex2_approx(f2_lo(t)), ex2_approx(f2_hi(t)));
  return f2_rcp(f2_add(e, f2_make(1.0f, 1.0f)));
}
// SiLU(u) = u·σ(u)
__device__ __forceinline__ V4 silu4(V4 u) { return {f2_mul(u.a, sigmoid2(u.a)), f2_mul(u.b, sigmoid2(u.b))}; }
// SiLU'(u) = σ(u)(1 + u(1 − σ(u)))
__device__ __forceinline__ f2 dsilu2(f2 u) {
  const f2 one = f2_make(1.0f, 1.0f);
  const f2 sg = sigmoid2(u);
  const f2 one_minus = f2_fma(sg, f2_make(-1.0f, -1.0f), one);
  return f2_mul(sg, f2_fma(u, one_minus, one));
}

template <int W>
__device__ __forceinline__ void load_taps(const ConvArgs& a, int h, int d0, V4 (&w)[W], V4& bias) {
  const float* wp = a.weight + ((size_t)h * a.D + d0) * W;  // [H][D][W]: four channels' taps are contiguous
#pragma unroll
  for (int k = 0; k < W; ++k) {
    w[k].a = f2_make(__ldg(wp + 0 * W + k), __ldg(wp + 1 * W + k));
    w[k].b = f2_make(__ldg(wp + 2 * W + k), __ldg(wp + 3 * W + k));
  }
  bias = a.bias ? ldg4(a.bias + (size_t)h * a.D + d0) : v4_zero();
}

// 8-byte asynchronous copy (rows of bf16 streams whose width is not a
// multiple of eight channels are only 8-byte aligned).
__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_addr(smem_dst)), "l"(gmem_src) : "memory");
}

// Queue the copy of `bytes` contiguous bytes (a multiple of 8; of 16 when
// `wide`) from global to shared memory, spread over the block's threads.
__device__ __forceinline__ void copy_span(void* dst, const void* src, int bytes, bool wide, int tid) {
  char* d = reinterpret_cast<char*>(dst);
  const char* s = reinterpret_cast<const char*>(src);
  if (wide) {
    for (int o = tid * 16; o < bytes; o += kConvThreads * 16) cp_async16(d + o, s + o);
  } else {
    for (int o = tid * 8; o < bytes; o += kConvThreads * 8) cp_async8(d + o, s + o);
  }
}

// The W − 1 input rows before a block's first token, at the end of the last
// stage buffer: x when the range does not start the sequence, else the
// carried window, else zeros.
template <typename IO, int W>
__device__ __forceinline__ void stage_halo(IO* halo, const IO* xg, const IO* win, long long T0, int D, int row,
                                           bool wide, int tid) {
  if (W == 1) return;
  if (T0 > 0) {
    copy_span(halo, xg + (T0 - (W - 1)) * D, (W - 1) * row, wide, tid);
  } else if (win) {
    copy_span(halo, win, (W - 1) * row, wide, tid);
  } else {
    for (int i = tid; i < (W - 1) * D; i += kConvThreads) halo[i] = from_f32<IO>(0.0f);
  }
}

// Forward: a block owns the token range [T0, T1) of one stream (b, h) and
// streams it through S shared-memory stages of TT tokens (all D channels; a
// stage is one contiguous span of x) with cp.async, S − 2 stages in flight
// while one is computed. Thread (g, c) computes tokens c·R … c·R+R−1 of a stage for
// channels 4g … 4g+3, reading its R+W−1 input rows from shared memory. The S
// stage buffers form one ring of S·TT rows; the rows before a stage are the
// end of the previous buffer (refilled only after the stage is done), and the
// W−1 rows before T0 sit at the end of the ring before the first stage.
template <typename IO, int W, bool ACT, int DC>
__global__ void __launch_bounds__(kConvThreads) kla_conv_kernel(const ConvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int R = kConvRows, S = conv_stages<IO>();
  // DC > 0: the row width is a compile-time constant (so are the stage
  // geometry and every row offset); DC = 0: any width, read from the arguments
  const int D = DC ? DC : a.D, G = D >> 2, T = a.T;
  const int cpb = DC ? kConvThreads / (DC / 4) : a.chunks_per_block, TT = cpb * R;
  const int tid = threadIdx.x, c = tid / G, g = tid - c * G, d0 = 4 * g, r0 = c * R;
  const long long bh = blockIdx.x;
  const int h = (int)(bh % a.H);
  const long long T0 = (long long)blockIdx.y * a.range, T1 = min(T0 + (long long)a.range, (long long)T);
  const int row = D * (int)sizeof(IO);
  const bool wide = row % 16 == 0;  // 16-byte copies; else 8-byte ones
  const IO* __restrict__ xg = reinterpret_cast<const IO*>(a.x) + bh * (long long)T * D;
  IO* __restrict__ yg = reinterpret_cast<IO*>(a.y) + bh * (long long)T * D;
  const IO* win = a.win ? reinterpret_cast<const IO*>(a.win) + bh * (long long)(W - 1) * D : nullptr;
  IO* ring = reinterpret_cast<IO*>(smem);
  const int ring_rows = S * TT;

  auto stage_copy = [&](int n) {
    const long long ts = T0 + (long long)n * TT;
    const int rows = (int)min((long long)TT, T1 - ts);
    if (rows > 0) copy_span(ring + (n % S) * TT * D, xg + ts * D, rows * row, wide, tid);
  };
  stage_halo<IO, W>(ring + (ring_rows - (W - 1)) * D, xg, win, T0, D, row, wide, tid);
#pragma unroll
  for (int n = 0; n < S - 1; ++n) {
    stage_copy(n);
    cp_async_commit();
  }

  V4 w[W], bias;
  load_taps<W>(a, h, d0, w, bias);
  // y of the token at row j of this thread, from input rows xr[j … j+W−1]
  auto output = [&](const V4 (&xr)[R + W - 1], int j) {
    V4 u = bias;
#pragma unroll
    for (int k = 0; k < W; ++k) u = fma4(w[k], xr[j + k], u);
    return ACT ? silu4(u) : u;
  };
  const int nst = (int)((T1 - T0 + TT - 1) / TT);
  for (int n = 0; n < nst; ++n) {
    cp_async_wait<S - 2>();
    __syncthreads();  // stage n (and the halo) landed for every thread
    const long long t_stage = T0 + (long long)n * TT;
    const int rows = (int)min((long long)TT, T1 - t_stage);  // tokens of this stage
    if (c < cpb && r0 < rows) {
      const int q0 = (n % S) * TT + r0 - (W - 1);
      V4 xr[R + W - 1];
#pragma unroll
      for (int i = 0; i < R + W - 1; ++i) {
        int q = q0 + i;
        q += q < 0 ? ring_rows : 0;
        xr[i] = lds4(ring + q * D + d0);  // rows past the stage's end are read but not used
      }
      IO* yo = yg + t_stage * D + d0 + r0 * D;
      if (r0 + R <= rows) {
#pragma unroll
        for (int j = 0; j < R; ++j) stg4(yo + j * D, output(xr, j));
      } else {
#pragma unroll
        for (int j = 0; j < R; ++j)
          if (r0 + j < rows) stg4(yo + j * D, output(xr, j));
      }
    }
    __syncthreads();  // nobody reads buffer (n − 1) any more
    stage_copy(n + S - 1);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // The window after the last token, written by the first block of the
  // stream: the last W−1 inputs of (window, x). Every value is read before
  // any is written, so the window out may be the window in.
  if (W > 1 && blockIdx.y == 0 && a.wout) {
    IO* wout = reinterpret_cast<IO*>(a.wout) + bh * (long long)(W - 1) * D;
    // item i = tid + q·256 < G·(W−1): window row i / G, channel group i % G (G ≤ 128)
    V4 v[W > 1 ? W - 1 : 1];
#pragma unroll
    for (int q = 0; q < W - 1; ++q) {
      const int i = tid + q * kConvThreads;
      v[q] = v4_zero();
      if (i < G * (W - 1)) {
        const int j = i / G, gg = i - j * G;
        const long long tau = (long long)T - (W - 1) + j;
        if (tau >= 0) v[q] = ldg4(xg + tau * D + 4 * gg);
        else if (win) v[q] = ldg4(win + (tau + W - 1) * D + 4 * gg);
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < W - 1; ++q) {
      const int i = tid + q * kConvThreads;
      if (i < G * (W - 1)) {
        const int j = i / G, gg = i - j * G;
        stg4(wout + (long long)j * D + 4 * gg, v[q]);
      }
    }
  }
}

// Backward: a block owns the token range [T0, T1) of one stream. gu is
// needed on [T0, T1e), T1e = min(T1 + W − 1, T) (gx of the range's last
// tokens reaches W − 1 tokens further), so x and gy stream through
// kConvBwdStages shared-memory stages over [T0, T1e) (x with the W − 1 rows
// before T0 at the end of its ring, as in the forward). Stage n: each thread
// forms gu of its R tokens × 4 channels into a two-stage fp32 ring in shared
// memory and adds its tokens below T1 to its tap and bias partial sums; then
// gx of stage n − 1 is complete and is written (gu rows past the stage come
// from stage n; tokens at or past T1e have gu = 0). The first block of a
// stream also writes the gradient of the window in (tokens −(W−1) … −1) once
// stage 0's gu exists.
template <typename IO, int W, bool ACT, int DC>
__global__ void __launch_bounds__(kConvThreads) kla_conv_bwd_kernel(const ConvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int R = kConvRows, S = kConvBwdStages;
  // DC > 0: the row width is a compile-time constant (so are the stage
  // geometry and every row offset); DC = 0: any width, read from the arguments
  const int D = DC ? DC : a.D, G = D >> 2, T = a.T;
  const int cpb = DC ? kConvThreads / (DC / 4) : a.chunks_per_block, TT = cpb * R;
  const int tid = threadIdx.x, c = tid / G, g = tid - c * G, d0 = 4 * g, r0 = c * R;
  const long long bh = blockIdx.x;
  const int h = (int)(bh % a.H);
  const long long T0 = (long long)blockIdx.y * a.range, T1 = min(T0 + (long long)a.range, (long long)T);
  const long long T1e = min(T1 + (W - 1), (long long)T);
  const int row = D * (int)sizeof(IO);
  const bool wide = row % 16 == 0;
  const int ring_rows = S * TT;
  IO* xs = reinterpret_cast<IO*>(smem);                           // x ring, S·TT rows
  IO* gys = xs + (size_t)ring_rows * D;                           // gy stages
  float* gus = reinterpret_cast<float*>(gys + (size_t)ring_rows * D);  // gu ring, 2·TT rows
  const long long off = bh * (long long)T * D;
  const IO* __restrict__ xg = reinterpret_cast<const IO*>(a.x) + off;
  const IO* __restrict__ gyg = a.gy ? reinterpret_cast<const IO*>(a.gy) + off : nullptr;  // null: zero
  IO* __restrict__ gxg = reinterpret_cast<IO*>(a.gx) + off;
  const long long woff = bh * (long long)(W - 1) * D;
  const IO* win = a.win ? reinterpret_cast<const IO*>(a.win) + woff : nullptr;
  const IO* gwo = a.gwout ? reinterpret_cast<const IO*>(a.gwout) + woff : nullptr;
  IO* gwin = a.gwin ? reinterpret_cast<IO*>(a.gwin) + woff : nullptr;
  const long long tail = (long long)T - (W - 1);  // first input copied into the window out

  auto stage_copy = [&](int n) {
    const long long ts = T0 + (long long)n * TT;
    const int rows = (int)min((long long)TT, T1e - ts);
    if (rows <= 0) return;
    copy_span(xs + (n % S) * TT * D, xg + ts * D, rows * row, wide, tid);
    if (gyg) copy_span(gys + (n % S) * TT * D, gyg + ts * D, rows * row, wide, tid);
  };
  stage_halo<IO, W>(xs + (ring_rows - (W - 1)) * D, xg, win, T0, D, row, wide, tid);
#pragma unroll
  for (int n = 0; n < S - 1; ++n) {
    stage_copy(n);
    cp_async_commit();
  }

  V4 w[W], bias, gw[W], gb = v4_zero();
  load_taps<W>(a, h, d0, w, bias);
#pragma unroll
  for (int k = 0; k < W; ++k) gw[k] = v4_zero();

  // gx of this thread's tokens in stage m from gu rows r0 … r0+R+W−2 of the
  // two-stage gu ring (rows past stage m are stage m + 1's). Positions are
  // 32-bit offsets from the stage start; a thread whose tokens are all below
  // T1, whose gu rows are all below T1e and which has no window-out gradient
  // takes the path without checks.
  auto emit = [&](int m) {
    if (c >= cpb) return;
    const long long sm0 = T0 + (long long)m * TT;
    const int lim1 = (int)min((long long)(2 * TT), T1 - sm0);    // rows below T1
    const int lim1e = (int)min((long long)(2 * TT), T1e - sm0);  // rows below T1e
    if (r0 >= lim1) return;
    const int q0 = (m & 1) * TT + r0;
    IO* go = gxg + sm0 * D + d0 + r0 * D;
    V4 gr[R + W - 1];
    const bool has_tail = gwo && sm0 + r0 + R - 1 >= tail;
    if (r0 + R <= lim1 && r0 + R + W - 1 <= lim1e && !has_tail) {
#pragma unroll
      for (int i = 0; i < R + W - 1; ++i) {
        int q = q0 + i;
        q -= q >= 2 * TT ? 2 * TT : 0;
        gr[i] = lds4(gus + q * D + d0);
      }
#pragma unroll
      for (int j = 0; j < R; ++j) {
        V4 gv = v4_zero();
#pragma unroll
        for (int k = 0; k < W; ++k) gv = fma4(w[k], gr[j + (W - 1) - k], gv);  // gu of token j + W−1−k
        stg4(go + j * D, gv);
      }
      return;
    }
    // row of the first input copied into the window out (a row of this stage
    // at or after it is a token within W − 1 of T, so clamping is exact)
    const int tl = (int)max(-8LL, min(tail - sm0, 2LL * TT + 1));
#pragma unroll
    for (int i = 0; i < R + W - 1; ++i) {
      int q = q0 + i;
      q -= q >= 2 * TT ? 2 * TT : 0;
      gr[i] = r0 + i < lim1e ? lds4(gus + q * D + d0) : v4_zero();  // gu past T1e is zero
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (r0 + j < lim1) {
        V4 gv = (gwo && r0 + j >= tl) ? ldg4(gwo + (r0 + j - tl) * D + d0) : v4_zero();
#pragma unroll
        for (int k = 0; k < W; ++k) gv = fma4(w[k], gr[j + (W - 1) - k], gv);
        stg4(go + j * D, gv);
      }
    }
  };
  // gradient of the window in: tokens −(W−1) … −1, all reached by stage 0's gu
  auto emit_window = [&]() {
    if constexpr (W == 1) return;
    if (blockIdx.y != 0 || !gwin) return;
    for (int i = tid; i < G * (W - 1); i += kConvThreads) {
      const int j = i / G, gg = i - j * G;
      const long long te = (long long)j - (W - 1);
      V4 gv = (gwo && te >= tail) ? ldg4(gwo + (te - tail) * D + 4 * gg) : v4_zero();
      V4 wg[W], bg;
      load_taps<W>(a, h, 4 * gg, wg, bg);
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const long long tt = te + (W - 1) - k;
        if (tt >= 0 && tt < T1e) gv = fma4(wg[k], lds4(gus + tt * D + 4 * gg), gv);  // stage 0: tt < W−1 ≤ TT
      }
      stg4(gwin + (long long)j * D + 4 * gg, gv);
    }
  };

  // gu of the token at row j of this thread, from gy and input rows
  // xr[j … j+W−1]; added to the partial sums when `own`
  auto grad_u = [&](const V4 (&xr)[R + W - 1], const IO* gyr, int j, bool own) {
    V4 gu = gyg ? lds4(gyr + j * D) : v4_zero();
    if (ACT) {
      V4 u = bias;
#pragma unroll
      for (int k = 0; k < W; ++k) u = fma4(w[k], xr[j + k], u);
      gu.a = f2_mul(gu.a, dsilu2(u.a));
      gu.b = f2_mul(gu.b, dsilu2(u.b));
    }
    if (own) {
      gb.a = f2_add(gb.a, gu.a);
      gb.b = f2_add(gb.b, gu.b);
#pragma unroll
      for (int k = 0; k < W; ++k) gw[k] = fma4(gu, xr[j + k], gw[k]);
    }
    return gu;
  };
  const int nst = (int)((T1e - T0 + TT - 1) / TT);
  for (int n = 0; n < nst; ++n) {
    cp_async_wait<S - 2>();
    __syncthreads();  // stage n landed; gx of stage n − 2 is done with its gu
    const long long t_stage = T0 + (long long)n * TT;
    const int rows = (int)min((long long)TT, T1e - t_stage);  // tokens whose gu is needed
    const int own = (int)max(0LL, min((long long)TT, T1 - t_stage));  // of those, tokens of this range
    if (c < cpb && r0 < rows) {
      const int q0 = (n % S) * TT + r0 - (W - 1);
      V4 xr[R + W - 1];
#pragma unroll
      for (int i = 0; i < R + W - 1; ++i) {
        int q = q0 + i;
        q += q < 0 ? ring_rows : 0;
        xr[i] = lds4(xs + q * D + d0);  // rows past the stage's end are read but not used
      }
      const IO* gyr = gys + ((n % S) * TT + r0) * D + d0;
      float* gu_out = gus + ((n & 1) * TT + r0) * D + d0;
      if (r0 + R <= own) {  // every token needed and of this range
#pragma unroll
        for (int j = 0; j < R; ++j) sts4(gu_out + j * D, grad_u(xr, gyr, j, true));
      } else {
#pragma unroll
        for (int j = 0; j < R; ++j) sts4(gu_out + j * D, r0 + j < rows ? grad_u(xr, gyr, j, r0 + j < own) : v4_zero());
      }
    }
    __syncthreads();  // gu of stage n visible; x and gy of stage n − 1 no longer read
    stage_copy(n + S - 1);
    cp_async_commit();
    if (n >= 1) emit(n - 1);
    else emit_window();
  }
  cp_async_wait<0>();
  if (nst >= 1) emit(nst - 1);
  else emit_window();  // T = 0: the window's gradient is the window out's

  if (!a.part) return;  // no tap or bias gradient wanted
  // Block partial: the threads of a channel group summed in chunk order,
  // through shared memory (all of it is free now: 16·(W+1)·256 bytes at
  // most, under the 20·TT·D ≥ 20·1024 bytes of the stages and the gu ring).
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);  // [cpb][G][W + 1] groups of four floats
  if (c < cpb) {
    float* r = red + ((size_t)c * G + g) * (W + 1) * 4;
#pragma unroll
    for (int k = 0; k < W; ++k) sts4(r + 4 * k, gw[k]);
    sts4(r + 4 * W, gb);
  }
  __syncthreads();
  for (int i = tid; i < G * (W + 1); i += kConvThreads) {
    const int gg = i / (W + 1), k = i - gg * (W + 1);
    float4 sum = *reinterpret_cast<const float4*>(red + ((size_t)gg * (W + 1) + k) * 4);
    for (int cc = 1; cc < cpb; ++cc) {
      const float4 v = *reinterpret_cast<const float4*>(red + (((size_t)cc * G + gg) * (W + 1) + k) * 4);
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    // partials [H][P][D][W + 1], P = B · gridDim.y, p = b · gridDim.y + blockIdx.y
    const long long b = bh / a.H;
    const long long p = b * gridDim.y + blockIdx.y;
    float* dst = a.part + (((size_t)h * a.nparts + p) * D + 4 * gg) * (W + 1) + k;
    dst[0] = sum.x;
    dst[W + 1] = sum.y;
    dst[2 * (W + 1)] = sum.z;
    dst[3 * (W + 1)] = sum.w;
  }
}

// gweight[h, d, k] and gbias[h, d]: the sum of the partials over p in order.
__global__ void __launch_bounds__(256) kla_conv_bwd_finish_kernel(const ConvArgs a, int W) {
  const long long n = (long long)a.H * a.D * (W + 1);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long h = i / ((long long)a.D * (W + 1));
    const long long r = i - h * a.D * (W + 1);  // d * (W + 1) + k
    float s = 0.f;
    for (long long p = 0; p < a.nparts; ++p) s += a.part[((size_t)h * a.nparts + p) * a.D * (W + 1) + r];
    const long long d = r / (W + 1), k = r - d * (W + 1);
    if (k < W) {
      if (a.gweight) a.gweight[(h * a.D + d) * W + k] = s;
    } else if (a.gbias) {
      a.gbias[h * a.D + d] = s;
    }
  }
}

// Raise kernel `Kernel`'s dynamic shared-memory limit to `smem_max` — the
// most any launch of that instantiation asks for (a stage holds at most 256
// threads' rows: TT·D ≤ 1024·kConvRows) — once per device.
template <auto Kernel>
cudaError_t prepare_kernel(size_t smem_max) {
  static std::atomic<int> done[kMaxDevices];  // one set per kernel instantiation
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  if ((e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max)) != cudaSuccess)
    return e;
  done[dev].store(1, std::memory_order_relaxed);
  return cudaSuccess;
}

template <typename IO, int W, bool ACT, int DC>
cudaError_t launch_fwd(ConvArgs a, int num_sms, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  a.chunks_per_block = kConvThreads / (a.D / 4);
  const long long TT = (long long)a.chunks_per_block * kConvRows;
  const size_t smem = (size_t)conv_stages<IO>() * TT * a.D * sizeof(IO);
  constexpr size_t smem_max = (size_t)conv_stages<IO>() * 1024 * kConvRows * sizeof(IO);
  auto fn = kla_conv_kernel<IO, W, ACT, DC>;
  const cudaError_t e = prepare_kernel<kla_conv_kernel<IO, W, ACT, DC>>(smem_max);
  if (e != cudaSuccess) return e;
  long long blocks_y = 0;
  a.range = conv_range(bh, a.T, TT, num_sms, kConvFwdMinStages, &blocks_y);
  fn<<<dim3((unsigned)bh, (unsigned)blocks_y), kConvThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename IO, int W, bool ACT, int DC>
cudaError_t launch_bwd(ConvArgs a, int num_sms, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  a.chunks_per_block = kConvThreads / (a.D / 4);
  const long long TT = (long long)a.chunks_per_block * kConvRows;
  const size_t smem = 2 * (size_t)kConvBwdStages * TT * a.D * sizeof(IO) + 2 * (size_t)TT * a.D * sizeof(float);
  constexpr size_t smem_max =
      (2 * (size_t)kConvBwdStages * sizeof(IO) + 2 * sizeof(float)) * 1024 * kConvRows;
  auto fn = kla_conv_bwd_kernel<IO, W, ACT, DC>;
  cudaError_t e = prepare_kernel<kla_conv_bwd_kernel<IO, W, ACT, DC>>(smem_max);
  if (e != cudaSuccess) return e;
  long long blocks_y = 0;
  a.range = conv_range(bh, a.T, TT, num_sms, kConvBwdMinStages, &blocks_y);  // as conv_partial_bytes()
  a.nparts = a.part ? (long long)a.B * blocks_y : 0;
  fn<<<dim3((unsigned)bh, (unsigned)blocks_y), kConvThreads, smem, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.gweight || a.gbias) {
    const long long n = (long long)a.H * a.D * (W + 1);
    const int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
    kla_conv_bwd_finish_kernel<<<blocks, 256, 0, s>>>(a, W);
    e = cudaGetLastError();
  }
  return e;
}

template <typename IO, int W, int DC>
cudaError_t launch_w(const ConvArgs& a, bool backward, int num_sms, cudaStream_t s) {
  if (backward)
    return a.act ? launch_bwd<IO, W, true, DC>(a, num_sms, s) : launch_bwd<IO, W, false, DC>(a, num_sms, s);
  return a.act ? launch_fwd<IO, W, true, DC>(a, num_sms, s) : launch_fwd<IO, W, false, DC>(a, num_sms, s);
}

template <typename IO, int DC>
cudaError_t launch_io(const ConvArgs& a, bool backward, int num_sms, cudaStream_t s) {
  switch (a.W) {
    case 1: return launch_w<IO, 1, DC>(a, backward, num_sms, s);
    case 2: return launch_w<IO, 2, DC>(a, backward, num_sms, s);
    case 3: return launch_w<IO, 3, DC>(a, backward, num_sms, s);
    case 4: return launch_w<IO, 4, DC>(a, backward, num_sms, s);
    case 5: return launch_w<IO, 5, DC>(a, backward, num_sms, s);
    case 6: return launch_w<IO, 6, DC>(a, backward, num_sms, s);
    case 7: return launch_w<IO, 7, DC>(a, backward, num_sms, s);
    case 8: return launch_w<IO, 8, DC>(a, backward, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Launch the forward (or the backward and its finish kernel) for row width
// DC (0: any width). kla_conv.cu instantiates DC = 0 and dispatches; the
// widths of the scan's common head sizes have their own translation units
// (kla_conv_d64.cu, kla_conv_d128.cu), compiled in parallel.
template <int DC>
cudaError_t conv_launch_dc(const ConvArgs& a, bool backward, int num_sms, cudaStream_t s) {
  return a.io == IO_BF16 ? launch_io<__nv_bfloat16, DC>(a, backward, num_sms, s)
                         : launch_io<float, DC>(a, backward, num_sms, s);
}

}  // namespace kla
