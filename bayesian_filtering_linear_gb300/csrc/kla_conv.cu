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
// Work layout: a thread owns four channels of one head and a chunk of L
// tokens, and walks them in order with the last W inputs (and, backward, the
// last W values of gu) in a register ring; the ring index of each token is a
// compile-time constant because the walk is unrolled by W. Threads of a block
// cover consecutive channel groups, then consecutive chunks of one (b, h), so
// each token row is read by consecutive threads. The chunk's first W−1 inputs
// (and, backward, its last W−1 values of gu) are the neighbouring chunk's and
// are recomputed, not exchanged. Both kernels stream from HBM: the bound is
// the bytes of x, y (and gy, gx).
//
// The backward's sums over (b, t) are deterministic: each thread sums its own
// chunk in token order, a block sums its threads in chunk order through
// shared memory, and a second kernel sums the blocks' partials in a fixed
// order. No atomics.
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>

#include "kla_device.cuh"
#include "kla_launch.h"

namespace kla {

namespace {

constexpr int kConvThreads = 256;
constexpr int kMaxDevices = 256;
// Consecutive tokens per thread and stage. With D ≤ 512 a stage holds at
// least two threads' rows, eight tokens, so it always covers the W − 1 ≤ 7
// rows that the next stage reads before its start.
constexpr int kConvRows = 4;
constexpr int kConvStages = 4;     // forward: shared-memory stages (three in flight)
constexpr int kConvBwdStages = 3;  // backward: stages of x and gy (two in flight)

__device__ __forceinline__ float4 load4ch(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4ch(const __nv_bfloat16* p) {
  const uint2 r = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
  const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ void store4ch(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4ch(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 r;
  r.x = *reinterpret_cast<const uint32_t*>(&lo);
  r.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = r;
}

// Four channels of one row from shared memory.
__device__ __forceinline__ float4 lds4ch(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 lds4ch(const __nv_bfloat16* p) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
  const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ float f4get(const float4& v, int e) { return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w; }
__device__ __forceinline__ void f4set(float4& v, int e, float s) {
  if (e == 0) v.x = s; else if (e == 1) v.y = s; else if (e == 2) v.z = s; else v.w = s;
}

// σ(u) with the hardware reciprocal; 0 for u below about −88 (e^−u overflows).
__device__ __forceinline__ float sigmoid_fast(float u) { return rcp_approx(1.0f + __expf(-u)); }

template <int W>
__device__ __forceinline__ void load_taps(const ConvArgs& a, int h, int d0, float4 (&w)[W], float4& bias) {
  const float* wp = a.weight + ((size_t)h * a.D + d0) * W;  // [H][D][W]: four channels' taps are contiguous
#pragma unroll
  for (int k = 0; k < W; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e) f4set(w[k], e, __ldg(wp + e * W + k));
  bias = a.bias ? __ldg(reinterpret_cast<const float4*>(a.bias + (size_t)h * a.D + d0)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// 8-byte asynchronous copy (rows of bf16 streams whose width is not a
// multiple of eight channels are only 8-byte aligned).
__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_addr(smem_dst)), "l"(gmem_src) : "memory");
}

// Forward: a block owns the token range [T0, T1) of one stream (b, h) and
// streams it through kConvStages shared-memory stages of TT tokens (all D
// channels; a stage is one contiguous span of x) with cp.async, kConvStages−1
// stages in flight. Thread (g, c) computes tokens c·R … c·R+R−1 of a stage for
// channels 4g … 4g+3, reading its R+W−1 input rows from shared memory (rows
// before the stage from the previous stage's buffer, which is refilled only
// after the stage is done). The W−1 rows before T0 — x, the carried window,
// or zeros — are placed at the end of the last buffer before the first stage.
template <typename IO, int W, bool ACT>
__global__ void __launch_bounds__(kConvThreads) kla_conv_kernel(const ConvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int R = kConvRows, S = kConvStages;
  const int D = a.D, G = D >> 2, T = a.T;
  const int cpb = a.chunks_per_block, TT = cpb * R;
  const int tid = threadIdx.x, c = tid / G, g = tid - c * G, d0 = 4 * g;
  const long long bh = blockIdx.x;
  const int h = (int)(bh % a.H);
  const long long T0 = (long long)blockIdx.y * a.range, T1 = min(T0 + (long long)a.range, (long long)T);
  const size_t row = (size_t)D * sizeof(IO);
  const size_t stage_bytes = (size_t)TT * row;
  const IO* __restrict__ xg = reinterpret_cast<const IO*>(a.x) + bh * (long long)T * D;
  IO* __restrict__ yg = reinterpret_cast<IO*>(a.y) + bh * (long long)T * D;
  const IO* win = a.win ? reinterpret_cast<const IO*>(a.win) + bh * (long long)(W - 1) * D : nullptr;
  auto buf = [&](long long n) { return reinterpret_cast<IO*>(smem + (size_t)(n % S) * stage_bytes); };
  const bool wide = row % 16 == 0;  // 16-byte copies; else 8-byte ones

  // Queue the copy of `bytes` contiguous bytes (a multiple of 8) into shared memory.
  auto copy_span = [&](void* dst, const void* src, size_t bytes) {
    char* d = reinterpret_cast<char*>(dst);
    const char* s0 = reinterpret_cast<const char*>(src);
    if (wide) {
      for (size_t o = (size_t)tid * 16; o < bytes; o += kConvThreads * 16) cp_async16(d + o, s0 + o);
    } else {
      for (size_t o = (size_t)tid * 8; o < bytes; o += kConvThreads * 8) cp_async8(d + o, s0 + o);
    }
  };
  auto stage_copy = [&](long long n) {
    const long long ts = T0 + n * TT, te = min(ts + TT, T1);
    if (ts < te) copy_span(buf(n), xg + ts * D, (size_t)(te - ts) * row);
  };

  // rows before T0, at the end of buffer S−1 (= the buffer before stage 0)
  if (W > 1) {
    IO* halo = reinterpret_cast<IO*>(smem + (size_t)(S - 1) * stage_bytes) + (size_t)(TT - (W - 1)) * D;
    if (T0 > 0) {
      copy_span(halo, xg + (T0 - (W - 1)) * D, (size_t)(W - 1) * row);
    } else if (win) {
      copy_span(halo, win, (size_t)(W - 1) * row);
    } else {
      for (int i = tid; i < (W - 1) * D; i += kConvThreads) halo[i] = from_f32<IO>(0.0f);
    }
  }
#pragma unroll
  for (int n = 0; n < S - 1; ++n) {
    stage_copy(n);
    cp_async_commit();
  }

  float4 w[W], bias;
  load_taps<W>(a, h, d0, w, bias);
  // y of one token from its W input rows xr[j … j+W−1]
  auto output = [&](const float4 (&xr)[R + W - 1], int j) {
    float4 u = bias;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const float4 xv = xr[j + k];
      u.x = fmaf(w[k].x, xv.x, u.x);
      u.y = fmaf(w[k].y, xv.y, u.y);
      u.z = fmaf(w[k].z, xv.z, u.z);
      u.w = fmaf(w[k].w, xv.w, u.w);
    }
    if (ACT) {
      u.x *= sigmoid_fast(u.x);
      u.y *= sigmoid_fast(u.y);
      u.z *= sigmoid_fast(u.z);
      u.w *= sigmoid_fast(u.w);
    }
    return u;
  };
  // The S stage buffers are one ring of S·TT rows; stage n starts at row
  // (n mod S)·TT, and the rows before it wrap from the ring's end. Offsets
  // inside a stage are 32-bit; the stage's global base is formed once.
  const IO* ring = reinterpret_cast<const IO*>(smem);
  const int ring_rows = S * TT, r0 = c * R;
  const int nst = (int)((T1 - T0 + TT - 1) / TT);
  for (int n = 0; n < nst; ++n) {
    cp_async_wait<S - 2>();
    __syncthreads();  // stage n (and the halo) landed for every thread
    const long long t_stage = T0 + (long long)n * TT;
    const int rows = (int)min((long long)TT, T1 - t_stage);  // tokens of this stage
    if (c < cpb && r0 < rows) {
      const int q0 = (n % S) * TT + r0 - (W - 1);
      float4 xr[R + W - 1];
#pragma unroll
      for (int i = 0; i < R + W - 1; ++i) {
        int q = q0 + i;
        q += q < 0 ? ring_rows : 0;
        xr[i] = lds4ch(ring + q * D + d0);  // rows past the stage's end are read but not used
      }
      IO* yo = yg + t_stage * D + d0 + r0 * D;
      if (r0 + R <= rows) {
#pragma unroll
        for (int j = 0; j < R; ++j) store4ch(yo + j * D, output(xr, j));
      } else {
#pragma unroll
        for (int j = 0; j < R; ++j)
          if (r0 + j < rows) store4ch(yo + j * D, output(xr, j));
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
    // item i = tid + q·256 < G·(W−1): window row i / G, channel group i % G (G ≤ 256)
    float4 v[W > 1 ? W - 1 : 1];
#pragma unroll
    for (int q = 0; q < W - 1; ++q) {
      const int i = tid + q * kConvThreads;
      v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < G * (W - 1)) {
        const int j = i / G, gg = i - j * G;
        const long long tau = (long long)T - (W - 1) + j;
        if (tau >= 0) v[q] = load4ch(xg + tau * D + 4 * gg);
        else if (win) v[q] = load4ch(win + (tau + W - 1) * D + 4 * gg);
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < W - 1; ++q) {
      const int i = tid + q * kConvThreads;
      if (i < G * (W - 1)) {
        const int j = i / G, gg = i - j * G;
        store4ch(wout + (long long)j * D + 4 * gg, v[q]);
      }
    }
  }
}

// Backward: a block owns the token range [T0, T1) of one stream. gu is
// needed on [T0, T1e), T1e = min(T1 + W − 1, T) (gx of the range's last
// tokens reaches W − 1 tokens further), so x and gy stream through
// kConvBwdStages shared-memory stages over [T0, T1e) (x with the W − 1 rows
// before T0 at the end of the last buffer, as in the forward). Stage n: each
// thread forms gu of its R tokens × 4 channels into a two-stage fp32 ring in
// shared memory and adds its tokens below T1 to its tap and bias partial
// sums; then gx of stage n − 1 is complete and is written (gu rows past the
// stage come from stage n; tokens at or past T1e have gu = 0). The first
// block of a stream also writes the gradient of the window in (tokens −(W−1)
// … −1) once stage 0's gu exists.
template <typename IO, int W, bool ACT>
__global__ void __launch_bounds__(kConvThreads) kla_conv_bwd_kernel(const ConvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int R = kConvRows, S = kConvBwdStages;
  const int D = a.D, G = D >> 2, T = a.T;
  const int cpb = a.chunks_per_block, TT = cpb * R;
  const int tid = threadIdx.x, c = tid / G, g = tid - c * G, d0 = 4 * g;
  const long long bh = blockIdx.x;
  const int h = (int)(bh % a.H);
  const long long T0 = (long long)blockIdx.y * a.range, T1 = min(T0 + (long long)a.range, (long long)T);
  const long long T1e = min(T1 + (W - 1), (long long)T);
  const size_t row = (size_t)D * sizeof(IO);
  const size_t stage_bytes = (size_t)TT * row;
  const size_t gu_stage = (size_t)TT * D;  // floats
  IO* xs = reinterpret_cast<IO*>(smem);
  IO* gys = reinterpret_cast<IO*>(smem + (size_t)S * stage_bytes);
  float* gus = reinterpret_cast<float*>(smem + 2 * (size_t)S * stage_bytes);
  const long long off = bh * (long long)T * D;
  const IO* __restrict__ xg = reinterpret_cast<const IO*>(a.x) + off;
  const IO* __restrict__ gyg = a.gy ? reinterpret_cast<const IO*>(a.gy) + off : nullptr;  // null: zero
  IO* __restrict__ gxg = reinterpret_cast<IO*>(a.gx) + off;
  const long long woff = bh * (long long)(W - 1) * D;
  const IO* win = a.win ? reinterpret_cast<const IO*>(a.win) + woff : nullptr;
  const IO* gwo = a.gwout ? reinterpret_cast<const IO*>(a.gwout) + woff : nullptr;
  IO* gwin = a.gwin ? reinterpret_cast<IO*>(a.gwin) + woff : nullptr;
  const long long tail = (long long)T - (W - 1);  // first input copied into the window out
  const bool wide = row % 16 == 0;

  auto copy_span = [&](void* dst, const void* src, size_t bytes) {
    char* d = reinterpret_cast<char*>(dst);
    const char* s0 = reinterpret_cast<const char*>(src);
    if (wide) {
      for (size_t o = (size_t)tid * 16; o < bytes; o += kConvThreads * 16) cp_async16(d + o, s0 + o);
    } else {
      for (size_t o = (size_t)tid * 8; o < bytes; o += kConvThreads * 8) cp_async8(d + o, s0 + o);
    }
  };
  auto stage_copy = [&](long long n) {
    const long long ts = T0 + n * TT, te = min(ts + TT, T1e);
    if (ts >= te) return;
    const size_t b = (size_t)(n % S) * stage_bytes;
    copy_span(reinterpret_cast<char*>(xs) + b, xg + ts * D, (size_t)(te - ts) * row);
    if (gyg) copy_span(reinterpret_cast<char*>(gys) + b, gyg + ts * D, (size_t)(te - ts) * row);
  };
  if (W > 1) {
    IO* halo = xs + (size_t)(S - 1) * TT * D + (size_t)(TT - (W - 1)) * D;
    if (T0 > 0) {
      copy_span(halo, xg + (T0 - (W - 1)) * D, (size_t)(W - 1) * row);
    } else if (win) {
      copy_span(halo, win, (size_t)(W - 1) * row);
    } else {
      for (int i = tid; i < (W - 1) * D; i += kConvThreads) halo[i] = from_f32<IO>(0.0f);
    }
  }
#pragma unroll
  for (int n = 0; n < S - 1; ++n) {
    stage_copy(n);
    cp_async_commit();
  }

  float4 w[W], bias, gw[W], gb = make_float4(0.f, 0.f, 0.f, 0.f);
  load_taps<W>(a, h, d0, w, bias);
#pragma unroll
  for (int k = 0; k < W; ++k) gw[k] = make_float4(0.f, 0.f, 0.f, 0.f);

  // gx of this thread's tokens in stage m: gu of stage m, and of m + 1 past
  // its end (the two gu buffers form a ring of 2·TT rows). Full stages away
  // from the sequence end take the path without per-token checks.
  const int r0 = c * R;
  auto emit = [&](int m) {
    if (c >= cpb) return;
    const long long sm0 = T0 + (long long)m * TT;
    const long long last = sm0 + r0 + R - 1;  // this thread's last token
    const int gq0 = (m & 1) * TT + r0 + (W - 1);  // gu row of token sm0 + r0 + W − 1
    IO* go = gxg + sm0 * D + d0 + r0 * D;
    auto gx_of = [&](int j, float4 gv) {
#pragma unroll
      for (int k = 0; k < W; ++k) {
        int q = gq0 + j - k;
        q -= q >= 2 * TT ? 2 * TT : 0;
        const float4 gu = lds4ch(gus + q * D + d0);
        gv.x = fmaf(w[k].x, gu.x, gv.x);
        gv.y = fmaf(w[k].y, gu.y, gv.y);
        gv.z = fmaf(w[k].z, gu.z, gv.z);
        gv.w = fmaf(w[k].w, gu.w, gv.w);
      }
      return gv;
    };
    if (last < T1 && last + (W - 1) < T1e && !(gwo && last >= tail)) {
#pragma unroll
      for (int j = 0; j < R; ++j) store4ch(go + j * D, gx_of(j, make_float4(0.f, 0.f, 0.f, 0.f)));
      return;
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const long long te = sm0 + r0 + j;
      if (te < T1) {
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (gwo && te >= tail) gv = load4ch(gwo + (te - tail) * D + d0);
#pragma unroll
        for (int k = 0; k < W; ++k) {
          if (te + (W - 1) - k < T1e) {  // gu of later tokens is zero
            int q = gq0 + j - k;
            q -= q >= 2 * TT ? 2 * TT : 0;
            const float4 gu = lds4ch(gus + q * D + d0);
            gv.x = fmaf(w[k].x, gu.x, gv.x);
            gv.y = fmaf(w[k].y, gu.y, gv.y);
            gv.z = fmaf(w[k].z, gu.z, gv.z);
            gv.w = fmaf(w[k].w, gu.w, gv.w);
          }
        }
        store4ch(go + j * D, gv);
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
      float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (gwo && te >= tail) gv = load4ch(gwo + (te - tail) * D + 4 * gg);
      const float* wp = a.weight + ((size_t)h * D + 4 * gg) * W;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const long long tt = te + (W - 1) - k;
        if (tt >= 0 && tt < T1e) {
          const float4 gu = lds4ch(gus + (size_t)tt * D + 4 * gg);  // stage 0 (tt < W − 1 ≤ TT)
          gv.x = fmaf(__ldg(wp + 0 * W + k), gu.x, gv.x);
          gv.y = fmaf(__ldg(wp + 1 * W + k), gu.y, gv.y);
          gv.z = fmaf(__ldg(wp + 2 * W + k), gu.z, gv.z);
          gv.w = fmaf(__ldg(wp + 3 * W + k), gu.w, gv.w);
        }
      }
      store4ch(gwin + (long long)j * D + 4 * gg, gv);
    }
  };

  // gu of one token (row j of this thread) from gy and its W input rows;
  // its terms are added to the partial sums when `own`
  auto grad_u = [&](const float4 (&xr)[R + W - 1], const IO* gyr, int j, bool own) {
    float4 gu = gyg ? lds4ch(gyr + j * D) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (ACT) {
      float4 u = bias;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        u.x = fmaf(w[k].x, xr[j + k].x, u.x);
        u.y = fmaf(w[k].y, xr[j + k].y, u.y);
        u.z = fmaf(w[k].z, xr[j + k].z, u.z);
        u.w = fmaf(w[k].w, xr[j + k].w, u.w);
      }
      float sg = sigmoid_fast(u.x);
      gu.x *= sg * fmaf(u.x, 1.0f - sg, 1.0f);
      sg = sigmoid_fast(u.y);
      gu.y *= sg * fmaf(u.y, 1.0f - sg, 1.0f);
      sg = sigmoid_fast(u.z);
      gu.z *= sg * fmaf(u.z, 1.0f - sg, 1.0f);
      sg = sigmoid_fast(u.w);
      gu.w *= sg * fmaf(u.w, 1.0f - sg, 1.0f);
    }
    if (own) {
      gb.x += gu.x; gb.y += gu.y; gb.z += gu.z; gb.w += gu.w;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        gw[k].x = fmaf(gu.x, xr[j + k].x, gw[k].x);
        gw[k].y = fmaf(gu.y, xr[j + k].y, gw[k].y);
        gw[k].z = fmaf(gu.z, xr[j + k].z, gw[k].z);
        gw[k].w = fmaf(gu.w, xr[j + k].w, gw[k].w);
      }
    }
    return gu;
  };
  const int ring_rows = S * TT;
  const int nst = (int)((T1e - T0 + TT - 1) / TT);
  for (int n = 0; n < nst; ++n) {
    cp_async_wait<S - 2>();
    __syncthreads();  // stage n landed; gx of stage n − 2 is done with its gu
    const long long t_stage = T0 + (long long)n * TT;
    const int rows = (int)min((long long)TT, T1e - t_stage);  // tokens whose gu is needed
    const int own = (int)max(0LL, min((long long)TT, T1 - t_stage));  // of those, tokens of this range
    if (c < cpb && r0 < rows) {
      const int q0 = (n % S) * TT + r0 - (W - 1);
      float4 xr[R + W - 1];
#pragma unroll
      for (int i = 0; i < R + W - 1; ++i) {
        int q = q0 + i;
        q += q < 0 ? ring_rows : 0;
        xr[i] = lds4ch(xs + q * D + d0);  // rows past the stage's end are read but not used
      }
      const IO* gyr = gys + ((n % S) * TT + r0) * D + d0;
      float* gu_out = gus + ((n & 1) * TT + r0) * D + d0;
      if (r0 + R <= own) {  // every token needed and of this range
#pragma unroll
        for (int j = 0; j < R; ++j) *reinterpret_cast<float4*>(gu_out + j * D) = grad_u(xr, gyr, j, true);
      } else {
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const float4 gu = r0 + j < rows ? grad_u(xr, gyr, j, r0 + j < own) : make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(gu_out + j * D) = gu;
        }
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
  float4* red = reinterpret_cast<float4*>(smem);  // [cpb][G][W + 1]
  if (c < cpb) {
    float4* r = red + ((size_t)c * G + g) * (W + 1);
#pragma unroll
    for (int k = 0; k < W; ++k) r[k] = gw[k];
    r[W] = gb;
  }
  __syncthreads();
  for (int i = tid; i < G * (W + 1); i += kConvThreads) {
    const int gg = i / (W + 1), k = i - gg * (W + 1);
    float4 sum = red[(size_t)gg * (W + 1) + k];
    for (int cc = 1; cc < cpb; ++cc) {
      const float4 v = red[((size_t)cc * G + gg) * (W + 1) + k];
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

// Blocks per SM of kernel `fn` with `smem_max` bytes of dynamic shared
// memory — the most any launch of that instantiation asks for (a stage holds
// at most 256 threads' rows: TT·D ≤ 1024·kConvRows) — with the kernel's shared-memory
// limit raised to it; looked up once per kernel and device and cached.
template <auto Kernel>
cudaError_t blocks_per_sm(size_t smem_max, int* occ) {
  static std::atomic<int> cache[kMaxDevices];  // one per kernel instantiation
  const auto fn = Kernel;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max)) != cudaSuccess)
      return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kConvThreads, smem_max)) != cudaSuccess)
      return e;
    n = std::max(n, 1);
    cache[dev].store(n, std::memory_order_relaxed);
  }
  *occ = n;
  return cudaSuccess;
}

// Forward launch: blocks of one stream split its tokens into ranges of whole
// stages, as many ranges as keep every block of the grid resident at once
// (one wave; streams beyond that are whole-sequence blocks in later waves).
template <typename IO, int W, bool ACT>
cudaError_t launch_fwd(ConvArgs a, int num_sms, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  a.chunks_per_block = kConvThreads / (a.D / 4);
  const long long TT = (long long)a.chunks_per_block * kConvRows;
  const size_t smem = (size_t)kConvStages * TT * a.D * sizeof(IO);
  constexpr size_t smem_max = (size_t)kConvStages * 1024 * kConvRows * sizeof(IO);
  auto fn = kla_conv_kernel<IO, W, ACT>;
  int occ = 0;
  const cudaError_t e = blocks_per_sm<kla_conv_kernel<IO, W, ACT>>(smem_max, &occ);
  if (e != cudaSuccess) return e;
  const long long slots = (long long)std::max(occ, 1) * num_sms;
  const long long nst = std::max(1LL, ((long long)a.T + TT - 1) / TT);
  const long long nsplit = std::max(1LL, std::min(nst, slots / bh));
  a.range = (int)(TT * ((nst + nsplit - 1) / nsplit));
  const long long blocks_y = a.T > 0 ? ((long long)a.T + a.range - 1) / a.range : 1;
  fn<<<dim3((unsigned)bh, (unsigned)blocks_y), kConvThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename IO, int W, bool ACT>
cudaError_t launch_bwd(ConvArgs a, int num_sms, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  a.chunks_per_block = kConvThreads / (a.D / 4);
  const long long TT = (long long)a.chunks_per_block * kConvRows;
  const size_t smem = 2 * (size_t)kConvBwdStages * TT * a.D * sizeof(IO) + 2 * (size_t)TT * a.D * sizeof(float);
  constexpr size_t smem_max =
      (2 * (size_t)kConvBwdStages * sizeof(IO) + 2 * sizeof(float)) * 1024 * kConvRows;
  auto fn = kla_conv_bwd_kernel<IO, W, ACT>;
  int occ = 0;
  cudaError_t e = blocks_per_sm<kla_conv_bwd_kernel<IO, W, ACT>>(smem_max, &occ);
  if (e != cudaSuccess) return e;
  const long long slots = (long long)std::max(occ, 1) * num_sms;
  const long long nst = std::max(1LL, ((long long)a.T + TT - 1) / TT);
  // never more ranges than the partial-sum workspace was sized for
  const long long nsplit =
      std::max(1LL, std::min({nst, slots / bh, conv_bwd_splits(bh, a.T, TT, num_sms)}));
  a.range = (int)(TT * ((nst + nsplit - 1) / nsplit));
  const long long blocks_y = a.T > 0 ? ((long long)a.T + a.range - 1) / a.range : 1;
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

template <typename IO, int W>
cudaError_t launch_w(const ConvArgs& a, bool backward, int num_sms, cudaStream_t s) {
  if (backward) return a.act ? launch_bwd<IO, W, true>(a, num_sms, s) : launch_bwd<IO, W, false>(a, num_sms, s);
  return a.act ? launch_fwd<IO, W, true>(a, num_sms, s) : launch_fwd<IO, W, false>(a, num_sms, s);
}

template <typename IO>
cudaError_t launch_io(const ConvArgs& a, bool backward, int num_sms, cudaStream_t s) {
  switch (a.W) {
    case 1: return launch_w<IO, 1>(a, backward, num_sms, s);
    case 2: return launch_w<IO, 2>(a, backward, num_sms, s);
    case 3: return launch_w<IO, 3>(a, backward, num_sms, s);
    case 4: return launch_w<IO, 4>(a, backward, num_sms, s);
    case 5: return launch_w<IO, 5>(a, backward, num_sms, s);
    case 6: return launch_w<IO, 6>(a, backward, num_sms, s);
    case 7: return launch_w<IO, 7>(a, backward, num_sms, s);
    case 8: return launch_w<IO, 8>(a, backward, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Ranges per stream of the backward: enough for two blocks per SM, at most
// one per stage of TT tokens.
long long conv_bwd_splits(long long bh, int T, long long TT, int num_sms) {
  const long long nst = std::max(1LL, ((long long)T + TT - 1) / TT);
  return std::max(1LL, std::min(nst, 2LL * num_sms / std::max(bh, 1LL)));
}

size_t conv_partial_bytes(int B, int H, int T, int D, int W, int num_sms) {
  const long long bh = (long long)B * H;
  if (bh == 0) return 0;
  const long long TT = (long long)(kConvThreads / (D / 4)) * kConvRows;
  const long long nst = std::max(1LL, ((long long)T + TT - 1) / TT);
  const long long nsplit = conv_bwd_splits(bh, T, TT, num_sms);
  const long long range = TT * ((nst + nsplit - 1) / nsplit);
  const long long blocks_y = T > 0 ? ((long long)T + range - 1) / range : 1;
  return (size_t)H * B * blocks_y * D * (W + 1) * sizeof(float);
}

cudaError_t launch_conv(const ConvArgs& a, int num_sms, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  if (bh == 0) return cudaSuccess;
  return a.io == IO_BF16 ? launch_io<__nv_bfloat16>(a, false, num_sms, s) : launch_io<float>(a, false, num_sms, s);
}

cudaError_t launch_conv_backward(const ConvArgs& a, int num_sms, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  if (bh > 0)
    return a.io == IO_BF16 ? launch_io<__nv_bfloat16>(a, true, num_sms, s) : launch_io<float>(a, true, num_sms, s);
  if (a.H > 0 && (a.gweight || a.gbias)) {  // no batch: the sums are zero
    const long long n = (long long)a.H * a.D * (a.W + 1);
    const int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
    ConvArgs z = a;
    z.nparts = 0;
    kla_conv_bwd_finish_kernel<<<blocks, 256, 0, s>>>(z, a.W);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace kla
