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

#include <cuda_bf16.h>

#include "kla_device.cuh"
#include "kla_launch.h"

namespace kla {

namespace {

constexpr int kConvThreads = 256;

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

__device__ __forceinline__ float f4get(const float4& v, int e) { return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w; }
__device__ __forceinline__ void f4set(float4& v, int e, float s) {
  if (e == 0) v.x = s; else if (e == 1) v.y = s; else if (e == 2) v.z = s; else v.w = s;
}

// σ(u) with the hardware reciprocal; 0 for u below about −88 (e^−u overflows).
__device__ __forceinline__ float sigmoid_fast(float u) { return rcp_approx(1.0f + __expf(-u)); }

// Thread → (channel group, chunk) of the block's (b, h).
struct ConvLane {
  int g, d0;         // channel group and its first channel
  long long chunk;   // token chunk index
  long long t0, t1;  // tokens [t0, t1) of the chunk
  bool active;
};
__device__ __forceinline__ ConvLane conv_lane(const ConvArgs& a) {
  ConvLane l;
  const int G = a.D >> 2;
  const int c = (int)threadIdx.x / G;
  l.g = (int)threadIdx.x - c * G;
  l.d0 = 4 * l.g;
  l.chunk = (long long)blockIdx.y * a.chunks_per_block + c;
  l.t0 = l.chunk * a.L;
  l.t1 = min(l.t0 + a.L, (long long)a.T);
  // chunk 0 always runs: it owns the windows, also when T = 0
  l.active = c < a.chunks_per_block && (l.chunk == 0 || l.t0 < a.T);
  return l;
}

template <int W>
__device__ __forceinline__ void load_taps(const ConvArgs& a, int h, int d0, float4 (&w)[W], float4& bias) {
  const float* wp = a.weight + ((size_t)h * a.D + d0) * W;  // [H][D][W]: four channels' taps are contiguous
#pragma unroll
  for (int k = 0; k < W; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e) f4set(w[k], e, __ldg(wp + e * W + k));
  bias = a.bias ? __ldg(reinterpret_cast<const float4*>(a.bias + (size_t)h * a.D + d0)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Input of token tau of this thread's stream: x for 0 ≤ tau < T, the carried
// window for tau < 0 (zeros without one), zeros past the end.
template <typename IO, int W>
__device__ __forceinline__ float4 input_at(const IO* x, const IO* win, long long tau, int T, int D) {
  if (tau >= 0) return tau < T ? load4ch(x + tau * D) : make_float4(0.f, 0.f, 0.f, 0.f);
  return win ? load4ch(win + (tau + W - 1) * D) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// u of the token in ring slot s (its window is slots s+1 … s+W, mod W).
template <int W>
__device__ __forceinline__ float4 preact(const float4 (&w)[W], const float4& bias, const float4 (&xr)[W], int s) {
  float4 u = bias;
#pragma unroll
  for (int k = 0; k < W; ++k) {
    const float4 xv = xr[(s + 1 + k) % W];
    u.x = fmaf(w[k].x, xv.x, u.x);
    u.y = fmaf(w[k].y, xv.y, u.y);
    u.z = fmaf(w[k].z, xv.z, u.z);
    u.w = fmaf(w[k].w, xv.w, u.w);
  }
  return u;
}

template <typename IO, int W, bool ACT>
__global__ void __launch_bounds__(kConvThreads) kla_conv_kernel(const ConvArgs a) {
  const ConvLane l = conv_lane(a);
  if (!l.active) return;
  const long long bh = blockIdx.x;
  const int h = (int)(bh % a.H);
  const int T = a.T, D = a.D;
  float4 w[W], bias;
  load_taps<W>(a, h, l.d0, w, bias);
  const IO* __restrict__ x = reinterpret_cast<const IO*>(a.x) + bh * (long long)T * D + l.d0;
  IO* __restrict__ y = reinterpret_cast<IO*>(a.y) + bh * (long long)T * D + l.d0;
  const IO* win = a.win ? reinterpret_cast<const IO*>(a.win) + bh * (long long)(W - 1) * D + l.d0 : nullptr;

  // Walk tokens tau = t0 − (W−1) + m, m ∈ [0, M): the first W−1 only fill the
  // ring; token m sits in slot m mod W.
  float4 xr[W];
  const long long base = l.t0 - (W - 1);
  const int M = (int)(l.t1 - l.t0) + W - 1;
#pragma unroll 2
  for (int mb = 0; mb < M; mb += W) {
#pragma unroll
    for (int s = 0; s < W; ++s) {
      const int m = mb + s;
      if (m < M) {
        const long long tau = base + m;
        xr[s] = input_at<IO, W>(x, win, tau, T, D);
        if (m >= W - 1) {
          float4 u = preact<W>(w, bias, xr, s);
          if (ACT) {
            u.x *= sigmoid_fast(u.x);
            u.y *= sigmoid_fast(u.y);
            u.z *= sigmoid_fast(u.z);
            u.w *= sigmoid_fast(u.w);
          }
          store4ch(y + tau * D, u);
        }
      }
    }
  }

  // The window after the last token, written by chunk 0's thread: the last
  // W−1 inputs of (window, x). All are read before any is written, so the
  // window out may be the window in.
  if (W > 1 && l.chunk == 0 && a.wout) {
    IO* wout = reinterpret_cast<IO*>(a.wout) + bh * (long long)(W - 1) * D + l.d0;
    float4 keep[W > 1 ? W - 1 : 1];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) keep[j] = input_at<IO, W>(x, win, (long long)T - (W - 1) + j, T, D);
#pragma unroll
    for (int j = 0; j < W - 1; ++j) store4ch(wout + (long long)j * D, keep[j]);
  }
}

template <typename IO, int W, bool ACT>
__global__ void __launch_bounds__(kConvThreads) kla_conv_bwd_kernel(const ConvArgs a) {
  extern __shared__ float4 red[];  // [chunks_per_block][G][W + 1] per-thread partial sums
  const ConvLane l = conv_lane(a);
  const long long bh = blockIdx.x;
  const int h = (int)(bh % a.H);
  const int T = a.T, D = a.D, G = D >> 2;
  const int c = (int)threadIdx.x / G;
  float4 gw[W], gb = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < W; ++k) gw[k] = make_float4(0.f, 0.f, 0.f, 0.f);

  if (l.active) {
    float4 w[W], bias;
    load_taps<W>(a, h, l.d0, w, bias);
    const long long off = bh * (long long)T * D + l.d0;
    const IO* __restrict__ x = reinterpret_cast<const IO*>(a.x) + off;
    const IO* __restrict__ gy = a.gy ? reinterpret_cast<const IO*>(a.gy) + off : nullptr;  // null: zero
    IO* __restrict__ gx = reinterpret_cast<IO*>(a.gx) + off;
    const long long woff = bh * (long long)(W - 1) * D + l.d0;
    const IO* win = a.win ? reinterpret_cast<const IO*>(a.win) + woff : nullptr;
    const IO* gwo = a.gwout ? reinterpret_cast<const IO*>(a.gwout) + woff : nullptr;
    IO* gwin = a.gwin ? reinterpret_cast<IO*>(a.gwin) + woff : nullptr;

    // Walk tau = t0 − (W−1) + m, m ∈ [0, M), M = L + 2(W−1): gu is formed for
    // tokens in [t0, min(t1 + W − 1, T)), and gx of token tau − (W−1) is
    // complete once gu of tau is. Chunk 0 also emits tokens −(W−1)…−1 (the
    // gradient of the window in).
    float4 xr[W], gr[W];
    const long long base = l.t0 - (W - 1);
    const long long emit_lo = l.chunk == 0 ? -(long long)(W - 1) : l.t0;
    const long long tail = (long long)T - (W - 1);  // first input copied into the window out
    const int M = (int)(l.t1 - l.t0) + 2 * (W - 1);
#pragma unroll 2
    for (int mb = 0; mb < M; mb += W) {
#pragma unroll
      for (int s = 0; s < W; ++s) {
        const int m = mb + s;
        if (m < M) {
          const long long tau = base + m;
          xr[s] = input_at<IO, W>(x, win, tau, T, D);
          float4 gu = make_float4(0.f, 0.f, 0.f, 0.f);
          if (tau >= l.t0 && tau < T) {
            const float4 u = preact<W>(w, bias, xr, s);
            if (gy) gu = load4ch(gy + tau * D);
            if (ACT) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float ue = f4get(u, e), sg = sigmoid_fast(ue);
                f4set(gu, e, f4get(gu, e) * (sg * fmaf(ue, 1.0f - sg, 1.0f)));
              }
            }
            if (tau < l.t1) {
              gb.x += gu.x; gb.y += gu.y; gb.z += gu.z; gb.w += gu.w;
#pragma unroll
              for (int k = 0; k < W; ++k) {
                const float4 xv = xr[(s + 1 + k) % W];
                gw[k].x = fmaf(gu.x, xv.x, gw[k].x);
                gw[k].y = fmaf(gu.y, xv.y, gw[k].y);
                gw[k].z = fmaf(gu.z, xv.z, gw[k].z);
                gw[k].w = fmaf(gu.w, xv.w, gw[k].w);
              }
            }
          }
          gr[s] = gu;
          const long long te = tau - (W - 1);  // the token whose gx is now complete
          if (te >= emit_lo && te < l.t1) {
            float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
            if (gwo && te >= tail) g = load4ch(gwo + (te - tail) * D);
#pragma unroll
            for (int k = 0; k < W; ++k) {
              const float4 gv = gr[(s - k + W) % W];  // gu of token tau − k
              g.x = fmaf(w[k].x, gv.x, g.x);
              g.y = fmaf(w[k].y, gv.y, g.y);
              g.z = fmaf(w[k].z, gv.z, g.z);
              g.w = fmaf(w[k].w, gv.w, g.w);
            }
            if (te >= 0) store4ch(gx + te * D, g);
            else if (gwin) store4ch(gwin + (te + W - 1) * D, g);
          }
        }
      }
    }
  }

  if (!a.part) return;  // no weight or bias gradient wanted
  // Block partial: threads of the same channel group summed in chunk order.
  const int cpb = a.chunks_per_block;
  if (c < cpb) {
    float4* r = red + ((size_t)c * G + l.g) * (W + 1);
#pragma unroll
    for (int k = 0; k < W; ++k) r[k] = gw[k];
    r[W] = gb;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * (W + 1); i += blockDim.x) {
    const int g = i / (W + 1), k = i - g * (W + 1);
    float4 s = red[(size_t)g * (W + 1) + k];
    for (int cc = 1; cc < cpb; ++cc) {
      const float4 v = red[((size_t)cc * G + g) * (W + 1) + k];
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    // partials [H][P][D][W + 1], P = B · gridDim.y, p = b · gridDim.y + blockIdx.y
    const long long b = bh / a.H;
    const long long p = b * gridDim.y + blockIdx.y;
    float* dst = a.part + (((size_t)h * a.nparts + p) * D + 4 * g) * (W + 1) + k;
    dst[0] = s.x;
    dst[W + 1] = s.y;
    dst[2 * (W + 1)] = s.z;
    dst[3 * (W + 1)] = s.w;
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

template <typename IO, int W>
cudaError_t launch_w(const ConvArgs& a, bool backward, dim3 grid, size_t smem, cudaStream_t s) {
  if (backward) {
    if (a.act) kla_conv_bwd_kernel<IO, W, true><<<grid, kConvThreads, smem, s>>>(a);
    else kla_conv_bwd_kernel<IO, W, false><<<grid, kConvThreads, smem, s>>>(a);
  } else {
    if (a.act) kla_conv_kernel<IO, W, true><<<grid, kConvThreads, 0, s>>>(a);
    else kla_conv_kernel<IO, W, false><<<grid, kConvThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_io(const ConvArgs& a, bool backward, dim3 grid, size_t smem, cudaStream_t s) {
  switch (a.W) {
    case 1: return launch_w<IO, 1>(a, backward, grid, smem, s);
    case 2: return launch_w<IO, 2>(a, backward, grid, smem, s);
    case 3: return launch_w<IO, 3>(a, backward, grid, smem, s);
    case 4: return launch_w<IO, 4>(a, backward, grid, smem, s);
    case 5: return launch_w<IO, 5>(a, backward, grid, smem, s);
    case 6: return launch_w<IO, 6>(a, backward, grid, smem, s);
    case 7: return launch_w<IO, 7>(a, backward, grid, smem, s);
    case 8: return launch_w<IO, 8>(a, backward, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

ConvPlan conv_plan(long long bh, int T, int D, int W, int num_sms) {
  ConvPlan p{};
  const int G = D / 4;
  p.chunks_per_block = kConvThreads / G;
  p.threads = kConvThreads;
  // Shortest chunk (≥ 16 tokens, a power of two) that keeps the grid within
  // about four blocks per SM — one wave at the kernels' occupancy — so the
  // recomputed W−1 inputs at each chunk start stay a small share.
  auto blocks_y = [&](long long L) {
    const long long chunks = T > 0 ? (T + L - 1) / L : 1;
    return (chunks + p.chunks_per_block - 1) / p.chunks_per_block;
  };
  long long L = 16;
  while (L < (1 << 20) && (bh * blocks_y(L) > 4LL * num_sms || blocks_y(L) > 65535)) L *= 2;
  p.L = (int)L;
  p.blocks_y = (int)blocks_y(L);
  p.nparts = 0;  // set per batch count by the caller: B · blocks_y
  p.smem_bwd = (size_t)p.chunks_per_block * G * (W + 1) * sizeof(float4);
  return p;
}

size_t conv_partial_bytes(int B, int H, int D, int W, const ConvPlan& p) {
  return (size_t)H * B * p.blocks_y * D * (W + 1) * sizeof(float);
}

cudaError_t launch_conv(const ConvArgs& a, const ConvPlan& p, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  if (bh == 0) return cudaSuccess;
  const dim3 grid((unsigned)bh, (unsigned)p.blocks_y);
  return a.io == IO_BF16 ? launch_io<__nv_bfloat16>(a, false, grid, 0, s) : launch_io<float>(a, false, grid, 0, s);
}

cudaError_t launch_conv_backward(const ConvArgs& a, const ConvPlan& p, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  if (bh > 0) {
    const dim3 grid((unsigned)bh, (unsigned)p.blocks_y);
    const cudaError_t e = a.io == IO_BF16 ? launch_io<__nv_bfloat16>(a, true, grid, p.smem_bwd, s)
                                          : launch_io<float>(a, true, grid, p.smem_bwd, s);
    if (e != cudaSuccess) return e;
  }
  if (a.H > 0 && (a.gweight || a.gbias)) {
    const long long n = (long long)a.H * a.D * (a.W + 1);
    const int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
    kla_conv_bwd_finish_kernel<<<blocks, 256, 0, s>>>(a, a.W);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace kla
