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
//  1. The forward scan kernel (sequential plan, no y) stores the scaled state
//     (P̃ = K·P, μ) of every element before every 16-token tile and at the
//     end into the workspace (kla_scan_kernel.cuh).
//  2. kla_bwd_kernel walks the chunks from last to first, each in sub-chunks
//     of kSub tokens from its end: it re-runs the forward from the chunk's
//     checkpoint to the sub-chunk, keeps the states before the sub-chunk's
//     tokens in shared memory, and runs the adjoint recursion back over them
//     (forward work per token: 2.25 steps besides the adjoint's own, no state
//     traffic to device memory).
//  3. kla_bwd_finish_kernel (only when a head's columns are split over
//     several blocks) adds the per-row partial sums of the blocks.
//
// Layout of a block: (head, column block of cc columns, all d_k rows). A lane
// owns one row and CPL = 8 (or, for few heads, 4 or 2) consecutive columns (fp32x2
// pairs), so every
// per-row sum (dq, dk, da, dp̄) is first a sum inside the lane; a warp covers
// RW = min(32, d_k) rows and 32/RW column groups; per-column sums (dv, dΛ^v)
// over the warp's rows are a butterfly reduce-scatter across its lanes. Sums
// across warps go through shared-memory atomics (their order is not fixed,
// so the last bits of those sums can differ from run to run).
#include <algorithm>

#include <cuda_runtime.h>

#include "kla_device.cuh"
#include "kla_launch.h"

namespace kla {
namespace {

constexpr int kChunk = 16;  // tokens per checkpoint interval and per staged tile
constexpr int kCpl = 8;     // columns per lane (4 or 2 when a block of 8 would have few warps)
constexpr int kSub = 4;     // tokens per reverse sub-chunk (states kept in shared memory)
static_assert(kChunk == kScanTile, "the forward scan checkpoints once per tile");

struct BwdParams {
  const void *q, *k, *v, *lam_v, *a, *pbar;
  const float *lam0, *eta0;
  const void* dy;
  const float *dlamT, *detaT;
  void *gq, *gk, *gv, *glam_v, *ga, *gpbar;  // per-token gradients (io dtype)
  float *dlam0, *deta0;
  float* ckpt;     // [nchunks + 1][2][elems]: (P, μ) at each chunk start, then at T
  float* rowpart;  // [B·H·T·d_k][4] fp32 per-row sums (dq, dk, da, dp̄) when ncb > 1, else null
  int T, dk, dv, cc, ncb, nchunks;
  int gates;        // kla_gate bits: a, p̄, Λ^v inputs are pre-activations
  long long elems;  // B·H·d_k·d_v
};

template <int DK, int CPL>
struct BwdGeo {
  static constexpr int RW = DK < 32 ? DK : 32;  // rows per warp
  static constexpr int CG = 32 / RW;            // column groups per warp
  static constexpr int WCOLS = CG * CPL;        // columns per warp
  static constexpr int NWR = DK / RW;           // warps along rows
};

// Shared memory of one block (fp32): staged per-row inputs (a, k, p̄, q)
// interleaved per (token, row) [kChunk][DK][4] (one 128-bit load gives a
// lane its row's four) and per-column inputs v, Λ^v, Λ^v·v, dy [kChunk][cc], the
// per-token accumulators of the row sums [kChunk][4][DK] and column sums
// [kChunk][2][cc], and each thread's states before the tokens of the current
// sub-chunk, [kSub][2][cpl/2][threads] fp32x2 (thread-fastest, so a warp's
// accesses are contiguous).
struct BwdSmem {
  float *rw, *v, *L, *Lv, *dy, *racc, *cacc, *st;
  unsigned char* raw;  // the next chunk's inputs as loaded (I/O dtype), filled by cp.async
  __device__ BwdSmem(float* base, int dk, int cc, int cpl) {
    rw = base;
    v = rw + 4 * kChunk * dk;
    L = v + kChunk * cc;
    Lv = L + kChunk * cc;
    dy = Lv + kChunk * cc;
    racc = dy + kChunk * cc;
    cacc = racc + kChunk * 4 * dk;
    st = cacc + kChunk * 2 * cc;
    raw = reinterpret_cast<unsigned char*>(st + kSub * 2 * cpl * (int)blockDim.x);
  }
  __host__ __device__ static size_t bytes(int dk, int cc, int threads, int cpl) {
    return sizeof(float) * ((size_t)kChunk * (4 * dk + 4 * cc) + (size_t)kChunk * 4 * dk + (size_t)kChunk * 2 * cc +
                            (size_t)kSub * 2 * cpl * threads + (size_t)kChunk * (4 * dk + 3 * cc));
  }
};

// UG consecutive column pairs (fp32x2) from 8·UG-byte aligned memory: one
// 128-bit load for two pairs, one 64-bit load for one.
template <int UG>
__device__ __forceinline__ void ld_pairs(const float* src, f2 (&out)[UG]) {
  if constexpr (UG == 2) {
    const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(src);
    out[0] = v.x;
    out[1] = v.y;
  } else {
    out[0] = *reinterpret_cast<const unsigned long long*>(src);
  }
}

template <typename IO>
__device__ __forceinline__ float ld(const void* base, size_t idx) {
  return to_f32<IO>(reinterpret_cast<const IO*>(base)[idx]);
}

// Queue 16-byte asynchronous copies of tokens [t0, t0 + tl) of the block's
// inputs (q, k, a, p̄ rows; v, Λ^v, dy columns) into s.raw, as stored.
template <typename IO>
__device__ void issue_raw(const BwdParams& p, const BwdSmem& s, long long bh, int jb, int t0, int tl) {
  const int nthr = blockDim.x;
  const size_t rowb = (size_t)kChunk * p.dk * sizeof(IO), colb = (size_t)kChunk * p.cc * sizeof(IO);
  const int rchunks = (int)((size_t)tl * p.dk * sizeof(IO) / 16);
  const size_t rsrc = ((size_t)bh * p.T + t0) * p.dk * sizeof(IO);
  const void* rows[4] = {p.q, p.k, p.a, p.pbar};
#pragma unroll
  for (int arr = 0; arr < 4; ++arr)
    for (int c = threadIdx.x; c < rchunks; c += nthr)
      cp_async16(s.raw + arr * rowb + (size_t)c * 16, static_cast<const char*>(rows[arr]) + rsrc + (size_t)c * 16);
  const int cpr = (int)(p.cc * sizeof(IO) / 16);  // 16-byte pieces per token row (a power of two)
  const int lcpr = __ffs(cpr) - 1;
  const size_t csrc = (((size_t)bh * p.T + t0) * p.dv + jb) * sizeof(IO), cstride = (size_t)p.dv * sizeof(IO);
  const void* cols[3] = {p.v, p.lam_v, p.dy};
  for (int arr = 0; arr < (p.dy ? 3 : 2); ++arr)
    for (int c = threadIdx.x; c < tl * cpr; c += nthr) {
      const int t = c >> lcpr, piece = c & (cpr - 1);
      cp_async16(s.raw + 4 * rowb + arr * colb + (size_t)c * 16,
                 static_cast<const char*>(cols[arr]) + csrc + t * cstride + (size_t)piece * 16);
    }
}

// Widen the staged chunk to fp32 (gates applied, Λ^v·v formed) and clear the
// chunk's sum accumulators.
template <typename IO>
__device__ void convert_raw(const BwdParams& p, const BwdSmem& s, int tl) {
  const int nthr = blockDim.x;
  const IO* r = reinterpret_cast<const IO*>(s.raw);
  const IO *rq = r, *rk = r + kChunk * p.dk, *ra = rk + kChunk * p.dk, *rp = ra + kChunk * p.dk;
  const IO *rv = rp + kChunk * p.dk, *rL = rv + kChunk * p.cc, *rg = rL + kChunk * p.cc;
  for (int x = threadIdx.x; x < tl * p.dk; x += nthr) {
    const float xa = to_f32<IO>(ra[x]);
    *reinterpret_cast<float4*>(s.rw + 4 * x) =
        make_float4(gate_a(xa, p.gates), to_f32<IO>(rk[x]), gate_pbar(to_f32<IO>(rp[x]), xa, p.gates),
                    to_f32<IO>(rq[x]));
  }
  for (int x = threadIdx.x; x < tl * p.cc; x += nthr) {
    s.v[x] = to_f32<IO>(rv[x]);
    s.L[x] = gate_lamv(to_f32<IO>(rL[x]), p.gates);
    s.Lv[x] = s.L[x] * s.v[x];
    s.dy[x] = p.dy ? to_f32<IO>(rg[x]) : 0.0f;
  }
  for (int x = threadIdx.x; x < kChunk * (4 * p.dk + 2 * p.cc); x += nthr) s.racc[x] = 0.0f;
}

// Lane geometry of the reverse kernel.
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

// Butterfly reduce-scatter of NV per-lane values over the RW lanes of a
// column group (lanes differing in their low log2(RW) bits). While a lane
// still holds more than one value, each round halves them (keeping one half,
// sending the other); after that the rounds add whole values. Afterwards v[0]
// holds the group sum of value `first`, and `owner` says whether this lane
// is the one of the lanes holding that same sum that should publish it.
template <int RW, int NV>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int lane, int& first, bool& owner) {
  first = 0;
  owner = true;
  int nv = NV;
#pragma unroll
  for (int m = RW / 2; m >= 1; m >>= 1) {
    if (nv > 1) {
      const int half = nv / 2;
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int u = 0; u < NV / 2; ++u) {
        if (u < half) {
          const float send = upper ? v[u] : v[u + half];
          const float keep = upper ? v[u + half] : v[u];
          v[u] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      if (upper) first += half;
      nv = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
      if (lane & m) owner = false;
    }
  }
}

// Pass 2: chunks from last to first. A chunk (kChunk tokens, staged in
// shared memory) is processed in sub-chunks of kSub tokens from its end: the
// state at the sub-chunk's start is recomputed from the chunk's checkpoint,
// the states before each of the sub-chunk's tokens are kept in registers,
// and the adjoint recursion runs back over them. Arithmetic is packed fp32x2
// over pairs of adjacent columns.

template <typename IO, int DK, int CPL>
__global__ void __launch_bounds__(512, 1) kla_bwd_kernel(const BwdParams p) {
  using G = BwdGeo<DK, CPL>;
  constexpr int NP = CPL / 2;            // column pairs per lane
  constexpr int UG = NP >= 2 ? 2 : 1;    // column pairs per shared- or global-memory load
  extern __shared__ __align__(16) float bwd_smem[];
  const BwdSmem s(bwd_smem, DK, p.cc, CPL);
  const long long bh = blockIdx.x;
  const int jb = blockIdx.y * p.cc;
  const BwdLane<DK, CPL> ln(p, bh, jb);
  const int lcc = __ffs(p.cc) - 1;  // cc is a power of two
  const int i = ln.i, jl = ln.jl;
  const f2 one2 = f2_make(1.0f, 1.0f), m1 = f2_make(-1.0f, -1.0f);

  auto load_pairs = [&](const float* src, f2 (&P)[NP], f2 (&M)[NP]) {
#pragma unroll
    for (int u = 0; u < NP; u += UG) {
      f2 pp[UG], mm[UG];
      ld_pairs<UG>(src + ln.e0 + 2 * u, pp);
      ld_pairs<UG>(src + p.elems + ln.e0 + 2 * u, mm);
#pragma unroll
      for (int x = 0; x < UG; ++x) {
        P[u + x] = pp[x];
        M[u + x] = mm[x];
      }
    }
  };
  // one forward token (staged token t) on the lane's column pairs
  auto fwd = [&](int t, f2 (&P)[NP], f2 (&M)[NP]) {
    const float4 r4 = *reinterpret_cast<const float4*>(s.rw + 4 * (t * DK + i));  // (a, k, p̄, q)
    const float at = r4.x, kt = r4.y;
    const f2 a1 = f2_make(at, at), a2 = f2_make(at * at, at * at), pb = f2_make(r4.z, r4.z);
    const f2 k1 = f2_make(kt, kt), k2 = f2_make(kt * kt, kt * kt);
#pragma unroll
    for (int u = 0; u < NP; u += UG) {
      f2 Ls[UG], Lvs[UG];
      ld_pairs<UG>(s.L + t * p.cc + jl + 2 * u, Ls);
      ld_pairs<UG>(s.Lv + t * p.cc + jl + 2 * u, Lvs);
#pragma unroll
      for (int x = 0; x < UG; ++x) {
        const f2 Pp = f2_fma(a2, P[u + x], pb);
        const f2 w = f2_rcp(f2_fma(f2_mul(k2, Ls[x]), Pp, one2));
        const f2 b = f2_mul(k1, Lvs[x]);
        const f2 uu = f2_fma(Pp, b, f2_mul(a1, M[u + x]));
        P[u + x] = f2_mul(w, Pp);
        M[u + x] = f2_mul(w, uu);
      }
    }
  };

  // The checkpoints hold the forward scan's scaled variance P̃ = K·P with
  // K = k² + 2^-40 of the token before (1 at the start).
  auto inv_scale = [&](int t) -> f2 {
    float K = 1.0f;
    if (t > 0) {
      const float kp = ld<IO>(p.k, ((size_t)bh * p.T + t - 1) * DK + i);
      K = fmaf(kp, kp, kK2Floor);
    }
    const float r = 1.0f / K;
    return f2_make(r, r);
  };
  auto load_state = [&](int idx, f2 rK, f2 (&P)[NP], f2 (&M)[NP]) {
    load_pairs(p.ckpt + (size_t)idx * 2 * p.elems, P, M);
#pragma unroll
    for (int u = 0; u < NP; ++u) P[u] = f2_mul(P[u], rK);
  };

  // terminal adjoints from dλ_T, dη_T through λ_T = 1/P_T, η_T = μ_T/P_T
  f2 Pb[NP], Mb[NP];
  {
    f2 PT[NP], MT[NP];
    if (p.nchunks > 0) {
      load_state(p.nchunks, inv_scale(p.T), PT, MT);
    } else {  // empty sequence: the final state is the initial one
#pragma unroll
      for (int u = 0; u < NP; ++u) {
        float pv[2], mv[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const size_t e = ln.e0 + 2 * u + h;
          pv[h] = p.lam0 ? 1.0f / p.lam0[e] : 1.0f;
          mv[h] = p.eta0 ? p.eta0[e] * pv[h] : 0.0f;
        }
        PT[u] = f2_make(pv[0], pv[1]);
        MT[u] = f2_make(mv[0], mv[1]);
      }
    }
#pragma unroll
    for (int u = 0; u < NP; ++u) {
      float pbv[2], mbv[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const size_t e = ln.e0 + 2 * u + h;
        const float dl = p.dlamT ? p.dlamT[e] : 0.0f, de = p.detaT ? p.detaT[e] : 0.0f;
        const float PTh = h ? f2_hi(PT[u]) : f2_lo(PT[u]), MTh = h ? f2_hi(MT[u]) : f2_lo(MT[u]);
        const float r = 1.0f / PTh;
        pbv[h] = -(dl + de * MTh) * r * r;
        mbv[h] = de * r;
      }
      Pb[u] = f2_make(pbv[0], pbv[1]);
      Mb[u] = f2_make(mbv[0], mbv[1]);
    }
  }

  auto chunk_len = [&](int c) { return min(kChunk, p.T - c * kChunk); };
  if (p.nchunks > 0) issue_raw<IO>(p, s, bh, jb, (p.nchunks - 1) * kChunk, chunk_len(p.nchunks - 1));
  cp_async_commit();
  for (int c = p.nchunks - 1; c >= 0; --c) {
    const int t0 = c * kChunk, tl = chunk_len(c);
    cp_async_wait<0>();
    __syncthreads();  // chunk c's inputs have landed; the previous chunk's staged data is no longer read
    convert_raw<IO>(p, s, tl);
    __syncthreads();  // staged; the raw buffer is free for the next chunk
    if (c > 0) issue_raw<IO>(p, s, bh, jb, t0 - kChunk, kChunk);
    cp_async_commit();
    const f2 rK = inv_scale(t0);
    for (int sb = (tl - 1) / kSub; sb >= 0; --sb) {
      const int ts = sb * kSub;
      f2 P[NP], M[NP];
      load_state(c, rK, P, M);
#pragma unroll 1
      for (int t = 0; t < ts; ++t) fwd(t, P, M);
      f2* st = reinterpret_cast<f2*>(s.st) + threadIdx.x;
      const int nthr = blockDim.x;
      auto Ps = [&](int r, int u) -> f2& { return st[((r * 2 + 0) * NP + u) * nthr]; };
      auto Ms = [&](int r, int u) -> f2& { return st[((r * 2 + 1) * NP + u) * nthr]; };
#pragma unroll
      for (int r = 0; r < kSub; ++r) {
#pragma unroll
        for (int u = 0; u < NP; ++u) {
          Ps(r, u) = P[u];
          Ms(r, u) = M[u];
        }
        if (r + 1 < kSub && ts + r < tl) fwd(ts + r, P, M);
      }
#pragma unroll
      for (int r = kSub - 1; r >= 0; --r) {
        const int t = ts + r;
        if (t >= tl) continue;
        const float4 r4 = *reinterpret_cast<const float4*>(s.rw + 4 * (t * DK + i));  // (a, k, p̄, q)
        const float at = r4.x, kt = r4.y, pt = r4.z, qt = r4.w;
        const f2 a1 = f2_make(at, at), a2 = f2_make(at * at, at * at), pb = f2_make(pt, pt);
        const f2 k1 = f2_make(kt, kt), k2 = f2_make(kt * kt, kt * kt), q1 = f2_make(qt, qt);
        const f2 nk2 = f2_make(-kt * kt, -kt * kt);
        const f2 zero = f2_make(0.0f, 0.0f);
        f2 rq = zero, rda1 = zero, rda2 = zero, rdp = zero, rdk1n = zero, rdk2 = zero;
        float cv[2 * CPL];  // per column: k²c̄, then k·b̄
#pragma unroll
        for (int u = 0; u < NP; u += UG) {
          f2 Ls[UG], Lvs[UG], gs[UG];
          ld_pairs<UG>(s.L + t * p.cc + jl + 2 * u, Ls);
          ld_pairs<UG>(s.Lv + t * p.cc + jl + 2 * u, Lvs);
          ld_pairs<UG>(s.dy + t * p.cc + jl + 2 * u, gs);
#pragma unroll
          for (int x = 0; x < UG; ++x) {
            const int uu2 = u + x;
            const f2 P0 = Ps(r, uu2), M0 = Ms(r, uu2);
            const f2 Pp = f2_fma(a2, P0, pb);
            const f2 cobs = f2_mul(k2, Ls[x]);
            const f2 w = f2_rcp(f2_fma(cobs, Pp, one2));
            const f2 b = f2_mul(k1, Lvs[x]);
            const f2 uu = f2_fma(Pp, b, f2_mul(a1, M0));
            const f2 mu_t = f2_mul(w, uu);
            const f2 mb = f2_fma(q1, gs[x], Mb[uu2]);
            rq = f2_fma(gs[x], mu_t, rq);
            const f2 ub = f2_mul(mb, w);
            // With 1 − cP⁻w = w and μ̄w = ū, uw = μ':
            //   P̄⁻ = P̄w + ūb − w̄cw² = P̄w² + ū(b − cμ'),
            //   −c̄ = w̄P⁻w² = P⁻(ūμ' + P̄w²P⁻).
            const f2 Pbw2 = f2_mul(Pb[uu2], f2_mul(w, w));
            const f2 Ppb = f2_fma(ub, f2_fma(f2_mul(cobs, mu_t), m1, b), Pbw2);
            const f2 cbn = f2_mul(Pp, f2_fma(Pbw2, Pp, f2_mul(ub, mu_t)));
            const f2 bb = f2_mul(ub, Pp);
            rda1 = f2_fma(ub, M0, rda1);
            rda2 = f2_fma(P0, Ppb, rda2);
            rdp = f2_add(rdp, Ppb);
            rdk1n = f2_fma(Ls[x], cbn, rdk1n);
            rdk2 = f2_fma(Lvs[x], bb, rdk2);
            // dΛ^v_j = Σ_i k²c̄ + v_j Σ_i k b̄ and dv_j = Λ^v_j Σ_i k b̄: per element
            // only −k²·(−c̄) and k·b̄ are summed over the rows.
            const f2 xl = f2_mul(nk2, cbn);
            const f2 zl = f2_mul(k1, bb);
            cv[2 * uu2] = f2_lo(xl);
            cv[2 * uu2 + 1] = f2_hi(xl);
            cv[CPL + 2 * uu2] = f2_lo(zl);
            cv[CPL + 2 * uu2 + 1] = f2_hi(zl);
            Pb[uu2] = f2_mul(a2, Ppb);
            Mb[uu2] = f2_mul(a1, ub);
          }
        }
        float* racc = s.racc + t * 4 * DK + i;
        atomicAdd(racc + 0 * DK, f2_lo(rq) + f2_hi(rq));
        atomicAdd(racc + 1 * DK, fmaf(-2.0f * kt, f2_lo(rdk1n) + f2_hi(rdk1n), f2_lo(rdk2) + f2_hi(rdk2)));
        atomicAdd(racc + 2 * DK, fmaf(2.0f * at, f2_lo(rda2) + f2_hi(rda2), f2_lo(rda1) + f2_hi(rda1)));
        atomicAdd(racc + 3 * DK, f2_lo(rdp) + f2_hi(rdp));
        int first;
        bool owner;
        reduce_scatter<G::RW, 2 * CPL>(cv, ln.lane, first, owner);
        constexpr int KEEP = (2 * CPL) / G::RW > 0 ? (2 * CPL) / G::RW : 1;
#pragma unroll
        for (int rr = 0; rr < KEEP; ++rr) {
          const int idx = first + rr;
          if (owner) atomicAdd(s.cacc + (t * 2 + idx / CPL) * p.cc + jl + idx % CPL, cv[rr]);
        }
      }
    }
    __syncthreads();
    // this chunk's gradients
    for (int x = threadIdx.x; x < tl * DK; x += blockDim.x) {
      const int t = x / DK, r = x - t * DK;
      const size_t g = ((size_t)bh * p.T + t0 + t) * DK + r;
      const float* acc = s.racc + t * 4 * DK + r;
      if (p.ncb == 1) {
        float gxa = acc[2 * DK], gxp = acc[3 * DK];
        if (p.gates) gate_chain_row(acc[2 * DK], acc[3 * DK], ld<IO>(p.a, g), ld<IO>(p.pbar, g), p.gates, gxa, gxp);
        reinterpret_cast<IO*>(p.gq)[g] = from_f32<IO>(acc[0]);
        reinterpret_cast<IO*>(p.gk)[g] = from_f32<IO>(acc[DK]);
        reinterpret_cast<IO*>(p.ga)[g] = from_f32<IO>(gxa);
        reinterpret_cast<IO*>(p.gpbar)[g] = from_f32<IO>(gxp);
      } else {  // other column blocks add to the same rows: accumulate in fp32
        atomicAdd(reinterpret_cast<float4*>(p.rowpart) + g, make_float4(acc[0], acc[DK], acc[2 * DK], acc[3 * DK]));
      }
    }
    for (int x = threadIdx.x; x < tl * p.cc; x += blockDim.x) {
      const int t = x >> lcc, j = x & (p.cc - 1);
      const size_t g = ((size_t)bh * p.T + t0 + t) * p.dv + jb + j;
      const float sz = s.cacc[(t * 2 + 1) * p.cc + j];  // Σ_i k b̄
      const float gL = fmaf(s.v[t * p.cc + j], sz, s.cacc[(t * 2) * p.cc + j]);
      reinterpret_cast<IO*>(p.glam_v)[g] = from_f32<IO>(p.gates ? gate_chain_lamv(gL, ld<IO>(p.lam_v, g), p.gates) : gL);
      reinterpret_cast<IO*>(p.gv)[g] = from_f32<IO>(s.L[t * p.cc + j] * sz);
    }
  }
  // initial-state gradients through P0 = 1/λ0, μ0 = η0/λ0
  if (p.dlam0) {
#pragma unroll
    for (int u = 0; u < NP; ++u) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const size_t e = ln.e0 + 2 * u + h;
        const float l0 = p.lam0 ? p.lam0[e] : 1.0f, n0 = p.eta0 ? p.eta0[e] : 0.0f;
        const float pbv = h ? f2_hi(Pb[u]) : f2_lo(Pb[u]), mbv = h ? f2_hi(Mb[u]) : f2_lo(Mb[u]);
        const float r = 1.0f / l0;
        p.dlam0[e] = -(pbv + mbv * n0) * r * r;
        p.deta0[e] = mbv * r;
      }
    }
  }
}

// Pass 3 (ncb > 1): convert the accumulated per-row sums to the I/O dtype.
template <typename IO>
__global__ void kla_bwd_finish_kernel(const BwdParams p, size_t BHTdk) {
  for (size_t g = blockIdx.x * (size_t)blockDim.x + threadIdx.x; g < BHTdk; g += (size_t)gridDim.x * blockDim.x) {
    const float4 acc = reinterpret_cast<const float4*>(p.rowpart)[g];
    float gxa = acc.z, gxp = acc.w;
    if (p.gates) gate_chain_row(acc.z, acc.w, ld<IO>(p.a, g), ld<IO>(p.pbar, g), p.gates, gxa, gxp);
    reinterpret_cast<IO*>(p.gq)[g] = from_f32<IO>(acc.x);
    reinterpret_cast<IO*>(p.gk)[g] = from_f32<IO>(acc.y);
    reinterpret_cast<IO*>(p.ga)[g] = from_f32<IO>(gxa);
    reinterpret_cast<IO*>(p.gpbar)[g] = from_f32<IO>(gxp);
  }
}

template <typename IO, int DK, int CPL>
cudaError_t launch_bwd_typed(const BwdParams& bp, dim3 grid, int threads, size_t smem, cudaStream_t s) {
  auto bw = kla_bwd_kernel<IO, DK, CPL>;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(bw, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const size_t BHTdk = (size_t)grid.x * bp.T * DK;
  if (bp.ncb > 1 && BHTdk > 0) {
    const cudaError_t e = cudaMemsetAsync(bp.rowpart, 0, BHTdk * 4 * sizeof(float), s);
    if (e != cudaSuccess) return e;
  }
  bw<<<grid, threads, smem, s>>>(bp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || bp.ncb == 1 || BHTdk == 0) return e;
  const unsigned blocks = (unsigned)std::min<size_t>((BHTdk + 255) / 256, 4096);
  kla_bwd_finish_kernel<IO><<<blocks, 256, 0, s>>>(bp, BHTdk);
  return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_bwd_io(int dk, int cpl, const BwdParams& bp, dim3 grid, int threads, size_t smem, cudaStream_t s) {
  switch (dk * 16 + cpl) {
    case 16 * 16 + 8: return launch_bwd_typed<IO, 16, 8>(bp, grid, threads, smem, s);
    case 32 * 16 + 8: return launch_bwd_typed<IO, 32, 8>(bp, grid, threads, smem, s);
    case 64 * 16 + 8: return launch_bwd_typed<IO, 64, 8>(bp, grid, threads, smem, s);
    case 128 * 16 + 8: return launch_bwd_typed<IO, 128, 8>(bp, grid, threads, smem, s);
    case 16 * 16 + 4: return launch_bwd_typed<IO, 16, 4>(bp, grid, threads, smem, s);
    case 32 * 16 + 4: return launch_bwd_typed<IO, 32, 4>(bp, grid, threads, smem, s);
    case 64 * 16 + 4: return launch_bwd_typed<IO, 64, 4>(bp, grid, threads, smem, s);
    case 128 * 16 + 4: return launch_bwd_typed<IO, 128, 4>(bp, grid, threads, smem, s);
    case 16 * 16 + 2: return launch_bwd_typed<IO, 16, 2>(bp, grid, threads, smem, s);
    case 32 * 16 + 2: return launch_bwd_typed<IO, 32, 2>(bp, grid, threads, smem, s);
    case 64 * 16 + 2: return launch_bwd_typed<IO, 64, 2>(bp, grid, threads, smem, s);
    case 128 * 16 + 2: return launch_bwd_typed<IO, 128, 2>(bp, grid, threads, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

BwdPlan backward_plan(long long bh, int T, int dk, int dv, int num_sms) {
  constexpr int kMaxWarps = 16;  // 512 threads at the reverse kernel's register budget
  constexpr size_t kMaxSmem = 220 * 1024;
  const int rw = dk < 32 ? dk : 32, nwr = dk / rw;
  // Column block and threads for `cpl` columns per lane.
  auto geometry = [&](int cpl) {
    BwdPlan b{};
    b.cpl = cpl;
    const int wcols = (32 / rw) * cpl;
    int cc = dv;
    while (cc > wcols &&
           (nwr * (cc / wcols) > kMaxWarps || BwdSmem::bytes(dk, cc, 32 * nwr * (cc / wcols), cpl) > kMaxSmem))
      cc /= 2;
    // Few heads: narrower column blocks, so that at least half the SMs get a
    // block (a block of up to 16 warps keeps an SM busy on its own).
    while (cc > wcols && 2 * bh * (dv / cc) < num_sms) cc /= 2;
    b.cc = cc;
    b.threads = 32 * nwr * (cc / wcols);
    b.smem = BwdSmem::bytes(dk, cc, b.threads, cpl);
    return b;
  };
  // Warps an SM holds at once: blocks per SM (as many as there are per SM,
  // within the shared-memory, thread and register limits) × warps per block.
  auto resident_warps = [&](const BwdPlan& b) {
    const long long blocks = bh * (dv / b.cc);
    const long long per_sm = (blocks + num_sms - 1) / num_sms;
    const long long by_smem = (long long)((228 * 1024) / (b.smem + 1024));
    const long long by_threads = 2048 / b.threads, by_regs = 65536 / (128LL * b.threads);
    const long long r = std::max(1LL, std::min(std::min(per_sm, by_smem), std::min(by_threads, by_regs)));
    return r * (b.threads / 32);
  };
  // Eight columns per lane amortise the per-row work best; four (then two)
  // columns double the warps of a block, which pays when eight would leave
  // the SMs with few warps to hide latency with (few heads).
  BwdPlan b = geometry(kCpl);
  for (int cpl = kCpl / 2; cpl >= 2 && resident_warps(b) < kMaxWarps; cpl /= 2) {
    const BwdPlan n = geometry(cpl);
    // (a staged column row must be at least 16 bytes in bf16: 8 columns)
    if (n.cc < 8 || resident_warps(n) <= resident_warps(b)) break;
    b = n;
  }
  b.ncb = dv / b.cc;
  b.nchunks = (T + kChunk - 1) / kChunk;
  const long long elems = bh * dk * dv;
  b.ckpt_bytes = (size_t)(b.nchunks + 1) * 2 * (size_t)elems * sizeof(float);
  b.rowpart_bytes = b.ncb > 1 ? (size_t)4 * (size_t)bh * T * dk * sizeof(float) : 0;
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
  bp.gates = f.gates;
  const dim3 grid((unsigned)bh, (unsigned)b.ncb);
  return f.io == IO_BF16 ? launch_bwd_io<__nv_bfloat16>(f.dk, b.cpl, bp, grid, b.threads, b.smem, s)
                         : launch_bwd_io<float>(f.dk, b.cpl, bp, grid, b.threads, b.smem, s);
}

}  // namespace kla
