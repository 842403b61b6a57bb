// KLA scan kernels for sm_103a: the sequential / chunk-apply scan, the
// chunk-map composition and the cross-chunk carry.
//
// The operation is the diagonal information-form Kalman filter of
// "Technische Samenvatting: Kalman Linear Attention (KLA)"
// (gist.science/nl/paper/2602.10743), Methodologie §1 (OU prior, observation
// through k with value precision Λ^v, posterior-mean readout through q) and
// §2 (Möbius precision recursion, associative composition, affine mean).
//
// ---------------------------------------------------------------------------
// Arithmetic of the scan (per element (i, j), token t; c = k²Λ^v, b = kΛ^v v)
//
// The filter is run in variance form, P = 1/λ and μ = η/λ, which needs one
// reciprocal per element-step instead of the two of the printed information
// form. The state is carried with a per-row scale so that the recurrence
// costs 7 fp32 operations and one hardware reciprocal per element-step:
//
//   K_t = k_t² + 2^-40 (per row), P̃ = K_{t-1}·P (K_{-1} := 1 at a chunk start)
//   ŝ  = A_t·P̃ + B_t          A_t = K_t a_t / K_{t-1},  B_t = K_t p̄_t / a_t
//   d  = ŝ·Λ^v_j + 1/a_t       (= (1 + c·s)/a with s = a²P + p̄ the predicted variance)
//   w̃  = 1/d                   (= a·w, w the Kalman weight 1/(1 + c s))
//   P̃  = ŝ·w̃                   (= K_t·P_t)
//   m  = (ŝ·Λ^v_j v_j)·(k_t/K_t) + μ
//   μ  = m·w̃                   (= w·(aμ + s·b), the posterior mean)
//   y_j += q_t·μ
//
// The per-row coefficients A, B, 1/a, k/K, q are computed once per (t, i) in
// shared memory and reused by all d_v columns of the block; Λ^v and Λ^v·v are
// computed once per (t, j). Only K_t and 1/a are floors-guarded (2^-40), so
// all scaled quantities stay normal fp32 numbers.
//
// Layout of work: a thread block owns one head (grid.x), a block of CC
// columns (grid.y) and one chunk of tokens (grid.z). A lane owns RL rows × 2
// columns; rows are paired so that every operation above is one packed
// fp32x2 instruction for two rows. A warp covers all d_k rows of WC columns.
// Tokens stream through shared memory in tiles of TC, staged one tile ahead
// with 16-byte asynchronous copies. The state stays in registers for the
// whole chunk and is never written per token.
// ---------------------------------------------------------------------------
#include <algorithm>

#include "kla_device.cuh"
#include "kla_launch.h"

namespace kla {

namespace {

constexpr int CL = 2;            // columns per lane
constexpr int kMaxThreads = 256;  // per block: leaves up to 255 registers per thread

template <int DK, int RL>
struct Geo {
  static constexpr int LANES_I = DK / RL;       // lanes along rows
  static constexpr int LANES_J = 32 / LANES_I;  // lanes along columns
  static constexpr int WC = LANES_J * CL;       // columns per warp
  static constexpr int NP = LANES_I / 2;        // partial sums per output after one exchange
  static_assert(LANES_I >= 2 && LANES_I <= 32 && RL % 4 == 0, "unsupported geometry");
};

struct KernelParams {
  const void *q, *k, *v, *lam_v, *a, *pbar;
  const float *lam0, *eta0;
  const float* starts;  // [S][2][elems] chunk-start (P, μ), or nullptr
  float* maps;          // compose output [S-1][7][elems]
  void* y;
  float *lamT, *etaT;
  int T, dv, chunk_len, cc, log2cc;
  long long elems;  // B·H·dk·dv
};

// Byte offsets inside the dynamic shared memory of one block.
template <typename IO, int DK, int TC>
struct Layout {
  int cc;
  __host__ __device__ explicit Layout(int cc_) : cc(cc_) {}
  __host__ __device__ size_t raw_i() const { return (size_t)TC * DK * sizeof(IO); }
  __host__ __device__ size_t raw_j() const { return (size_t)TC * cc * sizeof(IO); }
  __host__ __device__ size_t raw_buf() const { return 4 * raw_i() + 2 * raw_j(); }
  __host__ __device__ size_t coef() const { return 2 * raw_buf(); }
  __host__ __device__ size_t pj() const { return coef() + (size_t)TC * 5 * DK * sizeof(float); }
  __host__ __device__ size_t ypart() const { return pj() + (size_t)TC * cc * 4 * sizeof(float); }
  __host__ __device__ size_t kprev(int np) const { return ypart() + (size_t)TC * cc * np * sizeof(float); }
  __host__ __device__ size_t total(int np) const { return kprev(np) + 2 * DK * sizeof(float); }
};

// Queue the asynchronous copy of tokens [t0, t0 + tl) of this block's inputs
// into raw buffer `buf`: the four per-row arrays (contiguous tl × DK) and the
// two per-column arrays (tl rows of CC columns, row stride dv).
template <typename IO, int DK, int TC>
__device__ __forceinline__ void stage_tile(const KernelParams& p, unsigned char* buf, long long bh, int jb,
                                           int t0, int tl) {
  const Layout<IO, DK, TC> L(p.cc);
  const int tid = threadIdx.x, nthr = blockDim.x;
  const size_t row_i = (size_t)DK * sizeof(IO);
  const int chunks_i = (int)(tl * row_i / 16);
  const size_t base_i = ((size_t)bh * p.T + t0) * row_i;
#pragma unroll
  for (int arr = 0; arr < 4; ++arr) {
    const char* src = (const char*)(arr == 0 ? p.q : arr == 1 ? p.k : arr == 2 ? p.a : p.pbar) + base_i;
    unsigned char* dst = buf + arr * L.raw_i();
    for (int c = tid; c < chunks_i; c += nthr) cp_async16(dst + (size_t)c * 16, src + (size_t)c * 16);
  }
  const int cpr = (int)(p.cc * sizeof(IO) / 16);  // 16-byte chunks per staged row
  const int chunks_j = tl * cpr;
  const size_t row_j = (size_t)p.dv * sizeof(IO);
  const size_t base_j = ((size_t)bh * p.T + t0) * row_j + (size_t)jb * sizeof(IO);
#pragma unroll
  for (int arr = 0; arr < 2; ++arr) {
    const char* src = (const char*)(arr == 0 ? p.v : p.lam_v) + base_j;
    unsigned char* dst = buf + 4 * L.raw_i() + arr * L.raw_j();
    for (int c = tid; c < chunks_j; c += nthr) {
      const int row = c / cpr, col = c - row * cpr;
      cp_async16(dst + (size_t)c * 16, src + (size_t)row * row_j + (size_t)col * 16);
    }
  }
}

// Per-(t, j) column terms of a staged tile: (Λ^v, Λ^v, Λ^v·v, Λ^v·v), the
// duplicated pairs letting one packed instruction serve two rows.
template <typename IO, int DK, int TC>
__device__ __forceinline__ void column_terms(const KernelParams& p, const unsigned char* buf, float4* pj, int tl) {
  const Layout<IO, DK, TC> L(p.cc);
  const IO* rv = reinterpret_cast<const IO*>(buf + 4 * L.raw_i());
  const IO* rL = reinterpret_cast<const IO*>(buf + 4 * L.raw_i() + L.raw_j());
  for (int idx = threadIdx.x; idx < tl * p.cc; idx += blockDim.x) {
    const float lv = to_f32<IO>(rL[idx]);
    const float w = lv * to_f32<IO>(rv[idx]);
    pj[idx] = make_float4(lv, lv, w, w);
  }
}

}  // namespace

namespace {

// Sequential scan over one chunk of tokens (the whole sequence when there is
// one chunk). Chunk z starts from starts[z] when given, else from (λ0, η0);
// the last chunk writes (λ_T, η_T).
template <typename IO, int DK, int RL, int TC>
__global__ void __launch_bounds__(kMaxThreads) kla_scan_kernel(const KernelParams p) {
  using G = Geo<DK, RL>;
  constexpr int NPR = RL / 2;  // row pairs per lane
  extern __shared__ __align__(16) unsigned char smem[];
  const Layout<IO, DK, TC> L(p.cc);
  float* coef = reinterpret_cast<float*>(smem + L.coef());
  float4* pj = reinterpret_cast<float4*>(smem + L.pj());
  float* ypart = reinterpret_cast<float*>(smem + L.ypart());
  float* kprev = reinterpret_cast<float*>(smem + L.kprev(G::NP));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long bh = blockIdx.x;
  const int jb = blockIdx.y * p.cc;
  const int z = blockIdx.z;
  const int t_begin = z * p.chunk_len;
  const int t_end = min(p.T, t_begin + p.chunk_len);
  const int ntiles = (t_end - t_begin + TC - 1) / TC;

  const int li = lane % G::LANES_I, lj = lane / G::LANES_I;
  const int i0 = li * RL;
  const int cl0 = warp * G::WC + lj * CL;  // block-local first column of this lane
  const size_t E = (size_t)DK * p.dv;

  // ---- chunk-start state: P̃ = P (scale K := 1), μ ---------------------------
  f2 Pt[NPR][CL], Mu[NPR][CL];
#pragma unroll
  for (int r = 0; r < NPR; ++r) {
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      float P2[2], M2[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const size_t e = (size_t)bh * E + (size_t)(i0 + 2 * r + h) * p.dv + jb + cl0 + c;
        if (p.starts) {
          P2[h] = p.starts[(size_t)(2 * z) * p.elems + e];
          M2[h] = p.starts[(size_t)(2 * z + 1) * p.elems + e];
        } else if (p.lam0) {
          P2[h] = 1.0f / p.lam0[e];
          M2[h] = p.eta0[e] * P2[h];
        } else {
          P2[h] = 1.0f;
          M2[h] = 0.0f;
        }
      }
      Pt[r][c] = f2_make(P2[0], P2[1]);
      Mu[r][c] = f2_make(M2[0], M2[1]);
    }
  }
  for (int i = tid; i < DK; i += blockDim.x) kprev[i] = 1.0f;

  stage_tile<IO, DK, TC>(p, smem, bh, jb, t_begin, min(TC, t_end - t_begin));
  cp_async_commit();

  for (int n = 0; n < ntiles; ++n) {
    const int t0 = t_begin + n * TC;
    const int tl = min(TC, t_end - t0);
    if (n + 1 < ntiles) {
      const int t1 = t0 + TC;
      stage_tile<IO, DK, TC>(p, smem + ((n + 1) & 1) * L.raw_buf(), bh, jb, t1, min(TC, t_end - t1));
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    // ---- per-(t, i) row coefficients and per-(t, j) column terms ------------
    {
      const unsigned char* buf = smem + (n & 1) * L.raw_buf();
      const IO* rq = reinterpret_cast<const IO*>(buf);
      const IO* rk = rq + TC * DK;
      const IO* ra = rk + TC * DK;
      const IO* rp = ra + TC * DK;
      const float* kp_cur = kprev + (n & 1) * DK;
      float* kp_nxt = kprev + ((n + 1) & 1) * DK;
      for (int idx = tid; idx < tl * DK; idx += blockDim.x) {
        const int t = idx / DK, i = idx % DK;
        const float kt = to_f32<IO>(rk[idx]);
        const float at = fmaxf(to_f32<IO>(ra[idx]), kAMin);
        const float pt = to_f32<IO>(rp[idx]);
        const float Kt = fmaf(kt, kt, kK2Floor);
        float Kp;
        if (t == 0) {
          Kp = kp_cur[i];
        } else {
          const float km = to_f32<IO>(rk[idx - DK]);
          Kp = fmaf(km, km, kK2Floor);
        }
        const float aK = at * Kt;
        const float r = rcp_approx(aK * Kp);  // 1 / (a K_t K_{t-1})
        const float inv_Kp = aK * r;
        const float ainv = (Kt * Kp) * r;
        float* ct = coef + t * 5 * DK + i;
        ct[0 * DK] = aK * inv_Kp;           // A = K_t a / K_{t-1}
        ct[1 * DK] = (Kt * pt) * ainv;      // B = K_t p̄ / a
        ct[2 * DK] = ainv;                  // 1/a
        ct[3 * DK] = kt * (at * Kp * r);    // k / K_t
        ct[4 * DK] = to_f32<IO>(rq[idx]);   // q
        if (t == tl - 1) kp_nxt[i] = Kt;
      }
      column_terms<IO, DK, TC>(p, buf, pj, tl);
    }
    __syncthreads();

    // ---- the scan over this tile --------------------------------------------
    const bool odd = (li & 1) != 0;
    for (int t = 0; t < tl; ++t) {
      const float* ct = coef + t * 5 * DK + i0;
      f2 A[NPR], Bc[NPR], AI[NPR], KI[NPR], Q[NPR];
#pragma unroll
      for (int m = 0; m < NPR / 2; ++m) {
        const ulonglong2 a4 = *reinterpret_cast<const ulonglong2*>(ct + 0 * DK + 4 * m);
        const ulonglong2 b4 = *reinterpret_cast<const ulonglong2*>(ct + 1 * DK + 4 * m);
        const ulonglong2 i4 = *reinterpret_cast<const ulonglong2*>(ct + 2 * DK + 4 * m);
        const ulonglong2 k4 = *reinterpret_cast<const ulonglong2*>(ct + 3 * DK + 4 * m);
        const ulonglong2 q4 = *reinterpret_cast<const ulonglong2*>(ct + 4 * DK + 4 * m);
        A[2 * m] = a4.x;  A[2 * m + 1] = a4.y;
        Bc[2 * m] = b4.x; Bc[2 * m + 1] = b4.y;
        AI[2 * m] = i4.x; AI[2 * m + 1] = i4.y;
        KI[2 * m] = k4.x; KI[2 * m + 1] = k4.y;
        Q[2 * m] = q4.x;  Q[2 * m + 1] = q4.y;
      }
      float yc[CL];
#pragma unroll
      for (int c = 0; c < CL; ++c) {
        const ulonglong2 lv = *reinterpret_cast<const ulonglong2*>(pj + t * p.cc + cl0 + c);
        const f2 L2 = lv.x, V2 = lv.y;
        f2 y2 = f2_make(0.0f, 0.0f);
#pragma unroll
        for (int r = 0; r < NPR; ++r) {
          const f2 s = f2_fma(A[r], Pt[r][c], Bc[r]);
          const f2 d = f2_fma(s, L2, AI[r]);
          const f2 w = f2_rcp(d);
          Pt[r][c] = f2_mul(s, w);
          const f2 g = f2_mul(s, V2);
          const f2 m = f2_fma(g, KI[r], Mu[r][c]);
          Mu[r][c] = f2_mul(m, w);
          y2 = f2_fma(Q[r], Mu[r][c], y2);
        }
        yc[c] = f2_lo(y2) + f2_hi(y2);
      }
      // One exchange with the neighbouring row-lane halves the partial sums:
      // even lanes keep column 0, odd lanes column 1.
      const float send = odd ? yc[0] : yc[1];
      const float keep = odd ? yc[1] : yc[0];
      const float got = __shfl_xor_sync(0xffffffffu, send, 1);
      ypart[(t * p.cc + cl0 + (odd ? 1 : 0)) * G::NP + (li >> 1)] = keep + got;
    }
    __syncthreads();

    // ---- finish the d_k reduction and store y --------------------------------
    {
      IO* yout = reinterpret_cast<IO*>(p.y) + ((size_t)bh * p.T + t0) * p.dv + jb;
      for (int idx = tid; idx < tl * p.cc; idx += blockDim.x) {
        const int t = idx >> p.log2cc, c = idx & (p.cc - 1);
        const float* src = ypart + (size_t)idx * G::NP;
        float s = 0.0f;
#pragma unroll
        for (int q = 0; q < G::NP; ++q) s += src[q];
        yout[(size_t)t * p.dv + c] = from_f32<IO>(s);
      }
    }
  }

  // ---- final state of the last chunk: λ_T = K_last / P̃, η_T = μ λ_T ---------
  if (z == (int)gridDim.z - 1 && p.lamT) {
    const float* klast = kprev + (ntiles & 1) * DK;
#pragma unroll
    for (int r = 0; r < NPR; ++r) {
#pragma unroll
      for (int c = 0; c < CL; ++c) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = i0 + 2 * r + h;
          const size_t e = (size_t)bh * E + (size_t)i * p.dv + jb + cl0 + c;
          const float pt = h ? f2_hi(Pt[r][c]) : f2_lo(Pt[r][c]);
          const float mu = h ? f2_hi(Mu[r][c]) : f2_lo(Mu[r][c]);
          const float lam = klast[i] / pt;
          p.lamT[e] = lam;
          p.etaT[e] = mu * lam;
        }
      }
    }
  }
}

}  // namespace

namespace {

// Composition of one chunk's per-element map (the associative step of
// Methodologie §2, extended to the information mean).
//
// In homogeneous coordinates P = n/m, μ = e/m one token is LINEAR:
//   n' = a²n + p̄m,   m' = m + c·n',   e' = a·e + b·n'
// i.e. [n', m', e'] = M_t [n, m, e] with
//   M_t = [[a², p̄, 0], [c a², 1 + c p̄, 0], [b a², b p̄, a]],
// whose 2×2 block is the Möbius matrix of the precision recursion written
// for the variance. The product over a chunk keeps the shape
// [[A, B, 0], [C, D, 0], [E, F, G]]; it is built by pushing the two basis
// vectors (1,0,0) and (0,1,0) through the chunk (G is the running product of
// a). Every 8 tokens all seven entries are rescaled by the same power of two
// (exact) so that D stays in [1, 2); the map is homogeneous, so this changes
// nothing. Output: maps[z][0..6] = (A, B, C, D, E, F, G) per element.
template <typename IO, int DK, int RL, int TC>
__global__ void __launch_bounds__(kMaxThreads) kla_compose_kernel(const KernelParams p) {
  using G = Geo<DK, RL>;
  constexpr int NPR = RL / 2;
  extern __shared__ __align__(16) unsigned char smem[];
  const Layout<IO, DK, TC> L(p.cc);
  float* coef = reinterpret_cast<float*>(smem + L.coef());
  float4* pj = reinterpret_cast<float4*>(smem + L.pj());

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long bh = blockIdx.x;
  const int jb = blockIdx.y * p.cc;
  const int z = blockIdx.z;
  const int t_begin = z * p.chunk_len;
  const int t_end = min(p.T, t_begin + p.chunk_len);
  const int ntiles = (t_end - t_begin + TC - 1) / TC;
  const int li = lane % G::LANES_I, lj = lane / G::LANES_I;
  const int i0 = li * RL;
  const int cl0 = warp * G::WC + lj * CL;

  const f2 one = f2_make(1.0f, 1.0f), zero = f2_make(0.0f, 0.0f);
  f2 n1[NPR][CL], m1[NPR][CL], e1[NPR][CL], n2[NPR][CL], m2[NPR][CL], e2[NPR][CL], gg[NPR][CL];
#pragma unroll
  for (int r = 0; r < NPR; ++r)
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      n1[r][c] = one; m1[r][c] = zero; e1[r][c] = zero;
      n2[r][c] = zero; m2[r][c] = one; e2[r][c] = zero;
      gg[r][c] = one;
    }

  stage_tile<IO, DK, TC>(p, smem, bh, jb, t_begin, min(TC, t_end - t_begin));
  cp_async_commit();
  for (int n = 0; n < ntiles; ++n) {
    const int t0 = t_begin + n * TC;
    const int tl = min(TC, t_end - t0);
    if (n + 1 < ntiles) {
      const int t1 = t0 + TC;
      stage_tile<IO, DK, TC>(p, smem + ((n + 1) & 1) * L.raw_buf(), bh, jb, t1, min(TC, t_end - t1));
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    {
      const unsigned char* buf = smem + (n & 1) * L.raw_buf();
      const IO* rk = reinterpret_cast<const IO*>(buf) + TC * DK;
      const IO* ra = rk + TC * DK;
      const IO* rp = ra + TC * DK;
      for (int idx = tid; idx < tl * DK; idx += blockDim.x) {
        const int t = idx / DK, i = idx % DK;
        const float kt = to_f32<IO>(rk[idx]);
        const float at = fmaxf(to_f32<IO>(ra[idx]), kAMin);
        float* ct = coef + t * 5 * DK + i;
        ct[0 * DK] = at * at;                      // a²
        ct[1 * DK] = to_f32<IO>(rp[idx]);          // p̄
        ct[2 * DK] = fmaf(kt, kt, kK2Floor);       // k² (floored as in the scan)
        ct[3 * DK] = kt;                           // k
        ct[4 * DK] = at;                           // a
      }
      column_terms<IO, DK, TC>(p, buf, pj, tl);
    }
    __syncthreads();

    for (int t = 0; t < tl; ++t) {
      const float* ct = coef + t * 5 * DK + i0;
      f2 A2[NPR], PB[NPR], K2[NPR], KK[NPR], AA[NPR];
#pragma unroll
      for (int m = 0; m < NPR / 2; ++m) {
        const ulonglong2 x0 = *reinterpret_cast<const ulonglong2*>(ct + 0 * DK + 4 * m);
        const ulonglong2 x1 = *reinterpret_cast<const ulonglong2*>(ct + 1 * DK + 4 * m);
        const ulonglong2 x2 = *reinterpret_cast<const ulonglong2*>(ct + 2 * DK + 4 * m);
        const ulonglong2 x3 = *reinterpret_cast<const ulonglong2*>(ct + 3 * DK + 4 * m);
        const ulonglong2 x4 = *reinterpret_cast<const ulonglong2*>(ct + 4 * DK + 4 * m);
        A2[2 * m] = x0.x; A2[2 * m + 1] = x0.y;
        PB[2 * m] = x1.x; PB[2 * m + 1] = x1.y;
        K2[2 * m] = x2.x; K2[2 * m + 1] = x2.y;
        KK[2 * m] = x3.x; KK[2 * m + 1] = x3.y;
        AA[2 * m] = x4.x; AA[2 * m + 1] = x4.y;
      }
#pragma unroll
      for (int c = 0; c < CL; ++c) {
        const ulonglong2 lv = *reinterpret_cast<const ulonglong2*>(pj + t * p.cc + cl0 + c);
        const f2 Lw = lv.x, Vw = lv.y;
#pragma unroll
        for (int r = 0; r < NPR; ++r) {
          const f2 cc2 = f2_mul(K2[r], Lw);  // c = k²Λ^v
          const f2 bb2 = f2_mul(KK[r], Vw);  // b = kΛ^v v
          n1[r][c] = f2_fma(A2[r], n1[r][c], f2_mul(PB[r], m1[r][c]));
          m1[r][c] = f2_fma(cc2, n1[r][c], m1[r][c]);
          e1[r][c] = f2_fma(bb2, n1[r][c], f2_mul(AA[r], e1[r][c]));
          n2[r][c] = f2_fma(A2[r], n2[r][c], f2_mul(PB[r], m2[r][c]));
          m2[r][c] = f2_fma(cc2, n2[r][c], m2[r][c]);
          e2[r][c] = f2_fma(bb2, n2[r][c], f2_mul(AA[r], e2[r][c]));
          gg[r][c] = f2_mul(AA[r], gg[r][c]);
        }
      }
      if (((t0 + t - t_begin) & 7) == 7 || (n == ntiles - 1 && t == tl - 1)) {
#pragma unroll
        for (int r = 0; r < NPR; ++r)
#pragma unroll
          for (int c = 0; c < CL; ++c) {
            // 2^(127 - exponent(D)) for each half: brings D into [1, 2).
            const unsigned elo = min((__float_as_uint(f2_lo(m2[r][c])) >> 23) & 0xffu, 253u);
            const unsigned ehi = min((__float_as_uint(f2_hi(m2[r][c])) >> 23) & 0xffu, 253u);
            const f2 sc = f2_make(__uint_as_float((254u - elo) << 23), __uint_as_float((254u - ehi) << 23));
            n1[r][c] = f2_mul(n1[r][c], sc); m1[r][c] = f2_mul(m1[r][c], sc); e1[r][c] = f2_mul(e1[r][c], sc);
            n2[r][c] = f2_mul(n2[r][c], sc); m2[r][c] = f2_mul(m2[r][c], sc); e2[r][c] = f2_mul(e2[r][c], sc);
            gg[r][c] = f2_mul(gg[r][c], sc);
          }
      }
    }
    __syncthreads();
  }

  const size_t E = (size_t)DK * p.dv;
  float* out = p.maps + (size_t)z * 7 * p.elems;
#pragma unroll
  for (int r = 0; r < NPR; ++r)
#pragma unroll
    for (int c = 0; c < CL; ++c)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const size_t e = (size_t)bh * E + (size_t)(i0 + 2 * r + h) * p.dv + jb + cl0 + c;
        const f2 vals[7] = {n1[r][c], n2[r][c], m1[r][c], m2[r][c], e1[r][c], e2[r][c], gg[r][c]};
#pragma unroll
        for (int q = 0; q < 7; ++q) out[(size_t)q * p.elems + e] = h ? f2_hi(vals[q]) : f2_lo(vals[q]);
      }
}

// Cross-chunk carry: starts[0] = (1/λ0, η0/λ0); for each chunk z the map
// (A..G) takes (P, μ) at its start to its end:
//   n = A P + B,  m = C P + D,  e = E P + F + G μ;  P' = n/m,  μ' = e/m.
__global__ void kla_carry_kernel(const float* __restrict__ maps, float* __restrict__ starts,
                                 const float* __restrict__ lam0, const float* __restrict__ eta0,
                                 long long elems, int num_chunks) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= elems) return;
  float P = 1.0f, mu = 0.0f;
  if (lam0) {
    P = 1.0f / lam0[e];
    mu = eta0[e] * P;
  }
  starts[e] = P;
  starts[elems + e] = mu;
  for (int z = 0; z + 1 < num_chunks; ++z) {
    const float* m = maps + (size_t)z * 7 * elems + e;
    const float A = m[0], B = m[elems], C = m[2 * elems], D = m[3 * elems];
    const float E = m[4 * elems], F = m[5 * elems], Gm = m[6 * elems];
    const float nn = fmaf(A, P, B);
    const float mm = fmaf(C, P, D);
    const float ee = fmaf(E, P, fmaf(Gm, mu, F));
    P = nn / mm;
    mu = ee / mm;
    starts[(size_t)(2 * (z + 1)) * elems + e] = P;
    starts[(size_t)(2 * (z + 1) + 1) * elems + e] = mu;
  }
}

// T = 0: the final state is the initial one (λ0, η0, or 1 and 0).
__global__ void kla_init_state_kernel(const float* lam0, const float* eta0, float* lamT, float* etaT,
                                      long long elems) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= elems) return;
  const float l = lam0 ? lam0[e] : 1.0f;
  const float n = eta0 ? eta0[e] : 0.0f;
  if (lamT) lamT[e] = l;
  if (etaT) etaT[e] = n;
}

}  // namespace

// ---------------------------------------------------------------------------
// Host side: geometry and launchers.
// ---------------------------------------------------------------------------
int rows_per_lane_for(int dk) { return dk <= 32 ? 4 : 8; }
int tile_for(int dk, int io) { return (dk == 128 && io == IO_F32) ? 16 : 32; }
int warp_cols(int dk) { return (32 / (dk / rows_per_lane_for(dk))) * CL; }

namespace {
template <typename IO, int DK, int TC>
size_t layout_bytes(int cc) {
  const int np = DK / rows_per_lane_for(DK) / 2;
  return Layout<IO, DK, TC>(cc).total(np);
}
template <typename IO>
size_t smem_for(int dk, int cc, int tile) {
  if (tile == 16) {
    switch (dk) {
      case 16: return layout_bytes<IO, 16, 16>(cc);
      case 32: return layout_bytes<IO, 32, 16>(cc);
      case 64: return layout_bytes<IO, 64, 16>(cc);
      default: return layout_bytes<IO, 128, 16>(cc);
    }
  }
  switch (dk) {
    case 16: return layout_bytes<IO, 16, 32>(cc);
    case 32: return layout_bytes<IO, 32, 32>(cc);
    case 64: return layout_bytes<IO, 64, 32>(cc);
    default: return layout_bytes<IO, 128, 32>(cc);
  }
}
}  // namespace

size_t forward_smem_bytes(int dk, int io, int cc, int tile) {
  return io == IO_BF16 ? smem_for<__nv_bfloat16>(dk, cc, tile) : smem_for<float>(dk, cc, tile);
}
size_t compose_smem_bytes(int dk, int io, int cc, int tile) { return forward_smem_bytes(dk, io, cc, tile); }

size_t chunk_workspace_bytes(long long elems, int num_chunks) {
  if (num_chunks <= 1) return 0;
  return (size_t)(7 * (num_chunks - 1) + 2 * num_chunks) * (size_t)elems * sizeof(float);
}

namespace {

KernelParams make_params(const ForwardArgs& f, const Plan& p) {
  KernelParams kp{};
  kp.q = f.q; kp.k = f.k; kp.v = f.v; kp.lam_v = f.lam_v; kp.a = f.a; kp.pbar = f.pbar;
  kp.lam0 = f.lam0; kp.eta0 = f.eta0;
  kp.y = f.y; kp.lamT = f.lamT; kp.etaT = f.etaT;
  kp.T = f.T; kp.dv = f.dv; kp.chunk_len = p.chunk_len; kp.cc = p.cols_per_block;
  int l2 = 0;
  while ((1 << l2) < p.cols_per_block) ++l2;
  kp.log2cc = l2;
  kp.elems = (long long)f.B * f.H * f.dk * f.dv;
  return kp;
}

template <typename Kern>
cudaError_t launch_with_smem(Kern fn, dim3 grid, int threads, size_t smem, cudaStream_t s, const KernelParams& kp) {
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  fn<<<grid, threads, smem, s>>>(kp);
  return cudaGetLastError();
}

template <typename IO, int TC>
cudaError_t dispatch(bool compose, const ForwardArgs& f, const KernelParams& kp, dim3 grid, int threads,
                     size_t smem, cudaStream_t s) {
  switch (f.dk) {
    case 16:
      return launch_with_smem(compose ? kla_compose_kernel<IO, 16, 4, TC> : kla_scan_kernel<IO, 16, 4, TC>, grid,
                              threads, smem, s, kp);
    case 32:
      return launch_with_smem(compose ? kla_compose_kernel<IO, 32, 4, TC> : kla_scan_kernel<IO, 32, 4, TC>, grid,
                              threads, smem, s, kp);
    case 64:
      return launch_with_smem(compose ? kla_compose_kernel<IO, 64, 8, TC> : kla_scan_kernel<IO, 64, 8, TC>, grid,
                              threads, smem, s, kp);
    case 128:
      return launch_with_smem(compose ? kla_compose_kernel<IO, 128, 8, TC> : kla_scan_kernel<IO, 128, 8, TC>, grid,
                              threads, smem, s, kp);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_pass(bool compose, const ForwardArgs& f, const Plan& p, const KernelParams& kp, int nz,
                        cudaStream_t s) {
  const dim3 grid((unsigned)((long long)f.B * f.H), (unsigned)(f.dv / p.cols_per_block), (unsigned)nz);
  const int threads = 32 * (p.cols_per_block / warp_cols(f.dk));
  const size_t smem = forward_smem_bytes(f.dk, f.io, p.cols_per_block, p.tile);
  if (f.io == IO_BF16) {
    return p.tile == 16 ? dispatch<__nv_bfloat16, 16>(compose, f, kp, grid, threads, smem, s)
                        : dispatch<__nv_bfloat16, 32>(compose, f, kp, grid, threads, smem, s);
  }
  return p.tile == 16 ? dispatch<float, 16>(compose, f, kp, grid, threads, smem, s)
                      : dispatch<float, 32>(compose, f, kp, grid, threads, smem, s);
}

}  // namespace

cudaError_t launch_forward(const ForwardArgs& f, const Plan& p, const float* starts, cudaStream_t s) {
  KernelParams kp = make_params(f, p);
  kp.starts = starts;
  return launch_pass(false, f, p, kp, p.num_chunks, s);
}

cudaError_t launch_compose(const ForwardArgs& f, const Plan& p, float* maps, cudaStream_t s) {
  if (p.num_chunks <= 1) return cudaSuccess;
  KernelParams kp = make_params(f, p);
  kp.maps = maps;
  return launch_pass(true, f, p, kp, p.num_chunks - 1, s);
}

cudaError_t launch_carry(const ForwardArgs& f, const Plan& p, const float* maps, float* starts, cudaStream_t s) {
  const long long elems = (long long)f.B * f.H * f.dk * f.dv;
  const int threads = 256;
  const unsigned blocks = (unsigned)((elems + threads - 1) / threads);
  kla_carry_kernel<<<blocks, threads, 0, s>>>(maps, starts, f.lam0, f.eta0, elems, p.num_chunks);
  return cudaGetLastError();
}

cudaError_t launch_init_state(const ForwardArgs& f, cudaStream_t s) {
  const long long elems = (long long)f.B * f.H * f.dk * f.dv;
  if (elems == 0 || (!f.lamT && !f.etaT)) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = (unsigned)((elems + threads - 1) / threads);
  kla_init_state_kernel<<<blocks, threads, 0, s>>>(f.lam0, f.eta0, f.lamT, f.etaT, elems);
  return cudaGetLastError();
}

}  // namespace kla
