// Sequence scan of the KLA filter for sm_103a (the sequential path, and the
// re-run of each chunk on the chunk-parallel path): the kernel template. The
// host side is kla_scan.cu; kla_scan_inst_*.cu instantiate the kernel, one
// translation unit per readout mode so that they compile in parallel.
//
// The operation is the diagonal information-form Kalman filter of
// "Technische Samenvatting: Kalman Linear Attention (KLA)"
// (gist.science/nl/paper/2602.10743), Methodologie §1 (OU prior, observation
// through k with value precision Λ^v, posterior-mean readout through q) and
// §2 (Möbius precision recursion, affine information-mean recursion).
//
// ---------------------------------------------------------------------------
// Arithmetic (per element (i, j), token t; c = k²Λ^v, b = kΛ^v v)
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
// K_t and a_t are floored at 2^-40, so every scaled quantity stays a normal
// fp32 number.
//
// ---------------------------------------------------------------------------
// Work layout and pipeline
//
// A thread block owns one head (grid.x), a block of CC columns (grid.y) and
// one chunk of tokens (grid.z); all d_k rows of those columns. Each lane
// holds RL rows × CL columns in registers for the whole chunk — the state is
// never written per token. Tokens stream through shared memory in tiles of
// TC, double-buffered, between two groups of warps:
//
//   scan warps (CC/WC):   wait FULL[n%2]; scan tile n (coef/pj[n%2] → partial
//                         y sums ypart[n%2]); arrive EMPTY[n%2]
//   producer warps (4):   queue raw tile n+2 (16-byte cp.async); wait
//                         EMPTY[n%2]; store y of tile n (finish the d_k
//                         reduction from ypart); build the per-row
//                         coefficients and per-column terms of tile n+2 into
//                         coef/pj[n%2]; arrive FULL[n%2]
//
// (FULL/EMPTY are named barriers; bar.arrive does not wait.) The scan warps
// do nothing but the recurrence; the producers' work overlaps it, and their
// raw-tile loads have a whole tile of scanning to land. The per-row coefficients
// (A, B, 1/a, k/K, q) are computed once per (t, i) and serve all CC columns;
// the per-column terms (Λ^v, Λ^v v) once per (t, j) for all d_k rows. When a
// head's columns span several blocks, the coefficient pass (kla_coef_kernel)
// computes the per-row coefficients once for all of them and the producers
// (MODE 4) copy each tile's coefficients instead of building them.
// ---------------------------------------------------------------------------
#pragma once

#include <type_traits>

#include "kla_common.cuh"
#include "kla_launch.h"

namespace kla {

namespace {

constexpr int kTile = 16;  // tokens per shared-memory tile
// Named barrier ids of the scan's producer/consumer hand-off.
constexpr int kBarFull0 = 1;      // 1, 2: coefficients of buffer 0 / 1 are ready
constexpr int kBarEmpty0 = 3;     // 3, 4: the scan is done with buffer 0 / 1
constexpr int kBarProducers = 5;  // producer warps only (staged raw tile visible)

// Byte offsets of the double-buffered shared-memory regions of one block.
template <typename IO, int DK, int TC, int NP, int NC = 5, int NOUT = 1>
struct ScanLayout {
  int cc;
  // NC per-row coefficients per token; NOUT readouts (y, and y_var with both).
  __host__ __device__ explicit ScanLayout(int cc_) : cc(cc_) {}
  __host__ __device__ size_t raw_bytes() const { return RawTile<IO, DK, TC>::bytes(cc); }
  __host__ __device__ size_t coef_bytes() const { return (size_t)TC * NC * DK * sizeof(float); }
  __host__ __device__ size_t pj_bytes() const { return (size_t)TC * cc * sizeof(float4); }
  // Partial sums, token-major per (partial, column): [NP][cc][TC + 4] (the
  // padding keeps 128-bit stores of four tokens free of bank conflicts).
  static constexpr int TCP = TC + 4;
  __host__ __device__ size_t ypart_out() const { return (size_t)cc * NP * TCP; }  // floats per readout
  __host__ __device__ size_t ypart_bytes() const { return NOUT * ypart_out() * sizeof(float); }
  __host__ __device__ size_t raw(int b) const { return b * raw_bytes(); }
  __host__ __device__ size_t coef(int b) const { return 2 * raw_bytes() + b * coef_bytes(); }
  __host__ __device__ size_t pj(int b) const { return coef(2) + b * pj_bytes(); }
  __host__ __device__ size_t ypart(int b) const { return pj(2) + b * ypart_bytes(); }
  __host__ __device__ size_t kprev(int b) const { return ypart(2) + b * DK * sizeof(float); }
  __host__ __device__ size_t total() const { return kprev(2); }
};

// Per-row coefficients of one token for four consecutive rows, from the
// row's inputs k, a, p̄ (pre-activations when GATED) and K of the token
// before (1 at a chunk start): A = K_t a/K_{t-1}, B = K_t p̄/a, 1/a, k/K_t,
// K_t, and 1/K_t. The producers and the coefficient pass both call this, so
// the two paths give bit-identical coefficients.
template <bool GATED>
__device__ __forceinline__ void row_coef4(const float (&kv)[4], const float (&av)[4], const float (&pv)[4],
                                          const float (&kpv)[4], int gates, float (&A)[4], float (&B)[4],
                                          float (&AI)[4], float (&KI)[4], float (&Kt)[4], float (&rKo)[4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float at = fmaxf(GATED ? gate_a(av[u], gates) : av[u], kAMin);
    const float pbu = GATED ? gate_pbar(pv[u], av[u], gates) : pv[u];
    Kt[u] = fmaf(kv[u], kv[u], kK2Floor);
    const float aK = at * Kt[u];
    const float r = rcp_approx(aK * kpv[u]);  // 1 / (a K_t K_{t-1})
    AI[u] = (Kt[u] * kpv[u]) * r;             // 1/a
    A[u] = aK * (aK * r);                     // K_t a / K_{t-1}
    B[u] = (Kt[u] * pbu) * AI[u];             // K_t p̄ / a
    rKo[u] = at * kpv[u] * r;                 // 1 / K_t
    KI[u] = kv[u] * rKo[u];                   // k / K_t
  }
}

// Per-(t, i) row coefficients of a staged tile, four rows per thread:
// coef[t][0..4][i] = (A, B, 1/a, k/K, q); MODE 1 (variance readout only) has
// q²/K in place of q, MODE 2 (both readouts) adds q²/K as coef[t][5][i].
// kp_cur holds K of the row before the tile (1 at a chunk start); K of the
// tile's last row goes to kp_nxt.
template <typename IO, int DK, int TC, int MODE = 0, bool GATED = false>
__device__ __forceinline__ void row_coefficients(const unsigned char* raw, float* coef, const float* kp_cur,
                                                 float* kp_nxt, int tl, int tid, int nthr, int gates) {
  using R = RawTile<IO, DK, TC>;
  const IO* rq = reinterpret_cast<const IO*>(raw);
  const IO* rk = reinterpret_cast<const IO*>(raw + R::row_bytes());
  const IO* ra = reinterpret_cast<const IO*>(raw + 2 * R::row_bytes());
  const IO* rp = reinterpret_cast<const IO*>(raw + 3 * R::row_bytes());
  for (int g = tid; g < tl * (DK / 4); g += nthr) {
    const int t = g / (DK / 4), i = 4 * (g % (DK / 4));
    const int o = t * DK + i;
    const float4 k4 = load4<IO>(rk + o), a4 = load4<IO>(ra + o), p4 = load4<IO>(rp + o), q4 = load4<IO>(rq + o);
    float4 kp4;
    if (t == 0) {
      kp4 = *reinterpret_cast<const float4*>(kp_cur + i);
    } else {
      const float4 km = load4<IO>(rk + o - DK);
      kp4 = make_float4(fmaf(km.x, km.x, kK2Floor), fmaf(km.y, km.y, kK2Floor), fmaf(km.z, km.z, kK2Floor),
                        fmaf(km.w, km.w, kK2Floor));
    }
    const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, av[4] = {a4.x, a4.y, a4.z, a4.w};
    const float pv[4] = {p4.x, p4.y, p4.z, p4.w}, kpv[4] = {kp4.x, kp4.y, kp4.z, kp4.w};
    const float qv[4] = {q4.x, q4.y, q4.z, q4.w};
    float A[4], B[4], AI[4], KI[4], Kt[4], rK[4], QV[4];
    row_coef4<GATED>(kv, av, pv, kpv, gates, A, B, AI, KI, Kt, rK);
#pragma unroll
    for (int u = 0; u < 4; ++u) QV[u] = qv[u] * qv[u] * rK[u];  // q²/K_t (variance readout)
    constexpr int NC = MODE == 2 ? 6 : 5;
    float* ct = coef + t * NC * DK + i;
    *reinterpret_cast<float4*>(ct + 0 * DK) = make_float4(A[0], A[1], A[2], A[3]);
    *reinterpret_cast<float4*>(ct + 1 * DK) = make_float4(B[0], B[1], B[2], B[3]);
    *reinterpret_cast<float4*>(ct + 2 * DK) = make_float4(AI[0], AI[1], AI[2], AI[3]);
    *reinterpret_cast<float4*>(ct + 3 * DK) = make_float4(KI[0], KI[1], KI[2], KI[3]);
    if (MODE == 1)
      *reinterpret_cast<float4*>(ct + 4 * DK) = make_float4(QV[0], QV[1], QV[2], QV[3]);
    else
      *reinterpret_cast<float4*>(ct + 4 * DK) = q4;
    if (MODE == 2) *reinterpret_cast<float4*>(ct + 5 * DK) = make_float4(QV[0], QV[1], QV[2], QV[3]);
    if (t == tl - 1) *reinterpret_cast<float4*>(kp_nxt + i) = make_float4(Kt[0], Kt[1], Kt[2], Kt[3]);
  }
}

// The coefficient pass (scan MODE 4 reads its output): the per-row
// coefficients (A, B, 1/a, k/K, q) of every token of every head into
// coefs[B·H][T][5][d_k], each (t, i) once, however many column blocks of the
// head read them afterwards. K of the token before is 1 at t = 0. A block
// covers kCoefTokens tokens of one head (grid.x) for heads blockIdx.y,
// blockIdx.y + gridDim.y, ...; a thread handles four consecutive rows of a
// token, so loads and stores are 16-byte (fp32) or 8-byte (bf16) per thread
// and consecutive threads touch consecutive addresses.
constexpr int kCoefTokens = 64;
template <typename IO, int DK, bool GATED>
__global__ void __launch_bounds__(256) kla_coef_kernel(const KernelParams p, float* coefs, long long bh_count) {
  constexpr int R4 = DK / 4;
  const int t0 = blockIdx.x * kCoefTokens;
  const int tl = min(kCoefTokens, p.T - t0);
  for (long long bh = blockIdx.y; bh < bh_count; bh += gridDim.y) {
    const size_t row0 = (size_t)bh * p.T;
    for (int g = threadIdx.x; g < tl * R4; g += blockDim.x) {
      const int tt = g / R4, i = 4 * (g % R4), t = t0 + tt;
      const size_t o = (row0 + t) * DK + i;
      const float4 k4 = load4<IO>(reinterpret_cast<const IO*>(p.k) + o);
      const float4 a4 = load4<IO>(reinterpret_cast<const IO*>(p.a) + o);
      const float4 p4 = load4<IO>(reinterpret_cast<const IO*>(p.pbar) + o);
      const float4 q4 = load4<IO>(reinterpret_cast<const IO*>(p.q) + o);
      float4 kp4 = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
      if (t > 0) {
        const float4 km = load4<IO>(reinterpret_cast<const IO*>(p.k) + o - DK);
        kp4 = make_float4(fmaf(km.x, km.x, kK2Floor), fmaf(km.y, km.y, kK2Floor), fmaf(km.z, km.z, kK2Floor),
                          fmaf(km.w, km.w, kK2Floor));
      }
      const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, av[4] = {a4.x, a4.y, a4.z, a4.w};
      const float pv[4] = {p4.x, p4.y, p4.z, p4.w}, kpv[4] = {kp4.x, kp4.y, kp4.z, kp4.w};
      float A[4], B[4], AI[4], KI[4], Kt[4], rK[4];
      row_coef4<GATED>(kv, av, pv, kpv, p.gates, A, B, AI, KI, Kt, rK);
      float* ct = coefs + (row0 + t) * (5 * DK) + i;
      *reinterpret_cast<float4*>(ct + 0 * DK) = make_float4(A[0], A[1], A[2], A[3]);
      *reinterpret_cast<float4*>(ct + 1 * DK) = make_float4(B[0], B[1], B[2], B[3]);
      *reinterpret_cast<float4*>(ct + 2 * DK) = make_float4(AI[0], AI[1], AI[2], AI[3]);
      *reinterpret_cast<float4*>(ct + 3 * DK) = make_float4(KI[0], KI[1], KI[2], KI[3]);
      *reinterpret_cast<float4*>(ct + 4 * DK) = q4;
    }
  }
}

// Finish the d_k reduction of one tile (NP partial sums per output, layout
// [NP][cc][TCP]) and store y rows [t0, t0 + tl) of this block's columns; a
// thread handles one column and four tokens. cc = 2^log2cc.
template <typename IO, int NP, int TC, int TCP>
__device__ __forceinline__ void store_y(const float* ypart, IO* yout, int dv, int cc, int log2cc, int tl, int tid,
                                        int nthr) {
  // Columns vary fastest across threads: the partial-sum loads (columns
  // TCP floats apart) hit distinct banks and each y row is written by
  // consecutive threads.
  for (int g = tid; g < cc * (TC / 4); g += nthr) {
    const int col = g & (cc - 1), t4 = 4 * (g >> log2cc);
    if (t4 >= tl) continue;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(ypart + ((size_t)q * cc + col) * TCP + t4);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    const float sv[4] = {s.x, s.y, s.z, s.w};
    IO* dst = yout + (size_t)t4 * dv + col;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (t4 + u < tl) dst[(size_t)u * dv] = from_f32<IO>(sv[u]);
  }
}

// MODE 0: y. MODE 1: the variance readout y_var[t, j] = Σ_i q_i² P_t[i, j]
// instead of y (the mean recursion is skipped; y points at y_var). MODE 2:
// both, y into p.y and y_var into p.y_var. MODE 3: no readout; the state is
// stored into p.ckpt for the backward pass. MODE 4: y, as MODE 0, with the
// per-row coefficients copied from the coefficient pass's output p.coefs
// instead of built by the producers (one chunk, the sequential plan).
template <typename IO, int DK, int RL, int TC, int MODE = 0>
__global__ void __launch_bounds__(kMaxThreads + 32 * kProducerWarps, 1) kla_scan_kernel(const KernelParams p) {
  using G = Geo<DK, RL>;
  constexpr int NPR = RL / 2;  // row pairs per lane
  constexpr bool VAR = MODE == 1;
  constexpr bool CKPT = MODE == 3;
  constexpr bool PRE = MODE == 4;
  constexpr int NC = MODE == 2 ? 6 : 5, NOUT = MODE == 2 ? 2 : 1;
  extern __shared__ __align__(16) unsigned char smem[];
  const ScanLayout<IO, DK, TC, G::NP, NC, NOUT> L(p.cc);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Warps [0, ncons) scan; the last kProducerWarps warps stage raw tiles,
  // build per-row coefficients and per-column terms, and store y.
  const int ncons = (int)(blockDim.x >> 5) - kProducerWarps;
  const int nall = (int)blockDim.x;
  const long long bh = blockIdx.x;
  const int jb = blockIdx.y * p.cc;
  const int z = blockIdx.z;
  const int t_begin = z * p.chunk_len;
  const int t_end = min(p.T, t_begin + p.chunk_len);
  const int ntiles = (t_end - t_begin + TC - 1) / TC;
  const int li = lane / G::LANES_J, lj = lane % G::LANES_J;
  const int i0 = li * RL;
  const int cl0 = warp * G::WC + lj * CL;  // block-local first column of this lane
  // Register c of a lane holds column cl0 + (c ^ swz), swz = the low XR bits
  // of li bit-reversed into the top bits of the column index: then in every
  // exchange round each lane keeps the low half of its registers and sends
  // the high half (no per-lane select).
  constexpr int kLogCL = CL == 4 ? 2 : 1;
  int swz = 0;
#pragma unroll
  for (int r = 0; r < G::XR; ++r) swz |= ((li >> r) & 1) << (kLogCL - 1 - r);
  const size_t E = (size_t)DK * p.dv;
  IO* ybase = reinterpret_cast<IO*>(p.y) + ((size_t)bh * p.T) * p.dv + jb;
  IO* yvbase = reinterpret_cast<IO*>(p.y_var) + ((size_t)bh * p.T) * p.dv + jb;
  auto tile_len = [&](int n) { return min(TC, t_end - (t_begin + n * TC)); };

  if (warp >= ncons) {
    // ================= producer warps =================
    const int ptid = tid - 32 * ncons, pn = 32 * kProducerWarps;
    if constexpr (PRE) {
      // The same hand-off with the row coefficients copied, not built: tile
      // m's coefficients (tl·5·d_k contiguous floats) go straight into
      // coef[m % 2] once the scan is done with that buffer, while the store
      // of y of the tile before covers the copy's latency; only the
      // per-column terms are built here.
      auto fetch_coef = [&](int m) {
        const float* src = p.coefs + ((size_t)bh * p.T + t_begin + m * TC) * (5 * DK);
        float* dst = reinterpret_cast<float*>(smem + L.coef(m & 1));
        const int chunks = tile_len(m) * (5 * DK / 4);
        for (int c = ptid; c < chunks; c += pn) cp_async16(dst + 4 * c, src + 4 * c);
      };
      auto build_cols = [&](auto gated, int m) {
        column_terms<IO, DK, TC, decltype(gated)::value>(smem + L.raw(m & 1), reinterpret_cast<float4*>(smem + L.pj(m & 1)),
                                                         p.cc, tile_len(m), ptid, pn, p.gates);
      };
      auto cols = [&](int m) {
        if (p.gates) build_cols(std::true_type{}, m);
        else build_cols(std::false_type{}, m);
      };
      // K of the chunk's last token, for the final state (read by the scan
      // warps after the last tile, so after many FULL barriers)
      if (p.lamT && ntiles > 0) {
        float* klast = reinterpret_cast<float*>(smem + L.kprev(ntiles & 1));
        const IO* kl = reinterpret_cast<const IO*>(p.k) + ((size_t)bh * p.T + t_end - 1) * DK;
        for (int i = ptid; i < DK; i += pn) {
          const float kv = to_f32<IO>(kl[i]);
          klast[i] = fmaf(kv, kv, kK2Floor);
        }
      }
      stage_cols<IO, DK, TC>(p, smem + L.raw(0), bh, jb, t_begin, tile_len(0), ptid, pn);
      fetch_coef(0);
      cp_async_commit();
      if (ntiles > 1) {
        stage_cols<IO, DK, TC>(p, smem + L.raw(1), bh, jb, t_begin + TC, tile_len(1), ptid, pn);
        fetch_coef(1);
      }
      cp_async_commit();
      cp_async_wait<1>();
      named_sync(kBarProducers, pn);  // tile 0's columns and coefficients visible to all producers
      cols(0);
      named_arrive(kBarFull0, nall);
      if (ntiles > 1) {
        cp_async_wait<0>();
        named_sync(kBarProducers, pn);
        cols(1);
        named_arrive(kBarFull0 + 1, nall);
      }
      for (int n = 0; n < ntiles; ++n) {
        const int b = n & 1;
        if (n + 2 < ntiles) stage_cols<IO, DK, TC>(p, smem + L.raw(b), bh, jb, t_begin + (n + 2) * TC, tile_len(n + 2), ptid, pn);
        cp_async_commit();
        named_sync(kBarEmpty0 + b, nall);  // the scan of tile n is done with coef/pj[b] and ypart[b]
        if (n + 2 < ntiles) fetch_coef(n + 2);
        cp_async_commit();
        if (p.y)
          store_y<IO, G::NP, TC, L.TCP>(reinterpret_cast<const float*>(smem + L.ypart(b)),
                                        ybase + (size_t)(t_begin + n * TC) * p.dv, p.dv, p.cc, p.log2cc, tile_len(n), ptid, pn);
        if (n + 2 < ntiles) {
          cp_async_wait<0>();
          named_sync(kBarProducers, pn);
          cols(n + 2);
          named_arrive(kBarFull0 + b, nall);
        }
      }
      return;
    }
    float* kp0 = reinterpret_cast<float*>(smem + L.kprev(0));
    for (int i = ptid; i < DK; i += pn) kp0[i] = 1.0f;
    // coefficients of tile m into buffer m % 2; the gate activations are a
    // separate instantiation so that ungated producers carry no extra work
    auto build_tile = [&](auto gated, int m) {
      constexpr bool GT = decltype(gated)::value;
      const int bm = m & 1;
      row_coefficients<IO, DK, TC, MODE, GT>(smem + L.raw(bm), reinterpret_cast<float*>(smem + L.coef(bm)),
                                             reinterpret_cast<const float*>(smem + L.kprev(bm)),
                                             reinterpret_cast<float*>(smem + L.kprev(bm ^ 1)), tile_len(m), ptid, pn,
                                             p.gates);
      column_terms<IO, DK, TC, GT>(smem + L.raw(bm), reinterpret_cast<float4*>(smem + L.pj(bm)), p.cc,
                                   tile_len(m), ptid, pn, p.gates);
    };
    auto build = [&](int m) {
      if (p.gates) build_tile(std::true_type{}, m);
      else build_tile(std::false_type{}, m);
    };
    stage_raw<IO, DK, TC>(p, smem + L.raw(0), bh, jb, t_begin, tile_len(0), ptid, pn);
    cp_async_commit();
    if (ntiles > 1) stage_raw<IO, DK, TC>(p, smem + L.raw(1), bh, jb, t_begin + TC, tile_len(1), ptid, pn);
    cp_async_commit();
    cp_async_wait<1>();
    named_sync(kBarProducers, pn);  // raw tile 0 and kprev visible to all producers
    build(0);
    named_arrive(kBarFull0, nall);
    if (ntiles > 1) {
      cp_async_wait<0>();
      named_sync(kBarProducers, pn);
      build(1);
      named_arrive(kBarFull0 + 1, nall);
    }
    for (int n = 0; n < ntiles; ++n) {
      const int b = n & 1;
      // raw[b] held tile n, already consumed by build(n)
      if (n + 2 < ntiles) stage_raw<IO, DK, TC>(p, smem + L.raw(b), bh, jb, t_begin + (n + 2) * TC, tile_len(n + 2), ptid, pn);
      cp_async_commit();
      named_sync(kBarEmpty0 + b, nall);  // the scan of tile n is done with coef/pj[b] and ypart[b]
      if (!CKPT && p.y)
        store_y<IO, G::NP, TC, L.TCP>(reinterpret_cast<const float*>(smem + L.ypart(b)),
                                      ybase + (size_t)(t_begin + n * TC) * p.dv, p.dv, p.cc, p.log2cc, tile_len(n), ptid, pn);
      if (MODE == 2)
        store_y<IO, G::NP, TC, L.TCP>(reinterpret_cast<const float*>(smem + L.ypart(b)) + L.ypart_out(),
                                      yvbase + (size_t)(t_begin + n * TC) * p.dv, p.dv, p.cc, p.log2cc, tile_len(n), ptid, pn);
      if (n + 2 < ntiles) {
        cp_async_wait<0>();
        named_sync(kBarProducers, pn);
        build(n + 2);
        named_arrive(kBarFull0 + b, nall);
      }
    }
    return;
  }

  // ================= scan (consumer) warps =================
  // ---- chunk-start state: P̃ = P (scale K := 1), μ ---------------------------
  f2 Pt[NPR][CL], Mu[NPR][CL];
#pragma unroll
  for (int r = 0; r < NPR; ++r) {
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      float P2[2], M2[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const size_t e = (size_t)bh * E + (size_t)(i0 + 2 * r + h) * p.dv + jb + cl0 + (c ^ swz);
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
  // Checkpoints for the backward pass (sequential plan only): the scaled
  // state (P̃ = K_{t-1}·P, μ) before every tile and after the last token.
  auto checkpoint = [&](int idx) {
    float* ck = p.ckpt + (size_t)idx * 2 * p.elems;
#pragma unroll
    for (int r = 0; r < NPR; ++r)
#pragma unroll
      for (int c = 0; c < CL; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const size_t e = (size_t)bh * E + (size_t)(i0 + 2 * r + h) * p.dv + jb + cl0 + (c ^ swz);
          ck[e] = h ? f2_hi(Pt[r][c]) : f2_lo(Pt[r][c]);
          ck[p.elems + e] = h ? f2_hi(Mu[r][c]) : f2_lo(Mu[r][c]);
        }
  };
  for (int n = 0; n < ntiles; ++n) {
    const int b = n & 1;
    const int tl = tile_len(n);
    if constexpr (CKPT) checkpoint(n);
    named_sync(kBarFull0 + b, nall);  // coefficients of tile n are ready
    // ---- the scan over tile n ------------------------------------------------
    {
      const float* __restrict__ coef = reinterpret_cast<const float*>(smem + L.coef(b)) + i0;
      const float4* __restrict__ pj = reinterpret_cast<const float4*>(smem + L.pj(b)) + cl0;
      float* __restrict__ ypart = reinterpret_cast<float*>(smem + L.ypart(b));
      // Exchange rounds with the lanes holding neighbouring rows halve the
      // partial sums each time; after XR rounds a lane holds registers
      // 0..VALS-1, the sums over 2^XR row groups of columns cl0 + (u ^ swz)
      // (with VALS = 1: column cl0 + swz).
      // Readout o (0: y or, in MODE 1, y_var; 1: y_var in MODE 2) goes to
      // ypart + o·ypart_out().
      float* __restrict__ ydst = ypart + ((size_t)(li >> G::XR) * p.cc + cl0 + swz) * L.TCP;
      constexpr int NV = NOUT * G::VALS;  // partial sums a lane stores per token
      auto exchange = [&](const float* yc, float* ex) {
#pragma unroll
        for (int o = 0; o < NOUT; ++o) {
          float v[CL];
#pragma unroll
          for (int c = 0; c < CL; ++c) v[c] = yc[o * CL + c];
#pragma unroll
          for (int r = 0, nv = CL; r < G::XR; ++r, nv /= 2) {
#pragma unroll
            for (int u = 0; u < nv / 2; ++u) v[u] += __shfl_xor_sync(0xffffffffu, v[u + nv / 2], G::LANES_J << r);
          }
#pragma unroll
          for (int u = 0; u < G::VALS; ++u) ex[o * G::VALS + u] = v[u];
        }
      };
      auto slot = [&](int v) -> float* {  // destination of stored value v
        return ydst + (size_t)(v / G::VALS) * L.ypart_out() + (size_t)(v % G::VALS) * L.TCP;
      };
      f2 A[NPR], Bc[NPR], AI[NPR], KI[NPR], Q[NPR], QV[NPR], L2[CL], V2[CL];
      auto load_coef = [&](int t) {
        const float* ct = coef + t * NC * DK;
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
          if constexpr (!CKPT) {
            Q[2 * m] = q4.x;  Q[2 * m + 1] = q4.y;
          }
          if constexpr (MODE == 2) {
            const ulonglong2 v4 = *reinterpret_cast<const ulonglong2*>(ct + 5 * DK + 4 * m);
            QV[2 * m] = v4.x; QV[2 * m + 1] = v4.y;
          }
        }
#pragma unroll
        for (int c = 0; c < CL; ++c) {
          const ulonglong2 lv = *reinterpret_cast<const ulonglong2*>(pj + t * p.cc + (c ^ swz));
          L2[c] = lv.x; V2[c] = lv.y;
        }
      };
      // yc[c]: readout 0 of column register c; yc[CL + c]: readout 1 (MODE 2)
      auto compute = [&](float* yc) {
#pragma unroll
        for (int c = 0; c < CL; ++c) {
          f2 y2 = f2_make(0.0f, 0.0f), yv2 = f2_make(0.0f, 0.0f);
#pragma unroll
          for (int r = 0; r < NPR; ++r) {
            const f2 s = f2_fma(A[r], Pt[r][c], Bc[r]);
            const f2 d = f2_fma(s, L2[c], AI[r]);
            const f2 w = f2_rcp(d);
            Pt[r][c] = f2_mul(s, w);
            if constexpr (VAR) {
              y2 = f2_fma(Q[r], Pt[r][c], y2);  // (q²/K)·P̃ = q²·P
            } else {
              const f2 g = f2_mul(s, V2[c]);
              const f2 m = f2_fma(g, KI[r], Mu[r][c]);
              Mu[r][c] = f2_mul(m, w);
              if constexpr (!CKPT) y2 = f2_fma(Q[r], Mu[r][c], y2);
              if constexpr (MODE == 2) yv2 = f2_fma(QV[r], Pt[r][c], yv2);
            }
          }
          if constexpr (!CKPT) yc[c] = f2_lo(y2) + f2_hi(y2);
          if constexpr (MODE == 2) yc[CL + c] = f2_lo(yv2) + f2_hi(yv2);
        }
      };
      if constexpr (CKPT) {
        // State only (full tiles unrolled so that consecutive tokens' chains
        // overlap).
        if (tl == TC) {
#pragma unroll
          for (int t = 0; t < TC; ++t) {
            load_coef(t);
            compute(nullptr);
          }
        } else {
          for (int t = 0; t < tl; ++t) {
            load_coef(t);
            compute(nullptr);
          }
        }
      } else if (tl == TC) {
        // Full tile: tokens in batches of four. The previous batch's partial
        // sums are exchanged while this batch computes and stored with one
        // 128-bit store per value, so no store waits on a fresh result.
        // (Unrolled by at least two batches so that pb/cur are renamed, not
        // copied: a register move would cost a slot on the busy FMA pipe.
        // With eight rows per lane the whole tile is unrolled, which turns
        // the batch conditions and offsets into constants: 4-5% faster there,
        // 1% slower with four rows per lane.)
        constexpr int kBatchUnroll = RL == 8 ? TC / 4 : 2;
        float pb[4][NOUT * CL];
#pragma unroll kBatchUnroll
        for (int t4 = 0; t4 < TC; t4 += 4) {
          float cur[4][NOUT * CL], ex[4][NV];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            load_coef(t4 + u);
            if (t4 > 0) exchange(pb[u], ex[u]);
            compute(cur[u]);
          }
          if (t4 > 0) {
#pragma unroll
            for (int v = 0; v < NV; ++v)
              *reinterpret_cast<float4*>(slot(v) + t4 - 4) = make_float4(ex[0][v], ex[1][v], ex[2][v], ex[3][v]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int c = 0; c < NOUT * CL; ++c) pb[u][c] = cur[u][c];
        }
        float ex[4][NV];
#pragma unroll
        for (int u = 0; u < 4; ++u) exchange(pb[u], ex[u]);
#pragma unroll
        for (int v = 0; v < NV; ++v)
          *reinterpret_cast<float4*>(slot(v) + TC - 4) = make_float4(ex[0][v], ex[1][v], ex[2][v], ex[3][v]);
      } else {
        // Ragged last tile: one token at a time.
        for (int t = 0; t < tl; ++t) {
          float yc[NOUT * CL], ex[NV];
          load_coef(t);
          compute(yc);
          exchange(yc, ex);
#pragma unroll
          for (int v = 0; v < NV; ++v) slot(v)[t] = ex[v];
        }
      }
    }

    named_arrive(kBarEmpty0 + b, nall);
  }

  if constexpr (CKPT) checkpoint(ntiles);
  // ---- final state of the last chunk: λ_T = K_last / P̃, η_T = μ λ_T ---------
  if (z == (int)gridDim.z - 1 && p.lamT) {
    const float* klast = reinterpret_cast<const float*>(smem + L.kprev(ntiles & 1));
#pragma unroll
    for (int r = 0; r < NPR; ++r) {
#pragma unroll
      for (int c = 0; c < CL; ++c) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = i0 + 2 * r + h;
          const size_t e = (size_t)bh * E + (size_t)i * p.dv + jb + cl0 + (c ^ swz);
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

// Launch the MODE instantiation for (d_k, rows per lane).
template <typename IO, int MODE>
cudaError_t scan_launch_mode(int dk, int rl, dim3 grid, int threads, size_t smem, cudaStream_t s,
                             const KernelParams& kp) {
  switch (dk * 16 + rl) {
    case 16 * 16 + 4: return launch_kernel(kla_scan_kernel<IO, 16, 4, kTile, MODE>, grid, threads, smem, s, kp);
    case 32 * 16 + 4: return launch_kernel(kla_scan_kernel<IO, 32, 4, kTile, MODE>, grid, threads, smem, s, kp);
    case 64 * 16 + 4: return launch_kernel(kla_scan_kernel<IO, 64, 4, kTile, MODE>, grid, threads, smem, s, kp);
    case 64 * 16 + 8: return launch_kernel(kla_scan_kernel<IO, 64, 8, kTile, MODE>, grid, threads, smem, s, kp);
    case 128 * 16 + 4: return launch_kernel(kla_scan_kernel<IO, 128, 4, kTile, MODE>, grid, threads, smem, s, kp);
    case 128 * 16 + 8: return launch_kernel(kla_scan_kernel<IO, 128, 8, kTile, MODE>, grid, threads, smem, s, kp);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// One translation unit per mode (kla_scan_inst_*.cu) defines these.
cudaError_t scan_launch_y(int io, int dk, int rl, dim3 grid, int threads, size_t smem, cudaStream_t s,
                          const KernelParams& kp);
cudaError_t scan_launch_var(int io, int dk, int rl, dim3 grid, int threads, size_t smem, cudaStream_t s,
                            const KernelParams& kp);
cudaError_t scan_launch_y_var(int io, int dk, int rl, dim3 grid, int threads, size_t smem, cudaStream_t s,
                              const KernelParams& kp);
cudaError_t scan_launch_state(int io, int dk, int rl, dim3 grid, int threads, size_t smem, cudaStream_t s,
                              const KernelParams& kp);
cudaError_t scan_launch_y_pre(int io, int dk, int rl, dim3 grid, int threads, size_t smem, cudaStream_t s,
                              const KernelParams& kp);

}  // namespace kla
