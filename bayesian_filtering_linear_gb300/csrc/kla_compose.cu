// Chunk-parallel path over T for sm_103a: composition of each chunk's
// per-element map, the carry of the maps across chunks, and the state copy
// used when T = 0. The chunks are then re-run by the scan kernel
// (kla_scan_kernel.cuh) from their carried start states.
//
// Source: "Technische Samenvatting: Kalman Linear Attention (KLA)"
// (gist.science/nl/paper/2602.10743), Methodologie §2: the precision updates
// are Möbius maps that compose associatively, and the information-mean
// updates are affine, so a long sequence can be cut into chunks whose maps
// are built independently and then combined.
#include <type_traits>

#include "kla_common.cuh"
#include "kla_launch.h"

namespace kla {

namespace {

constexpr int kComposeTile = 16;

// Shared memory of the composition kernel: two raw tiles, one tile of row
// coefficients (a², p̄, K, k, a) and one of column terms.
template <typename IO, int DK, int TC>
struct ComposeLayout {
  int cc;
  __host__ __device__ explicit ComposeLayout(int cc_) : cc(cc_) {}
  __host__ __device__ size_t raw(int b) const { return b * RawTile<IO, DK, TC>::bytes(cc); }
  __host__ __device__ size_t coef() const { return raw(2); }
  __host__ __device__ size_t pj() const { return coef() + (size_t)TC * 5 * DK * sizeof(float); }
  __host__ __device__ size_t total() const { return pj() + (size_t)TC * cc * sizeof(float4); }
};

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
  const ComposeLayout<IO, DK, TC> L(p.cc);
  float* coef = reinterpret_cast<float*>(smem + L.coef());
  float4* pj = reinterpret_cast<float4*>(smem + L.pj());

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long bh = blockIdx.x;
  const int jb = blockIdx.y * p.cc;
  const int z = blockIdx.z;
  const int t_begin = z * p.chunk_len;
  const int t_end = min(p.T, t_begin + p.chunk_len);
  const int ntiles = (t_end - t_begin + TC - 1) / TC;
  const int li = lane / G::LANES_J, lj = lane % G::LANES_J;
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

  stage_raw<IO, DK, TC>(p, smem + L.raw(0), bh, jb, t_begin, min(TC, t_end - t_begin), tid, blockDim.x);
  cp_async_commit();
  for (int n = 0; n < ntiles; ++n) {
    const int t0 = t_begin + n * TC;
    const int tl = min(TC, t_end - t0);
    if (n + 1 < ntiles) {
      const int t1 = t0 + TC;
      stage_raw<IO, DK, TC>(p, smem + L.raw((n + 1) & 1), bh, jb, t1, min(TC, t_end - t1), tid, blockDim.x);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    {
      const unsigned char* buf = smem + L.raw(n & 1);
      const IO* rk = reinterpret_cast<const IO*>(buf) + TC * DK;
      const IO* ra = rk + TC * DK;
      const IO* rp = ra + TC * DK;
      // (the gate activations are a separate instantiation: no extra work
      // without them)
      auto coefficients = [&](auto gated) {
        constexpr bool GT = decltype(gated)::value;
        for (int idx = tid; idx < tl * DK; idx += blockDim.x) {
          const int t = idx / DK, i = idx % DK;
          const float kt = to_f32<IO>(rk[idx]);
          const float xa = to_f32<IO>(ra[idx]);
          const float at = fmaxf(GT ? gate_a(xa, p.gates) : xa, kAMin);
          const float xp = to_f32<IO>(rp[idx]);
          float* ct = coef + t * 5 * DK + i;
          ct[0 * DK] = at * at;                                 // a²
          ct[1 * DK] = GT ? gate_pbar(xp, xa, p.gates) : xp;   // p̄
          ct[2 * DK] = fmaf(kt, kt, kK2Floor);                 // k² (floored as in the scan)
          ct[3 * DK] = kt;                                      // k
          ct[4 * DK] = at;                                      // a
        }
        column_terms<IO, DK, TC, GT>(buf, pj, p.cc, tl, tid, blockDim.x, p.gates);
      };
      if (p.gates) coefficients(std::true_type{});
      else coefficients(std::false_type{});
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

// Context-parallel sharding over T: the start state of a shard from the maps
// of the shards before it, applied in order to (λ0, η0) (or 1 and 0), in
// information form: λ = 1/P, η = μ/P. Each thread reads its element's
// initial state before writing, so the output may alias lam0/eta0.
__global__ void kla_shard_start_kernel(const float* __restrict__ maps, int n_maps, const float* lam0,
                                       const float* eta0, float* lamS, float* etaS, long long elems) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= elems) return;
  float P = 1.0f, mu = 0.0f;
  if (lam0) {
    P = 1.0f / lam0[e];
    mu = eta0[e] * P;
  }
  for (int z = 0; z < n_maps; ++z) {
    const float* m = maps + (size_t)z * 7 * elems + e;
    const float A = m[0], B = m[elems], C = m[2 * elems], D = m[3 * elems];
    const float E = m[4 * elems], F = m[5 * elems], Gm = m[6 * elems];
    const float nn = fmaf(A, P, B);
    const float mm = fmaf(C, P, D);
    const float ee = fmaf(E, P, fmaf(Gm, mu, F));
    P = nn / mm;
    mu = ee / mm;
  }
  lamS[e] = 1.0f / P;
  etaS[e] = mu / P;
}

// The identity map (A, D, G = 1; B, C, E, F = 0): the map of an empty shard.
__global__ void kla_identity_map_kernel(float* maps, long long elems) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= elems) return;
#pragma unroll
  for (int q = 0; q < 7; ++q) maps[(size_t)q * elems + e] = (q == 0 || q == 3 || q == 6) ? 1.0f : 0.0f;
}

}  // namespace

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {
template <typename IO>
size_t compose_smem(int dk, int cc) {
  switch (dk) {
    case 16: return ComposeLayout<IO, 16, kComposeTile>(cc).total();
    case 32: return ComposeLayout<IO, 32, kComposeTile>(cc).total();
    case 64: return ComposeLayout<IO, 64, kComposeTile>(cc).total();
    default: return ComposeLayout<IO, 128, kComposeTile>(cc).total();
  }
}

template <typename IO>
cudaError_t compose_dispatch(int dk, dim3 grid, int threads, size_t smem, cudaStream_t s, const KernelParams& kp) {
  switch (dk) {
    case 16:
      return launch_kernel(kla_compose_kernel<IO, 16, RowsPerLane<16>::value, kComposeTile>, grid, threads, smem, s, kp);
    case 32:
      return launch_kernel(kla_compose_kernel<IO, 32, RowsPerLane<32>::value, kComposeTile>, grid, threads, smem, s, kp);
    case 64:
      return launch_kernel(kla_compose_kernel<IO, 64, RowsPerLane<64>::value, kComposeTile>, grid, threads, smem, s, kp);
    case 128:
      return launch_kernel(kla_compose_kernel<IO, 128, RowsPerLane<128>::value, kComposeTile>, grid, threads, smem, s, kp);
    default:
      return cudaErrorInvalidValue;
  }
}
}  // namespace

size_t compose_smem_bytes(int dk, int io, int cc, int /*tile*/) {
  return io == IO_BF16 ? compose_smem<__nv_bfloat16>(dk, cc) : compose_smem<float>(dk, cc);
}

size_t chunk_workspace_bytes(long long elems, int num_chunks) {
  if (num_chunks <= 1) return 0;
  return (size_t)(7 * (num_chunks - 1) + 2 * num_chunks) * (size_t)elems * sizeof(float);
}

cudaError_t launch_compose(const ForwardArgs& f, const Plan& p, float* maps, cudaStream_t s) {
  if (p.num_chunks <= 1) return cudaSuccess;
  KernelParams kp = make_params(f, p);
  kp.maps = maps;
  const dim3 grid((unsigned)((long long)f.B * f.H), (unsigned)(f.dv / p.cols_per_block), (unsigned)(p.num_chunks - 1));
  const int threads = 32 * (p.cols_per_block / warp_cols(f.dk, rows_per_lane_for(f.dk)));
  const size_t smem = compose_smem_bytes(f.dk, f.io, p.cols_per_block, 0);
  return f.io == IO_BF16 ? compose_dispatch<__nv_bfloat16>(f.dk, grid, threads, smem, s, kp)
                         : compose_dispatch<float>(f.dk, grid, threads, smem, s, kp);
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

namespace kla {

cudaError_t launch_shard_start(const float* maps, int n_maps, const float* lam0, const float* eta0, float* lamS,
                               float* etaS, long long elems, cudaStream_t s) {
  if (elems == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = (unsigned)((elems + threads - 1) / threads);
  kla_shard_start_kernel<<<blocks, threads, 0, s>>>(maps, n_maps, lam0, eta0, lamS, etaS, elems);
  return cudaGetLastError();
}

cudaError_t launch_identity_map(float* maps, long long elems, cudaStream_t s) {
  if (elems == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = (unsigned)((elems + threads - 1) / threads);
  kla_identity_map_kernel<<<blocks, threads, 0, s>>>(maps, elems);
  return cudaGetLastError();
}

}  // namespace kla
