// Scan kernel instantiations for MODE 4 (the readout y with per-row
// coefficients from the coefficient pass), both I/O types, and the
// coefficient pass itself.
#include <algorithm>

#include "kla_scan_kernel.cuh"

namespace kla {

cudaError_t scan_launch_y_pre(int io, int dk, int rl, dim3 grid, int threads, size_t smem, cudaStream_t s,
                              const KernelParams& kp) {
  return io == IO_BF16 ? scan_launch_mode<__nv_bfloat16, 4>(dk, rl, grid, threads, smem, s, kp)
                       : scan_launch_mode<float, 4>(dk, rl, grid, threads, smem, s, kp);
}

size_t coef_workspace_bytes(long long bh, int T, int dk) {
  return (size_t)bh * (size_t)T * 5 * (size_t)dk * sizeof(float);
}

namespace {
template <typename IO, int DK>
cudaError_t coef_launch(const KernelParams& kp, float* coefs, long long bh, dim3 grid, cudaStream_t s) {
  if (kp.gates)
    kla_coef_kernel<IO, DK, true><<<grid, 256, 0, s>>>(kp, coefs, bh);
  else
    kla_coef_kernel<IO, DK, false><<<grid, 256, 0, s>>>(kp, coefs, bh);
  return cudaGetLastError();
}
template <typename IO>
cudaError_t coef_launch_io(int dk, const KernelParams& kp, float* coefs, long long bh, dim3 grid, cudaStream_t s) {
  switch (dk) {
    case 16: return coef_launch<IO, 16>(kp, coefs, bh, grid, s);
    case 32: return coef_launch<IO, 32>(kp, coefs, bh, grid, s);
    case 64: return coef_launch<IO, 64>(kp, coefs, bh, grid, s);
    case 128: return coef_launch<IO, 128>(kp, coefs, bh, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_coef(const ForwardArgs& f, float* coefs, cudaStream_t s) {
  const long long bh = (long long)f.B * f.H;
  if (bh == 0 || f.T == 0) return cudaSuccess;
  KernelParams kp{};
  kp.q = f.q; kp.k = f.k; kp.a = f.a; kp.pbar = f.pbar;
  kp.T = f.T;
  kp.gates = f.gates;
  // token blocks along x (up to 2^31 - 1), heads along y in a grid-stride loop
  const dim3 grid((unsigned)((f.T + kCoefTokens - 1) / kCoefTokens), (unsigned)std::min<long long>(bh, 65535));
  return f.io == IO_BF16 ? coef_launch_io<__nv_bfloat16>(f.dk, kp, coefs, bh, grid, s)
                         : coef_launch_io<float>(f.dk, kp, coefs, bh, grid, s);
}

}  // namespace kla
