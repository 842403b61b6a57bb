// Scan kernel instantiations for MODE 1 (the variance readout alone), both I/O types.
#include "kla_scan_kernel.cuh"

namespace kla {

cudaError_t scan_launch_var(int io, int dk, int rl, dim3 grid, int threads, size_t smem, cudaStream_t s,
                            const KernelParams& kp) {
  return io == IO_BF16 ? scan_launch_mode<__nv_bfloat16, 1>(dk, rl, grid, threads, smem, s, kp)
                       : scan_launch_mode<float, 1>(dk, rl, grid, threads, smem, s, kp);
}

}  // namespace kla
