// Scan kernel instantiations for MODE 0 (the readout y), both I/O types.
#include "kla_scan_kernel.cuh"

namespace kla {

cudaError_t scan_launch_y(int io, int dk, int rl, dim3 grid, int threads, size_t smem, cudaStream_t s,
                          const KernelParams& kp) {
  return io == IO_BF16 ? scan_launch_mode<__nv_bfloat16, 0>(dk, rl, grid, threads, smem, s, kp)
                       : scan_launch_mode<float, 0>(dk, rl, grid, threads, smem, s, kp);
}

}  // namespace kla
