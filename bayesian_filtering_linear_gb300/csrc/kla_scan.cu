// Sequence scan of the KLA filter, host side: geometry queries, shared-memory
// sizes and the launch of the kernel in kla_scan_kernel.cuh (instantiated in
// kla_scan_inst_*.cu).
#include "kla_scan_kernel.cuh"

namespace kla {

// ---------------------------------------------------------------------------
// Host side: geometry and launch.
// ---------------------------------------------------------------------------
int rows_per_lane_for(int dk) {
  switch (dk) {
    case 16: return RowsPerLane<16>::value;
    case 32: return RowsPerLane<32>::value;
    case 64: return RowsPerLane<64>::value;
    default: return RowsPerLane<128>::value;
  }
}
int scan_rows_per_lane(int dk, int* rl_out) {
  // d_k <= 32: four rows per lane only (a warp covers the head's rows with
  // no more than 8 lanes); 64 and 128: eight rows per lane, or four for
  // finer column blocks (more blocks for few heads).
  if (dk <= 32) {
    rl_out[0] = 4;
    return 1;
  }
  rl_out[0] = 8;
  rl_out[1] = 4;
  return 2;
}
int tile_for(int /*dk*/, int /*io*/) { return kTile; }
int max_threads() { return kMaxThreads; }
int producer_warps() { return kProducerWarps; }
int warp_cols(int dk, int rl) { return (32 / (dk / rl)) * CL; }

namespace {
template <typename IO, int DK, int RL>
size_t scan_smem(int cc, int mode) {
  using G = Geo<DK, RL>;
  return mode == 2 ? ScanLayout<IO, DK, kTile, G::NP, 6, 2>(cc).total() : ScanLayout<IO, DK, kTile, G::NP>(cc).total();
}
template <typename IO>
size_t scan_smem_io(int dk, int rl, int cc, int mode) {
  switch (dk * 16 + rl) {
    case 16 * 16 + 4: return scan_smem<IO, 16, 4>(cc, mode);
    case 32 * 16 + 4: return scan_smem<IO, 32, 4>(cc, mode);
    case 64 * 16 + 4: return scan_smem<IO, 64, 4>(cc, mode);
    case 64 * 16 + 8: return scan_smem<IO, 64, 8>(cc, mode);
    case 128 * 16 + 4: return scan_smem<IO, 128, 4>(cc, mode);
    case 128 * 16 + 8: return scan_smem<IO, 128, 8>(cc, mode);
    default: return 0;
  }
}
cudaError_t scan_dispatch(int io, int dk, int rl, int mode, dim3 grid, int threads, size_t smem, cudaStream_t s,
                          const KernelParams& kp) {
  switch (mode) {
    case 0: return scan_launch_y(io, dk, rl, grid, threads, smem, s, kp);
    case 1: return scan_launch_var(io, dk, rl, grid, threads, smem, s, kp);
    case 2: return scan_launch_y_var(io, dk, rl, grid, threads, smem, s, kp);
    case 4: return scan_launch_y_pre(io, dk, rl, grid, threads, smem, s, kp);
    default: return scan_launch_state(io, dk, rl, grid, threads, smem, s, kp);
  }
}
}  // namespace

size_t forward_smem_bytes(int dk, int rl, int io, int cc, int /*tile*/, int mode) {
  return io == IO_BF16 ? scan_smem_io<__nv_bfloat16>(dk, rl, cc, mode) : scan_smem_io<float>(dk, rl, cc, mode);
}

static_assert(kTile == kScanTile, "checkpoints are taken once per tile");

cudaError_t launch_forward(const ForwardArgs& f, const Plan& p, const float* starts, cudaStream_t s, float* ckpt,
                           int mode, const float* coefs) {
  KernelParams kp = make_params(f, p);
  kp.starts = starts;
  kp.ckpt = ckpt;
  kp.coefs = coefs;
  if (ckpt) mode = 3;
  if (coefs) mode = 4;  // y with the coefficient pass's output (one chunk)
  const dim3 grid((unsigned)((long long)f.B * f.H), (unsigned)(f.dv / p.cols_per_block), (unsigned)p.num_chunks);
  const int threads = 32 * (p.cols_per_block / warp_cols(f.dk, p.rows_per_lane) + kProducerWarps);
  const size_t smem = forward_smem_bytes(f.dk, p.rows_per_lane, f.io, p.cols_per_block, p.tile, mode);
  return scan_dispatch(f.io, f.dk, p.rows_per_lane, mode, grid, threads, smem, s, kp);
}

}  // namespace kla
