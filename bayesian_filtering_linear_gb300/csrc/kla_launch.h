// Host-side interface between the C ABI (kla_api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace kla {

enum IoType { IO_F32 = 0, IO_BF16 = 1 };

struct ForwardArgs {
  const void *q, *k, *v, *lam_v, *a, *pbar;
  const float *lam0, *eta0;
  void* y;
  float *lamT, *etaT;
  int B, H, T, dk, dv;
  int io;      // IoType
  int gates;   // kla_gate bits: Λ^v, a, p̄ given as pre-activations
  void* y_var; // variance readout [B,H,T,dv] (scan mode 2), or null
};

// Launch geometry shared by the planner and the launchers.
struct Plan {
  int strategy;        // 1 sequential, 2 chunked
  int chunk_len;       // tokens per chunk (multiple of the tile length)
  int num_chunks;
  int cols_per_block;  // CC: d_v columns per thread block
  int rows_per_lane;   // RL: d_k rows held by one lane of the scan kernel
  int tile;            // TC: tokens staged per shared-memory tile
  int coef_pass;       // 1: the sequential plan reads per-row coefficients from the coefficient pass
  size_t ws_bytes;
};

// Geometry of the sequential / apply (scan) kernel and of the chunk
// composition kernel. The scan kernel is built for every RL that
// scan_rows_per_lane() lists for d_k; composition always uses
// rows_per_lane_for(d_k).
int rows_per_lane_for(int dk);
int scan_rows_per_lane(int dk, int* rl_out);  // the RL choices for d_k (at most 2); returns their count
int tile_for(int dk, int io);
int warp_cols(int dk, int rl);  // columns covered by one warp
int max_threads();              // largest number of scanning threads in a block
int producer_warps();           // extra warps per scan block that feed the scanning warps
size_t forward_smem_bytes(int dk, int rl, int io, int cc, int tile, int mode = 0);
size_t compose_smem_bytes(int dk, int io, int cc, int tile);

// Workspace layout for the chunked path (fp32 elements):
//   maps   [S-1][7][B·H·dk·dv]  per-chunk homogeneous maps (A,B,C,D,E,F,G)
//   starts [S][2][B·H·dk·dv]    chunk-start (P, μ)
size_t chunk_workspace_bytes(long long elems, int num_chunks);

// mode 0: y; 1: the variance readout y_var = Σ_i q_i² P_t into f.y instead
// of y (no mean); 2: both, y into f.y and y_var into f.y_var. With ckpt (a
// sequential plan only) the scan runs without a readout and stores the
// backward's checkpoints there instead (mode is then ignored).
cudaError_t launch_forward(const ForwardArgs& f, const Plan& p, const float* starts, cudaStream_t s,
                           float* ckpt = nullptr, int mode = 0, const float* coefs = nullptr);
// The coefficient pass: per-row coefficients of every token into `coefs`
// ([B·H][T][5][d_k] fp32, coef_workspace_bytes), read by the scan in mode 4.
cudaError_t launch_coef(const ForwardArgs& f, float* coefs, cudaStream_t s);
size_t coef_workspace_bytes(long long bh, int T, int dk);
// The scan stores its checkpoints every kScanTile tokens.
constexpr int kScanTile = 16;
cudaError_t launch_compose(const ForwardArgs& f, const Plan& p, float* maps, cudaStream_t s);
cudaError_t launch_carry(const ForwardArgs& f, const Plan& p, const float* maps, float* starts,
                         cudaStream_t s);
cudaError_t launch_init_state(const ForwardArgs& f, cudaStream_t s);
// Context-parallel sharding over T (kla_shard_map / kla_shard_start): the
// start state (λ, η) of a shard from the maps [n_maps][7][elems] of the shards
// before it, and the identity map (an empty shard).
cudaError_t launch_shard_start(const float* maps, int n_maps, const float* lam0, const float* eta0, float* lamS,
                               float* etaS, long long elems, cudaStream_t s);
cudaError_t launch_identity_map(float* maps, long long elems, cudaStream_t s);

// Backward pass (kla_backward.cu): gradients of a loss given dL/dy and
// optionally dL/dλ_T, dL/dη_T.
struct BackwardArgs {
  const void *q, *k, *v, *lam_v, *a, *pbar;
  const float *lam0, *eta0;
  const void* dy;                              // [B,H,T,dv] io, or null (zero)
  const float *dlamT, *detaT;                  // [B,H,dk,dv] fp32, or null (zero)
  void *dq, *dk_, *da, *dpbar, *dv_, *dlam_v;  // per-token gradients, io
  float *dlam0, *deta0;                        // [B,H,dk,dv] fp32, or null
  int B, H, T, dk, dv;
  int io;
  int gates;
};
struct BwdPlan {
  int cc, cpl, threads, ncb, nchunks;
  size_t ckpt_bytes, rowpart_bytes, smem;
};
BwdPlan backward_plan(long long bh, int T, int dk, int dv, int num_sms);
cudaError_t launch_backward(const BackwardArgs& f, const BwdPlan& b, void* workspace, cudaStream_t s);

struct StepArgs {
  const void *q, *k, *v, *lam_v, *a, *pbar;
  float *lam, *eta;
  void* y;
  int B, H, dk, dv;
  int io;
  int gates;
};
cudaError_t launch_step(const StepArgs& a, cudaStream_t s);

// Causal depthwise convolution with optional SiLU (kla_conv.cu), forward and
// backward. x, y, gy, gx: [B,H,T,D] io; weight [H,D,W], bias [H,D] fp32;
// windows [B,H,W-1,D] io. Null optional pointers mean zeros / not wanted.
struct ConvArgs {
  const void* x;
  const float *weight, *bias;
  const void* win;    // carried inputs before token 0
  void *y, *wout;     // forward outputs
  const void *gy, *gwout;
  void *gx, *gwin;    // backward outputs (io)
  float *gweight, *gbias;
  float* part;        // backward block partials [H][nparts][D][W+1], or null (no gweight/gbias)
  long long nparts;   // B · blocks along T; set by the backward launcher
  int B, H, T, D, W;
  int io, act;
  int chunks_per_block;  // token groups (of four or eight) per stage; set by the launchers
  int range;             // tokens per block; set by the launchers
};
// Both launchers choose their geometry (tokens per block from conv_range()
// for `num_sms` SMs). The backward's per-block partial sums of the tap and
// bias gradients need conv_partial_bytes() of workspace in `part`.
int conv_range(long long bh, int T, long long TT, int num_sms, int min_stages, long long* blocks_y);
size_t conv_partial_bytes(int B, int H, int T, int D, int W, int num_sms);
cudaError_t launch_conv(const ConvArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_conv_backward(const ConvArgs& a, int num_sms, cudaStream_t s);

}  // namespace kla
