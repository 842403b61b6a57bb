// C ABI of the KLA scan library: argument validation, the launch planner and
// the entry points declared in include/kla.h. Host code only; the kernels are
// in kla_scan_kernel.cuh (sequence scan; launched from kla_scan.cu),
// kla_compose.cu (chunk compose and carry),
// kla_noalloc.cu (the allocation-free chunked path), kla_step.cu (decode step)
// and kla_backward.cu (backward pass).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "kla.h"
#include "kla_launch.h"

namespace {

using kla::Plan;

constexpr size_t kMaxSmem = 227 * 1024;
constexpr int kChunkAlign = 32;  // chunk lengths are multiples of the largest tile

bool valid_d(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t io_size(int io) { return io == KLA_BF16 ? 2 : 4; }

// Shape checks shared by every entry point that takes (B, H, T, dk, dv).
kla_status check_shape(int B, int H, int T, int dk, int dv) {
  if (B < 0 || H < 0 || T < 0) return KLA_ERR_INVALID_ARG;
  if (!valid_d(dk) || !valid_d(dv)) return KLA_ERR_UNSUPPORTED_SHAPE;
  const long long bh = (long long)B * H;
  if (bh > INT_MAX) return KLA_ERR_UNSUPPORTED_SHAPE;
  // Element counts must fit comfortably in 64-bit offsets.
  if (bh > 0 && (long long)T > (1LL << 46) / (bh * 128)) return KLA_ERR_UNSUPPORTED_SHAPE;
  return KLA_OK;
}

// Options for a head of dk rows (dk already checked).
bool valid_gates(int g) {
  return (g & ~15) == 0 && !((g & KLA_GATE_PBAR_SOFTPLUS) && (g & KLA_GATE_PBAR_OU));
}

kla_status check_options(const kla_options* opt, int dk) {
  if (!opt) return KLA_OK;
  if (!valid_gates(opt->gates)) return KLA_ERR_INVALID_ARG;
  if (opt->strategy < KLA_AUTO || opt->strategy > KLA_CHUNKED) return KLA_ERR_INVALID_ARG;
  if (opt->chunk_len < 0 || opt->chunk_len % kChunkAlign != 0) return KLA_ERR_INVALID_ARG;
  if (opt->coef_pass < KLA_COEF_AUTO || opt->coef_pass > KLA_COEF_ON) return KLA_ERR_INVALID_ARG;
  if (opt->rows_per_lane != 0) {  // must be a geometry the scan kernel is built for
    int rls[2];
    const int nrl = kla::scan_rows_per_lane(dk, rls);
    bool ok = false;
    for (int n = 0; n < nrl; ++n) ok = ok || rls[n] == opt->rows_per_lane;
    if (!ok) return KLA_ERR_INVALID_ARG;
  }
  return KLA_OK;
}

// ---- planner -----------------------------------------------------------------
//
// Cost model in sub-partition (SMSP) cycles. A warp advancing one token does
// RL·2·32 element-steps, each needing one MUFU reciprocal at 4 per SMSP-cycle.
// Blocks of CC columns (CC/wc warps) are spread evenly over the SMs and a
// block's warps over the 4 sub-partitions, so the busiest sub-partition
// carries ceil(ceil(blocks/SMs) · warps/4) warps. Per-row coefficients cost
// about 4.5 columns' worth of work per block; a sub-partition with a single
// warp issues at ~0.7 of its rate (latency), two or more at ~0.9. With four
// rows per lane the per-element share of coefficient loads and readout is
// larger: ~1.15× the work per element-step at d_k = 64 and ~1.45× at 128
// (sixteen partial sums per output instead of eight). Chunk composition costs ~1.6× a
// scan step. Fixed costs: ~2 tiles of pipeline fill per block, ~4000 cycles
// per kernel launch, and the carry kernel's traffic (9 floats per element per
// chunk at ~6.6 TB/s, ~1.95 GHz).
constexpr double kLaunchCycles = 4000.0;
constexpr double kCyclesPerByte = 1.95e9 / 6.6e12;

struct Candidate {
  int cc, rl;
  double cost;
};

int blocks_per_sm_limit(int dk, int rl, int io, int cc, int tile, int wc, bool compose) {
  const size_t smem =
      compose ? kla::compose_smem_bytes(dk, io, cc, tile) : kla::forward_smem_bytes(dk, rl, io, cc, tile);
  if (smem == 0 || smem > kMaxSmem) return 0;
  if (32 * (cc / wc) > kla::max_threads()) return 0;
  const int threads = 32 * (cc / wc) + (compose ? 0 : 32 * kla::producer_warps());
  const int by_smem = (int)((kMaxSmem + 1024) / (smem + 1024));
  const int by_threads = 2048 / threads;
  return std::max(0, std::min(by_smem, by_threads));
}

// One pass (scan, or composition when `compose`) over `tokens` tokens of
// every block: bh heads × dv/cc column blocks × blocks_z chunks.
double pass_cost(long long bh, int dk, int rl, int dv, int io, int cc, int tile, int num_sms, long long blocks_z,
                 bool compose, long long tokens) {
  const int wc = kla::warp_cols(dk, rl);
  const int bps = blocks_per_sm_limit(dk, rl, io, cc, tile, wc, compose);
  if (bps == 0) return INFINITY;
  const long long blocks = bh * (dv / cc) * blocks_z;
  const long long per_sm = (blocks + num_sms - 1) / num_sms;
  const long long waves = (per_sm + bps - 1) / bps;
  const long long resident = std::min<long long>(per_sm, bps);
  const long long warps_sm = resident * (cc / wc);
  const long long warps_smsp = (warps_sm + 3) / 4;
  const double eff = warps_smsp >= 2 ? 0.9 : 0.7;
  const double step_cost = (compose ? 1.6 : 1.0) * (rl == 4 && dk >= 64 ? (dk == 64 ? 1.15 : 1.45) : 1.0);
  const double warp_token = 8.0 * rl * 2;  // cycles per warp per token
  return kLaunchCycles + (double)waves * (double)(tokens + 2 * tile) * (double)warps_smsp * warp_token *
                             (step_cost + 4.5 / cc) / eff;
}

// The coefficient pass (kla_coef_pass) under KLA_COEF_AUTO: taken when a
// head's columns span at least kCoefMinBlocks blocks (each would build the
// same per-row coefficients) of at most kCoefMaxCols columns (a block's
// per-row work is shared by its columns, so it weighs more in narrow
// blocks), and its buffer is at most kCoefMaxBytes. Measured on GB300: 4 or
// 8 blocks of 16 columns 10-12% faster with the pass; 4 blocks of 32 columns
// 1% slower, 2 blocks of 32 columns 8% slower, one block of 64 14% slower.
constexpr int kCoefMinBlocks = 4;
constexpr int kCoefMaxCols = 16;
constexpr size_t kCoefMaxBytes = (size_t)16 << 30;

// allow_coef: the caller can run the coefficient pass (kla_forward's plain
// readout; not the uncertainty readout or the allocation-free entry point).
kla_status make_plan(int B, int H, int T, int dk, int dv, int io, const kla_options* opt, int num_sms,
                     Plan* out, bool allow_coef = true) {
  kla_status st = check_shape(B, H, T, dk, dv);
  if (st != KLA_OK) return st;
  if ((st = check_options(opt, dk)) != KLA_OK) return st;
  if (io != KLA_F32 && io != KLA_BF16) return KLA_ERR_INVALID_ARG;
  if (num_sms < 1) return KLA_ERR_INVALID_ARG;
  const int strategy = opt ? opt->strategy : KLA_AUTO;
  const int fixed_len = opt ? opt->chunk_len : 0;
  const long long bh = (long long)B * H;
  const long long elems = bh * dk * dv;
  const int tile = kla::tile_for(dk, io);
  int rls[2];
  int nrl = kla::scan_rows_per_lane(dk, rls);
  if (opt && opt->rows_per_lane != 0) {  // fixed by the caller (checked above)
    rls[0] = opt->rows_per_lane;
    nrl = 1;
  }
  const int rl_compose = kla::rows_per_lane_for(dk);

  // Cheapest (column block, rows per lane) for a split into num_chunks
  // chunks of chunk_len tokens.
  auto best_geometry = [&](int num_chunks, int chunk_len) {
    Candidate best{0, 0, INFINITY};
    for (int n = 0; n < nrl; ++n) {
      const int rl = rls[n], wc = kla::warp_cols(dk, rl);
      int cc_min = std::max<int>(wc, (int)(16 / io_size(io)));
      if (num_chunks > 1) cc_min = std::max(cc_min, kla::warp_cols(dk, rl_compose));
      if (n == 0) best = {cc_min, rl, INFINITY};  // kept only if nothing fits
      const int cc_max = std::min(dv, kla::max_threads() / 32 * wc);
      for (int cc = cc_max; cc >= cc_min; cc /= 2) {
        double c = pass_cost(bh, dk, rl, dv, io, cc, tile, num_sms, num_chunks, false, chunk_len);
        if (num_chunks > 1) {
          c += pass_cost(bh, dk, rl_compose, dv, io, cc, tile, num_sms, num_chunks - 1, true, chunk_len);
          c += kLaunchCycles + kCyclesPerByte * 36.0 * (double)num_chunks * (double)elems;
        }
        if (c < best.cost) best = {cc, rl, c};
      }
    }
    return best;
  };

  Plan p{};
  p.tile = tile;
  const long long Tl = std::max(T, 1);
  const Candidate seq = best_geometry(1, (int)Tl);
  p.strategy = KLA_SEQUENTIAL;
  p.chunk_len = (int)Tl;
  p.num_chunks = 1;
  p.cols_per_block = seq.cc;
  p.rows_per_lane = seq.rl;

  if (strategy == KLA_CHUNKED || strategy == KLA_AUTO) {
    int best_len = 0;
    Candidate best_c{0, 0, INFINITY};
    auto consider = [&](long long len) {
      len = ((len + kChunkAlign - 1) / kChunkAlign) * kChunkAlign;
      if (len < kChunkAlign) len = kChunkAlign;
      const long long S = (Tl + len - 1) / len;
      if (S < 2 || S > 65535) return;
      const Candidate c = best_geometry((int)S, (int)len);
      if (c.cost < best_c.cost) {
        best_c = c;
        best_len = (int)len;
      }
    };
    if (fixed_len > 0) {
      consider(fixed_len);
    } else {
      for (int S = 2; S <= 256; S = S < 8 ? S + 1 : S * 2) consider((Tl + S - 1) / S);
    }
    const bool take = strategy == KLA_CHUNKED ? best_len > 0 : (best_len > 0 && best_c.cost < seq.cost);
    if (take) {
      p.strategy = KLA_CHUNKED;
      p.chunk_len = best_len;
      p.num_chunks = (int)((Tl + best_len - 1) / best_len);
      p.cols_per_block = best_c.cc;
      p.rows_per_lane = best_c.rl;
    }
  }
  const int coef = opt ? opt->coef_pass : KLA_COEF_AUTO;
  if (allow_coef && p.strategy == KLA_SEQUENTIAL && bh > 0 && T > 0 && coef != KLA_COEF_OFF) {
    const bool split = dv / p.cols_per_block >= kCoefMinBlocks && p.cols_per_block <= kCoefMaxCols;
    p.coef_pass = coef == KLA_COEF_ON || (split && kla::coef_workspace_bytes(bh, T, dk) <= kCoefMaxBytes);
  }
  p.ws_bytes = p.strategy == KLA_CHUNKED ? kla::chunk_workspace_bytes(elems, p.num_chunks)
               : p.coef_pass          ? kla::coef_workspace_bytes(bh, T, dk)
                                      : 0;
  *out = p;
  return KLA_OK;
}

// Per-device SM count, queried once.
std::atomic<int> g_sms[256];

kla_status device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KLA_ERR_CUDA;
  if (dev < 0 || dev >= 256) return KLA_ERR_CUDA;
  int n = g_sms[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return KLA_ERR_CUDA;
    g_sms[dev].store(n, std::memory_order_relaxed);
  }
  *sms = n;
  return KLA_OK;
}

bool overlaps_partially(const void* x, const void* y, size_t bytes) {
  if (!x || !y || x == y) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(y);
  return a < b + bytes && b < a + bytes;
}

// Byte ranges [x, x + nx) and [y, y + ny) intersect (null or empty ranges never do).
bool ranges_overlap(const void* x, size_t nx, const void* y, size_t ny) {
  if (!x || !y || nx == 0 || ny == 0) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(y);
  return a < b + ny && b < a + nx;
}

// Shape checks of the causal convolution entry points.
kla_status check_conv_shape(int B, int H, int T, int D, int W) {
  if (B < 0 || H < 0 || T < 0) return KLA_ERR_INVALID_ARG;
  if (D < 4 || D > 512 || D % 4 != 0 || W < 1 || W > 8) return KLA_ERR_UNSUPPORTED_SHAPE;
  const long long bh = (long long)B * H;
  if (bh > INT_MAX) return KLA_ERR_UNSUPPORTED_SHAPE;
  if (bh > 0 && (long long)T > (1LL << 46) / (bh * D)) return KLA_ERR_UNSUPPORTED_SHAPE;
  return KLA_OK;
}

void fill_info(const Plan& p, kla_plan_info* out) {
  out->strategy = p.strategy;
  out->chunk_len = p.chunk_len;
  out->num_chunks = p.num_chunks;
  out->cols_per_block = p.cols_per_block;
  out->workspace_bytes = p.ws_bytes;
  out->rows_per_lane = p.rows_per_lane;
  out->coef_pass = p.coef_pass;
}


// kla_forward, and with y_var the variance readout of kla_forward_uncertainty.
kla_status forward_impl(const void* q, const void* k, const void* v, const void* lam_v, const void* a,
                       const void* pbar, const float* lam0, const float* eta0, void* y, float* lamT,
                       float* etaT, int B, int H, int T, int dk, int dv, kla_dtype io, void* workspace,
                       size_t ws_bytes, const kla_options* opt, void* stream, void* y_var) {
  // ---- validation: no CUDA call before it passes ---------------------------
  kla_status st = check_shape(B, H, T, dk, dv);
  if (st != KLA_OK) return st;
  if ((st = check_options(opt, dk)) != KLA_OK) return st;
  if (io != KLA_F32 && io != KLA_BF16) return KLA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  const long long tokens = bh * T;
  if ((lam0 == nullptr) != (eta0 == nullptr)) return KLA_ERR_INVALID_ARG;
  if ((lamT == nullptr) != (etaT == nullptr)) return KLA_ERR_INVALID_ARG;
  if (tokens > 0 && (!q || !k || !v || !lam_v || !a || !pbar || !y)) return KLA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, lam_v, a, pbar, lam0, eta0, y, lamT, etaT, y_var};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KLA_ERR_MISALIGNED;
  const size_t state_bytes = (size_t)bh * dk * dv * sizeof(float);
  if (overlaps_partially(lamT, lam0, state_bytes) || overlaps_partially(etaT, eta0, state_bytes) ||
      overlaps_partially(lamT, eta0, state_bytes) || overlaps_partially(etaT, lam0, state_bytes) ||
      (lamT && lamT == (const float*)eta0) || (etaT && etaT == (const float*)lam0))
    return KLA_ERR_INVALID_ARG;
  if (lamT && overlaps_partially(lamT, etaT, state_bytes)) return KLA_ERR_INVALID_ARG;
  if (lamT && lamT == etaT) return KLA_ERR_INVALID_ARG;
  if (y_var && (y_var == y || overlaps_partially(y_var, y, (size_t)tokens * dv * (io == KLA_BF16 ? 2 : 4))))
    return KLA_ERR_INVALID_ARG;
  if (bh == 0) return KLA_OK;

  int sms = 0;
  if ((st = device_sms(&sms)) != KLA_OK) return st;
  Plan p{};
  if ((st = make_plan(B, H, T, dk, dv, io, opt, sms, &p, y_var == nullptr)) != KLA_OK) return st;
  if (p.ws_bytes > 0 && (!workspace || ws_bytes < p.ws_bytes)) return KLA_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return KLA_ERR_MISALIGNED;

  kla::ForwardArgs f{q, k, v, lam_v, a, pbar, lam0, eta0, y, lamT, etaT, B, H, T, dk, dv, (int)io,
                     opt ? opt->gates : 0};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  // The variance readout (when asked for) is fused into the scan (mode 2)
  // when that kernel's shared memory fits; otherwise it is a separate pass
  // without the mean (mode 1), run before the main pass, which may
  // overwrite λ0/η0 in place.
  const bool fused = y_var && kla::forward_smem_bytes(dk, p.rows_per_lane, io, p.cols_per_block, p.tile, 2) <=
                                  kMaxSmem;
  f.y_var = fused ? y_var : nullptr;
  kla::ForwardArgs fv = f;
  fv.y = y_var;
  fv.y_var = nullptr;
  fv.lamT = fv.etaT = nullptr;
  const int main_mode = fused ? 2 : 0;
  const bool var_pass = y_var && !fused;
  if (T == 0) {
    e = kla::launch_init_state(f, s);
  } else if (p.strategy == KLA_SEQUENTIAL && p.coef_pass) {  // no y_var here (allow_coef above)
    float* coefs = reinterpret_cast<float*>(workspace);
    e = kla::launch_coef(f, coefs, s);
    if (e == cudaSuccess) e = kla::launch_forward(f, p, nullptr, s, nullptr, 0, coefs);
  } else if (p.strategy == KLA_SEQUENTIAL) {
    e = var_pass ? kla::launch_forward(fv, p, nullptr, s, nullptr, 1) : cudaSuccess;
    if (e == cudaSuccess) e = kla::launch_forward(f, p, nullptr, s, nullptr, main_mode);
  } else {
    const long long elems = bh * dk * dv;
    float* maps = reinterpret_cast<float*>(workspace);
    float* starts = maps + (size_t)7 * (p.num_chunks - 1) * elems;
    e = kla::launch_compose(f, p, maps, s);
    if (e == cudaSuccess) e = kla::launch_carry(f, p, maps, starts, s);
    if (e == cudaSuccess && var_pass) e = kla::launch_forward(fv, p, starts, s, nullptr, 1);
    if (e == cudaSuccess) e = kla::launch_forward(f, p, starts, s, nullptr, main_mode);
  }
  return e == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* kla_status_string(kla_status s) {
  switch (s) {
    case KLA_OK: return "ok";
    case KLA_ERR_INVALID_ARG: return "invalid argument";
    case KLA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (d_k, d_v must be 16, 32, 64 or 128)";
    case KLA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case KLA_ERR_WORKSPACE: return "workspace missing or too small";
    case KLA_ERR_CUDA: return "CUDA error";
    case KLA_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

int kla_version(void) { return 100; }

kla_status kla_plan_for_sms(int B, int H, int T, int dk, int dv, kla_dtype io, const kla_options* opt,
                            int num_sms, kla_plan_info* out) {
  if (!out) return KLA_ERR_INVALID_ARG;
  Plan p{};
  const kla_status st = make_plan(B, H, T, dk, dv, io, opt, num_sms, &p);
  if (st == KLA_OK) fill_info(p, out);
  return st;
}

kla_status kla_plan(int B, int H, int T, int dk, int dv, kla_dtype io, const kla_options* opt,
                    kla_plan_info* out) {
  if (!out) return KLA_ERR_INVALID_ARG;
  Plan p{};
  kla_status st = make_plan(B, H, T, dk, dv, io, opt, 1, &p);  // validates first, no CUDA call
  if (st != KLA_OK) return st;
  int sms = 0;
  if ((st = device_sms(&sms)) != KLA_OK) return st;
  if ((st = make_plan(B, H, T, dk, dv, io, opt, sms, &p)) != KLA_OK) return st;
  fill_info(p, out);
  return KLA_OK;
}

size_t kla_forward_workspace_size(int B, int H, int T, int dk, int dv, const kla_options* opt) {
  Plan p{};
  if (make_plan(B, H, T, dk, dv, KLA_F32, opt, 1, &p) != KLA_OK) return (size_t)-1;
  int sms = 0;
  if (device_sms(&sms) != KLA_OK) return (size_t)-1;
  size_t ws = 0;
  for (int io = KLA_F32; io <= KLA_BF16; ++io) {
    if (make_plan(B, H, T, dk, dv, io, opt, sms, &p) != KLA_OK) return (size_t)-1;
    ws = std::max(ws, p.ws_bytes);
  }
  return ws;
}

kla_status kla_forward(const void* q, const void* k, const void* v, const void* lam_v, const void* a,
                       const void* pbar, const float* lam0, const float* eta0, void* y, float* lamT,
                       float* etaT, int B, int H, int T, int dk, int dv, kla_dtype io, void* workspace,
                       size_t ws_bytes, const kla_options* opt, void* stream) {
  return forward_impl(q, k, v, lam_v, a, pbar, lam0, eta0, y, lamT, etaT, B, H, T, dk, dv, io, workspace,
                      ws_bytes, opt, stream, nullptr);
}

kla_status kla_forward_uncertainty(const void* q, const void* k, const void* v, const void* lam_v, const void* a,
                                   const void* pbar, const float* lam0, const float* eta0, void* y, void* y_var,
                                   float* lamT, float* etaT, int B, int H, int T, int dk, int dv, kla_dtype io,
                                   void* workspace, size_t ws_bytes, const kla_options* opt, void* stream) {
  if ((long long)B * H * T > 0 && !y_var) return KLA_ERR_INVALID_ARG;
  return forward_impl(q, k, v, lam_v, a, pbar, lam0, eta0, y, lamT, etaT, B, H, T, dk, dv, io, workspace,
                      ws_bytes, opt, stream, y_var);
}

kla_status kla_step_gated(const void* q, const void* k, const void* v, const void* lam_v, const void* a,
                          const void* pbar, float* lam, float* eta, void* y, int B, int H, int dk, int dv,
                          kla_dtype io, int gates, void* stream) {
  kla_status st = check_shape(B, H, 1, dk, dv);
  if (st != KLA_OK) return st;
  if (io != KLA_F32 && io != KLA_BF16) return KLA_ERR_INVALID_ARG;
  if (!valid_gates(gates)) return KLA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  if (bh > 0 && (!q || !k || !v || !lam_v || !a || !pbar || !lam || !eta || !y)) return KLA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, lam_v, a, pbar, lam, eta, y};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KLA_ERR_MISALIGNED;
  const size_t state_bytes = (size_t)bh * dk * dv * sizeof(float);
  if (lam && (lam == eta || overlaps_partially(lam, eta, state_bytes))) return KLA_ERR_INVALID_ARG;
  if (bh == 0) return KLA_OK;
  kla::StepArgs sa{q, k, v, lam_v, a, pbar, lam, eta, y, B, H, dk, dv, (int)io, gates};
  const cudaError_t e = kla::launch_step(sa, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

kla_status kla_step(const void* q, const void* k, const void* v, const void* lam_v, const void* a,
                    const void* pbar, float* lam, float* eta, void* y, int B, int H, int dk, int dv, kla_dtype io,
                    void* stream) {
  return kla_step_gated(q, k, v, lam_v, a, pbar, lam, eta, y, B, H, dk, dv, io, 0, stream);
}

kla_status kla_shard_map(const void* q, const void* k, const void* v, const void* lam_v, const void* a,
                         const void* pbar, float* map, int B, int H, int T, int dk, int dv, kla_dtype io, int gates,
                         void* stream) {
  // ---- validation: no CUDA call before it passes ---------------------------
  kla_status st = check_shape(B, H, T, dk, dv);
  if (st != KLA_OK) return st;
  if (io != KLA_F32 && io != KLA_BF16) return KLA_ERR_INVALID_ARG;
  if (!valid_gates(gates)) return KLA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  if (bh > 0 && !map) return KLA_ERR_INVALID_ARG;
  if (bh > 0 && T > 0 && (!q || !k || !v || !lam_v || !a || !pbar)) return KLA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, lam_v, a, pbar, map};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KLA_ERR_MISALIGNED;
  if (bh == 0) return KLA_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long elems = bh * dk * dv;
  if (T == 0) return kla::launch_identity_map(map, elems, s) == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
  int sms = 0;
  if ((st = device_sms(&sms)) != KLA_OK) return st;
  // The whole shard is one chunk of the composition kernel (grid.z = 1).
  // Column block: the widest that still gives two blocks per SM, else the
  // narrowest the kernel allows (more blocks for few heads).
  const int wc = kla::warp_cols(dk, kla::rows_per_lane_for(dk));
  const int cc_min = std::max<int>(wc, (int)(16 / io_size(io)));
  const int cc_max = std::min(dv, kla::max_threads() / 32 * wc);
  int cc = cc_min;
  for (int c = cc_min; c <= cc_max; c *= 2)
    if (bh * (dv / c) >= 2LL * sms) cc = c;
  if (kla::compose_smem_bytes(dk, io, cc, kla::tile_for(dk, io)) > kMaxSmem) return KLA_ERR_UNSUPPORTED_SHAPE;
  Plan p{};
  p.strategy = KLA_CHUNKED;
  p.chunk_len = T;
  p.num_chunks = 2;
  p.cols_per_block = cc;
  p.rows_per_lane = kla::rows_per_lane_for(dk);
  p.tile = kla::tile_for(dk, io);
  kla::ForwardArgs f{q, k, v, lam_v, a, pbar, nullptr, nullptr, nullptr, nullptr, nullptr, B, H, T, dk, dv,
                     (int)io, gates};
  return kla::launch_compose(f, p, map, s) == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

kla_status kla_shard_start(const float* maps, int n_maps, const float* lam0, const float* eta0, float* lam_start,
                           float* eta_start, int B, int H, int dk, int dv, void* stream) {
  kla_status st = check_shape(B, H, 0, dk, dv);
  if (st != KLA_OK) return st;
  if (n_maps < 0) return KLA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  if ((lam0 == nullptr) != (eta0 == nullptr)) return KLA_ERR_INVALID_ARG;
  if (bh > 0 && (!lam_start || !eta_start || (n_maps > 0 && !maps))) return KLA_ERR_INVALID_ARG;
  const void* ptrs[] = {maps, lam0, eta0, lam_start, eta_start};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KLA_ERR_MISALIGNED;
  const size_t state_bytes = (size_t)bh * dk * dv * sizeof(float);
  if (overlaps_partially(lam_start, lam0, state_bytes) || overlaps_partially(eta_start, eta0, state_bytes) ||
      overlaps_partially(lam_start, eta0, state_bytes) || overlaps_partially(eta_start, lam0, state_bytes) ||
      (lam_start && (lam_start == (const float*)eta0 || lam_start == eta_start)) ||
      (eta_start && eta_start == (const float*)lam0) || overlaps_partially(lam_start, eta_start, state_bytes))
    return KLA_ERR_INVALID_ARG;
  if (maps && n_maps > 0) {
    const size_t map_bytes = (size_t)n_maps * 7 * state_bytes;
    for (const float* o : {lam_start, eta_start}) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(maps), b0 = reinterpret_cast<uintptr_t>(o);
      if (a0 < b0 + state_bytes && b0 < a0 + map_bytes) return KLA_ERR_INVALID_ARG;
    }
  }
  if (bh == 0) return KLA_OK;
  const cudaError_t e = kla::launch_shard_start(maps, n_maps, lam0, eta0, lam_start, eta_start, bh * dk * dv,
                                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

size_t kla_backward_workspace_size(int B, int H, int T, int dk, int dv) {
  if (check_shape(B, H, T, dk, dv) != KLA_OK) return (size_t)-1;
  const long long bh = (long long)B * H;
  if (bh == 0) return 0;
  int sms = 0;
  if (device_sms(&sms) != KLA_OK) return (size_t)-1;
  const kla::BwdPlan b = kla::backward_plan(bh, T, dk, dv, sms);
  return b.ckpt_bytes + b.rowpart_bytes;
}

kla_status kla_backward_plan_for_sms(int B, int H, int T, int dk, int dv, int num_sms,
                                     kla_backward_plan_info* out) {
  if (!out) return KLA_ERR_INVALID_ARG;
  const kla_status st = check_shape(B, H, T, dk, dv);
  if (st != KLA_OK) return st;
  if (num_sms < 1) return KLA_ERR_INVALID_ARG;
  *out = kla_backward_plan_info{};
  const long long bh = (long long)B * H;
  if (bh == 0) return KLA_OK;
  const kla::BwdPlan b = kla::backward_plan(bh, T, dk, dv, num_sms);
  out->cols_per_block = b.cc;
  out->cols_per_lane = b.cpl;
  out->threads = b.threads;
  out->column_blocks = b.ncb;
  out->workspace_bytes = b.ckpt_bytes + b.rowpart_bytes;
  return KLA_OK;
}

kla_status kla_backward(const void* q, const void* k, const void* v, const void* lam_v, const void* a,
                        const void* pbar, const float* lam0, const float* eta0, const void* gy,
                        const float* glamT, const float* getaT, void* gq, void* gk, void* gv, void* glam_v,
                        void* ga, void* gpbar, float* glam0, float* geta0, int B, int H, int T, int dk, int dv,
                        kla_dtype io, int gates, void* workspace, size_t ws_bytes, void* stream) {
  // ---- validation: no CUDA call before it passes ---------------------------
  kla_status st = check_shape(B, H, T, dk, dv);
  if (st != KLA_OK) return st;
  if (io != KLA_F32 && io != KLA_BF16) return KLA_ERR_INVALID_ARG;
  if (!valid_gates(gates)) return KLA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  const long long tokens = bh * T;
  if ((lam0 == nullptr) != (eta0 == nullptr)) return KLA_ERR_INVALID_ARG;
  if ((glam0 == nullptr) != (geta0 == nullptr)) return KLA_ERR_INVALID_ARG;
  if (tokens > 0 && (!q || !k || !v || !lam_v || !a || !pbar || !gq || !gk || !gv || !glam_v || !ga || !gpbar))
    return KLA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, lam_v, a, pbar, lam0, eta0, gy, glamT, getaT,
                        gq, gk, gv, glam_v, ga, gpbar, glam0, geta0};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KLA_ERR_MISALIGNED;
  if (glam0 && (glam0 == geta0 || overlaps_partially(glam0, geta0, (size_t)bh * dk * dv * sizeof(float))))
    return KLA_ERR_INVALID_ARG;
  if (bh == 0) return KLA_OK;

  int sms = 0;
  if ((st = device_sms(&sms)) != KLA_OK) return st;
  const kla::BwdPlan b = kla::backward_plan(bh, T, dk, dv, sms);
  if (!workspace || ws_bytes < b.ckpt_bytes + b.rowpart_bytes) return KLA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KLA_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T > 0) {  // forward scan storing its state every 16 tokens (no y)
    const kla_options seq{KLA_SEQUENTIAL, 0, 0, gates, KLA_COEF_OFF};
    Plan fp{};
    if ((st = make_plan(B, H, T, dk, dv, io, &seq, sms, &fp)) != KLA_OK) return st;
    kla::ForwardArgs ff{q, k, v, lam_v, a, pbar, lam0, eta0, nullptr, nullptr, nullptr, B, H, T, dk, dv, (int)io,
                        gates};
    if (kla::launch_forward(ff, fp, nullptr, s, reinterpret_cast<float*>(workspace)) != cudaSuccess)
      return KLA_ERR_CUDA;
  }
  kla::BackwardArgs f{q,  k,  v,  lam_v, a,     pbar, lam0, eta0, gy, glamT, getaT, gq, gk, ga,
                      gpbar, gv, glam_v, glam0, geta0, B, H, T, dk, dv, (int)io, gates};
  const cudaError_t e = kla::launch_backward(f, b, workspace, s);
  return e == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

kla_status kla_conv(const void* x, const float* weight, const float* bias, const void* window_in, void* y,
                    void* window_out, int B, int H, int T, int D, int W, kla_dtype io, int activation,
                    void* stream) {
  // ---- validation: no CUDA call before it passes ---------------------------
  kla_status st = check_conv_shape(B, H, T, D, W);
  if (st != KLA_OK) return st;
  if (io != KLA_F32 && io != KLA_BF16) return KLA_ERR_INVALID_ARG;
  if (activation != KLA_ACT_NONE && activation != KLA_ACT_SILU) return KLA_ERR_INVALID_ARG;
  if (W == 1) window_in = window_out = nullptr;  // empty windows
  const long long bh = (long long)B * H;
  if (bh > 0 && !weight) return KLA_ERR_INVALID_ARG;
  if (bh * T > 0 && (!x || !y)) return KLA_ERR_INVALID_ARG;
  const void* ptrs[] = {x, weight, bias, window_in, y, window_out};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KLA_ERR_MISALIGNED;
  const size_t xb = (size_t)bh * T * D * io_size(io), wb = (size_t)bh * (W - 1) * D * io_size(io);
  const size_t tb = (size_t)H * D * W * sizeof(float), bb = (size_t)H * D * sizeof(float);
  const void* ins[] = {x, weight, bias, window_in};
  const size_t in_bytes[] = {xb, tb, bb, wb};
  for (int i = 0; i < 4; ++i) {
    if (ranges_overlap(y, xb, ins[i], in_bytes[i])) return KLA_ERR_INVALID_ARG;
    if (i != 3 && ranges_overlap(window_out, wb, ins[i], in_bytes[i])) return KLA_ERR_INVALID_ARG;
  }
  if (overlaps_partially(window_out, window_in, wb) || ranges_overlap(window_out, wb, y, xb))
    return KLA_ERR_INVALID_ARG;
  if (bh == 0) return KLA_OK;
  int sms = 0;
  if ((st = device_sms(&sms)) != KLA_OK) return st;
  kla::ConvArgs a{};
  a.x = x; a.weight = weight; a.bias = bias; a.win = window_in; a.y = y; a.wout = window_out;
  a.B = B; a.H = H; a.T = T; a.D = D; a.W = W; a.io = (int)io; a.act = activation;
  return kla::launch_conv(a, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KLA_OK : KLA_ERR_CUDA;
}

size_t kla_conv_backward_workspace_size(int B, int H, int T, int D, int W) {
  if (check_conv_shape(B, H, T, D, W) != KLA_OK) return (size_t)-1;
  const long long bh = (long long)B * H;
  if (bh == 0) return 0;
  int sms = 0;
  if (device_sms(&sms) != KLA_OK) return (size_t)-1;
  return kla::conv_partial_bytes(B, H, T, D, W, sms);
}

kla_status kla_conv_backward(const void* x, const float* weight, const float* bias, const void* window_in,
                             const void* gy, const void* gwindow_out, void* gx, float* gweight, float* gbias,
                             void* gwindow, int B, int H, int T, int D, int W, kla_dtype io, int activation,
                             void* workspace, size_t ws_bytes, void* stream) {
  // ---- validation: no CUDA call before it passes ---------------------------
  kla_status st = check_conv_shape(B, H, T, D, W);
  if (st != KLA_OK) return st;
  if (io != KLA_F32 && io != KLA_BF16) return KLA_ERR_INVALID_ARG;
  if (activation != KLA_ACT_NONE && activation != KLA_ACT_SILU) return KLA_ERR_INVALID_ARG;
  if (W == 1) window_in = gwindow_out = gwindow = nullptr;  // empty windows
  const long long bh = (long long)B * H;
  if (bh > 0 && !weight) return KLA_ERR_INVALID_ARG;
  if (bh * T > 0 && (!x || !gx)) return KLA_ERR_INVALID_ARG;
  const void* ptrs[] = {x, weight, bias, window_in, gy, gwindow_out, gx, gweight, gbias, gwindow, workspace};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KLA_ERR_MISALIGNED;
  const size_t xb = (size_t)bh * T * D * io_size(io), wb = (size_t)bh * (W - 1) * D * io_size(io);
  const size_t tb = (size_t)H * D * W * sizeof(float), bb = (size_t)H * D * sizeof(float);
  const void* ins[] = {x, weight, bias, window_in, gy, gwindow_out};
  const size_t in_bytes[] = {xb, tb, bb, wb, xb, wb};
  const void* outs[] = {gx, gweight, gbias, gwindow};
  const size_t out_bytes[] = {xb, tb, bb, wb};
  for (int o = 0; o < 4; ++o) {
    for (int i = 0; i < 6; ++i)
      if (ranges_overlap(outs[o], out_bytes[o], ins[i], in_bytes[i])) return KLA_ERR_INVALID_ARG;
    for (int p = o + 1; p < 4; ++p)
      if (ranges_overlap(outs[o], out_bytes[o], outs[p], out_bytes[p])) return KLA_ERR_INVALID_ARG;
  }
  const bool want_sums = gweight || gbias;
  if (bh == 0 && !(want_sums && H > 0)) return KLA_OK;
  int sms = 0;
  if ((st = device_sms(&sms)) != KLA_OK) return st;
  const size_t part_bytes = kla::conv_partial_bytes(B, H, T, D, W, sms);
  if (want_sums && part_bytes > 0 && (!workspace || ws_bytes < part_bytes)) return KLA_ERR_WORKSPACE;
  if (want_sums && part_bytes > 0)
    for (int o = 0; o < 4; ++o)
      if (ranges_overlap(workspace, part_bytes, outs[o], out_bytes[o])) return KLA_ERR_INVALID_ARG;
  kla::ConvArgs a{};
  a.x = x; a.weight = weight; a.bias = bias; a.win = window_in;
  a.gy = gy; a.gwout = gwindow_out; a.gx = gx; a.gwin = gwindow; a.gweight = gweight; a.gbias = gbias;
  a.part = want_sums && part_bytes > 0 ? reinterpret_cast<float*>(workspace) : nullptr;
  a.B = B; a.H = H; a.T = T; a.D = D; a.W = W; a.io = (int)io; a.act = activation;
  return kla::launch_conv_backward(a, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KLA_OK
                                                                                                  : KLA_ERR_CUDA;
}

}  // extern "C"
