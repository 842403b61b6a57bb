// Causal depthwise 1-D convolution with SiLU: launch geometry, the
// partial-sum workspace and the dispatch over row widths. The kernels are in
// kla_conv_kernels.cuh (the operation and its work layout are described
// there); this unit compiles the any-width kernels, kla_conv_d{16,32,64,128}.cu
// the fixed-width ones for the scan's head sizes.
#include "kla_conv_kernels.cuh"

namespace kla {

// Tokens per block. Both kernels are issue-bound on their busiest SM, whose
// time is the total work of the blocks it runs, so each stream is cut into
// the number n of ranges (of whole stages) that minimises the busiest SM's
// share, ceil(B·H·n / SMs) / n — for 128 streams on 152 SMs, n = 7 is within
// 2% of an even spread — with at least `min_stages` stages per range so that
// a block's pipeline fill (and, backward, its extra tail stage) stays a small
// part of its work: 8 forward, 32 backward (measured: at 128 streams of 64
// stages, 7 ranges per stream made the backward 5% slower than 2). Ties go to
// the larger n (more blocks resident to hide latency).
int conv_range(long long bh, int T, long long TT, int num_sms, int min_stages, long long* blocks_y) {
  const long long nst = std::max(1LL, ((long long)T + TT - 1) / TT);
  const long long nmax = std::min(512LL, std::max(1LL, nst / min_stages));
  const long long sms = std::max(num_sms, 1);
  long long best = 1;
  long long best_num = (bh + sms - 1) / sms, best_den = 1;  // cost = num / den
  for (long long n = 2; n <= nmax; ++n) {
    const long long num = (bh * n + sms - 1) / sms;
    if (num * best_den <= best_num * n) {
      best = n;
      best_num = num;
      best_den = n;
    }
  }
  const long long range = TT * ((nst + best - 1) / best);
  *blocks_y = T > 0 ? ((long long)T + range - 1) / range : 1;
  return (int)range;
}

size_t conv_partial_bytes(int B, int H, int T, int D, int W, int num_sms) {
  const long long bh = (long long)B * H;
  if (bh == 0) return 0;
  const long long TT = (long long)(kConvThreads / (D / 4)) * kConvRows;
  long long blocks_y = 0;
  conv_range(bh, T, TT, num_sms, kConvBwdMinStages, &blocks_y);
  return (size_t)H * B * blocks_y * D * (W + 1) * sizeof(float);
}

template cudaError_t conv_launch_dc<0>(const ConvArgs&, bool, int, cudaStream_t);
extern template cudaError_t conv_launch_dc<16>(const ConvArgs&, bool, int, cudaStream_t);
extern template cudaError_t conv_launch_dc<32>(const ConvArgs&, bool, int, cudaStream_t);
extern template cudaError_t conv_launch_dc<64>(const ConvArgs&, bool, int, cudaStream_t);
extern template cudaError_t conv_launch_dc<128>(const ConvArgs&, bool, int, cudaStream_t);

namespace {
cudaError_t conv_dispatch(const ConvArgs& a, bool backward, int num_sms, cudaStream_t s) {
  switch (a.D) {
    case 16: return conv_launch_dc<16>(a, backward, num_sms, s);
    case 32: return conv_launch_dc<32>(a, backward, num_sms, s);
    case 64: return conv_launch_dc<64>(a, backward, num_sms, s);
    case 128: return conv_launch_dc<128>(a, backward, num_sms, s);
    default: return conv_launch_dc<0>(a, backward, num_sms, s);
  }
}
}  // namespace

cudaError_t launch_conv(const ConvArgs& a, int num_sms, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  if (bh == 0) return cudaSuccess;
  return conv_dispatch(a, false, num_sms, s);
}

cudaError_t launch_conv_backward(const ConvArgs& a, int num_sms, cudaStream_t s) {
  const long long bh = (long long)a.B * a.H;
  if (bh > 0) return conv_dispatch(a, true, num_sms, s);
  if (a.H > 0 && (a.gweight || a.gbias)) {  // no batch: the sums are zero
    const long long n = (long long)a.H * a.D * (a.W + 1);
    const int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
    ConvArgs z = a;
    z.nparts = 0;
    kla_conv_bwd_finish_kernel<<<blocks, 256, 0, s>>>(z, a.W);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace kla
