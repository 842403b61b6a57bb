// The causal convolution's kernels for streams of 128 channels (a
// compile-time row width); see kla_conv_kernels.cuh.
#include "kla_conv_kernels.cuh"

namespace kla {
template cudaError_t conv_launch_dc<128>(const ConvArgs&, bool, int, cudaStream_t);
}  // namespace kla
