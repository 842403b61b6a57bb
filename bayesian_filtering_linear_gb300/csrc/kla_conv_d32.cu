// The causal convolution's kernels for streams of 32 channels (a
// compile-time row width); see kla_conv_kernels.cuh.
#include "kla_conv_kernels.cuh"

namespace kla {
template cudaError_t conv_launch_dc<32>(const ConvArgs&, bool, int, cudaStream_t);
}  // namespace kla
