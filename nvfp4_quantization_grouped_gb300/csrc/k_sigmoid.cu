// Instantiates the fused grouped scaled activation + quantization kernel
// (forward/backward x MXFP8/NVFP4) for one activation.
#include "gsa_kernel.cuh"

namespace gsa {
GSA_DEFINE_ACT(ACT_SIGMOID, sigmoid)
}  // namespace gsa
