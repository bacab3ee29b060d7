// fc_conv_bf16.cu -- the fused conv3x3 kernel instantiated for bf16 inputs on BF16 tensor cores
// in single CTAs (M = 128 MMAs), one variant per (pool or full output) x (erf-GELU, Mish, Mish twice).
#include "fc_conv_kernel.cuh"

namespace fc {
namespace convk {

FC_CONV_LAUNCH_DECL(launch_main_bf16)
{
    FC_CONV_LAUNCH_BODY(true, false, false, false)
}

}  // namespace convk
}  // namespace fc
