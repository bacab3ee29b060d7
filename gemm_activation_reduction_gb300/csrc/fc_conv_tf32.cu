// fc_conv_tf32.cu -- the fused conv3x3 kernel instantiated for fp32 inputs on TF32 tensor cores
// in single CTAs (M = 128 MMAs), one variant per (pool or full output) x (erf-GELU, Mish, Mish twice).
#include "fc_conv_kernel.cuh"

namespace fc {
namespace convk {

FC_CONV_LAUNCH_DECL(launch_main_tf32)
{
    FC_CONV_LAUNCH_BODY(false, false, false, false)
}

}  // namespace convk
}  // namespace fc
