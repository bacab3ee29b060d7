// fc_conv_tf32_pair.cu -- the fused conv3x3 kernel instantiated for fp32 inputs on TF32 tensor cores
// in CTA pairs (M = 256 MMAs), one variant per (pool or full output) x (erf-GELU, Mish, Mish twice).
#include "fc_conv_kernel.cuh"

namespace fc {
namespace convk {

FC_CONV_LAUNCH_DECL(launch_main_tf32_pair)
{
    FC_CONV_LAUNCH_BODY(false, true, false, false)
}

}  // namespace convk
}  // namespace fc
