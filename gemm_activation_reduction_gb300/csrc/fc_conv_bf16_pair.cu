// fc_conv_bf16_pair.cu -- the fused conv3x3 kernel instantiated for bf16 inputs on BF16 tensor cores
// in CTA pairs (M = 256 MMAs), one variant per (pool or full output) x (erf-GELU, Mish, Mish twice).
#include "fc_conv_kernel.cuh"

namespace fc {
namespace convk {

FC_CONV_LAUNCH_DECL(launch_main_bf16_pair)
{
    FC_CONV_LAUNCH_BODY(true, true, false, false)
}

}  // namespace convk
}  // namespace fc
