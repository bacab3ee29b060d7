// fc_conv_tf32_nhwc.cu -- the fused conv3x3 kernel for fp32 inputs on TF32 tensor cores in single CTAs (M = 128 MMAs),
// NHWC (channels-last) input and full output: TMA boxes of channels land straight in the staged strip.
#include "fc_conv_kernel.cuh"

namespace fc {
namespace convk {

FC_CONV_LAUNCH_DECL(launch_main_tf32_nhwc)
{
    FC_CONV_LAUNCH_BODY(false, false, false, true)
}

}  // namespace convk
}  // namespace fc
