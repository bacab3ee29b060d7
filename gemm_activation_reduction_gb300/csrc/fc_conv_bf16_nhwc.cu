// fc_conv_bf16_nhwc.cu -- the fused conv3x3 kernel for bf16 inputs on BF16 tensor cores in single CTAs (M = 128 MMAs),
// NHWC (channels-last) input and full output: TMA boxes of channels land straight in the staged strip.
#include "fc_conv_kernel.cuh"

namespace fc {
namespace convk {

FC_CONV_LAUNCH_DECL(launch_main_bf16_nhwc)
{
    FC_CONV_LAUNCH_BODY(true, false, false, true)
}

}  // namespace convk
}  // namespace fc
