// fc_conv_bf16_padx.cu -- the fused conv3x3 kernel for bf16 inputs on BF16 tensor cores in single CTAs (M = 128 MMAs),
// with zero padding whose column shift is not a 16-byte multiple (XP extra staged columns).
#include "fc_conv_kernel.cuh"

namespace fc {
namespace convk {

FC_CONV_LAUNCH_DECL(launch_main_bf16_padx)
{
    FC_CONV_LAUNCH_BODY(true, false, true, false)
}

}  // namespace convk
}  // namespace fc
