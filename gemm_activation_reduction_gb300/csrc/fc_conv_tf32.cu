// fc_conv_tf32.cu -- the fused conv3x3 kernel instantiated for fp32 inputs on TF32 tensor cores
// in single CTAs (M = 128 MMAs), one variant per (pool or full output) x (erf-GELU, Mish, Mish twice).
#include "fc_conv_kernel.cuh"

namespace fc {
namespace convk {

FC_CONV_LAUNCH_DECL(launch_main_tf32)
{
    switch (pool * 3 + act) {
    case 0: return launch_variant<false, false, 0, false>(tmx, a, grid, smem_bytes, stream);
    case 1: return launch_variant<false, false, 1, false>(tmx, a, grid, smem_bytes, stream);
    case 2: return launch_variant<false, false, 2, false>(tmx, a, grid, smem_bytes, stream);
    case 3: return launch_variant<false, true, 0, false>(tmx, a, grid, smem_bytes, stream);
    case 4: return launch_variant<false, true, 1, false>(tmx, a, grid, smem_bytes, stream);
    case 5: return launch_variant<false, true, 2, false>(tmx, a, grid, smem_bytes, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace convk
}  // namespace fc
