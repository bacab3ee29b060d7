// fc_conv_tf32_pair.cu -- the fused conv3x3 kernel instantiated for fp32 inputs on TF32 tensor cores
// in CTA pairs (M = 256 MMAs), one variant per (pool or full output) x (erf-GELU, Mish, Mish twice).
#include "fc_conv_kernel.cuh"

namespace fc {
namespace convk {

FC_CONV_LAUNCH_DECL(launch_main_tf32_pair)
{
    switch (pool * 3 + act) {
    case 0: return launch_variant<false, false, 0, true>(tmx, a, grid, smem_bytes, stream);
    case 1: return launch_variant<false, false, 1, true>(tmx, a, grid, smem_bytes, stream);
    case 2: return launch_variant<false, false, 2, true>(tmx, a, grid, smem_bytes, stream);
    case 3: return launch_variant<false, true, 0, true>(tmx, a, grid, smem_bytes, stream);
    case 4: return launch_variant<false, true, 1, true>(tmx, a, grid, smem_bytes, stream);
    case 5: return launch_variant<false, true, 2, true>(tmx, a, grid, smem_bytes, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace convk
}  // namespace fc
