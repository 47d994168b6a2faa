// Kernels whose tiles are fetched by cp.async (K not a multiple of 16, or A / B not
// 16-byte aligned): same swizzled shared-memory layout as TMA writes, zero fill past K.
#include "launch.h"

namespace mslkb {

const VariantInfo kVariantsCpAsync[] = {
    make_variant<KernelCfg<128, 6, false, false, false, 8>>("stacked_tile128x128_cpasync"),
    make_variant<KernelCfg<128, 6, false, false, true, 8>>("dynamic_tile128x128_cpasync"),
    make_variant<KernelCfg<16, 11, true, false, false>>("stacked_swap_w128xa16_cpasync"),
    make_variant<KernelCfg<16, 11, true, false, true>>("dynamic_swap_w128xa16_cpasync"),
};
const int kNumVariantsCpAsync = sizeof(kVariantsCpAsync) / sizeof(kVariantsCpAsync[0]);

}  // namespace mslkb
