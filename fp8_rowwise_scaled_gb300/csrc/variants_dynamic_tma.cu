// Dynamic (padded) layout kernels fed by TMA.
#include "launch.h"

namespace mslkb {

const VariantInfo kVariantsDynamicTma[] = {
    make_variant<KernelCfg<256, 4, false, true, true, 8>>("dynamic_tile128x256_tma"),
    make_variant<KernelCfg<128, 6, false, true, true, 8>>("dynamic_tile128x128_tma"),
    make_variant<KernelCfg<16, 11, true, true, true>>("dynamic_swap_w128xa16_tma"),
    make_variant<KernelCfg<32, 10, true, true, true>>("dynamic_swap_w128xa32_tma"),
    make_variant<KernelCfg<64, 8, true, true, true>>("dynamic_swap_w128xa64_tma"),
    make_variant<KernelCfg<256, 6, false, true, true, 8, true>>("dynamic_pair256x256_tma"),
};
const int kNumVariantsDynamicTma = sizeof(kVariantsDynamicTma) / sizeof(kVariantsDynamicTma[0]);

}  // namespace mslkb
