// Stacked-layout kernels fed by TMA.
#include "launch.h"

namespace mslkb {

const VariantInfo kVariantsStackedTma[] = {
    make_variant<KernelCfg<256, 4, false, true, false, 8>>("stacked_tile128x256_tma"),
    make_variant<KernelCfg<128, 6, false, true, false, 8>>("stacked_tile128x128_tma"),
    make_variant<KernelCfg<16, 11, true, true, false>>("stacked_swap_w128xa16_tma"),
    make_variant<KernelCfg<32, 10, true, true, false>>("stacked_swap_w128xa32_tma"),
    make_variant<KernelCfg<64, 8, true, true, false>>("stacked_swap_w128xa64_tma"),
    make_variant<KernelCfg<256, 6, false, true, false, 8, true>>("stacked_pair256x256_tma"),
};
const int kNumVariantsStackedTma = sizeof(kVariantsStackedTma) / sizeof(kVariantsStackedTma[0]);

}  // namespace mslkb
