// Block-scaled (groupwise) stacked kernels fed by TMA: one K block per TMEM chunk, each
// chunk scaled on its way into the fp32 registers.
#include "launch.h"

namespace mslkb {

const VariantInfo kVariantsBlockScale[] = {
    make_variant<KernelCfg<256, 4, false, true, false, 8, false, 0, true>>(
        "blockscale_tile128x256_tma"),
    make_variant<KernelCfg<128, 6, false, true, false, 8, false, 0, true>>(
        "blockscale_tile128x128_tma"),
    make_variant<KernelCfg<16, 11, true, true, false, 4, false, 0, true>>(
        "blockscale_swap_w128xa16_tma"),
    make_variant<KernelCfg<32, 10, true, true, false, 4, false, 0, true>>(
        "blockscale_swap_w128xa32_tma"),
};
const int kNumVariantsBlockScale = sizeof(kVariantsBlockScale) / sizeof(kVariantsBlockScale[0]);

}  // namespace mslkb
