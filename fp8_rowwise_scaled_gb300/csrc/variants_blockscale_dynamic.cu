// Block-scaled (groupwise) slab kernels (dynamic and batched layouts) fed by TMA: one K
// block per TMEM chunk, each chunk scaled on its way into the fp32 registers; padding rows
// of a slab are written +0.0.
#include "launch.h"

namespace mslkb {

const VariantInfo kVariantsBlockScaleDynamic[] = {
    make_variant<KernelCfg<256, 4, false, true, true, 8, false, 0, true>>(
        "dynamic_blockscale_tile128x256_tma"),
    make_variant<KernelCfg<128, 6, false, true, true, 8, false, 0, true>>(
        "dynamic_blockscale_tile128x128_tma"),
    make_variant<KernelCfg<16, 11, true, true, true, 4, false, 0, true>>(
        "dynamic_blockscale_swap_w128xa16_tma"),
    make_variant<KernelCfg<32, 10, true, true, true, 4, false, 0, true>>(
        "dynamic_blockscale_swap_w128xa32_tma"),
};
const int kNumVariantsBlockScaleDynamic =
    sizeof(kVariantsBlockScaleDynamic) / sizeof(kVariantsBlockScaleDynamic[0]);

}  // namespace mslkb
