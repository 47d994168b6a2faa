// Kernels for the ragged-K layout (groups slice the contraction), fed by TMA.
#include "launch.h"

namespace mslkb {

const VariantInfo kVariantsRaggedK[] = {
    make_variant<KernelCfg<256, 4, false, true, false, 8, false, 2>>("ragk_tile128x256_tma"),
    make_variant<KernelCfg<128, 6, false, true, false, 8, false, 2>>("ragk_tile128x128_tma"),
    make_variant<KernelCfg<32, 10, true, true, false, 4, false, 2>>("ragk_swap_w128xa32_tma"),
};
const int kNumVariantsRaggedK = sizeof(kVariantsRaggedK) / sizeof(kVariantsRaggedK[0]);

}  // namespace mslkb
