// Kernels for the ragged-N layout (groups partition the weight rows / output columns),
// fed by TMA.
#include "launch.h"

namespace mslkb {

const VariantInfo kVariantsRaggedN[] = {
    make_variant<KernelCfg<256, 4, false, true, false, 8, false, 1>>("ragn_tile128x256_tma"),
    make_variant<KernelCfg<128, 6, false, true, false, 8, false, 1>>("ragn_tile128x128_tma"),
    make_variant<KernelCfg<32, 10, true, true, false, 4, false, 1>>("ragn_swap_w128xa32_tma"),
};
const int kNumVariantsRaggedN = sizeof(kVariantsRaggedN) / sizeof(kVariantsRaggedN[0]);

}  // namespace mslkb
