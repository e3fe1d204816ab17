// Kernel instantiations for bf16 tensors (all three wire types).
#include "ar_dispatch.h"

namespace tps {

const Kernels &kernels_bf16(int wire) {
    static const Kernels table[3] = {make_kernels<kBF16, kF32>(), make_kernels<kBF16, kF16>(),
                                     make_kernels<kBF16, kBF16>()};
    return table[wire];
}

}  // namespace tps
