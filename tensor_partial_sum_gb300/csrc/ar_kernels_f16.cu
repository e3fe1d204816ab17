// Kernel instantiations for f16 tensors (all three wire types).
#include "ar_dispatch.h"

namespace tps {

const Kernels &kernels_f16(int wire) {
    static const Kernels table[3] = {make_kernels<kF16, kF32>(), make_kernels<kF16, kF16>(),
                                     make_kernels<kF16, kBF16>()};
    return table[wire];
}

}  // namespace tps
