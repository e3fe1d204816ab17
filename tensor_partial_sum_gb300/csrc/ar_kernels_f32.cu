// Kernel instantiations for f32 tensors (all three wire types).
#include "ar_dispatch.h"

namespace tps {

const Kernels &kernels_f32(int wire) {
    static const Kernels table[3] = {make_kernels<kF32, kF32>(), make_kernels<kF32, kF16>(),
                                     make_kernels<kF32, kBF16>()};
    return table[wire];
}

}  // namespace tps
