// Host-side view of the kernel instantiations: one table per (dst, wire)
// type pair, filled by the per-type translation units (ar_kernels_*.cu).
#pragma once

#include "ar_kernels.cuh"
#include "ar_kernels_ex.cuh"
#include "ar_kernels_tma.cuh"

namespace tps {

using KernelFn = void (*)(ArParams);

// One vector width with its two rank-batch sizes, each as [NC] pair
// (0 = coherent loads because a destination is also a source, 1 = read-only
// loads).
struct VecKernels {
    KernelFn few[2];   // R <= 2: ranks loaded two at a time
    KernelFn many[2];  // R >= 3: ranks loaded four at a time
};

using ExKernelFn = void (*)(ArExParams);
using TmaKernelFn = void (*)(ArParams, TmaPlan);
using PackKernelFn = void (*)(const void *, void *, unsigned long long, int, int);

struct Kernels {
    ExKernelFn ex[2][2][2];  // [R >= 3][residual][16-byte vectors]
    ExKernelFn ex32[2][2];   // [R >= 3][residual], 32-byte vectors (f32 only, else nullptr)
    PackKernelFn pack[2];    // [16-byte vectors]
    PackKernelFn pack32;     // 32-byte source vectors (f32 only, else nullptr)
    VecKernels v16;    // 16-byte vectors, unrolled loops: the latency launch
    VecKernels bw16;   // 16-byte vectors, rolled loops: the bandwidth launch
    VecKernels wide;   // the bandwidth launch's widest: 32-byte vectors for f32, bw16 otherwise
    int wide_bytes;    // 32 or 16
    KernelFn scalar[2];  // [NC]
    KernelFn naive;
    TmaKernelFn tma;     // shared-memory staging with bulk copies
};

// Defined in ar_kernels_f32.cu / ar_kernels_f16.cu / ar_kernels_bf16.cu.
const Kernels &kernels_f32(int wire);
const Kernels &kernels_f16(int wire);
const Kernels &kernels_bf16(int wire);

// UNR: rank and destination loops unrolled (the latency launch).
template <int Td, int Tw, int VB, bool UNR>
VecKernels make_vec_kernels() {
    return VecKernels{
        {ar_reduce_kernel<Td, Tw, VB, 1, 2, false, UNR>, ar_reduce_kernel<Td, Tw, VB, 1, 2, true, UNR>},
        {ar_reduce_kernel<Td, Tw, VB, 1, 4, false, UNR>, ar_reduce_kernel<Td, Tw, VB, 1, 4, true, UNR>}};
}

// Kernel set of one (dst, wire) pair.
template <int Td, int Tw>
Kernels make_kernels() {
    Kernels k{};
    k.v16 = make_vec_kernels<Td, Tw, 16, true>();
    k.bw16 = make_vec_kernels<Td, Tw, 16, false>();
    if constexpr (Td == kF32) {
        k.wide = make_vec_kernels<Td, Tw, 32, false>();
        k.wide_bytes = 32;
    } else {
        k.wide = k.bw16;
        k.wide_bytes = 16;
    }
    k.ex[0][0][0] = ar_reduce_ex_kernel<Td, Tw, 2, false, false>;
    k.ex[0][0][1] = ar_reduce_ex_kernel<Td, Tw, 2, false, true>;
    k.ex[0][1][0] = ar_reduce_ex_kernel<Td, Tw, 2, true, false>;
    k.ex[0][1][1] = ar_reduce_ex_kernel<Td, Tw, 2, true, true>;
    k.ex[1][0][0] = ar_reduce_ex_kernel<Td, Tw, 4, false, false>;
    k.ex[1][0][1] = ar_reduce_ex_kernel<Td, Tw, 4, false, true>;
    k.ex[1][1][0] = ar_reduce_ex_kernel<Td, Tw, 4, true, false>;
    k.ex[1][1][1] = ar_reduce_ex_kernel<Td, Tw, 4, true, true>;
    k.pack[0] = ar_pack_kernel<Td, Tw, false>;
    k.pack[1] = ar_pack_kernel<Td, Tw, true>;
    if constexpr (Td == kF32) {
        k.ex32[0][0] = ar_reduce_ex_kernel<Td, Tw, 2, false, true, 32>;
        k.ex32[0][1] = ar_reduce_ex_kernel<Td, Tw, 2, true, true, 32>;
        k.ex32[1][0] = ar_reduce_ex_kernel<Td, Tw, 4, false, true, 32>;
        k.ex32[1][1] = ar_reduce_ex_kernel<Td, Tw, 4, true, true, 32>;
        k.pack32 = ar_pack_kernel<Td, Tw, true, 32>;
    }
    k.scalar[0] = ar_scalar_kernel<Td, Tw, false>;
    k.scalar[1] = ar_scalar_kernel<Td, Tw, true>;
    k.naive = ar_naive_kernel<Td, Tw>;
    k.tma = ar_tma_kernel<Td, Tw>;
    return k;
}

}  // namespace tps
