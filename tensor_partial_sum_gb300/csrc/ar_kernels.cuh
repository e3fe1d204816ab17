// Device code of the partial-sum reduction for sm_103a.
//
// Every kernel computes, for each element i it owns,
//     acc = float(wire(src[0][i])); acc += float(wire(src[r][i])) for r = 1..R-1;
//     dst[d][i] = T_dst(acc) for every destination d,
// the formula of ggml_cuda_ar_kernel phase 3 and ggml_cuda_ar_add_kernel
// (ggml-cuda allreduce.cu, toy 0.8.0 vendored ggml), folded over R ranks in
// ascending order as in DEFINE_ALLREDUCE_THREAD_DMA_1D (ggml-hexagon
// htp/allreduce-ops.c).  Narrowing casts use the hardware's round-to-nearest-
// even conversions (cvt.rn, no flush to zero); widening is exact; adds are
// add.rn.f32.  The wire rounding never touches memory on one GPU: it happens
// in registers, so the bytes moved are (R + n_dsts) * nelem * sizeof(T_dst).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace tps {

constexpr int kF32 = 0;
constexpr int kF16 = 1;
constexpr int kBF16 = 2;
constexpr int kMaxRanks = 16;
constexpr int kMaxDsts = 16;

// Kernel arguments, passed by value (272 bytes) as a __grid_constant__.
struct ArParams {
    const void *src[kMaxRanks];
    void *dst[kMaxDsts];
    unsigned long long nelem;
    int R;
    int n_dsts;
};

template <int T>
struct Elem;
template <>
struct Elem<kF32> {
    using storage = uint32_t;
    static constexpr int bytes = 4;
};
template <>
struct Elem<kF16> {
    using storage = uint16_t;
    static constexpr int bytes = 2;
};
template <>
struct Elem<kBF16> {
    using storage = uint16_t;
    static constexpr int bytes = 2;
};

// ---- packed conversions -------------------------------------------------
// cvt.rn.{bf16x2,f16x2}.f32 d, a, b puts a in the upper half and b in the
// lower half of d; the helpers take (lo, hi) in element order.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// bfloat16 is the upper half of a float: widening is a shift.
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float f16_lo(uint32_t v) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, l; }" : "=f"(f) : "r"(v));
    return f;
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(v));
    return f;
}

// Widen two packed elements of type T (element 2k in the low half).
template <int T>
__device__ __forceinline__ void widen2(uint32_t v, float &lo, float &hi) {
    if constexpr (T == kBF16) {
        lo = bf16_lo(v);
        hi = bf16_hi(v);
    } else {
        lo = f16_lo(v);
        hi = f16_hi(v);
    }
}

// Round two floats to T and pack them.
template <int T>
__device__ __forceinline__ uint32_t narrow2(float lo, float hi) {
    if constexpr (T == kBF16) {
        return pack_bf16x2(lo, hi);
    } else {
        return pack_f16x2(lo, hi);
    }
}

// True when rounding a T_dst value through T_wire can change it: a value of
// a format rounds to itself, and every format here is a subset of float.
template <int Td, int Tw>
constexpr bool kWireRounds = (Tw != kF32) && (Tw != Td);

// Round a pair of widened operands through the wire type and widen back.
template <int Td, int Tw>
__device__ __forceinline__ void wire2(float &a, float &b) {
    if constexpr (kWireRounds<Td, Tw>) {
        widen2<Tw>(narrow2<Tw>(a, b), a, b);
    }
}

// ---- 16-byte vectors ----------------------------------------------------
template <int Td>
constexpr int kVec = 16 / Elem<Td>::bytes;

template <bool NC>
__device__ __forceinline__ uint4 load16(const uint4 *p) {
    if constexpr (NC) {
        uint4 v;
        asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
            : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
            : "l"(p));
        return v;
    } else {
        return *p;
    }
}

// The operands of one 16-byte source vector, rounded through the wire type.
template <int Td, int Tw>
__device__ __forceinline__ void operands(const uint4 &v, float (&x)[kVec<Td>]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (Td == kF32) {
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = __uint_as_float(w[k]);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) widen2<Td>(w[k], x[2 * k], x[2 * k + 1]);
    }
#pragma unroll
    for (int k = 0; k < kVec<Td>; k += 2) wire2<Td, Tw>(x[k], x[k + 1]);
}

template <int Td>
__device__ __forceinline__ uint4 pack_result(const float (&acc)[kVec<Td>]) {
    uint32_t w[4];
    if constexpr (Td == kF32) {
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = __float_as_uint(acc[k]);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = narrow2<Td>(acc[2 * k], acc[2 * k + 1]);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---- one element at a time ----------------------------------------------
template <int Td, bool NC>
__device__ __forceinline__ float load_elem(const void *base, size_t i) {
    if constexpr (Td == kF32) {
        const float *p = static_cast<const float *>(base) + i;
        return NC ? __ldg(p) : *p;
    } else {
        const unsigned short *p = static_cast<const unsigned short *>(base) + i;
        const uint32_t h = NC ? __ldg(p) : *p;
        float lo, hi;
        widen2<Td>(h, lo, hi);
        return lo;
    }
}

template <int Td, int Tw, bool NC>
__device__ __forceinline__ float elem_operand(const void *base, size_t i) {
    float a = load_elem<Td, NC>(base, i);
    float b = a;
    wire2<Td, Tw>(a, b);
    return a;
}

template <int Td>
__device__ __forceinline__ void store_elem(void *base, size_t i, float v) {
    if constexpr (Td == kF32) {
        static_cast<float *>(base)[i] = v;
    } else {
        static_cast<unsigned short *>(base)[i] = static_cast<unsigned short>(narrow2<Td>(v, v) & 0xFFFFu);
    }
}

template <int Td, int Tw, bool NC>
__device__ __forceinline__ void reduce_elem(const ArParams &p, size_t i) {
    float acc = elem_operand<Td, Tw, NC>(p.src[0], i);
    for (int r = 1; r < p.R; ++r) acc = __fadd_rn(acc, elem_operand<Td, Tw, NC>(p.src[r], i));
    for (int d = 0; d < p.n_dsts; ++d) store_elem<Td>(p.dst[d], i, acc);
}

// ---- kernels ------------------------------------------------------------

// Vector kernel: each thread owns U 16-byte vectors per tile (one per
// blockDim.x stride, so every load instruction of a warp covers 512
// contiguous bytes).  U = 1 with a grid covering the tensor is the latency
// variant; larger U with a grid of a few CTAs per SM that strides over tiles
// is the bandwidth variant.  The last CTA also does the tail of fewer than
// one vector's worth of elements, element by element.
template <int Td, int Tw, int U, bool NC>
__global__ void __launch_bounds__(256) ar_vec_kernel(const __grid_constant__ ArParams p) {
    constexpr int V = kVec<Td>;
    const size_t nvec = p.nelem / V;
    const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x * U;
    for (size_t base = static_cast<size_t>(blockIdx.x) * blockDim.x * U + threadIdx.x; base < nvec;
         base += step) {
        float acc[U][V];
        {
            const uint4 *s = static_cast<const uint4 *>(p.src[0]);
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t idx = base + static_cast<size_t>(u) * blockDim.x;
                v[u] = idx < nvec ? load16<NC>(s + idx) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) operands<Td, Tw>(v[u], acc[u]);
        }
        for (int r = 1; r < p.R; ++r) {
            const uint4 *s = static_cast<const uint4 *>(p.src[r]);
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t idx = base + static_cast<size_t>(u) * blockDim.x;
                v[u] = idx < nvec ? load16<NC>(s + idx) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float x[V];
                operands<Td, Tw>(v[u], x);
#pragma unroll
                for (int k = 0; k < V; ++k) acc[u][k] = __fadd_rn(acc[u][k], x[k]);
            }
        }
        uint4 out[U];
#pragma unroll
        for (int u = 0; u < U; ++u) out[u] = pack_result<Td>(acc[u]);
        for (int d = 0; d < p.n_dsts; ++d) {
            uint4 *o = static_cast<uint4 *>(p.dst[d]);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t idx = base + static_cast<size_t>(u) * blockDim.x;
                if (idx < nvec) __stcs(o + idx, out[u]);
            }
        }
    }
    if (blockIdx.x == gridDim.x - 1) {
        const size_t i = nvec * V + threadIdx.x;
        if (i < p.nelem) reduce_elem<Td, Tw, NC>(p, i);
    }
}

// Element-wise grid-stride kernel: the path for pointers that are not all
// 16-byte aligned.  Same arithmetic as the vector kernel, one element per
// thread per iteration.
template <int Td, int Tw, bool NC>
__global__ void __launch_bounds__(256) ar_scalar_kernel(const __grid_constant__ ArParams p) {
    const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.nelem; i += step)
        reduce_elem<Td, Tw, NC>(p, i);
}

// Naive cross-check kernel in the style of ggml_cuda_ar_add_kernel: one
// element per thread, grid-stride, plain loads and stores, no vectors.
template <int Td, int Tw>
__global__ void __launch_bounds__(256) ar_naive_kernel(const __grid_constant__ ArParams p) {
    const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.nelem; i += step) {
        float acc = 0.0f;
        for (int r = 0; r < p.R; ++r) {
            const float x = elem_operand<Td, Tw, false>(p.src[r], i);
            acc = (r == 0) ? x : __fadd_rn(acc, x);
        }
        for (int d = 0; d < p.n_dsts; ++d) store_elem<Td>(p.dst[d], i, acc);
    }
}

}  // namespace tps
