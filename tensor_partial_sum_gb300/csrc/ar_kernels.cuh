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
    // Work plan of ar_reduce_kernel, computed by the host for the launch's
    // grid: `rounds` rounds of `chunk` vectors per CTA (see the kernel).
    unsigned long long chunk;
    unsigned long long rounds;
    int R;
    int n_dsts;
};

// Programmatic dependent launch: when a launch opts in, the next kernel on
// the stream may start while this one runs; griddepcontrol.wait then holds
// it until this grid has completed and its writes are visible, so results
// never depend on the overlap.  Without the opt-in both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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

// Round one widened value through the wire type.
template <int Td, int Tw>
__device__ __forceinline__ float wire1(float a) {
    float b = a;
    wire2<Td, Tw>(a, b);
    return a;
}

// One element of every rank: all R loads are issued (predicated on r < R)
// before the first is used, so the element path waits for memory once, not
// once per rank; then the operands are folded in ascending rank order.
template <int Td, int Tw, bool NC>
__device__ __forceinline__ void reduce_elem(const ArParams &p, size_t i) {
    float v[kMaxRanks];
#pragma unroll
    for (int r = 0; r < kMaxRanks; ++r)
        if (r < p.R) v[r] = load_elem<Td, NC>(p.src[r], i);
    float acc = wire1<Td, Tw>(v[0]);
#pragma unroll
    for (int r = 1; r < kMaxRanks; ++r)
        if (r < p.R) acc = __fadd_rn(acc, wire1<Td, Tw>(v[r]));
    for (int d = 0; d < p.n_dsts; ++d) store_elem<Td>(p.dst[d], i, acc);
}

// ---- kernels ------------------------------------------------------------

// ---- words of a wide vector ----------------------------------------------
// A vector of VB bytes (16 or 32) held as VB/4 32-bit words.  32-byte
// accesses (ld/st .v8.b32) need 32-byte-aligned addresses and halve the
// number of memory instructions per byte.
template <int VB, bool NC>
__device__ __forceinline__ void load_words(const void *p, uint32_t (&w)[VB / 4]) {
    static_assert(VB == 16 || VB == 32, "vector width");
    if constexpr (VB == 16) {
        if constexpr (NC) {
            asm("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
                : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                : "l"(p));
        } else {
            asm volatile("ld.global.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "l"(p)
                         : "memory");
        }
    } else {
        if constexpr (NC) {
            asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                  "=r"(w[7])
                : "l"(p));
        } else {
            asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
                           "=r"(w[7])
                         : "l"(p)
                         : "memory");
        }
    }
}

template <int VB>
__device__ __forceinline__ void store_words(void *p, const uint32_t (&w)[VB / 4]) {
    if constexpr (VB == 16) {
        asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                     "r"(w[3])
                     : "memory");
    } else {
        asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                     "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    }
}

// The operands held in NW words of T_dst, rounded through the wire type.
template <int Td, int Tw, int NW>
__device__ __forceinline__ void word_operands(const uint32_t (&w)[NW], float (&x)[NW * 4 / Elem<Td>::bytes]) {
    if constexpr (Td == kF32) {
#pragma unroll
        for (int k = 0; k < NW; ++k) x[k] = __uint_as_float(w[k]);
    } else {
#pragma unroll
        for (int k = 0; k < NW; ++k) widen2<Td>(w[k], x[2 * k], x[2 * k + 1]);
    }
#pragma unroll
    for (int k = 0; k < NW * 4 / Elem<Td>::bytes; k += 2) wire2<Td, Tw>(x[k], x[k + 1]);
}

template <int Td, int NW>
__device__ __forceinline__ void word_pack(const float (&acc)[NW * 4 / Elem<Td>::bytes], uint32_t (&w)[NW]) {
    if constexpr (Td == kF32) {
#pragma unroll
        for (int k = 0; k < NW; ++k) w[k] = __float_as_uint(acc[k]);
    } else {
#pragma unroll
        for (int k = 0; k < NW; ++k) w[k] = narrow2<Td>(acc[2 * k], acc[2 * k + 1]);
    }
}

// The vectors [first, end) of one thread block, RB ranks per batch, U
// vectors per thread per tile; see ar_bw_kernel.
template <int Td, int Tw, int VB, int U, int RB, bool NC>
__device__ __forceinline__ void reduce_span(const ArParams &p, size_t first, size_t end) {
    constexpr int NW = VB / 4;
    constexpr int V = VB / Elem<Td>::bytes;
    const size_t tile = static_cast<size_t>(blockDim.x) * U;
    for (size_t base = first + threadIdx.x; base < end; base += tile) {
        float acc[U][V];
        for (int r0 = 0; r0 < p.R; r0 += RB) {
            uint32_t w[RB][U][NW];
#pragma unroll
            for (int j = 0; j < RB; ++j) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const size_t idx = base + static_cast<size_t>(u) * blockDim.x;
                    if (r0 + j < p.R && idx < end) {
                        load_words<VB, NC>(static_cast<const char *>(p.src[r0 + j]) + idx * VB, w[j][u]);
                    } else {
#pragma unroll
                        for (int k = 0; k < NW; ++k) w[j][u][k] = 0u;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < RB; ++j) {
                if (r0 + j < p.R) {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        float x[V];
                        word_operands<Td, Tw, NW>(w[j][u], x);
                        if (r0 + j == 0) {
#pragma unroll
                            for (int k = 0; k < V; ++k) acc[u][k] = x[k];
                        } else {
#pragma unroll
                            for (int k = 0; k < V; ++k) acc[u][k] = __fadd_rn(acc[u][k], x[k]);
                        }
                    }
                }
            }
        }
        uint32_t out[U][NW];
#pragma unroll
        for (int u = 0; u < U; ++u) word_pack<Td, NW>(acc[u], out[u]);
        for (int d = 0; d < p.n_dsts; ++d) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t idx = base + static_cast<size_t>(u) * blockDim.x;
                if (idx < end) store_words<VB>(static_cast<char *>(p.dst[d]) + idx * VB, out[u]);
            }
        }
    }
}

// The reduction kernel.  G CTAs of T threads cover nvec vectors of VB bytes
// in K = ceil(nvec / (G*T*U)) rounds: in round k, CTA b takes the c vectors
// starting at (k*G + b)*c, with c = ceil(nvec / (K*G)) <= T*U.  Launched
// with G = ceil(nvec / (T*U)) this is one round and one vector (U = 1) per
// thread, and the hardware block scheduler balances the CTAs; launched with
// a smaller, persistent grid the CTAs move through the tensors together in
// one window and each CTA's total differs from the others' by at most one
// chunk.  Ranks are loaded RB at a time: all RB*U loads of a batch are
// issued before the first conversion (RB*U*VB bytes in flight per thread),
// then the batch's operands are added in ascending rank order.  Each warp
// access covers 32 adjacent vectors.  The last CTA also does the tail of
// fewer than one vector's elements, on its highest threads.
template <int Td, int Tw, int VB, int U, int RB, bool NC>
__global__ void __launch_bounds__(256) ar_reduce_kernel(const __grid_constant__ ArParams p) {
    constexpr int V = VB / Elem<Td>::bytes;
    const size_t nvec = p.nelem / V;
    const size_t G = gridDim.x;
    const size_t b = blockIdx.x;
    pdl_launch_dependents();
    pdl_wait();
    {
        const size_t K = p.rounds;  // ceil(nvec / (G * blockDim.x * U)), from the host
        const size_t c = p.chunk;   // ceil(nvec / (K * G)), from the host
        for (size_t k = 0; k < K; ++k) {
            const size_t first = (k * G + b) * c;
            if (first >= nvec) break;
            reduce_span<Td, Tw, VB, U, RB, NC>(p, first, first + c < nvec ? first + c : nvec);
        }
    }
    if (blockIdx.x == gridDim.x - 1) {
        // the tail goes to the block's highest threads: when the host leaves
        // them without a vector (it does whenever there is a tail), the tail's
        // loads overlap the vectors' instead of following them
        const size_t i = nvec * V + (blockDim.x - 1 - threadIdx.x);
        if (i < p.nelem) reduce_elem<Td, Tw, NC>(p, i);
    }
}

// Element-wise grid-stride kernel: the path for pointers that are not all
// 16-byte aligned.  Same arithmetic as ar_reduce_kernel, one element per
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

// ==== extended layouts: row strides, inactive ranks, residual / bias ======
namespace tps {

// Kernel arguments of ar_reduce_ex_kernel (by value, about 560 bytes).
struct ArExParams {
    const void *src[kMaxRanks];
    void *dst[kMaxDsts];
    long long src_stride[kMaxRanks];  // row strides in bytes
    long long dst_stride[kMaxDsts];
    const void *residual;             // nullptr: none
    long long res_stride;             // 0: one row broadcast to every row
    unsigned long long ne0;           // elements per row
    unsigned long long ne1;           // rows
    unsigned inactive;                // bit r: rank r contributes +0
    int R;
    int n_dsts;
};

// Operand r of element i of row `row`, rounded through the wire type; +0
// for an inactive rank (the reduction of a zeroed partial).
template <int Td, int Tw>
__device__ __forceinline__ float ex_operand(const ArExParams &p, int r, size_t row, size_t i) {
    if ((p.inactive >> r) & 1u) return 0.0f;
    const char *base = static_cast<const char *>(p.src[r]) + static_cast<long long>(row) * p.src_stride[r];
    return wire1<Td, Tw>(load_elem<Td, false>(base, i));
}

// One element of a row, rank after rank (row tails and unaligned layouts;
// kept sequential so the vector path's register budget is not raised).
template <int Td, int Tw, bool RES>
__device__ __forceinline__ void ex_reduce_elem(const ArExParams &p, size_t row, size_t i) {
    float acc = ex_operand<Td, Tw>(p, 0, row, i);
    for (int r = 1; r < p.R; ++r) acc = __fadd_rn(acc, ex_operand<Td, Tw>(p, r, row, i));
    if constexpr (RES) {
        const char *rb = static_cast<const char *>(p.residual) + static_cast<long long>(row) * p.res_stride;
        acc = __fadd_rn(acc, load_elem<Td, false>(rb, i));
    }
    for (int d = 0; d < p.n_dsts; ++d)
        store_elem<Td>(static_cast<char *>(p.dst[d]) + static_cast<long long>(row) * p.dst_stride[d], i, acc);
}

// Reduction over ne1 rows of ne0 elements.  blockIdx.y strides over rows;
// within a row, thread t of CTA x owns VB-byte vector x*blockDim.x + t,
// loading RB ranks at a time (inactive ranks are not loaded: their operand
// is +0), then adds the residual (not rounded through the wire type) after
// the rank fold, casts once and stores to every destination.  The last CTA
// in x does the row's tail of fewer than one vector, element by element.
// VEC = false runs every element through that element-wise path (buffers
// or strides not 16-byte aligned).
template <int Td, int Tw, int RB, bool RES, bool VEC, int VB = 16>
__global__ void __launch_bounds__(256) ar_reduce_ex_kernel(const __grid_constant__ ArExParams p) {
    constexpr int NW = VB / 4;
    constexpr int V = VB / Elem<Td>::bytes;
    const size_t vpr = VEC ? p.ne0 / V : 0;  // whole vectors per row
    const size_t tail0 = vpr * V;
    for (size_t row = blockIdx.y; row < p.ne1; row += gridDim.y) {
        if constexpr (VEC) {
            const size_t v = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
            if (v < vpr) {
                float acc[V];
                for (int r0 = 0; r0 < p.R; r0 += RB) {
                    uint32_t w[RB][NW];
#pragma unroll
                    for (int j = 0; j < RB; ++j) {
                        const int r = r0 + j;
                        if (r < p.R && !((p.inactive >> r) & 1u)) {
                            const char *base = static_cast<const char *>(p.src[r]) +
                                               static_cast<long long>(row) * p.src_stride[r] + v * VB;
                            load_words<VB, false>(base, w[j]);
                        } else {
#pragma unroll
                            for (int k = 0; k < NW; ++k) w[j][k] = 0u;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < RB; ++j) {
                        if (r0 + j < p.R) {
                            float x[V];
                            word_operands<Td, Tw, NW>(w[j], x);
#pragma unroll
                            for (int k = 0; k < V; ++k) acc[k] = (r0 + j == 0) ? x[k] : __fadd_rn(acc[k], x[k]);
                        }
                    }
                }
                if constexpr (RES) {
                    uint32_t rw[NW];
                    load_words<VB, false>(static_cast<const char *>(p.residual) +
                                              static_cast<long long>(row) * p.res_stride + v * VB,
                                          rw);
                    float x[V];
                    word_operands<Td, Td, NW>(rw, x);  // widened, no wire rounding
#pragma unroll
                    for (int k = 0; k < V; ++k) acc[k] = __fadd_rn(acc[k], x[k]);
                }
                uint32_t out[NW];
                word_pack<Td, NW>(acc, out);
                for (int d = 0; d < p.n_dsts; ++d)
                    store_words<VB>(static_cast<char *>(p.dst[d]) + static_cast<long long>(row) * p.dst_stride[d] +
                                        v * VB,
                                    out);
            }
            if (blockIdx.x == gridDim.x - 1) {
                const size_t i = tail0 + threadIdx.x;
                if (i < p.ne0) ex_reduce_elem<Td, Tw, RES>(p, row, i);
            }
        } else {
            for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.ne0;
                 i += static_cast<size_t>(gridDim.x) * blockDim.x)
                ex_reduce_elem<Td, Tw, RES>(p, row, i);
        }
    }
}

// Wire pack: wire[i] = T_wire(value(src[i])), the buffer a transport would
// send (phase 1 of ggml_cuda_ar_kernel in ggml-cuda allreduce.cu).  VEC:
// each thread converts one VB-byte vector of sources (16 or 32 bytes); the
// last CTA does the tail element by element.
template <int Td, int Tw, bool VEC, int VB = 16>
__global__ void __launch_bounds__(256) ar_pack_kernel(const void *src, void *wire, unsigned long long nelem) {
    constexpr int NW = VB / 4;
    constexpr int V = VB / Elem<Td>::bytes;
    constexpr int WB = V * Elem<Tw>::bytes;  // output bytes per vector: 8, 16 or 32
    auto one = [&](size_t i) {
        float a = load_elem<Td, false>(src, i);
        if constexpr (Tw == kF32) {
            static_cast<float *>(wire)[i] = a;
        } else {
            float b = a;
            static_cast<unsigned short *>(wire)[i] = static_cast<unsigned short>(narrow2<Tw>(a, b) & 0xFFFFu);
        }
    };
    if constexpr (VEC) {
        const size_t nvec = nelem / V;
        const size_t v = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        if (v < nvec) {
            uint32_t w[NW];
            load_words<VB, false>(static_cast<const char *>(src) + v * VB, w);  // may run in place
            float x[V];
            word_operands<Td, Td, NW>(w, x);  // exact values
            char *o = static_cast<char *>(wire) + v * WB;
            constexpr int OW = WB / 4;  // output words: 2, 4 or 8
            uint32_t ow[OW];
            if constexpr (Tw == kF32) {
#pragma unroll
                for (int k = 0; k < V; ++k) ow[k] = __float_as_uint(x[k]);
            } else {
#pragma unroll
                for (int k = 0; k < V / 2; ++k) ow[k] = narrow2<Tw>(x[2 * k], x[2 * k + 1]);
            }
            if constexpr (OW == 2) {
                asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(o), "r"(ow[0]), "r"(ow[1]) : "memory");
            } else if constexpr (OW == 4) {
                store_words<16>(o, reinterpret_cast<uint32_t(&)[4]>(ow));
            } else {
                store_words<32>(o, reinterpret_cast<uint32_t(&)[8]>(ow));
            }
        }
        if (blockIdx.x == gridDim.x - 1) {
            const size_t i = nvec * V + threadIdx.x;
            if (i < nelem) one(i);
        }
    } else {
        for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nelem;
             i += static_cast<size_t>(gridDim.x) * blockDim.x)
            one(i);
    }
}

}  // namespace tps

// ==== TMA bulk-copy variant ===============================================
// The bandwidth variant with shared-memory staging: a producer warp streams
// the R source tiles of each stage into shared memory with 1-D bulk copies
// (cp.async.bulk, completion counted on an mbarrier), eight consumer warps
// fold each tile into an output tile, and one elected consumer writes that
// tile to every destination with bulk stores.  Every wait is bounded by
// %globaltimer; a wait that runs out sets *status and the kernel drains its
// own copies (also bounded) and returns, so it cannot hang.
namespace tps {

struct TmaPlan {
    unsigned long long vec_bytes;  // bytes of each buffer covered by 16-byte vectors
    unsigned long long ntiles;     // ceil(vec_bytes / tile_bytes)
    unsigned tile_bytes;           // per rank per stage, a multiple of 1024
    unsigned stages;               // 2 .. kTmaMaxStages
    unsigned *status;              // device word: bit 0 = a wait timed out
    unsigned long long timeout_ns; // bound of every wait
    unsigned long long drop_tile;  // test hook: this tile's loads are never issued (~0 = none)
};

constexpr int kTmaMaxStages = 8;
constexpr int kTmaHeaderBytes = 256;  // mbarriers and the abort flag, before the tiles
constexpr int kTmaConsumers = 256;                // eight consumer warps
constexpr int kTmaThreads = kTmaConsumers + 32;   // plus one producer warp

__device__ __forceinline__ unsigned smem_u32(const void *p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(unsigned long long *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Wait for the phase with the given parity to complete, for at most
// timeout_ns (globaltimer).  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, unsigned parity, unsigned long long timeout_ns) {
    const unsigned a = smem_u32(bar);
    const unsigned long long deadline = global_ns() + timeout_ns;
    while (true) {
        unsigned done;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
            : "=r"(done)
            : "r"(a), "r"(parity), "r"(1000u)
            : "memory");
        if (done) return true;
        if (global_ns() > deadline) return false;
    }
}
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, unsigned bytes, unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_store(void *gdst, const void *smem_src, unsigned bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(smem_src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kTmaConsumers) : "memory"); }
// Barrier of the consumer warps that also ORs a flag over them: every
// consumer gets the same answer, so they all leave a loop together.
__device__ __forceinline__ bool consumer_sync_or(bool v) {
    unsigned r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 q, %1, 0; bar.red.or.pred p, 1, %2, q; selp.u32 %0, 1, 0, p; }"
        : "=r"(r)
        : "r"(static_cast<unsigned>(v)), "n"(kTmaConsumers)
        : "memory");
    return r != 0;
}

// Dynamic shared memory: full[kTmaMaxStages], empty[kTmaMaxStages] mbarriers,
// a flag word, then (from byte kTmaHeaderBytes) in[stages][R][tile] and
// out[2][tile].
template <int Td, int Tw>
__global__ void __launch_bounds__(kTmaThreads) ar_tma_kernel(const __grid_constant__ ArParams p,
                                                                const __grid_constant__ TmaPlan plan) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned long long *full = reinterpret_cast<unsigned long long *>(smem);
    unsigned long long *empty = full + kTmaMaxStages;
    volatile unsigned *abort_flag = reinterpret_cast<volatile unsigned *>(empty + kTmaMaxStages);
    unsigned char *in = smem + kTmaHeaderBytes;
    const unsigned T = plan.tile_bytes, S = plan.stages;
    unsigned char *out = in + static_cast<size_t>(S) * p.R * T;
    const int tid = threadIdx.x;
    const unsigned long long G = gridDim.x;
    // this CTA's tiles: b, b + G, b + 2G, ...
    const unsigned long long my_tiles =
        plan.ntiles > blockIdx.x ? (plan.ntiles - blockIdx.x + G - 1) / G : 0;

    if (tid == 0) {
        for (unsigned s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        *abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const unsigned long long timeout = plan.timeout_ns;

    if (tid < 32) {
        // ---- producer warp (lane 0 issues) ----
        if (tid == 0) {
            unsigned long long issued = 0;
            for (unsigned long long k = 0; k < my_tiles; ++k) {
                const unsigned s = static_cast<unsigned>(k % S);
                if (k >= S && !mbar_wait(&empty[s], static_cast<unsigned>((k / S - 1) & 1), timeout)) {
                    atomicOr(plan.status, 1u);
                    *abort_flag = 1u;
                    break;
                }
                if (*abort_flag) break;
                const unsigned long long off = (blockIdx.x + k * G) * T;
                const unsigned bytes = static_cast<unsigned>(min(static_cast<unsigned long long>(T), plan.vec_bytes - off));
                if (blockIdx.x + k * G != plan.drop_tile) {  // the hook leaves the stage's barrier waiting
                    mbar_expect_tx(&full[s], bytes * p.R);
                    for (int r = 0; r < p.R; ++r)
                        bulk_load(in + (static_cast<size_t>(s) * p.R + r) * T,
                                  static_cast<const char *>(p.src[r]) + off, bytes, &full[s]);
                }
                issued = k + 1;
            }
            // before leaving, every copy this warp started must have landed
            // (bounded: a copy that never completes only costs the deadline)
            for (unsigned long long k = issued > S ? issued - S : 0; k < issued; ++k)
                mbar_wait(&full[k % S], static_cast<unsigned>((k / S) & 1), timeout);
        }
    } else {
        // ---- consumer warps ----
        const int ct = tid - 32;
        constexpr int V = 16 / Elem<Td>::bytes;
        for (unsigned long long k = 0; k < my_tiles; ++k) {
            const unsigned s = static_cast<unsigned>(k % S);
            const bool ok = mbar_wait(&full[s], static_cast<unsigned>((k / S) & 1), timeout);
            if (!ok) {
                atomicOr(plan.status, 1u);
                *abort_flag = 1u;
            }
            if (ct == 0) bulk_wait_read_1();  // the store that last read out[k % 2] is done reading
            if (consumer_sync_or(!ok || *abort_flag)) break;  // uniform: all consumers leave together
            const unsigned long long off = (blockIdx.x + k * G) * T;
            const unsigned bytes = static_cast<unsigned>(min(static_cast<unsigned long long>(T), plan.vec_bytes - off));
            unsigned char *o = out + (k & 1) * T;
            for (unsigned v = ct; v < bytes / 16; v += kTmaConsumers) {
                float acc[V];
                for (int r = 0; r < p.R; ++r) {
                    const uint4 w4 =
                        *reinterpret_cast<const uint4 *>(in + (static_cast<size_t>(s) * p.R + r) * T + v * 16);
                    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
                    float x[V];
                    word_operands<Td, Tw, 4>(w, x);
#pragma unroll
                    for (int e = 0; e < V; ++e) acc[e] = (r == 0) ? x[e] : __fadd_rn(acc[e], x[e]);
                }
                uint32_t ow[4];
                word_pack<Td, 4>(acc, ow);
                *reinterpret_cast<uint4 *>(o + v * 16) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // st.shared -> bulk store
            consumer_sync();
            if (ct == 0) {
                mbar_arrive(&empty[s]);  // this stage's inputs are free
                for (int d = 0; d < p.n_dsts; ++d) bulk_store(static_cast<char *>(p.dst[d]) + off, o, bytes);
                bulk_commit();
            }
        }
        if (ct == 0) bulk_wait_all();
    }
    // the tail of fewer than 16 bytes, element by element, by the last CTA
    if (blockIdx.x == gridDim.x - 1) {
        constexpr int V = 16 / Elem<Td>::bytes;
        const size_t i = plan.vec_bytes / Elem<Td>::bytes + tid;
        if (tid < V && i < p.nelem) reduce_elem<Td, Tw, false>(p, i);
    }
}

}  // namespace tps
