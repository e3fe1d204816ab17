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

// Kernel arguments, passed by value (296 bytes) as a __grid_constant__.
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
    // Elements before the (aligned) buffer starts that belong to the call:
    // when every buffer is misaligned by the same amount, the host shifts the
    // pointers forward to alignment and the first `head` elements sit at
    // indices -head .. -1.
    int head;
    // CTAs 0 .. prefetch_ctas-1 (the ones resident from the start, so the
    // ones that may run while the kernel ahead of this one on the stream is
    // still draining) ask L2 for the source vectors of their first round
    // before waiting for that kernel (see prefetch_first_round); 0 = none.
    int prefetch_ctas;
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
__device__ __forceinline__ float load_elem(const void *base, long long i) {
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
__device__ __forceinline__ float elem_operand(const void *base, long long i) {
    float a = load_elem<Td, NC>(base, i);
    float b = a;
    wire2<Td, Tw>(a, b);
    return a;
}

template <int Td>
__device__ __forceinline__ void store_elem(void *base, long long i, float v) {
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
__device__ __forceinline__ void reduce_elem(const ArParams &p, long long i) {
    float v[kMaxRanks];
#pragma unroll
    for (int r = 0; r < kMaxRanks; ++r)
        if (r < p.R) v[r] = load_elem<Td, NC>(p.src[r], i);
    float acc = wire1<Td, Tw>(v[0]);
#pragma unroll
    for (int r = 1; r < kMaxRanks; ++r)
        if (r < p.R) acc = __fadd_rn(acc, wire1<Td, Tw>(v[r]));
#pragma unroll
    for (int d = 0; d < kMaxDsts; ++d)
        if (d < p.n_dsts) store_elem<Td>(p.dst[d], i, acc);
}

// ---- kernels ------------------------------------------------------------

// ---- words of a wide vector ----------------------------------------------
// A vector of VB bytes (16 or 32) held as VB/4 32-bit words.  32-byte
// accesses (ld/st .v8.b32) need 32-byte-aligned addresses and halve the
// number of memory instructions per byte.  NC loads take the non-coherent
// path, valid only when nothing the kernel writes is read; the others are
// coherent.  Neither allocates in L1: every byte is read once.
template <int VB, bool NC>
__device__ __forceinline__ void load_words(const void *p, uint32_t (&w)[VB / 4]) {
    static_assert(VB == 16 || VB == 32, "vector width");
    if constexpr (VB == 16) {
        if constexpr (NC) {
            asm("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
                : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                : "l"(p));
        } else {
            asm volatile("ld.global.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
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
            asm volatile("ld.global.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
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
// vectors per thread per tile; see ar_reduce_kernel.  UNR unrolls the rank
// and destination loops to kMaxRanks / kMaxDsts so that every pointer is
// read from the kernel parameters at a constant offset: a runtime index
// goes through a computed address, which on GB300 costs about 0.1-0.25 us
// of latency per launch (decode-sized calls gain 5%), while the rolled
// loops keep the bandwidth launches 0.2-0.5% faster.
template <int Td, int Tw, int VB, int U, int RB, bool NC, bool UNR>
__device__ __forceinline__ void reduce_span(const ArParams &p, size_t first, size_t end) {
    constexpr int NW = VB / 4;
    constexpr int V = VB / Elem<Td>::bytes;
    const size_t tile = static_cast<size_t>(blockDim.x) * U;
    for (size_t base = first + threadIdx.x; base < end; base += tile) {
        float acc[U][V];
        // ranks r0 .. r0+RB-1: all loads first, then the adds in rank order
        auto batch = [&](int r0) {
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
        };
        if constexpr (UNR) {
#pragma unroll
            for (int r0 = 0; r0 < kMaxRanks; r0 += RB) {
                if (r0 >= p.R) break;
                batch(r0);
            }
        } else {
            for (int r0 = 0; r0 < p.R; r0 += RB) batch(r0);
        }
        uint32_t out[U][NW];
#pragma unroll
        for (int u = 0; u < U; ++u) word_pack<Td, NW>(acc[u], out[u]);
        auto store = [&](int d) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const size_t idx = base + static_cast<size_t>(u) * blockDim.x;
                if (idx < end) store_words<VB>(static_cast<char *>(p.dst[d]) + idx * VB, out[u]);
            }
        };
        if constexpr (UNR) {
#pragma unroll
            for (int d = 0; d < kMaxDsts; ++d) {
                if (d >= p.n_dsts) break;
                store(d);
            }
        } else {
            for (int d = 0; d < p.n_dsts; ++d) store(d);
        }
    }
}

// Ask L2 for the source vectors this thread loads in its first round (one
// prefetch.global.L2 per rank), before pdl_wait.  Launched as a programmatic
// dependent, the first wave of CTAs runs this while the kernel ahead of it on
// the stream drains, so DRAM starts on this kernel's sources instead of
// idling through the hand-over.  A prefetch returns no data: it only moves
// lines into L2, the point where every write of the earlier kernel lands as
// well, so a line it brings in is updated by any later write to it, and the
// loads that use the data still come after pdl_wait.  Later waves start after
// the hand-over and would only add a second request per load, so the host
// limits the prefetch to the CTAs resident from the start.
template <int VB, bool UNR>
__device__ __forceinline__ void prefetch_first_round(const ArParams &p, size_t first, size_t end) {
    const size_t idx = first + threadIdx.x;
    if (idx >= end) return;
    auto one = [&](int r) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char *>(p.src[r]) + idx * VB));
    };
    if constexpr (UNR) {
#pragma unroll
        for (int r = 0; r < kMaxRanks; ++r) {
            if (r >= p.R) break;
            one(r);
        }
    } else {
        for (int r = 0; r < p.R; ++r) one(r);
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
// fewer than one vector's elements, on its highest threads, and CTA 0 the
// head before an aligned start (see ArParams::head), on its highest threads.
template <int Td, int Tw, int VB, int U, int RB, bool NC, bool UNR>
__global__ void __launch_bounds__(256) ar_reduce_kernel(const __grid_constant__ ArParams p) {
    constexpr int V = VB / Elem<Td>::bytes;
    const size_t nvec = p.nelem / V;
    const size_t G = gridDim.x;
    const size_t b = blockIdx.x;
    pdl_launch_dependents();
    if (U == 1 && b < static_cast<size_t>(p.prefetch_ctas) && p.rounds > 0 && b * p.chunk < nvec)
        prefetch_first_round<VB, UNR>(p, b * p.chunk, b * p.chunk + p.chunk < nvec ? b * p.chunk + p.chunk : nvec);
    pdl_wait();
    {
        const size_t K = p.rounds;  // ceil(nvec / (G * blockDim.x * U)), from the host
        const size_t c = p.chunk;   // ceil(nvec / (K * G)), from the host
        for (size_t k = 0; k < K; ++k) {
            const size_t first = (k * G + b) * c;
            if (first >= nvec) break;
            reduce_span<Td, Tw, VB, U, RB, NC, UNR>(p, first, first + c < nvec ? first + c : nvec);
        }
    }
    if (blockIdx.x == gridDim.x - 1) {
        // the tail goes to the block's highest threads: when the host leaves
        // them without a vector (it does whenever there is a tail), the tail's
        // loads overlap the vectors' instead of following them
        const size_t i = nvec * V + (blockDim.x - 1 - threadIdx.x);
        if (i < p.nelem) reduce_elem<Td, Tw, NC>(p, static_cast<long long>(i));
    }
    if (blockIdx.x == 0) {
        // the head before the aligned start (fewer than one vector)
        const int k = static_cast<int>(blockDim.x) - 1 - static_cast<int>(threadIdx.x);
        if (k < p.head) reduce_elem<Td, Tw, NC>(p, -1 - k);
    }
}

// Element-wise grid-stride kernel: the path for buffers at different
// offsets from a vector boundary.  Same arithmetic as ar_reduce_kernel.  Each
// thread takes E elements a grid stride apart per iteration (every warp
// access stays coalesced) and loads them for four ranks at a time before
// folding, so 4*E loads are in flight per thread instead of R.
template <int Td, int Tw, bool NC>
__global__ void __launch_bounds__(256) ar_scalar_kernel(const __grid_constant__ ArParams p) {
    constexpr int E = 4;
    constexpr int RB = 4;
    const size_t step = static_cast<size_t>(gridDim.x) * blockDim.x;
    pdl_launch_dependents();
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (blockIdx.x < static_cast<unsigned>(p.prefetch_ctas)) {
        // the first iteration's elements into L2 before the wait (as in
        // prefetch_first_round)
        for (int r = 0; r < p.R; ++r)
#pragma unroll
            for (int e = 0; e < E; ++e)
                if (i + e * step < p.nelem)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char *>(p.src[r]) +
                                                                  (i + e * step) * Elem<Td>::bytes));
    }
    pdl_wait();
    for (; i + (E - 1) * step < p.nelem; i += E * step) {
        float acc[E];
#pragma unroll
        for (int r0 = 0; r0 < kMaxRanks; r0 += RB) {  // constant parameter offsets (see reduce_span)
            if (r0 >= p.R) break;
            float v[RB][E];
#pragma unroll
            for (int j = 0; j < RB; ++j)
#pragma unroll
                for (int e = 0; e < E; ++e)
                    v[j][e] = r0 + j < p.R ? load_elem<Td, NC>(p.src[r0 + j], static_cast<long long>(i + e * step))
                                           : 0.0f;
#pragma unroll
            for (int j = 0; j < RB; ++j)
                if (r0 + j < p.R) {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float w = wire1<Td, Tw>(v[j][e]);
                        acc[e] = (r0 + j == 0) ? w : __fadd_rn(acc[e], w);
                    }
                }
        }
#pragma unroll
        for (int d = 0; d < kMaxDsts; ++d) {
            if (d >= p.n_dsts) break;
#pragma unroll
            for (int e = 0; e < E; ++e) store_elem<Td>(p.dst[d], static_cast<long long>(i + e * step), acc[e]);
        }
    }
    for (; i < p.nelem; i += step) reduce_elem<Td, Tw, NC>(p, static_cast<long long>(i));
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
