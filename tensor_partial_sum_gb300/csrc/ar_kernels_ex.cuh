// Device code of the extended entry points: ar_reduce_ex (row strides,
// inactive ranks, residual / bias) and ar_wire_pack.  Built on the casts and
// element helpers of ar_kernels.cuh.
#pragma once

#include "ar_kernels.cuh"

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
    int prefetch_ctas;                // CTAs (in launch order) that prefetch before the wait
};

// Operand r of element i of row `row`, rounded through the wire type; +0
// for an inactive rank (the reduction of a zeroed partial).
template <int Td, int Tw>
__device__ __forceinline__ float ex_operand(const ArExParams &p, int r, size_t row, size_t i) {
    if ((p.inactive >> r) & 1u) return 0.0f;
    const char *base = static_cast<const char *>(p.src[r]) + static_cast<long long>(row) * p.src_stride[r];
    return wire1<Td, Tw>(load_elem<Td, false>(base, i));
}

// One element of a row, rank after rank: the row heads and tails of the
// vector path.  Kept sequential, which keeps that kernel at the register
// count it runs fastest with (the batched form below cut it from 48 to 40
// registers per thread, and the extra resident CTAs made aligned layouts
// 1.5% slower).
template <int Td, int Tw, bool RES>
__device__ __forceinline__ void ex_reduce_elem_seq(const ArExParams &p, size_t row, size_t i) {
    float acc = ex_operand<Td, Tw>(p, 0, row, i);
    for (int r = 1; r < p.R; ++r) acc = __fadd_rn(acc, ex_operand<Td, Tw>(p, r, row, i));
    if constexpr (RES) {
        const char *rb = static_cast<const char *>(p.residual) + static_cast<long long>(row) * p.res_stride;
        acc = __fadd_rn(acc, load_elem<Td, false>(rb, i));
    }
    for (int d = 0; d < p.n_dsts; ++d)
        store_elem<Td>(static_cast<char *>(p.dst[d]) + static_cast<long long>(row) * p.dst_stride[d], i, acc);
}

// One element of a row (the element-wise loop's last elements): the loads of
// four ranks at a time are issued before any of them is rounded and added (a
// load whose result is used before the next is issued would leave one memory
// latency per rank on this thread).
template <int Td, int Tw, bool RES>
__device__ __forceinline__ void ex_reduce_elem(const ArExParams &p, size_t row, size_t i) {
    float resv = 0.0f;
    if constexpr (RES) {
        const char *rb = static_cast<const char *>(p.residual) + static_cast<long long>(row) * p.res_stride;
        resv = load_elem<Td, false>(rb, static_cast<long long>(i));
    }
    float acc = 0.0f;
    for (int r0 = 0; r0 < p.R; r0 += 4) {
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = r0 + j;
            const char *b = (r < p.R && !((p.inactive >> r) & 1u))
                                ? static_cast<const char *>(p.src[r]) + static_cast<long long>(row) * p.src_stride[r]
                                : nullptr;
            v[j] = b ? load_elem<Td, false>(b, static_cast<long long>(i)) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (r0 + j < p.R) {
                const float x = wire1<Td, Tw>(v[j]);
                acc = (r0 + j == 0) ? x : __fadd_rn(acc, x);
            }
    }
    if constexpr (RES) acc = __fadd_rn(acc, resv);
    for (int d = 0; d < p.n_dsts; ++d)
        store_elem<Td>(static_cast<char *>(p.dst[d]) + static_cast<long long>(row) * p.dst_stride[d], i, acc);
}

// Reduction over ne1 rows of ne0 elements.  blockIdx.y strides over rows;
// within a row, thread t of CTA x owns VB-byte vector x*blockDim.x + t,
// loading RB ranks at a time (inactive ranks are not loaded: their operand
// is +0), then adds the residual (not rounded through the wire type) after
// the rank fold, casts once and stores to every destination.  With VEC the
// host guarantees that in every row all buffers sit at one common offset
// from a VB-byte boundary (read here from destination 0); the vectors start
// at the first boundary, and the row's head before it and tail after the
// last whole vector go element by element to the threads left without a
// vector, so their loads overlap the vectors' instead of following them.
// The host launches at least ne0/V + 2V - 2 threads in x, which leaves
// enough idle ones for any head and tail (fewer than V elements each).
// VEC = false runs every element through the element-wise path (buffers
// whose row starts sit at different offsets).
template <int Td, int Tw, int RB, bool RES, bool VEC, int VB = 16>
__global__ void __launch_bounds__(256) ar_reduce_ex_kernel(const __grid_constant__ ArExParams p) {
    constexpr int NW = VB / 4;
    constexpr int V = VB / Elem<Td>::bytes;
    pdl_launch_dependents();
    if constexpr (VEC) {
        // the first wave asks L2 for its first row's operands (as in
        // ar_reduce_kernel's prefetch_first_round)
        const size_t cta = static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x;
        const size_t row = blockIdx.y;
        if (cta < static_cast<size_t>(p.prefetch_ctas) && row < p.ne1) {
            const unsigned off = static_cast<unsigned>(
                (reinterpret_cast<uintptr_t>(p.dst[0]) + static_cast<long long>(row) * p.dst_stride[0]) % VB);
            size_t h = off ? (VB - off) / Elem<Td>::bytes : 0;
            if (h > p.ne0) h = p.ne0;
            const size_t vpr = (p.ne0 - h) / V;
            const size_t v = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
            const size_t at = h * Elem<Td>::bytes + v * VB;
            if (v < vpr) {
                for (int r = 0; r < p.R; ++r)
                    if (!((p.inactive >> r) & 1u))
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char *>(p.src[r]) +
                                                                      static_cast<long long>(row) * p.src_stride[r] +
                                                                      at));
                if constexpr (RES)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char *>(p.residual) +
                                                                  static_cast<long long>(row) * p.res_stride + at));
            }
        }
    }
    pdl_wait();  // the kernel before this one on the stream has finished
    for (size_t row = blockIdx.y; row < p.ne1; row += gridDim.y) {
        if constexpr (VEC) {
            // elements of the row before its first VB-byte boundary
            const unsigned off = static_cast<unsigned>(
                (reinterpret_cast<uintptr_t>(p.dst[0]) + static_cast<long long>(row) * p.dst_stride[0]) % VB);
            size_t h = off ? (VB - off) / Elem<Td>::bytes : 0;
            if (h > p.ne0) h = p.ne0;
            const size_t vpr = (p.ne0 - h) / V;  // whole vectors in the row
            const size_t t = p.ne0 - h - vpr * V;  // tail elements
            const size_t hb = h * Elem<Td>::bytes;
            const size_t v = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
            if (v < vpr) {
                // the residual's load is issued first so that it overlaps the
                // ranks'; it is still added after the fold
                uint32_t rw[NW];
                if constexpr (RES)
                    load_words<VB, false>(static_cast<const char *>(p.residual) +
                                              static_cast<long long>(row) * p.res_stride + hb + v * VB,
                                          rw);
                float acc[V];
                for (int r0 = 0; r0 < p.R; r0 += RB) {
                    uint32_t w[RB][NW];
#pragma unroll
                    for (int j = 0; j < RB; ++j) {
                        const int r = r0 + j;
                        if (r < p.R && !((p.inactive >> r) & 1u)) {
                            const char *base = static_cast<const char *>(p.src[r]) +
                                               static_cast<long long>(row) * p.src_stride[r] + hb + v * VB;
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
                    float x[V];
                    word_operands<Td, Td, NW>(rw, x);  // widened, no wire rounding
#pragma unroll
                    for (int k = 0; k < V; ++k) acc[k] = __fadd_rn(acc[k], x[k]);
                }
                uint32_t out[NW];
                word_pack<Td, NW>(acc, out);
                for (int d = 0; d < p.n_dsts; ++d)
                    store_words<VB>(static_cast<char *>(p.dst[d]) + static_cast<long long>(row) * p.dst_stride[d] +
                                        hb + v * VB,
                                    out);
            }
            // the threads after the last vector take the head's elements,
            // then the tail's
            const size_t u = v - vpr;
            if (v >= vpr && u < h + t) ex_reduce_elem_seq<Td, Tw, RES>(p, row, u < h ? u : u + vpr * V);
        } else {
            // E elements a grid stride apart per thread, their loads for four
            // ranks at a time in flight before the fold
            constexpr int E = 4;
            const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
            size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
            for (; i + (E - 1) * stride < p.ne0; i += E * stride) {
                float acc[E];
                for (int r0 = 0; r0 < p.R; r0 += 4) {
                    // the batch's row pointers first (NULL for an absent or
                    // inactive rank, whose operand is +0), then all its loads,
                    // then the wire rounding and the adds in rank order
                    const char *rb[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = r0 + j;
                        rb[j] = (r < p.R && !((p.inactive >> r) & 1u))
                                    ? static_cast<const char *>(p.src[r]) + static_cast<long long>(row) * p.src_stride[r]
                                    : nullptr;
                    }
                    float v[4][E];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            v[j][e] = rb[j] ? load_elem<Td, false>(rb[j], static_cast<long long>(i + e * stride)) : 0.0f;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (r0 + j < p.R) {
#pragma unroll
                            for (int e = 0; e < E; ++e) {
                                const float x = wire1<Td, Tw>(v[j][e]);
                                acc[e] = (r0 + j == 0) ? x : __fadd_rn(acc[e], x);
                            }
                        }
                }
                if constexpr (RES) {
                    const char *rb = static_cast<const char *>(p.residual) + static_cast<long long>(row) * p.res_stride;
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[e] = __fadd_rn(acc[e], load_elem<Td, false>(rb, i + e * stride));
                }
                for (int d = 0; d < p.n_dsts; ++d) {
                    char *db = static_cast<char *>(p.dst[d]) + static_cast<long long>(row) * p.dst_stride[d];
#pragma unroll
                    for (int e = 0; e < E; ++e) store_elem<Td>(db, static_cast<long long>(i + e * stride), acc[e]);
                }
            }
            for (; i < p.ne0; i += stride) ex_reduce_elem<Td, Tw, RES>(p, row, i);
        }
    }
}

// Wire pack: wire[i] = T_wire(value(src[i])), the buffer a transport would
// send (phase 1 of ggml_cuda_ar_kernel in ggml-cuda allreduce.cu).  VEC:
// each thread converts one VB-byte vector of sources (16 or 32 bytes); the
// last CTA does the tail element by element, and CTA 0 the `head` elements
// at indices -head .. -1 (the host shifts both pointers forward past them
// when the buffers start off a vector boundary).  Otherwise element-wise,
// eight elements in flight per thread.
template <int Td, int Tw, bool VEC, int VB = 16>
__global__ void __launch_bounds__(256) ar_pack_kernel(const void *src, void *wire, unsigned long long nelem,
                                                      int head, int prefetch_ctas) {
    constexpr int NW = VB / 4;
    constexpr int V = VB / Elem<Td>::bytes;
    constexpr int WB = V * Elem<Tw>::bytes;  // output bytes per vector: 8, 16 or 32
    auto put = [&](long long i, float a) {
        if constexpr (Tw == kF32) {
            static_cast<float *>(wire)[i] = a;
        } else {
            float b = a;
            static_cast<unsigned short *>(wire)[i] = static_cast<unsigned short>(narrow2<Tw>(a, b) & 0xFFFFu);
        }
    };
    auto one = [&](long long i) { put(i, load_elem<Td, false>(src, i)); };
    pdl_launch_dependents();
    if constexpr (VEC) {
        // the first wave asks L2 for its source vector before the wait
        const size_t v = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        if (blockIdx.x < static_cast<unsigned>(prefetch_ctas) && v < nelem / V)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char *>(src) + v * VB));
    }
    pdl_wait();  // the kernel before this one on the stream has finished
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
            if (i < nelem) one(static_cast<long long>(i));
        }
        if (blockIdx.x == 0) {
            const int k = static_cast<int>(blockDim.x) - 1 - static_cast<int>(threadIdx.x);
            if (k < head) one(-1 - k);
        }
    } else {
        // eight elements a grid stride apart per thread: loads first, then
        // stores (8 measured 7% faster than 4 here; the reductions keep 4)
        constexpr int E = 8;
        const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
        size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        for (; i + (E - 1) * stride < nelem; i += E * stride) {
            float a[E];
#pragma unroll
            for (int e = 0; e < E; ++e) a[e] = load_elem<Td, false>(src, static_cast<long long>(i + e * stride));
#pragma unroll
            for (int e = 0; e < E; ++e) put(static_cast<long long>(i + e * stride), a[e]);
        }
        for (; i < nelem; i += stride) one(static_cast<long long>(i));
    }
}

}  // namespace tps
