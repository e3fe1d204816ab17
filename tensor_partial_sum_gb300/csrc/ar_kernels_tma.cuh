// Device code of the TMA bulk-copy variant of the reduction (opt-in).
// Built on the casts and element helpers of ar_kernels.cuh.
#pragma once

#include "ar_kernels.cuh"

// ==== TMA bulk-copy variant ===============================================
// The bandwidth variant with shared-memory staging: a producer warp streams
// the R source tiles of each stage into shared memory with 1-D bulk copies
// (cp.async.bulk, completion counted on an mbarrier), sixteen consumer warps
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
constexpr int kTmaConsumers = 512;                // sixteen consumer warps (8: 1.7% slower)
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
    pdl_launch_dependents();
    if (threadIdx.x < static_cast<unsigned>(p.R) && blockIdx.x < static_cast<unsigned>(p.prefetch_ctas)) {
        // the first stages' tiles of rank threadIdx.x into L2 while the
        // kernel ahead drains (a prefetch returns no data, so the bulk loads
        // after the wait still see that kernel's writes); tiles start on
        // 1 KiB boundaries of 16-byte aligned buffers and span whole vectors
        for (unsigned k = 0; k < plan.stages; ++k) {
            const unsigned long long t = blockIdx.x + static_cast<unsigned long long>(k) * gridDim.x;
            if (t >= plan.ntiles) break;
            const unsigned long long off = t * plan.tile_bytes;
            const unsigned bytes =
                static_cast<unsigned>(min(static_cast<unsigned long long>(plan.tile_bytes), plan.vec_bytes - off));
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const char *>(
                             p.src[threadIdx.x]) + off),
                         "r"(bytes)
                         : "memory");
        }
    }
    pdl_wait();  // the kernel before this one on the stream has finished
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
