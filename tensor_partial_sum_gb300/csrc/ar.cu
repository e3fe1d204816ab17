// C ABI of the partial-sum reduction: context, argument checks, variant
// dispatch and launches.  The operation, its arguments and its error
// behaviour are specified in include/ar.h.
//
// Structure follows the hook trio of the pages (init / allreduce / free in
// ggml-cuda allreduce.cu: ggml_cuda_ar_pipeline_init, ggml_cuda_ar_allreduce,
// ggml_cuda_ar_pipeline_free) without the transport: on one GPU the R
// partials are plain device buffers, so a call is one kernel launch on the
// caller's stream.  ggml_cuda_ar_allreduce chooses its strategy by byte
// count; here the byte count chooses the launch shape of one kernel family:
// 16-byte vectors in 128-thread blocks below the switch, the widest aligned
// vectors in 256-thread blocks above it.  Status codes instead of asserts
// follow validate_allreduce / op_allreduce in ggml-hexagon
// htp/allreduce-ops.c.
#include "ar.h"

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ar_dispatch.h"

using tps::ArParams;

namespace {

constexpr int kLatencyThreads = 128;
constexpr int kBandwidthThreads = 256;
constexpr int kScalarThreads = 256;
constexpr int64_t kDefaultLatencyMaxBytes = 16ll << 20;  // measured crossover on GB300
// ar_reduce_host cuts a call into chunks of this many bytes per buffer (at
// most kMaxHostChunks chunks) so that host->device copies, kernels and
// device->host copies of different chunks overlap.
constexpr int64_t kDefaultHostChunkBytes = 4ll << 20;
constexpr int kMaxHostChunks = 64;

// Streams and events of the ar_reduce_host pipeline, made once at ar_init.
struct HostPipe {
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t copied[kMaxHostChunks] = {};
    cudaEvent_t reduced[kMaxHostChunks] = {};
};

struct Context {
    bool ready = false;
    int R = 0;
    size_t max_elems = 0;
    int device = -1;
    int sm_count = 0;
    int64_t latency_max_bytes = kDefaultLatencyMaxBytes;
    int forced_variant = AR_VARIANT_AUTO;
    int last_variant = AR_VARIANT_AUTO;
    int fault_inject = 0;
    int bw_blocks_per_sm = 0;
    int64_t host_chunk_bytes = kDefaultHostChunkBytes;
    HostPipe pipe;
    unsigned *dev_status = nullptr;  // device word the TMA variant sets when a wait runs out
    int tma_stages = 3;              // AR_TMA_STAGES (2..8)
    int tma_tile = 16384;            // AR_TMA_TILE: largest tile, bytes (1024 .. 32768, 1 KiB multiples)
    int tma_ctas_per_sm = 2;         // AR_TMA_CTAS_PER_SM (1..4)
    int64_t tma_drop_tile = -1;      // test hook (AR_Q_TMA_DROP_TILE), -1 = off
    int pdl = 1;                     // AR_PDL: kernels launch as programmatic dependents
    int l2_prefetch = 1;             // AR_L2_PREFETCH: the first wave prefetches its sources before the wait
};

void destroy_pipe(HostPipe &p) {
    for (cudaStream_t *s : {&p.h2d, &p.comp, &p.d2h})
        if (*s) cudaStreamDestroy(*s), *s = nullptr;
    for (cudaEvent_t *e : {&p.start, &p.done})
        if (*e) cudaEventDestroy(*e), *e = nullptr;
    for (int k = 0; k < kMaxHostChunks; ++k) {
        if (p.copied[k]) cudaEventDestroy(p.copied[k]), p.copied[k] = nullptr;
        if (p.reduced[k]) cudaEventDestroy(p.reduced[k]), p.reduced[k] = nullptr;
    }
}

bool create_pipe(HostPipe &p) {
    const unsigned ev = cudaEventDisableTiming;
    bool ok = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.start, ev) == cudaSuccess &&
              cudaEventCreateWithFlags(&p.done, ev) == cudaSuccess;
    for (int k = 0; ok && k < kMaxHostChunks; ++k)
        ok = cudaEventCreateWithFlags(&p.copied[k], ev) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.reduced[k], ev) == cudaSuccess;
    if (!ok) destroy_pipe(p);
    return ok;
}

std::mutex g_mu;
Context g_ctx;
// Held by a staged ar_reduce_host for its whole call (the context's pipeline
// streams and events are one set), and by ar_init and ar_free while they
// replace the context.  Lock order: g_pipe_mu before g_mu.
std::mutex g_pipe_mu;
// Incremented (under g_mu) by every ar_init and ar_free: a call that drops
// the lock half way through can tell whether the context was replaced.
unsigned long long g_ctx_gen = 0;

// Forget the cached device addresses of the no-allocation staging area (a
// new context may follow a device reset, after which the area can sit at a
// new address).  Called with g_mu held.
void forget_noalloc_addresses();

size_t elem_bytes(int dtype) {
    switch (dtype) {
        case AR_F32: return 4;
        case AR_F16: return 2;
        case AR_BF16: return 2;
        default: return 0;
    }
}

bool ranges_overlap(uintptr_t a, uintptr_t b, size_t bytes) { return a < b + bytes && b < a + bytes; }

using tps::KernelFn;
using tps::Kernels;

const Kernels &kernels_for(int dst, int wire) {
    if (dst == AR_F32) return tps::kernels_f32(wire);
    if (dst == AR_F16) return tps::kernels_f16(wire);
    return tps::kernels_bf16(wire);
}

// Resident CTAs per SM of a kernel at a block size (queried once, then
// cached in an open-addressed table keyed by the kernel's address and the
// block size; guarded by g_mu).
struct OccEntry {
    const void *fn;
    int threads;
    int blocks;
};
constexpr int kOccSlots = 1024;  // more than twice the (kernel, block size) pairs queried
OccEntry g_occ[kOccSlots];

// The slot holding (fn, threads), or the empty slot where it belongs (-1: full).
int occ_slot(const void *fn, int threads) {
    size_t h = ((reinterpret_cast<uintptr_t>(fn) >> 4) ^ static_cast<uintptr_t>(threads)) % kOccSlots;
    for (int probe = 0; probe < kOccSlots; ++probe, h = (h + 1) % kOccSlots) {
        if (g_occ[h].fn == nullptr || (g_occ[h].fn == fn && g_occ[h].threads == threads)) return static_cast<int>(h);
    }
    return -1;
}

template <typename Fn>
int blocks_per_sm(Fn *fn, int threads) {
    const void *f = reinterpret_cast<const void *>(fn);
    const int h = occ_slot(f, threads);
    if (h >= 0 && g_occ[h].fn == f) return g_occ[h].blocks;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, f, threads, 0) != cudaSuccess || b < 1) {
        cudaGetLastError();
        b = 1;
    }
    if (h >= 0) g_occ[h] = OccEntry{f, threads, b};
    return b;
}

// CTAs of a launch that the GPU holds from the start (its first wave), for
// the L2 prefetch before the dependent-launch wait.  Makes no CUDA call, so
// it is safe inside a stream capture: the cached occupancy when ar_init
// queried it, else the bound that the SM's thread limit sets.
template <typename Fn>
int first_wave(Fn *fn, int threads, int sms) {
    const void *f = reinterpret_cast<const void *>(fn);
    const int h = occ_slot(f, threads);
    const int per_sm = (h >= 0 && g_occ[h].fn == f) ? g_occ[h].blocks : 2048 / threads;
    return per_sm * sms;
}

// Occupancy of every kernel a prefetching launch uses at its usual block
// size, queried once (at ar_init, outside any stream capture).
void warm_occupancy() {
    const int dtypes[3] = {AR_F32, AR_F16, AR_BF16};
    for (int dst : dtypes)
        for (int wire : dtypes) {
            const Kernels &k = kernels_for(dst, wire);
            for (int nc = 0; nc < 2; ++nc) {
                blocks_per_sm(k.v16.few[nc], kLatencyThreads);
                blocks_per_sm(k.v16.many[nc], kLatencyThreads);
                blocks_per_sm(k.bw16.few[nc], kBandwidthThreads);
                blocks_per_sm(k.bw16.many[nc], kBandwidthThreads);
                blocks_per_sm(k.wide.few[nc], kBandwidthThreads);
                blocks_per_sm(k.wide.many[nc], kBandwidthThreads);
                blocks_per_sm(k.pack[nc], 256);
                blocks_per_sm(k.scalar[nc], kScalarThreads);
            }
            if (k.pack32) blocks_per_sm(k.pack32, 256);
            for (int many = 0; many < 2; ++many)
                for (int res = 0; res < 2; ++res) {
                    blocks_per_sm(k.ex[many][res][1], 256);
                    if (k.ex32[many][res]) blocks_per_sm(k.ex32[many][res], 256);
                }
        }
}

int parse_variant(const char *s) {
    if (!s || !*s || !strcmp(s, "auto")) return AR_VARIANT_AUTO;
    if (!strcmp(s, "tma")) return AR_VARIANT_TMA;
    if (!strcmp(s, "naive")) return AR_VARIANT_NAIVE;
    if (!strcmp(s, "latency")) return AR_VARIANT_LATENCY;
    if (!strcmp(s, "bandwidth")) return AR_VARIANT_BANDWIDTH;
    if (!strcmp(s, "scalar")) return AR_VARIANT_SCALAR;
    return -1;
}

const char *variant_name(int v) {
    switch (v) {
        case AR_VARIANT_NAIVE: return "naive";
        case AR_VARIANT_LATENCY: return "latency";
        case AR_VARIANT_BANDWIDTH: return "bandwidth";
        case AR_VARIANT_SCALAR: return "scalar";
        case AR_VARIANT_TMA: return "tma";
        default: return "auto";
    }
}

// Launch a kernel that runs griddepcontrol.launch_dependents and
// griddepcontrol.wait before it loads or stores anything: as a programmatic
// dependent of the kernel before it on the stream when `pdl`, else plainly.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*fn)(Params...), dim3 grid, unsigned threads, size_t smem, cudaStream_t stream,
                             bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // Not on the default streams: their implicit ordering against other
    // streams is left exactly as a plain launch has it.
    const bool default_stream = stream == nullptr || stream == cudaStreamLegacy || stream == cudaStreamPerThread;
    cfg.numAttrs = (pdl && !default_stream) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, fn, args...);
}

int grid_cap(long long want, long long cap) {
    if (want < 1) want = 1;
    if (want > cap) want = cap;
    return static_cast<int>(want);
}

// TMA variant: 3 stages of R source tiles plus two output tiles in shared
// memory, the tile as large as fits (1 KiB multiples, at most 16 KiB), two
// CTAs per SM (or grid_blocks), every wait bounded by 100 ms.
constexpr size_t kTmaSmemBudget = 224 * 1024;  // per SM

int launch_tma_locked(const Kernels &k, const ArParams &p, size_t nelem, size_t esize, int grid_blocks,
                      cudaStream_t stream) {
    Context &c = g_ctx;
    tps::TmaPlan plan{};
    plan.vec_bytes = (static_cast<unsigned long long>(nelem) * esize) / 16 * 16;
    const size_t S = static_cast<size_t>(c.tma_stages);
    const size_t budget = kTmaSmemBudget / static_cast<size_t>(c.tma_ctas_per_sm) - tps::kTmaHeaderBytes - 1024;
    size_t tile = budget / (S * p.R + 2) / 1024 * 1024;
    if (tile > static_cast<size_t>(c.tma_tile)) tile = static_cast<size_t>(c.tma_tile);
    if (tile < 1024) return AR_ERR_UNSUPPORTED;
    plan.tile_bytes = static_cast<unsigned>(tile);
    plan.stages = static_cast<unsigned>(S);
    plan.ntiles = (plan.vec_bytes + tile - 1) / tile;
    plan.status = c.dev_status;
    plan.timeout_ns = 100ull * 1000 * 1000;
    plan.drop_tile = c.tma_drop_tile < 0 ? ~0ull : static_cast<unsigned long long>(c.tma_drop_tile);
    const size_t smem = tps::kTmaHeaderBytes + (S * p.R + 2) * tile;
    if (cudaFuncSetAttribute(reinterpret_cast<const void *>(k.tma), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return AR_ERR_CUDA;
    long long grid = grid_blocks > 0 ? grid_blocks : static_cast<long long>(c.sm_count) * c.tma_ctas_per_sm;
    if (grid > static_cast<long long>(plan.ntiles)) grid = static_cast<long long>(plan.ntiles);
    if (grid < 1) grid = 1;
    ArParams pt = p;  // every CTA of the persistent grid is resident from the start
    pt.prefetch_ctas = c.l2_prefetch ? static_cast<int>(grid) : 0;
    if (launch_dependent(k.tma, dim3(static_cast<unsigned>(grid)), tps::kTmaThreads, smem, stream, c.pdl != 0, pt,
                         plan) != cudaSuccess) {
        cudaGetLastError();
        return AR_ERR_CUDA;
    }
    c.last_variant = AR_VARIANT_TMA;
    return AR_OK;
}

// Launch one reduction; the caller holds g_mu and has validated the arguments.
int launch_locked(const void *const *srcs, void *const *dsts, int n_dsts, size_t nelem, int dst_dtype,
                  int wire_dtype, int variant, int grid_blocks, cudaStream_t stream, bool explicit_variant,
                  bool device_buffers = true) {
    Context &c = g_ctx;
    if (nelem == 0) return AR_OK;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
    if (dev != c.device) return AR_ERR_INVALID_ARG;

    bool alias = false;
    for (int d = 0; d < n_dsts; ++d)
        for (int r = 0; r < c.R; ++r) alias |= (dsts[d] == srcs[r]);
    // The offset every buffer has from an M-byte boundary when they all share
    // one, else -1.  A shared offset lets the vector kernels run on buffers
    // shifted forward to alignment, with the few elements before handled
    // one by one (the "head").
    auto common_offset = [&](uintptr_t M) -> long long {
        const uintptr_t m0 = reinterpret_cast<uintptr_t>(srcs[0]) % M;
        for (int r = 1; r < c.R; ++r)
            if (reinterpret_cast<uintptr_t>(srcs[r]) % M != m0) return -1;
        for (int d = 0; d < n_dsts; ++d)
            if (reinterpret_cast<uintptr_t>(dsts[d]) % M != m0) return -1;
        return static_cast<long long>(m0);
    };
    const long long off16 = common_offset(16), off32 = common_offset(32);
    const bool aligned = off16 >= 0;  // vector paths possible (after a head)

    const size_t esize = elem_bytes(dst_dtype);
    if (variant == AR_VARIANT_AUTO) variant = c.forced_variant;
    if (variant == AR_VARIANT_AUTO) {
        const double bytes = static_cast<double>(c.R + n_dsts) * static_cast<double>(nelem) * esize;
        variant = bytes < static_cast<double>(c.latency_max_bytes) ? AR_VARIANT_LATENCY : AR_VARIANT_BANDWIDTH;
    }
    if (!aligned && (variant == AR_VARIANT_LATENCY || variant == AR_VARIANT_BANDWIDTH || variant == AR_VARIANT_TMA)) {
        if (explicit_variant) return AR_ERR_INVALID_ARG;
        variant = AR_VARIANT_SCALAR;
    }
    if (variant == AR_VARIANT_TMA && off16 != 0) {
        // bulk copies need 16-byte starts; a shared offset still suits the vector kernel
        if (explicit_variant) return AR_ERR_INVALID_ARG;
        variant = AR_VARIANT_BANDWIDTH;
    }
    if (c.fault_inject) return AR_ERR_CUDA;

    ArParams p;
    memset(&p, 0, sizeof p);
    for (int r = 0; r < c.R; ++r) p.src[r] = srcs[r];
    for (int d = 0; d < n_dsts; ++d) p.dst[d] = dsts[d];
    p.nelem = nelem;
    p.R = c.R;
    p.n_dsts = n_dsts;

    // A destination that is also a source is written while it is being
    // read, so those calls use coherent loads instead of the read-only path.
    const int nc = alias ? 0 : 1;
    const Kernels &k = kernels_for(dst_dtype, wire_dtype);
    const long long sms = c.sm_count;
    KernelFn fn = nullptr;
    int threads = 0, grid = 0;
    int plan_vec_bytes = 0;  // vector width of an ar_reduce_kernel launch, 0 for the other kernels
    // Shift every buffer forward past the head to the vector boundary.
    auto peel = [&](int vec_bytes, long long offset) {
        long long head = offset ? (vec_bytes - offset) / static_cast<long long>(esize) : 0;
        if (head > static_cast<long long>(nelem)) head = static_cast<long long>(nelem);
        for (int r = 0; r < c.R; ++r) p.src[r] = static_cast<const char *>(srcs[r]) + head * esize;
        for (int d = 0; d < n_dsts; ++d) p.dst[d] = static_cast<char *>(dsts[d]) + head * esize;
        p.nelem = nelem - static_cast<size_t>(head);
        p.head = static_cast<int>(head);
    };
    switch (variant) {
        case AR_VARIANT_LATENCY: {
            // 16-byte vectors, one per thread, a grid that covers the tensor
            const tps::VecKernels &vk = k.v16;
            fn = (c.R <= 2 ? vk.few : vk.many)[nc];
            threads = kLatencyThreads;
            plan_vec_bytes = 16;
            peel(16, off16);
            const long long V = static_cast<long long>(16 / esize);
            const long long nv = static_cast<long long>(p.nelem) / V;
            // with a tail, at most threads - V vectors per CTA, so the last CTA
            // has idle threads for the tail
            const long long per_cta = (static_cast<long long>(p.nelem) % V) ? threads - V : threads;
            grid = grid_cap((nv + per_cta - 1) / per_cta, 0x7FFFFFFFll);
            break;
        }
        case AR_VARIANT_BANDWIDTH: {
            // the widest vectors the buffers' common offset allows, one per
            // thread; a grid that covers the tensor unless a persistent grid
            // is asked for
            const bool wide = k.wide_bytes == 32 && off32 >= 0;
            const tps::VecKernels &vk = wide ? k.wide : k.bw16;
            const int vec_bytes = wide ? k.wide_bytes : 16;
            fn = (c.R <= 2 ? vk.few : vk.many)[nc];
            threads = kBandwidthThreads;
            plan_vec_bytes = vec_bytes;
            peel(vec_bytes, wide ? off32 : off16);
            const long long V = static_cast<long long>(vec_bytes / esize);
            const long long nv = static_cast<long long>(p.nelem) / V;
            const long long per_cta = (static_cast<long long>(p.nelem) % V) ? threads - V : threads;
            const long long full = (nv + per_cta - 1) / per_cta;
            if (grid_blocks > 0) {
                grid = grid_blocks;
            } else if (c.bw_blocks_per_sm > 0) {
                const int occ = blocks_per_sm(fn, threads);
                grid = grid_cap(full, sms * (c.bw_blocks_per_sm < occ ? c.bw_blocks_per_sm : occ));
            } else {
                grid = grid_cap(full, 0x7FFFFFFFll);
            }
            break;
        }
        case AR_VARIANT_SCALAR: {
            fn = k.scalar[nc];
            threads = kScalarThreads;
            const long long cap = grid_blocks > 0 ? grid_blocks : sms * blocks_per_sm(fn, threads);
            grid = grid_cap(grid_blocks > 0 ? cap : (static_cast<long long>(nelem) + threads - 1) / threads, cap);
            // the first wave prefetches its first elements before the wait
            if (c.l2_prefetch && device_buffers) p.prefetch_ctas = first_wave(fn, threads, c.sm_count);
            break;
        }
        case AR_VARIANT_TMA:
            return launch_tma_locked(k, p, nelem, esize, grid_blocks, stream);
        case AR_VARIANT_NAIVE: {
            fn = k.naive;
            threads = kScalarThreads;
            const long long cap = grid_blocks > 0 ? grid_blocks : sms * 16;
            grid = grid_cap(grid_blocks > 0 ? cap : (static_cast<long long>(nelem) + threads - 1) / threads, cap);
            break;
        }
        default: return AR_ERR_INVALID_ARG;
    }

    if (plan_vec_bytes > 0) {
        // rounds and chunk of ar_reduce_kernel for this grid (one vector per thread per round)
        const unsigned long long nv = p.nelem / (plan_vec_bytes / esize);
        const unsigned long long per_round = static_cast<unsigned long long>(grid) * threads;
        p.rounds = (nv + per_round - 1) / per_round;
        p.chunk = p.rounds ? (nv + p.rounds * grid - 1) / (p.rounds * grid) : 0;
        // the first wave (the CTAs the GPU holds at once) prefetches its
        // sources into L2 before waiting for the kernel ahead of it; device
        // memory only: host buffers read over the CPU-GPU link are left to
        // the loads
        if (c.l2_prefetch && device_buffers) p.prefetch_ctas = first_wave(fn, threads, c.sm_count);
    }
    // The kernels wait (griddepcontrol.wait) for the kernel before them on
    // the stream before they load or store anything (their first wave only
    // prefetches into L2 before it), so they may be launched as programmatic
    // dependents: the launch then overlaps that kernel's last wave.  The
    // naive cross-check kernel has no such wait and launches plainly.
    if (launch_dependent(fn, dim3(static_cast<unsigned>(grid)), static_cast<unsigned>(threads), 0, stream,
                         c.pdl != 0 && variant != AR_VARIANT_NAIVE, p) != cudaSuccess) {
        cudaGetLastError();
        return AR_ERR_CUDA;
    }
    c.last_variant = variant;
    return AR_OK;
}

// Device address of host memory the GPU can reach (pinned or managed), or
// nullptr for memory it cannot (pageable, or unknown to CUDA).
void *device_view(const void *host) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeManaged) return const_cast<void *>(host);
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    return nullptr;
}

// ar_reduce_host without staging buffers: the kernel loads the host
// partials and stores the host results itself, over the CPU-GPU link
// (NVLink-C2C on GB300), with one persistent CTA per SM.
int reduce_host_direct_locked(const void *const *h_srcs, void *const *h_dsts, int n_dsts, size_t nelem,
                              int dst_dtype, int wire_dtype, cudaStream_t stream) {
    const Context &c = g_ctx;
    if (n_dsts < 1 || n_dsts > AR_MAX_DSTS) return AR_ERR_INVALID_ARG;
    const void *s[AR_MAX_RANKS];
    void *d[AR_MAX_DSTS];
    for (int r = 0; r < c.R; ++r) {
        if (!h_srcs[r] && nelem) return AR_ERR_INVALID_ARG;
        s[r] = nelem ? device_view(h_srcs[r]) : h_srcs[r];
        if (nelem && !s[r]) return AR_ERR_INVALID_ARG;
    }
    for (int k = 0; k < n_dsts; ++k) {
        if (!h_dsts[k] && nelem) return AR_ERR_INVALID_ARG;
        d[k] = nelem ? device_view(h_dsts[k]) : h_dsts[k];
        if (nelem && !d[k]) return AR_ERR_INVALID_ARG;
    }
    const int st = ar_check_args(c.R, s, d, n_dsts, nelem, c.max_elems, dst_dtype, wire_dtype);
    if (st != AR_OK || nelem == 0) return st;
    // one CTA per SM; buffers at different offsets from a vector boundary
    // fall back to the element-wise kernel on the same grid
    return launch_locked(s, d, n_dsts, nelem, dst_dtype, wire_dtype, AR_VARIANT_BANDWIDTH, c.sm_count, stream,
                         false, false);
}

}  // namespace

extern "C" {

const char *ar_status_string(int status) {
    switch (status) {
        case AR_OK: return "ok";
        case AR_ERR_INVALID_ARG: return "invalid argument";
        case AR_ERR_UNSUPPORTED: return "unsupported dtype or device";
        case AR_ERR_TOO_LARGE: return "nelem exceeds max_elems";
        case AR_ERR_NOT_INITIALIZED: return "ar_init has not succeeded";
        case AR_ERR_OVERLAP: return "a destination partly overlaps another buffer";
        case AR_ERR_CUDA: return "CUDA call failed";
        default: return "unknown status";
    }
}

int ar_check_args(int R, const void *const *srcs, void *const *dsts, int n_dsts, size_t nelem, size_t max_elems,
                  int dst_dtype, int wire_dtype) {
    if (R < 1 || R > AR_MAX_RANKS) return AR_ERR_INVALID_ARG;
    if (n_dsts < 1 || n_dsts > AR_MAX_DSTS) return AR_ERR_INVALID_ARG;
    if (!srcs || !dsts) return AR_ERR_INVALID_ARG;
    const size_t esize = elem_bytes(dst_dtype);
    if (!esize || !elem_bytes(wire_dtype)) return AR_ERR_UNSUPPORTED;
    if (nelem > max_elems) return AR_ERR_TOO_LARGE;
    if (nelem == 0) return AR_OK;
    for (int r = 0; r < R; ++r) {
        if (!srcs[r]) return AR_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(srcs[r]) % esize) return AR_ERR_INVALID_ARG;
    }
    for (int d = 0; d < n_dsts; ++d) {
        if (!dsts[d]) return AR_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(dsts[d]) % esize) return AR_ERR_INVALID_ARG;
    }
    if (nelem > SIZE_MAX / esize) return AR_ERR_TOO_LARGE;
    const size_t bytes = nelem * esize;
    for (int d = 0; d < n_dsts; ++d) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(dsts[d]);
        if (a > UINTPTR_MAX - bytes) return AR_ERR_INVALID_ARG;
        for (int r = 0; r < R; ++r) {
            const uintptr_t b = reinterpret_cast<uintptr_t>(srcs[r]);
            if (a != b && ranges_overlap(a, b, bytes)) return AR_ERR_OVERLAP;
        }
        for (int e = 0; e < d; ++e) {
            if (ranges_overlap(a, reinterpret_cast<uintptr_t>(dsts[e]), bytes)) return AR_ERR_OVERLAP;
        }
    }
    return AR_OK;
}

int ar_init(int R, size_t max_elems) {
    if (R < 1 || R > AR_MAX_RANKS || max_elems < 1) return AR_ERR_INVALID_ARG;
    if (max_elems > SIZE_MAX / 4) return AR_ERR_INVALID_ARG;
    const int variant = parse_variant(getenv("AR_VARIANT"));
    if (variant < 0) return AR_ERR_INVALID_ARG;

    std::lock_guard<std::mutex> pipe_lock(g_pipe_mu);
    std::lock_guard<std::mutex> lock(g_mu);
    destroy_pipe(g_ctx.pipe);
    if (g_ctx.dev_status) cudaFree(g_ctx.dev_status);
    g_ctx = Context{};
    ++g_ctx_gen;
    forget_noalloc_addresses();
    int dev = -1, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return AR_ERR_CUDA;
    // The library carries sm_103a code only: make sure this device runs it.
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, reinterpret_cast<const void *>(kernels_for(AR_F32, AR_F32).v16.few[1])) !=
        cudaSuccess) {
        cudaGetLastError();
        return AR_ERR_UNSUPPORTED;
    }
    Context c;
    c.R = R;
    c.max_elems = max_elems;
    c.device = dev;
    c.sm_count = sms;
    c.forced_variant = variant;
    auto env_int = [](const char *name, int lo, int hi, int *out) {
        const char *s = getenv(name);
        if (!s) return true;
        char *end = nullptr;
        const long v = strtol(s, &end, 10);
        if (end == s || v < lo || v > hi) return false;
        *out = static_cast<int>(v);
        return true;
    };
    if (!env_int("AR_TMA_STAGES", 2, tps::kTmaMaxStages, &c.tma_stages) ||
        !env_int("AR_TMA_TILE", 1024, 32768, &c.tma_tile) || c.tma_tile % 1024 ||
        !env_int("AR_TMA_CTAS_PER_SM", 1, 4, &c.tma_ctas_per_sm) || !env_int("AR_PDL", 0, 1, &c.pdl) ||
        !env_int("AR_L2_PREFETCH", 0, 1, &c.l2_prefetch))
        return AR_ERR_INVALID_ARG;
    if (const char *s = getenv("AR_LATENCY_MAX_BYTES")) {
        char *end = nullptr;
        const long long v = strtoll(s, &end, 10);
        if (end == s || v < 0) return AR_ERR_INVALID_ARG;
        c.latency_max_bytes = v;
    }
    warm_occupancy();
    if (!create_pipe(c.pipe)) return AR_ERR_CUDA;
    if (cudaMalloc(reinterpret_cast<void **>(&c.dev_status), 64) != cudaSuccess ||
        cudaMemset(c.dev_status, 0, 64) != cudaSuccess) {
        destroy_pipe(c.pipe);
        return AR_ERR_CUDA;
    }
    c.ready = true;
    g_ctx = c;
    if (const char *s = getenv("AR_LOG"); s && !strcmp(s, "1")) {
        fprintf(stderr, "[ar] init: R=%d max_elems=%zu device=%d SMs=%d latency_max_bytes=%lld variant=%s\n", R,
                max_elems, dev, sms, static_cast<long long>(c.latency_max_bytes), variant_name(variant));
    }
    return AR_OK;
}

void ar_free(void) {
    std::lock_guard<std::mutex> pipe_lock(g_pipe_mu);
    std::lock_guard<std::mutex> lock(g_mu);
    destroy_pipe(g_ctx.pipe);
    if (g_ctx.dev_status) cudaFree(g_ctx.dev_status);
    g_ctx = Context{};
    ++g_ctx_gen;
    forget_noalloc_addresses();
}

int ar_reduce_variant(const void *const *srcs, void *const *dsts, int n_dsts, size_t nelem, int dst_dtype,
                      int wire_dtype, int variant, int grid_blocks, cudaStream_t stream) {
    if (variant < AR_VARIANT_AUTO || variant > AR_VARIANT_TMA || grid_blocks < 0) return AR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ctx.ready) return AR_ERR_NOT_INITIALIZED;
    const int st = ar_check_args(g_ctx.R, srcs, dsts, n_dsts, nelem, g_ctx.max_elems, dst_dtype, wire_dtype);
    if (st != AR_OK) return st;
    return launch_locked(srcs, dsts, n_dsts, nelem, dst_dtype, wire_dtype, variant, grid_blocks, stream,
                         variant != AR_VARIANT_AUTO);
}

int ar_reduce(const void *const *srcs, void *const *dsts, int n_dsts, size_t nelem, int dst_dtype, int wire_dtype,
              cudaStream_t stream) {
    return ar_reduce_variant(srcs, dsts, n_dsts, nelem, dst_dtype, wire_dtype, AR_VARIANT_AUTO, 0, stream);
}

int ar_query(int key, int64_t *value) {
    if (!value) return AR_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ctx.ready) return AR_ERR_NOT_INITIALIZED;
    const Context &c = g_ctx;
    switch (key) {
        case AR_Q_RANKS: *value = c.R; break;
        case AR_Q_MAX_ELEMS: *value = static_cast<int64_t>(c.max_elems); break;
        case AR_Q_DEVICE: *value = c.device; break;
        case AR_Q_SM_COUNT: *value = c.sm_count; break;
        case AR_Q_LATENCY_MAX_BYTES: *value = c.latency_max_bytes; break;
        case AR_Q_FORCED_VARIANT: *value = c.forced_variant; break;
        case AR_Q_LAST_VARIANT: *value = c.last_variant; break;
        case AR_Q_FAULT_INJECT: *value = c.fault_inject; break;
        case AR_Q_BW_BLOCKS_PER_SM: *value = c.bw_blocks_per_sm; break;
        case AR_Q_HOST_CHUNK_BYTES: *value = c.host_chunk_bytes; break;
        case AR_Q_TMA_DROP_TILE: *value = c.tma_drop_tile; break;
        case AR_Q_DEVICE_STATUS: {
            unsigned v = 0;
            if (cudaMemcpy(&v, c.dev_status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return AR_ERR_CUDA;
            *value = v;
            break;
        }
        default: return AR_ERR_INVALID_ARG;
    }
    return AR_OK;
}

int ar_set_option(int key, int64_t value) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ctx.ready) return AR_ERR_NOT_INITIALIZED;
    Context &c = g_ctx;
    switch (key) {
        case AR_Q_LATENCY_MAX_BYTES:
            if (value < 0) return AR_ERR_INVALID_ARG;
            c.latency_max_bytes = value;
            break;
        case AR_Q_FORCED_VARIANT:
            if (value < AR_VARIANT_AUTO || value > AR_VARIANT_TMA) return AR_ERR_INVALID_ARG;
            c.forced_variant = static_cast<int>(value);
            break;
        case AR_Q_FAULT_INJECT: c.fault_inject = value ? 1 : 0; break;
        case AR_Q_BW_BLOCKS_PER_SM:
            if (value < 0 || value > 64) return AR_ERR_INVALID_ARG;
            c.bw_blocks_per_sm = static_cast<int>(value);
            break;
        case AR_Q_HOST_CHUNK_BYTES:
            if (value < 1) return AR_ERR_INVALID_ARG;
            c.host_chunk_bytes = value;
            break;
        case AR_Q_TMA_DROP_TILE:
            if (value < -1) return AR_ERR_INVALID_ARG;
            c.tma_drop_tile = value;
            break;
        case AR_Q_DEVICE_STATUS:
            if (value != 0) return AR_ERR_INVALID_ARG;
            if (cudaMemset(c.dev_status, 0, 64) != cudaSuccess) return AR_ERR_CUDA;
            break;
        default: return AR_ERR_INVALID_ARG;
    }
    return AR_OK;
}

int ar_reduce_host(const void *const *h_srcs, void *const *h_dsts, int n_dsts, size_t nelem, int dst_dtype,
                   int wire_dtype, void *const *d_srcs, void *const *d_dsts, cudaStream_t stream) {
    if (!d_srcs && !d_dsts) {  // direct mode: one launch, under the library lock like every launch
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_ctx.ready) return AR_ERR_NOT_INITIALIZED;
        if (!h_srcs || !h_dsts) return AR_ERR_INVALID_ARG;
        return reduce_host_direct_locked(h_srcs, h_dsts, n_dsts, nelem, dst_dtype, wire_dtype, stream);
    }
    // Staged mode.  g_pipe_mu gives this call the context's pipeline streams
    // and events (and keeps them alive: ar_init and ar_free take it too).
    // The copies are enqueued without g_mu, because a copy from or to
    // pageable host memory can block the calling thread until its stream
    // gets there, and other library calls must not wait behind it; each
    // chunk's launch takes g_mu.
    std::lock_guard<std::mutex> pipe_lock(g_pipe_mu);
    int R = 0;
    size_t chunk = 0;
    HostPipe pp;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_ctx.ready) return AR_ERR_NOT_INITIALIZED;
        const Context &c = g_ctx;
        if (!h_srcs || !h_dsts) return AR_ERR_INVALID_ARG;
        if (!d_srcs || !d_dsts) return AR_ERR_INVALID_ARG;
        const void *srcs_c[AR_MAX_RANKS];
        for (int r = 0; r < c.R; ++r) srcs_c[r] = d_srcs[r];
        int st = ar_check_args(c.R, srcs_c, d_dsts, n_dsts, nelem, c.max_elems, dst_dtype, wire_dtype);
        if (st != AR_OK) return st;
        if (nelem == 0) return AR_OK;
        // The host buffers obey the same rules.  A host destination that partly
        // overlaps a host source would be written (copy back of chunk k) before
        // a later chunk's copy in has read the source bytes it shares.
        st = ar_check_args(c.R, h_srcs, h_dsts, n_dsts, nelem, c.max_elems, dst_dtype, wire_dtype);
        if (st != AR_OK) return st;
        // the launches check the device too, but only after copies would be queued
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
        if (dev != c.device) return AR_ERR_INVALID_ARG;
        if (c.fault_inject) return AR_ERR_CUDA;
        // Chunks of whole 256-element groups (so every chunk keeps the buffers'
        // alignment); chunking never changes a result bit.
        chunk = static_cast<size_t>(c.host_chunk_bytes) / elem_bytes(dst_dtype);
        const size_t min_chunk = (nelem + kMaxHostChunks - 1) / kMaxHostChunks;
        if (chunk < min_chunk) chunk = min_chunk;
        chunk = (chunk + 255) / 256 * 256;
        R = c.R;
        pp = c.pipe;
    }
    const size_t esize = elem_bytes(dst_dtype);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // everything the caller enqueued on `stream` before this call comes first
    if (!ok(cudaEventRecord(pp.start, stream)) || !ok(cudaStreamWaitEvent(pp.h2d, pp.start, 0)) ||
        !ok(cudaStreamWaitEvent(pp.comp, pp.start, 0)) || !ok(cudaStreamWaitEvent(pp.d2h, pp.start, 0)))
        return AR_ERR_CUDA;
    const void *cs[AR_MAX_RANKS];
    void *cd[AR_MAX_DSTS];
    int k = 0;
    for (size_t off = 0; off < nelem; off += chunk, ++k) {
        const size_t n = nelem - off < chunk ? nelem - off : chunk;
        const size_t boff = off * esize, nb = n * esize;
        for (int r = 0; r < R; ++r) {
            char *dptr = static_cast<char *>(d_srcs[r]) + boff;
            if (!ok(cudaMemcpyAsync(dptr, static_cast<const char *>(h_srcs[r]) + boff, nb, cudaMemcpyHostToDevice,
                                    pp.h2d)))
                return AR_ERR_CUDA;
            cs[r] = dptr;
        }
        for (int d = 0; d < n_dsts; ++d) cd[d] = static_cast<char *>(d_dsts[d]) + boff;
        if (!ok(cudaEventRecord(pp.copied[k], pp.h2d)) || !ok(cudaStreamWaitEvent(pp.comp, pp.copied[k], 0)))
            return AR_ERR_CUDA;
        {
            std::lock_guard<std::mutex> lock(g_mu);
            const int lst =
                launch_locked(cs, cd, n_dsts, n, dst_dtype, wire_dtype, AR_VARIANT_AUTO, 0, pp.comp, false);
            if (lst != AR_OK) return lst;
        }
        if (!ok(cudaEventRecord(pp.reduced[k], pp.comp)) || !ok(cudaStreamWaitEvent(pp.d2h, pp.reduced[k], 0)))
            return AR_ERR_CUDA;
        for (int d = 0; d < n_dsts; ++d)
            if (!ok(cudaMemcpyAsync(static_cast<char *>(h_dsts[d]) + boff, cd[d], nb, cudaMemcpyDeviceToHost, pp.d2h)))
                return AR_ERR_CUDA;
    }
    // the caller's stream continues once the last copy back has finished
    if (!ok(cudaEventRecord(pp.done, pp.d2h)) || !ok(cudaStreamWaitEvent(stream, pp.done, 0))) return AR_ERR_CUDA;
    return AR_OK;
}

// ---- extended layouts --------------------------------------------------------

namespace {

// Byte span [start, end) a buffer of ne1 rows at `stride` touches.
struct Span {
    uintptr_t start, end;
    int64_t stride;
};

bool make_span(const void *p, int64_t stride, size_t ne0, size_t ne1, size_t es, Span *out) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const unsigned __int128 len = static_cast<unsigned __int128>(ne1 - 1) * static_cast<uint64_t>(stride) +
                                  static_cast<unsigned __int128>(ne0) * es;
    if (len > static_cast<unsigned __int128>(UINTPTR_MAX - a)) return false;
    *out = Span{a, a + static_cast<uintptr_t>(len), stride};
    return true;
}

bool spans_overlap(const Span &x, const Span &y) { return x.start < y.end && y.start < x.end; }

bool valid_stride(int64_t stride, size_t ne0, size_t es) {
    return stride >= 0 && static_cast<uint64_t>(stride) >= ne0 * es && stride % static_cast<int64_t>(es) == 0;
}

}  // namespace

int ar_check_layout(int R, const void *const *srcs, void *const *dsts, int n_dsts, const ar_layout *L,
                    size_t max_elems, int dst_dtype, int wire_dtype) {
    if (R < 1 || R > AR_MAX_RANKS || n_dsts < 1 || n_dsts > AR_MAX_DSTS) return AR_ERR_INVALID_ARG;
    if (!srcs || !dsts || !L) return AR_ERR_INVALID_ARG;
    const size_t es = elem_bytes(dst_dtype);
    if (!es || !elem_bytes(wire_dtype)) return AR_ERR_UNSUPPORTED;
    if (R < 32 && (L->inactive_mask >> R) != 0) return AR_ERR_INVALID_ARG;
    if (L->ne0 && L->ne1 > SIZE_MAX / L->ne0) return AR_ERR_TOO_LARGE;
    const size_t nelem = L->ne0 * L->ne1;
    if (nelem > max_elems) return AR_ERR_TOO_LARGE;
    if (nelem == 0) return AR_OK;
    const int64_t packed = static_cast<int64_t>(L->ne0 * es);
    Span dsp[AR_MAX_DSTS], ssp[AR_MAX_RANKS], rsp{};
    bool active[AR_MAX_RANKS];
    for (int r = 0; r < R; ++r) {
        active[r] = !((L->inactive_mask >> r) & 1u);
        if (!active[r]) continue;
        const int64_t st = L->src_row_bytes ? L->src_row_bytes[r] : packed;
        if (!srcs[r] || reinterpret_cast<uintptr_t>(srcs[r]) % es) return AR_ERR_INVALID_ARG;
        if (L->ne1 > 1 && !valid_stride(st, L->ne0, es)) return AR_ERR_INVALID_ARG;
        if (!make_span(srcs[r], L->ne1 > 1 ? st : packed, L->ne0, L->ne1, es, &ssp[r])) return AR_ERR_INVALID_ARG;
    }
    for (int d = 0; d < n_dsts; ++d) {
        const int64_t st = L->dst_row_bytes ? L->dst_row_bytes[d] : packed;
        if (!dsts[d] || reinterpret_cast<uintptr_t>(dsts[d]) % es) return AR_ERR_INVALID_ARG;
        if (L->ne1 > 1 && !valid_stride(st, L->ne0, es)) return AR_ERR_INVALID_ARG;
        if (!make_span(dsts[d], L->ne1 > 1 ? st : packed, L->ne0, L->ne1, es, &dsp[d])) return AR_ERR_INVALID_ARG;
    }
    const bool bcast = L->residual && L->residual_row_bytes == 0;
    if (L->residual) {
        if (reinterpret_cast<uintptr_t>(L->residual) % es) return AR_ERR_INVALID_ARG;
        if (!bcast && L->ne1 > 1 && !valid_stride(L->residual_row_bytes, L->ne0, es)) return AR_ERR_INVALID_ARG;
        const int64_t st = (bcast || L->ne1 <= 1) ? packed : L->residual_row_bytes;
        if (!make_span(L->residual, st, L->ne0, bcast ? 1 : L->ne1, es, &rsp)) return AR_ERR_INVALID_ARG;
    }
    for (int d = 0; d < n_dsts; ++d) {
        for (int r = 0; r < R; ++r) {
            if (!active[r] || !spans_overlap(dsp[d], ssp[r])) continue;
            const bool same = dsp[d].start == ssp[r].start && (L->ne1 <= 1 || dsp[d].stride == ssp[r].stride);
            if (!same) return AR_ERR_OVERLAP;
        }
        if (L->residual && spans_overlap(dsp[d], rsp)) {
            const bool same = !bcast && dsp[d].start == rsp.start && (L->ne1 <= 1 || dsp[d].stride == rsp.stride);
            if (!same) return AR_ERR_OVERLAP;
        }
        for (int e = 0; e < d; ++e)
            if (spans_overlap(dsp[d], dsp[e])) return AR_ERR_OVERLAP;
    }
    return AR_OK;
}

int ar_reduce_ex(const void *const *srcs, void *const *dsts, int n_dsts, const ar_layout *L, int dst_dtype,
                 int wire_dtype, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ctx.ready) return AR_ERR_NOT_INITIALIZED;
    Context &c = g_ctx;
    const int st = ar_check_layout(c.R, srcs, dsts, n_dsts, L, c.max_elems, dst_dtype, wire_dtype);
    if (st != AR_OK || L->ne0 * L->ne1 == 0) return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
    if (dev != c.device) return AR_ERR_INVALID_ARG;
    if (c.fault_inject) return AR_ERR_CUDA;

    const size_t es = elem_bytes(dst_dtype);
    const int64_t packed = static_cast<int64_t>(L->ne0 * es);
    tps::ArExParams p;
    memset(&p, 0, sizeof p);
    p.ne0 = L->ne0;
    p.ne1 = L->ne1;
    p.R = c.R;
    p.n_dsts = n_dsts;
    p.inactive = L->inactive_mask;
    // The vector kernels need every row of every buffer to start at one
    // common offset from an M-byte boundary (the kernel reduces the elements
    // before it one by one): the start addresses agree modulo M, and so do
    // the row strides when there is more than one row.
    uintptr_t addr[tps::kMaxRanks + tps::kMaxDsts + 1], stride[tps::kMaxRanks + tps::kMaxDsts + 1];
    int nbuf = 0;
    auto add = [&](const void *a, long long st) {
        addr[nbuf] = reinterpret_cast<uintptr_t>(a);
        stride[nbuf++] = static_cast<uintptr_t>(st);
    };
    for (int r = 0; r < c.R; ++r) {
        if ((L->inactive_mask >> r) & 1u) continue;
        p.src[r] = srcs[r];
        p.src_stride[r] = L->src_row_bytes ? L->src_row_bytes[r] : packed;
        add(srcs[r], p.src_stride[r]);
    }
    for (int d = 0; d < n_dsts; ++d) {
        p.dst[d] = dsts[d];
        p.dst_stride[d] = L->dst_row_bytes ? L->dst_row_bytes[d] : packed;
        add(dsts[d], p.dst_stride[d]);
    }
    if (L->residual) {
        p.residual = L->residual;
        p.res_stride = L->residual_row_bytes;
        add(L->residual, L->residual_row_bytes);
    }
    auto common = [&](uintptr_t M) {
        for (int b = 1; b < nbuf; ++b) {
            if (addr[b] % M != addr[0] % M) return false;
            if (L->ne1 > 1 && stride[b] % M != stride[0] % M) return false;
        }
        return true;
    };
    const bool vec = common(16);
    const tps::Kernels &k = kernels_for(dst_dtype, wire_dtype);
    const bool vec32 = k.ex32[0][0] != nullptr && common(32);
    const tps::ExKernelFn fn =
        vec32 ? k.ex32[c.R > 2][L->residual != nullptr] : k.ex[c.R > 2][L->residual != nullptr][vec];
    const size_t VB = vec32 ? 32 : 16;
    const size_t V = VB / es;
    int threads = 256;
    long long gx;
    if (vec) {
        // threads per row: one per whole vector, plus, when a row can have a
        // head or a tail (fewer than V elements each), enough idle ones for
        // both (the kernel relies on them), with the CTA size that wastes
        // the fewest threads
        const bool ragged =
            L->ne0 % V != 0 || addr[0] % VB != 0 || (L->ne1 > 1 && stride[0] % VB != 0);
        const long long need = static_cast<long long>(L->ne0 / V) + (ragged ? 2 * static_cast<long long>(V) - 2 : 0);
        if (need <= 256) {
            threads = static_cast<int>(need < 32 ? 32 : (need + 31) / 32 * 32);
        } else if (ragged) {
            long long best = 0;
            for (int t = 256; t >= 128; t -= 32) {
                const long long cover = (need + t - 1) / t * t;
                if (best == 0 || cover < best) best = cover, threads = t;
            }
        }
        gx = (need + threads - 1) / threads;
    } else {
        // four elements per thread (the element-wise path's batch)
        gx = (static_cast<long long>(L->ne0) + 4ll * threads - 1) / (4ll * threads);
        if (gx > 1024) gx = 1024;
    }
    if (gx < 1) gx = 1;
    const unsigned gy = L->ne1 < 65535 ? static_cast<unsigned>(L->ne1) : 65535u;
    // the first wave of the vector kernel prefetches its first row's operands
    // into L2 before the wait (in the element-wise kernel, measured, it did
    // not help: R=2 unchanged, R=8 2.7% slower)
    if (c.l2_prefetch && vec) p.prefetch_ctas = first_wave(fn, threads, c.sm_count);
    if (launch_dependent(fn, dim3(static_cast<unsigned>(gx), gy), static_cast<unsigned>(threads), 0, stream, c.pdl != 0,
                         p) != cudaSuccess) {
        cudaGetLastError();
        return AR_ERR_CUDA;
    }
    c.last_variant = vec ? AR_VARIANT_BANDWIDTH : AR_VARIANT_SCALAR;
    return AR_OK;
}

int ar_wire_pack(const void *src, void *wire, size_t nelem, int dst_dtype, int wire_dtype, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ctx.ready) return AR_ERR_NOT_INITIALIZED;
    const Context &c = g_ctx;
    const size_t es = elem_bytes(dst_dtype), ew = elem_bytes(wire_dtype);
    if (!es || !ew) return AR_ERR_UNSUPPORTED;
    if (nelem > c.max_elems) return AR_ERR_TOO_LARGE;
    if (nelem == 0) return AR_OK;
    if (!src || !wire) return AR_ERR_INVALID_ARG;
    const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(wire);
    if (a % es || b % ew) return AR_ERR_INVALID_ARG;
    if (a < b + nelem * ew && b < a + nelem * es && !(a == b && es == ew)) return AR_ERR_OVERLAP;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
    if (dev != c.device) return AR_ERR_INVALID_ARG;
    if (c.fault_inject) return AR_ERR_CUDA;
    const tps::Kernels &k = kernels_for(dst_dtype, wire_dtype);
    // 32-byte source vectors when both buffers allow them, else 16, else
    // element-wise.  A buffer pair off a vector boundary still qualifies when
    // skipping the same few elements (the head) aligns both.
    auto head_for = [&](size_t vb) -> long long {  // -1: this vector size does not fit
        const size_t h = (vb - a % vb) % vb / es;
        const size_t out_bytes = vb / es * ew;  // wire bytes per source vector
        const size_t out_align = vb == 32 || out_bytes > 16 ? out_bytes : 16;
        return (b + h * ew) % out_align == 0 ? static_cast<long long>(h) : -1;
    };
    long long head = k.pack32 != nullptr ? head_for(32) : -1;
    const bool vec32 = head >= 0;
    if (!vec32) head = head_for(16);
    const bool vec = head >= 0;
    const size_t V = (vec32 ? 32 : 16) / es;
    const tps::PackKernelFn fn = vec32 ? k.pack32 : k.pack[vec];
    long long grid;
    if (vec) {
        if (head > static_cast<long long>(nelem)) head = static_cast<long long>(nelem);
        nelem -= static_cast<size_t>(head);
        grid = (static_cast<long long>(nelem / V) + 255) / 256;
    } else {
        head = 0;
        grid = (static_cast<long long>(nelem) + 255) / 256;
        if (grid > c.sm_count * 8ll) grid = c.sm_count * 8ll;
    }
    if (grid < 1) grid = 1;
    const void *s0 = static_cast<const char *>(src) + head * es;
    void *w0 = static_cast<char *>(wire) + head * ew;
    const int prefetch_ctas = (c.l2_prefetch && vec) ? first_wave(fn, 256, c.sm_count) : 0;
    if (launch_dependent(fn, dim3(static_cast<unsigned>(grid)), 256u, 0, stream, g_ctx.pdl != 0, s0, w0,
                         static_cast<unsigned long long>(nelem), static_cast<int>(head), prefetch_ctas) !=
        cudaSuccess) {
        cudaGetLastError();
        return AR_ERR_CUDA;
    }
    g_ctx.last_variant = vec ? AR_VARIANT_BANDWIDTH : AR_VARIANT_SCALAR;
    return AR_OK;
}

}  // extern "C"

// ---- staging without allocation ---------------------------------------------
//
// ar_reduce_host_noalloc stages host partials through this fixed array
// instead of device buffers the caller would have to allocate.  It is part of
// the library image, so every GPU that loads the library holds it (64 MiB)
// until the process exits; it is shared by every call on that GPU.

namespace {

static_assert(AR_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");
static __device__ __align__(256) unsigned char g_noalloc_scratch[AR_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch per device ordinal, looked up by the
// first call on that device after each ar_init (guarded by g_mu).  In host
// code the array's name is only a host-side handle, never an address a kernel
// may use.
constexpr int kMaxScratchDevices = 64;
void *g_noalloc_addr[kMaxScratchDevices] = {};

void forget_noalloc_addresses() {
    for (void *&a : g_noalloc_addr) a = nullptr;
}

}  // namespace

extern "C" {

int ar_reduce_host_noalloc(const void *const *h_srcs, void *const *h_dsts, int n_dsts, size_t nelem, int dst_dtype,
                           int wire_dtype, cudaStream_t stream) {
    // Under the lock: check the call and find the staging area.  The copies
    // are enqueued without the lock, because a copy from or to pageable host
    // memory can block the calling thread until the stream gets there, and
    // other library calls must not wait behind it.
    int R = 0;
    unsigned long long gen = 0;
    size_t bytes = 0, slot = 0;
    char *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_ctx.ready) return AR_ERR_NOT_INITIALIZED;
        const Context &c = g_ctx;
        if (!h_srcs || !h_dsts) return AR_ERR_INVALID_ARG;
        // the rules of ar_reduce, applied to the host buffers: counts, types,
        // NULL pointers, element alignment, partial overlap
        const int st = ar_check_args(c.R, h_srcs, h_dsts, n_dsts, nelem, c.max_elems, dst_dtype, wire_dtype);
        if (st != AR_OK || nelem == 0) return st;
        // every staged buffer starts on a 256-byte boundary of the array
        bytes = nelem * elem_bytes(dst_dtype);
        slot = (bytes + 255) / 256 * 256;
        if (slot < bytes || static_cast<size_t>(c.R + n_dsts) > AR_NOALLOC_SCRATCH_BYTES / slot)
            return AR_ERR_TOO_LARGE;
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
        if (dev != c.device || dev < 0 || dev >= kMaxScratchDevices) return AR_ERR_INVALID_ARG;
        if (!g_noalloc_addr[dev]) {
            // first call on this device since ar_init (the device is current here)
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
                cudaGetLastError();
                return AR_ERR_CUDA;
            }
            g_noalloc_addr[dev] = ptr;
        }
        if (c.fault_inject) return AR_ERR_CUDA;
        base = static_cast<char *>(g_noalloc_addr[dev]);
        R = c.R;
        gen = g_ctx_gen;
    }
    const void *d_srcs[AR_MAX_RANKS];
    void *d_dsts[AR_MAX_DSTS];
    for (int r = 0; r < R; ++r) {
        d_srcs[r] = base + static_cast<size_t>(r) * slot;
        if (cudaMemcpyAsync(const_cast<void *>(d_srcs[r]), h_srcs[r], bytes, cudaMemcpyHostToDevice, stream) !=
            cudaSuccess)
            return AR_ERR_CUDA;
    }
    for (int d = 0; d < n_dsts; ++d) d_dsts[d] = base + static_cast<size_t>(R + d) * slot;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        // ar_init or ar_free on another thread since the checks: the staging
        // area may have moved, so stop before the launch (only the staging
        // area has been written)
        if (!g_ctx.ready || g_ctx_gen != gen) return AR_ERR_NOT_INITIALIZED;
        const int st = launch_locked(d_srcs, d_dsts, n_dsts, nelem, dst_dtype, wire_dtype, AR_VARIANT_AUTO, 0,
                                     stream, false);
        if (st != AR_OK) return st;
    }
    for (int d = 0; d < n_dsts; ++d)
        if (cudaMemcpyAsync(h_dsts[d], d_dsts[d], bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
            return AR_ERR_CUDA;
    return AR_OK;
}

}  // extern "C"
