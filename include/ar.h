/*
 * ar.h -- C ABI of the GB300 partial-sum reduction (libtps_ar.so).
 *
 * The operation is the reduction step of a tensor-parallel AllReduce, done
 * on one GPU: R partial tensors ("ranks") of one activation, each in its own
 * device allocation, are each rounded through a narrower wire type, summed
 * in float in ascending rank order, and the sum is cast back to the tensor
 * type and written to every destination buffer:
 *
 *   for every element i:
 *     acc = float(wire(src[0][i]))
 *     acc = acc + float(wire(src[r][i]))        r = 1 .. R-1, in this order
 *     dst[d][i] = T_dst(acc)                     d = 0 .. n_dsts-1
 *
 * wire(x) and T_dst(x) round to nearest, ties to even, keep subnormals and
 * overflow to infinity; float(x) is exact; the adds are float adds rounded
 * to nearest.  The result is bit-for-bit the same for every variant, grid
 * size and alignment (NaN payloads aside).
 *
 * Where this comes from:
 *   - ggml-cuda allreduce.cu (toy 0.8.0 vendored ggml), ggml_cuda_ar_kernel,
 *     phases 1 and 3, and ggml_cuda_ar_add_kernel: both operands are rounded
 *     through the wire type, widened to float, added in float and the sum is
 *     cast back to the tensor type, so that every rank computes identical
 *     bits; ggml_cuda_ar_allreduce picks the wire type (bf16 for f32 tensors)
 *     and the strategy by tensor size.
 *   - ggml-hexagon htp/allreduce-ops.c (char-fork/llama.cpp),
 *     DEFINE_ALLREDUCE_THREAD_DMA_1D: the ranks are folded left to right and
 *     the result is written to each of n_dsts destinations; validate_allreduce
 *     and op_allreduce return status codes instead of asserting.
 *   - The float accumulator for R > 2, the start from rank 0's operand (not
 *     from zero) and the rounding rules are this library's readings where the
 *     pages are silent.
 *
 * Conventions for every call below:
 *   - Device pointers are CUDA addresses the device that was current at
 *     ar_init can access: device memory, or pinned/managed host memory
 *     (which the kernel then reads or writes over the CPU-GPU link); host
 *     pointers are ordinary (ideally pinned) host memory.  The caller owns
 *     every buffer and the stream; the library keeps no pointer after a call
 *     returns and allocates nothing per call.
 *   - Calls that take a stream only enqueue work on it and return; results
 *     are ready when the stream reaches that point.  No call synchronizes
 *     (a host call given pageable memory waits for CUDA's synchronous
 *     pageable copies, see ar_reduce_host and ar_reduce_host_noalloc), so ar_reduce and
 *     ar_reduce_variant can be captured in a CUDA graph.
 *   - On any status other than AR_OK nothing has been enqueued or written,
 *     except AR_ERR_CUDA from a launch, after which the stream's state is
 *     whatever CUDA reports.
 *   - All calls are thread-safe; they share one process-wide context.
 */
#ifndef TPS_AR_H
#define TPS_AR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle (identical to its own typedef). */
typedef struct CUstream_st *cudaStream_t;

/* Element types.  Sources and destinations hold T_dst; T_wire is the type
 * every operand is rounded through before the float sum. */
typedef enum { AR_F32 = 0, AR_F16 = 1, AR_BF16 = 2 } ar_dtype;

typedef enum {
    AR_OK = 0,
    AR_ERR_INVALID_ARG = 1,     /* bad count, NULL pointer, wrong device, ... */
    AR_ERR_UNSUPPORTED = 2,     /* unknown dtype, or the GPU cannot run the kernels */
    AR_ERR_TOO_LARGE = 3,       /* nelem > max_elems given to ar_init */
    AR_ERR_NOT_INITIALIZED = 4, /* ar_init has not succeeded */
    AR_ERR_OVERLAP = 5,         /* a destination partly overlaps another buffer */
    AR_ERR_CUDA = 6             /* a CUDA call failed */
} ar_status;

/* Limits: at most 16 ranks and 16 destinations per call (the pages cap
 * their rank arrays at compile-time maxima of this order:
 * GGML_CUDA_MAX_DEVICES in allreduce.cu, HTP_ALLREDUCE_MAX_RANKS in
 * allreduce-ops.c). */
#define AR_MAX_RANKS 16
#define AR_MAX_DSTS 16

/* Kernel variants.  AUTO picks LATENCY or BANDWIDTH by the call's byte
 * count.  The vector variants want every source and destination at the same
 * offset from a 16-byte boundary (32 for BANDWIDTH's wide f32 vectors, else
 * 16): they then shift past the few elements before the boundary, which they
 * reduce one by one.  When the offsets differ AUTO takes SCALAR.  Every
 * variant computes the same bits. */
typedef enum {
    AR_VARIANT_AUTO = 0,
    AR_VARIANT_NAIVE = 1,     /* one element per thread, grid-stride: a cross-check */
    AR_VARIANT_LATENCY = 2,   /* one 16-byte vector per thread, 128-thread CTAs */
    AR_VARIANT_BANDWIDTH = 3, /* one 32-byte (f32) or 16-byte vector per thread, 256-thread
                                 CTAs; all loads of two or four ranks issued together */
    AR_VARIANT_SCALAR = 4,    /* element-wise path used when the buffers' offsets differ */
    AR_VARIANT_TMA = 5        /* shared-memory staging: a producer warp bulk-copies (cp.async.bulk)
                                 R source tiles per stage, sixteen warps fold them, one thread
                                 bulk-stores the result tile to every destination; two CTAs per SM.
                                 Needs 16-byte aligned buffers.  Never chosen by AUTO (an
                                 AR_VARIANT environment override with offset buffers takes
                                 BANDWIDTH, or SCALAR when the offsets differ).  Its internal waits are bounded: a wait
                                 that runs out sets bit 0 of AR_Q_DEVICE_STATUS and the call's
                                 results are then unspecified (the call still ends). */
} ar_variant;

/*
 * ar_init -- create the process-wide context on the current CUDA device.
 *   R          number of ranks (partials) every ar_reduce call sums, 1..16.
 *   max_elems  largest nelem any later call may pass (>= 1).
 * Reads the environment once: AR_VARIANT (auto|naive|latency|bandwidth|
 * scalar|tma), AR_LATENCY_MAX_BYTES (size switch, bytes of sources plus
 * destinations), AR_TMA_STAGES (2..8, default 3), AR_TMA_TILE (largest
 * tile in bytes, a multiple of 1024 up to 32768, default 16384),
 * AR_TMA_CTAS_PER_SM (1..4, default 2), AR_PDL (1 = default: on a created
 * stream, every kernel but NAIVE's launches as a programmatic dependent of
 * the kernel before it on the stream, which it waits for before touching
 * memory; launches on the default streams stay plain; 0 = plain launches
 * everywhere), AR_L2_PREFETCH (1 = default: the first wave of CTAs of the
 * LATENCY and BANDWIDTH kernels asks L2 for its source vectors before that
 * wait, so they load while the kernel ahead drains; 0 = off; results are the
 * same either way), AR_LOG=1 (one line per init to stderr).
 * Calling it again replaces the context.  Returns AR_OK, AR_ERR_INVALID_ARG,
 * AR_ERR_UNSUPPORTED (the device is not sm_103) or AR_ERR_CUDA (no device).
 */
int ar_init(int R, size_t max_elems);

/*
 * ar_reduce -- enqueue one reduction on `stream`.
 *   srcs       host array of R device pointers, each to nelem elements of
 *              dst_dtype (contiguous); read only.
 *   dsts       host array of n_dsts device pointers, each to nelem elements
 *              of dst_dtype; all receive the same bits.  A destination may
 *              be exactly one of the sources (in-place reduction) but may
 *              not partly overlap any source or other destination.
 *   n_dsts     1..16.
 *   nelem      elements per buffer, <= max_elems; 0 is a no-op (AR_OK).
 *   dst_dtype  ar_dtype of sources and destinations.
 *   wire_dtype ar_dtype every operand is rounded through (any of the three).
 *   stream     CUDA stream of the init device (0 = legacy default stream).
 * Any element-aligned pointer works; buffers that all share one offset from
 * a 16-byte boundary take the vector paths.  Returns an ar_status.
 */
int ar_reduce(const void *const *srcs, void *const *dsts, int n_dsts, size_t nelem,
              int dst_dtype, int wire_dtype, cudaStream_t stream);

/* ar_free -- drop the context.  Safe to call when not initialized. */
void ar_free(void);

/* Static English text for a status code (never NULL). */
const char *ar_status_string(int status);

/*
 * ar_check_args -- the host-side validation ar_reduce runs before any CUDA
 * call, on explicit R and max_elems instead of the context's.  Makes no CUDA
 * call and touches no device memory, so it runs without a GPU.
 */
int ar_check_args(int R, const void *const *srcs, void *const *dsts, int n_dsts,
                  size_t nelem, size_t max_elems, int dst_dtype, int wire_dtype);

/*
 * ar_reduce_variant -- ar_reduce with the kernel variant forced.
 *   variant     an ar_variant; AUTO behaves exactly like ar_reduce.
 *   grid_blocks CTAs to launch for BANDWIDTH/NAIVE/SCALAR (0 = the library's
 *               choice); ignored by LATENCY, whose grid covers the tensor.
 *               A BANDWIDTH grid smaller than the tensor needs is persistent:
 *               its CTAs sweep the tensors together in rounds.
 * The result bits do not depend on either argument.  LATENCY or BANDWIDTH
 * asked for with buffers at different offsets from a 16-byte boundary, or
 * TMA with any buffer off that boundary, returns AR_ERR_INVALID_ARG.
 */
int ar_reduce_variant(const void *const *srcs, void *const *dsts, int n_dsts, size_t nelem,
                      int dst_dtype, int wire_dtype, int variant, int grid_blocks,
                      cudaStream_t stream);

/* Keys for ar_query / ar_set_option. */
typedef enum {
    AR_Q_RANKS = 0,             /* R fixed at ar_init (query only) */
    AR_Q_MAX_ELEMS = 1,         /* max_elems (query only) */
    AR_Q_DEVICE = 2,            /* CUDA device ordinal (query only) */
    AR_Q_SM_COUNT = 3,          /* SMs on that device (query only) */
    AR_Q_LATENCY_MAX_BYTES = 4, /* AUTO uses LATENCY below this many bytes */
    AR_Q_FORCED_VARIANT = 5,    /* variant AUTO resolves to when nonzero */
    AR_Q_LAST_VARIANT = 6,      /* variant the last successful launch used (query only); after
                                   ar_reduce_ex or ar_wire_pack: BANDWIDTH for their vector
                                   kernel, SCALAR for their element-wise one */
    AR_Q_FAULT_INJECT = 7,      /* nonzero: the next launches fail with AR_ERR_CUDA
                                   before anything is enqueued (host-side test hook) */
    AR_Q_BW_BLOCKS_PER_SM = 8,  /* 0: the BANDWIDTH grid covers the tensor (default); n > 0: a
                                   persistent grid of n CTAs per SM (capped by occupancy) */
    AR_Q_HOST_CHUNK_BYTES = 9,  /* ar_reduce_host pipeline chunk, bytes per buffer (default 4 MiB;
                                   at most 64 chunks per call) */
    AR_Q_DEVICE_STATUS = 10,    /* device-side status word (bit 0: a bounded wait of the TMA
                                   variant ran out); reading it synchronises with the device;
                                   set it to 0 to clear it */
    AR_Q_TMA_DROP_TILE = 11     /* test hook for failure detection, -1 (default) = off: TMA
                                   launches never load tile n, so the CTA that owns it waits
                                   for data that never comes until its bound (100 ms) runs out,
                                   reports through AR_Q_DEVICE_STATUS and returns; the results of
                                   such a launch are unspecified and the context stays usable */
} ar_key;

/* Read one context value into *value.  AR_ERR_NOT_INITIALIZED before init. */
int ar_query(int key, int64_t *value);

/* Change one settable context value.  Not to be called while a stream
 * capture that uses the library is in progress. */
int ar_set_option(int key, int64_t value);

/*
 * ar_reduce_host -- the same reduction for callers whose partials live in
 * host memory; the results are written back to host memory.
 *   h_srcs, h_dsts  R and n_dsts host pointers, nelem elements each.
 * Two ways to move the data, chosen by the staging arguments:
 *   d_srcs, d_dsts  R and n_dsts device buffers of nelem elements: each host
 *                   source is copied into its staging buffer, the reduction
 *                   writes the staging destinations, and those are copied
 *                   back to the host.  The work is cut into chunks (see
 *                   AR_Q_HOST_CHUNK_BYTES) and pipelined over three streams
 *                   the context owns, so copies in, kernels and copies out of
 *                   different chunks overlap.  Pinned host memory makes the
 *                   copies asynchronous; pageable memory also works, but CUDA
 *                   copies it synchronously, so the call then waits for its
 *                   copies.  It waits without holding the library lock:
 *                   other threads' calls go on, except another staged
 *                   ar_reduce_host (the pipeline is one per context) and
 *                   ar_init / ar_free, which wait for this call to end.
 *   both NULL       no staging: the kernel itself loads the host partials and
 *                   stores the host results over the CPU-GPU link (NVLink-C2C
 *                   on GB300), with no copies at all.  Every host buffer must
 *                   be memory the GPU can reach (cudaHostAlloc /
 *                   cudaHostRegister pinned memory, or managed memory);
 *                   otherwise AR_ERR_INVALID_ARG.
 * Everything else as for ar_reduce, and the host buffers obey ar_reduce's
 * buffer rules too: element-aligned, and a host destination may be exactly
 * a host source but may not partly overlap any host source or other host
 * destination (AR_ERR_OVERLAP, nothing enqueued).  Either way the work
 * starts after what is already enqueued on `stream`, and `stream` reaches
 * the end of this call only when the host results are complete.  Results
 * are identical to one ar_reduce over device copies of the same tensors.
 */
int ar_reduce_host(const void *const *h_srcs, void *const *h_dsts, int n_dsts, size_t nelem,
                   int dst_dtype, int wire_dtype, void *const *d_srcs, void *const *d_dsts,
                   cudaStream_t stream);

/*
 * Layout of an extended reduction (ar_reduce_ex): a 2-D tensor of ne1 rows
 * of ne0 elements with per-buffer row strides, ranks that may be inactive,
 * and an optional residual or bias added after the rank fold.
 *
 * Where this comes from:
 *   - row strides: the 2-D DMA variant DEFINE_ALLREDUCE_THREAD_DMA_2D of
 *     ggml-hexagon htp/allreduce-ops.c walks every source and destination
 *     row by row through its nb[1] byte stride;
 *   - residual and bias: the ALLREDUCE_ADD variants of the same file add one
 *     more tensor after the ranks (add_bcast adds one row to every row);
 *   - inactive ranks: ggml_cuda_ar_allreduce in ggml-cuda allreduce.cu zeroes
 *     the data of shards that did not compute, so they contribute zeros.
 * Readings taken where the pages are silent: the residual is added in float
 * after the rank fold and before the one final cast, and is not rounded
 * through the wire type (it never crosses the wire); an inactive rank
 * contributes +0 to every element, which is not the same as leaving it out
 * (-0 + +0 = +0).
 */
typedef struct {
    size_t ne0;                   /* elements per row */
    size_t ne1;                   /* rows; ne0 * ne1 <= max_elems */
    const int64_t *src_row_bytes; /* R row strides in bytes (>= ne0 * element size, a multiple of
                                     the element size), or NULL: every source's rows are packed */
    const int64_t *dst_row_bytes; /* n_dsts row strides in bytes, or NULL: packed */
    const void *residual;         /* NULL, or a T_dst tensor added after the rank fold */
    int64_t residual_row_bytes;   /* residual row stride in bytes; 0: the residual is one row of
                                     ne0 elements added to every row (a bias) */
    uint32_t inactive_mask;       /* bit r set: rank r contributes +0 everywhere and srcs[r] is not
                                     read (it may be NULL); bits >= R must be clear */
} ar_layout;

/*
 * ar_reduce_ex -- the reduction over an ar_layout, enqueued on `stream`:
 *   dst[d][row][i] = T_dst( fold_r wire(src[r][row][i]) (+ residual[row][i]) )
 * with the fold, casts and rounding of ar_reduce.  srcs has R entries (NULL
 * allowed for inactive ranks), dsts has n_dsts.  A destination may be
 * exactly a source or exactly the residual (same pointer and same row
 * stride: an in-place update such as x = x + allreduce(partials)); any other
 * overlap of the buffers' row spans is AR_ERR_OVERLAP (the check is
 * conservative: interleaved rows that never touch are also refused).
 * When every buffer's start agrees modulo 16 bytes, and (with more than one
 * row) so does every row stride, every row of every buffer starts at one
 * common offset from a 16-byte boundary: the vector path runs, reducing each
 * row's few elements before that boundary one by one.  Any other
 * element-aligned layout works element by element with the same bits.
 * Statuses as for ar_reduce; nothing is enqueued unless AR_OK.
 */
int ar_reduce_ex(const void *const *srcs, void *const *dsts, int n_dsts, const ar_layout *layout,
                 int dst_dtype, int wire_dtype, cudaStream_t stream);

/* Host-only validation of an ar_reduce_ex call on explicit R and max_elems
 * (no CUDA call; runs without a GPU). */
int ar_check_layout(int R, const void *const *srcs, void *const *dsts, int n_dsts, const ar_layout *layout,
                    size_t max_elems, int dst_dtype, int wire_dtype);

/*
 * ar_wire_pack -- materialise the wire copy of one partial:
 *   wire[i] = T_wire(src[i]) for i < nelem,
 * the buffer a transport sends to the other ranks (phase 1 of
 * ggml_cuda_ar_kernel in ggml-cuda allreduce.cu writes exactly this; its
 * copy-engine path converts to bf16 into a temporary before copying).
 *   src   nelem elements of dst_dtype (device-accessible).
 *   wire  nelem elements of wire_dtype; may be src itself when both types
 *         have the same size, otherwise must not overlap it.
 * Vector kernel when skipping the same first few elements aligns both
 * buffers (they are then converted one by one), element-wise otherwise; the
 * bits are the same.  Needs ar_init (nelem <= max_elems).  Statuses as for
 * ar_reduce.
 */
int ar_wire_pack(const void *src, void *wire, size_t nelem, int dst_dtype, int wire_dtype,
                 cudaStream_t stream);

/*
 * ar_reduce_host_noalloc -- ar_reduce_host for callers that cannot allocate
 * device memory.  (The pages have no counterpart: this entry point exists
 * for callers of this library, not because of the method.)
 *
 * Who needs it: code that may not call cudaMalloc -- for example a plug-in
 * running inside a framework whose caching allocator owns the whole device
 * memory budget, or a latency-critical path that cannot afford cudaMalloc /
 * cudaFree and the device-wide synchronisation they can cause.  Such
 * callers cannot provide the device staging buffers ar_reduce_host wants.
 *
 * What it does: copies each host source into a fixed staging area built into
 * the library, reduces there, and copies every destination back to its host
 * buffer, all enqueued on `stream` (results are valid once `stream` reaches
 * the end of this call).  It allocates nothing: no cudaMalloc, no cudaFree,
 * no allocating library routine.  Same arguments, buffer rules (partial
 * overlap of host buffers is AR_ERR_OVERLAP) and results as ar_reduce_host
 * with NULL staging arrays, except that the host buffers may be ordinary
 * pageable memory.  CUDA copies pageable memory synchronously, so with
 * pageable buffers the call itself waits until `stream` has reached its
 * copies; it holds no library lock while it waits, so other threads' calls
 * go on.
 *
 * Limits and rules:
 *   - The staging area is AR_NOALLOC_SCRATCH_BYTES (64 MiB) of device
 *     memory that every GPU which loads the library holds until the process
 *     exits.  A call needs R + n_dsts buffers of nelem elements, each rounded
 *     up to 256 bytes; a call that needs more returns AR_ERR_TOO_LARGE and
 *     does nothing.
 *   - The first call on a device after each ar_init looks up the staging
 *     area's device address (once, with that device current); make that
 *     first call before any stream capture.  ar_init and ar_free forget the
 *     address, so a context created after cudaDeviceReset finds the area
 *     where the new device context holds it.  If another thread runs
 *     ar_init or ar_free while a call is under way, the call may return
 *     AR_ERR_NOT_INITIALIZED after its copies into the staging area were
 *     enqueued (the caller's buffers are then not written).
 *   - Every call on a GPU uses the same staging area, and each call leaves
 *     its data there: nothing in it has to start at zero, because every call
 *     writes its inputs before reading them.  Calls whose work overlaps on
 *     the GPU (two streams, or two threads) race on the staging area and may
 *     produce wrong results: serialise them, e.g. on one stream.
 */
#define AR_NOALLOC_SCRATCH_BYTES (64u << 20)
int ar_reduce_host_noalloc(const void *const *h_srcs, void *const *h_dsts, int n_dsts, size_t nelem,
                           int dst_dtype, int wire_dtype, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TPS_AR_H */
