/*
 * Scalar CPU oracle for the tensor-parallel partial-sum reduction.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this code: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA library; the two meet only in the seeded input
 * generators, which hold none of the arithmetic below.
 *
 * What it computes (per element i, one element at a time, in this order):
 *
 *     acc  = widen( round<T_wire>( value(src[0][i]) ) )
 *     acc  = acc + widen( round<T_wire>( value(src[r][i]) ) )   r = 1 .. R-1
 *     y    = round<T_dst>( acc )
 *     dst[d][i] = y                                             d = 0 .. n_dsts-1
 *
 * Sources:
 *   - ggml-cuda allreduce.cu (toy 0.8.0 vendored ggml), ggml_cuda_ar_kernel,
 *     "Phase 3": the local operand is rounded through the wire type exactly
 *     like the peer's, both are widened to float, added in float and the sum
 *     is cast back to the destination type; ggml_cuda_ar_add_kernel applies
 *     the same formula.
 *   - ggml-hexagon htp/allreduce-ops.c (char-fork/llama.cpp),
 *     DEFINE_ALLREDUCE_THREAD_DMA_1D: ranks are folded left to right
 *     (s0 + s1, then + s2, ...) and the one result is written to every
 *     destination buffer.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - the accumulator is float for the whole fold, with one final cast;
 *   - the fold starts from the first operand, not from zero (this keeps -0);
 *   - every narrowing cast is IEEE-754 round-to-nearest, ties-to-even, with
 *     gradual underflow and overflow to infinity; float adds round to nearest;
 *   - a NaN stays a NaN (its payload is not specified).
 *
 * Pins (tests that tie this code to something other than itself): the casts
 * are checked exhaustively against library conversions (numpy float16,
 * torch bfloat16) and against a brute-force nearest-value search over every
 * value of the target format; the widen is checked exhaustively against
 * library decoders; the fold is checked against closed forms (R = 1 wire
 * round-trip, R = 2 symmetry, exact small-integer sums, an order-sensitive
 * constructed case) and against a per-step-rounded exact rational fold.
 */
#ifndef TPS_ORACLE_H
#define TPS_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types, numbered like the library's public enum but defined here on
 * their own so that the oracle includes nothing from the product. */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* Size in bytes of one stored element, or 0 for an unknown type. */
size_t orc_elem_size(int dtype);

/* Exact value of one stored element (bit pattern in the low bits). */
float orc_widen(int dtype, uint32_t bits);

/* Bit pattern of x rounded to nearest, ties to even, in the given type. */
uint32_t orc_round(int dtype, float x);

/* Array forms of the two casts above (n elements). */
void orc_widen_array(int dtype, const void *in, float *out, size_t n);
void orc_round_array(int dtype, const float *in, void *out, size_t n);

/* The reduction over elements [begin, end) of R source arrays of T_dst,
 * writing the same result into each of n_dsts destination arrays.
 * Returns 0, or -1 for an unknown type or a bad count. */
int orc_reduce_range(int R, const void *const *srcs, void *const *dsts, int n_dsts,
                     size_t begin, size_t end, int dst_dtype, int wire_dtype);

/* The reduction over all nelem elements. */
int orc_reduce(int R, const void *const *srcs, void *const *dsts, int n_dsts,
               size_t nelem, int dst_dtype, int wire_dtype);

/*
 * The reduction over a 2-D tensor of ne1 rows of ne0 elements, with the
 * three extensions the pages describe around the same fold:
 *   - row strides in bytes for every source and destination (NULL: rows
 *     packed), as the 2-D DMA variant of ggml-hexagon allreduce-ops.c
 *     (DEFINE_ALLREDUCE_THREAD_DMA_2D) walks rows through nb[1];
 *   - inactive ranks: bit r of inactive_mask set means rank r contributes
 *     +0 for every element (its source may be NULL), as
 *     ggml_cuda_ar_allreduce in ggml-cuda allreduce.cu zeroes the data of
 *     shards without the compute flag before reducing;
 *   - a residual in T_dst added after the rank fold and before the final
 *     cast (the ALLREDUCE_ADD variants of allreduce-ops.c add the residual
 *     after the ranks); residual_stride is its row stride in bytes, 0 means
 *     one row broadcast to every row (the row-broadcast "add_bcast"
 *     variant).  The residual does not cross the wire, so it is not rounded
 *     through the wire type; it is added in float.
 * Per element (row j, column i):
 *     acc = w_0; acc = acc + w_r for r = 1..R-1   (w_r = +0 for an inactive rank)
 *     if residual: acc = acc + value(residual[j][i])
 *     dst[d][j][i] = round<T_dst>(acc)
 */
int orc_reduce_2d(int R, const void *const *srcs, const long long *src_strides, unsigned inactive_mask,
                  const void *residual, long long residual_stride, void *const *dsts,
                  const long long *dst_strides, int n_dsts, size_t ne0, size_t ne1, int dst_dtype,
                  int wire_dtype);

/*
 * The wire cast materialised: wire[i] = round<T_wire>(value(src[i])), the
 * buffer phase 1 of ggml_cuda_ar_kernel (ggml-cuda allreduce.cu) writes
 * before sending it to the peer.
 */
int orc_wire_pack(const void *src, void *wire, size_t nelem, int dst_dtype, int wire_dtype);

#ifdef __cplusplus
}
#endif

#endif /* TPS_ORACLE_H */
