/*
 * Scalar CPU oracle for the tensor-parallel partial-sum reduction.
 * TEST INFRASTRUCTURE ONLY -- see oracle.h for what it computes, the
 * passages it follows, the readings it takes and what pins it.
 *
 * Build: plain C11, -O2 -ffp-contract=off, no fast-math.  Every float
 * operation here is a single IEEE-754 binary32 or binary64 operation.
 */
#include "oracle.h"

#include <float.h>
#include <math.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float arithmetic evaluated in float (FLT_EVAL_METHOD == 0)"
#endif

/*
 * A binary floating-point format narrower than float, described the way
 * IEEE-754 describes binary16 (and bfloat16 by the same rules):
 *   p     precision in bits, the implicit leading bit included
 *   emin  exponent of the smallest normal number
 *   emax  exponent of the largest finite number (also the exponent bias)
 *   ebits width of the stored exponent field
 * The stored fraction field is p - 1 bits wide.
 */
typedef struct {
    int p;
    int emin;
    int emax;
    int ebits;
} orc_format;

/* IEEE-754 binary16: 11-bit precision, normal exponents -14 .. 15. */
static const orc_format FMT_F16 = {11, -14, 15, 5};
/* bfloat16: float's exponent range (-126 .. 127) with 8-bit precision. */
static const orc_format FMT_BF16 = {8, -126, 127, 8};

static const orc_format *format_of(int dtype) {
    if (dtype == ORC_F16) return &FMT_F16;
    if (dtype == ORC_BF16) return &FMT_BF16;
    return NULL;
}

size_t orc_elem_size(int dtype) {
    switch (dtype) {
        case ORC_F32: return 4;
        case ORC_F16: return 2;
        case ORC_BF16: return 2;
        default: return 0;
    }
}

/* Value of a stored element of a narrow format, from its three fields. */
static double decode(const orc_format *f, uint32_t bits) {
    const int mbits = f->p - 1;
    const uint32_t fraction = bits & ((1u << mbits) - 1u);
    const uint32_t expfield = (bits >> mbits) & ((1u << f->ebits) - 1u);
    const int negative = (int)((bits >> (mbits + f->ebits)) & 1u);
    double v;
    if (expfield == (1u << f->ebits) - 1u) {
        v = fraction ? (double)NAN : (double)INFINITY;
    } else if (expfield == 0) {
        /* subnormal (or zero): fraction * 2^(emin - (p-1)) */
        v = ldexp((double)fraction, f->emin - mbits);
    } else {
        /* normal: (2^(p-1) + fraction) * 2^(E - bias - (p-1)) */
        v = ldexp((double)(fraction + (1u << mbits)), (int)expfield - f->emax - mbits);
    }
    return negative ? -v : v;
}

/*
 * x rounded to the nearest value of format f, ties to the value whose
 * significand is even; magnitudes that round to 2^(emax+1) or beyond become
 * infinity; below 2^emin the grid spacing stays 2^(emin-(p-1)) (gradual
 * underflow).  Returns the stored bit pattern.
 */
static uint32_t round_to(const orc_format *f, float x) {
    const int mbits = f->p - 1;
    const uint32_t sign = signbit(x) ? (1u << (mbits + f->ebits)) : 0u;
    const uint32_t exp_all_ones = ((1u << f->ebits) - 1u) << mbits;

    if (isnan(x)) return sign | exp_all_ones | (1u << (mbits - 1)); /* quiet NaN */
    if (isinf(x)) return sign | exp_all_ones;

    const double a = fabs((double)x); /* exact */
    if (a == 0.0) return sign;

    /* a lies in [2^e, 2^(e+1)); below the normal range the spacing is fixed. */
    int k;
    (void)frexp(a, &k); /* a = m * 2^k with m in [0.5, 1) */
    int e = k - 1;
    if (e < f->emin) e = f->emin;
    const double spacing = ldexp(1.0, e - mbits);

    /* a / spacing is exact: a has at most 24 significant bits. */
    const double n = a / spacing;
    const double below = floor(n);
    const double frac = n - below;
    double r;
    if (frac > 0.5) {
        r = below + 1.0;
    } else if (frac < 0.5) {
        r = below;
    } else {
        r = (fmod(below, 2.0) == 0.0) ? below : below + 1.0;
    }
    const double y = r * spacing; /* exact */

    if (y >= ldexp(1.0, f->emax + 1)) return sign | exp_all_ones; /* overflow */
    if (y == 0.0) return sign;

    int ky;
    (void)frexp(y, &ky);
    const int ey = ky - 1;
    if (ey < f->emin) {
        /* subnormal: the stored fraction is y / 2^(emin - (p-1)) */
        const uint32_t fraction = (uint32_t)(y / ldexp(1.0, f->emin - mbits));
        return sign | fraction;
    }
    const uint32_t significand = (uint32_t)(y / ldexp(1.0, ey - mbits));
    const uint32_t fraction = significand - (1u << mbits);
    const uint32_t expfield = (uint32_t)(ey + f->emax);
    return sign | (expfield << mbits) | fraction;
}

float orc_widen(int dtype, uint32_t bits) {
    if (dtype == ORC_F32) {
        float v;
        memcpy(&v, &bits, sizeof v);
        return v;
    }
    const orc_format *f = format_of(dtype);
    if (!f) return NAN;
    /* every value of a narrower format is a float, so this cast is exact */
    return (float)decode(f, bits);
}

uint32_t orc_round(int dtype, float x) {
    if (dtype == ORC_F32) {
        uint32_t bits;
        memcpy(&bits, &x, sizeof bits);
        return bits;
    }
    const orc_format *f = format_of(dtype);
    if (!f) return 0;
    return round_to(f, x);
}

static uint32_t load_bits(int dtype, const void *base, size_t i) {
    if (dtype == ORC_F32) {
        uint32_t b;
        memcpy(&b, (const char *)base + 4 * i, 4);
        return b;
    }
    uint16_t h;
    memcpy(&h, (const char *)base + 2 * i, 2);
    return h;
}

static void store_bits(int dtype, void *base, size_t i, uint32_t bits) {
    if (dtype == ORC_F32) {
        memcpy((char *)base + 4 * i, &bits, 4);
    } else {
        const uint16_t h = (uint16_t)bits;
        memcpy((char *)base + 2 * i, &h, 2);
    }
}

void orc_widen_array(int dtype, const void *in, float *out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_widen(dtype, load_bits(dtype, in, i));
}

void orc_round_array(int dtype, const float *in, void *out, size_t n) {
    for (size_t i = 0; i < n; ++i) store_bits(dtype, out, i, orc_round(dtype, in[i]));
}

/* One operand as it enters the sum: its exact value rounded once to the wire
 * type, then widened back to float (exact). */
static float wire_operand(int dst_dtype, int wire_dtype, const void *src, size_t i) {
    const float value = orc_widen(dst_dtype, load_bits(dst_dtype, src, i));
    return orc_widen(wire_dtype, orc_round(wire_dtype, value));
}

int orc_reduce_range(int R, const void *const *srcs, void *const *dsts, int n_dsts,
                     size_t begin, size_t end, int dst_dtype, int wire_dtype) {
    if (R < 1 || n_dsts < 1 || !srcs || !dsts) return -1;
    if (!orc_elem_size(dst_dtype) || !orc_elem_size(wire_dtype)) return -1;
    for (int r = 0; r < R; ++r)
        if (!srcs[r]) return -1;
    for (int d = 0; d < n_dsts; ++d)
        if (!dsts[d]) return -1;

    for (size_t i = begin; i < end; ++i) {
        /* the fold starts from rank 0's operand and adds ranks in order */
        float acc = wire_operand(dst_dtype, wire_dtype, srcs[0], i);
        for (int r = 1; r < R; ++r) {
            acc = acc + wire_operand(dst_dtype, wire_dtype, srcs[r], i);
        }
        const uint32_t y = orc_round(dst_dtype, acc);
        for (int d = 0; d < n_dsts; ++d) store_bits(dst_dtype, dsts[d], i, y);
    }
    return 0;
}

int orc_reduce(int R, const void *const *srcs, void *const *dsts, int n_dsts,
               size_t nelem, int dst_dtype, int wire_dtype) {
    return orc_reduce_range(R, srcs, dsts, n_dsts, 0, nelem, dst_dtype, wire_dtype);
}

/* Element i of a row that starts at byte offset row_off of base. */
static uint32_t load_bits_at(int dtype, const void *base, long long row_off, size_t i) {
    return load_bits(dtype, (const char *)base + row_off, i);
}

int orc_reduce_2d(int R, const void *const *srcs, const long long *src_strides, unsigned inactive_mask,
                  const void *residual, long long residual_stride, void *const *dsts,
                  const long long *dst_strides, int n_dsts, size_t ne0, size_t ne1, int dst_dtype,
                  int wire_dtype) {
    const size_t es = orc_elem_size(dst_dtype);
    if (R < 1 || R > 32 || n_dsts < 1 || !srcs || !dsts) return -1;
    if (!es || !orc_elem_size(wire_dtype)) return -1;
    for (int r = 0; r < R; ++r)
        if (!srcs[r] && !((inactive_mask >> r) & 1u)) return -1;
    for (int d = 0; d < n_dsts; ++d)
        if (!dsts[d]) return -1;
    const long long packed = (long long)(ne0 * es);

    for (size_t j = 0; j < ne1; ++j) {
        for (size_t i = 0; i < ne0; ++i) {
            float acc = 0.0f;
            for (int r = 0; r < R; ++r) {
                float w;
                if ((inactive_mask >> r) & 1u) {
                    /* an inactive rank's data are zeros: its operand is +0 */
                    w = orc_widen(wire_dtype, orc_round(wire_dtype, 0.0f));
                } else {
                    const long long stride = src_strides ? src_strides[r] : packed;
                    const float v = orc_widen(dst_dtype, load_bits_at(dst_dtype, srcs[r], (long long)j * stride, i));
                    w = orc_widen(wire_dtype, orc_round(wire_dtype, v));
                }
                acc = (r == 0) ? w : acc + w;
            }
            if (residual) {
                const long long off = (long long)j * residual_stride;
                acc = acc + orc_widen(dst_dtype, load_bits_at(dst_dtype, residual, off, i));
            }
            const uint32_t y = orc_round(dst_dtype, acc);
            for (int d = 0; d < n_dsts; ++d) {
                const long long stride = dst_strides ? dst_strides[d] : packed;
                store_bits(dst_dtype, (char *)dsts[d] + (long long)j * stride, i, y);
            }
        }
    }
    return 0;
}

int orc_wire_pack(const void *src, void *wire, size_t nelem, int dst_dtype, int wire_dtype) {
    if (!src || !wire || !orc_elem_size(dst_dtype) || !orc_elem_size(wire_dtype)) return -1;
    for (size_t i = 0; i < nelem; ++i) {
        const float v = orc_widen(dst_dtype, load_bits(dst_dtype, src, i));
        store_bits(wire_dtype, wire, i, orc_round(wire_dtype, v));
    }
    return 0;
}
