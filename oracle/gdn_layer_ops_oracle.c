/*
 * gdn_layer_ops_oracle.c -- plain sequential CPU oracle for the two steps either
 * side of the GDN recurrence that "The inference stack behind OCRia" (LlamaIndex
 * engineering blog, section "Avoiding unnecessary memory transfers") names among
 * its fused kernels: the causal convolution of the GDN layers, and the gated
 * RMSNorm followed by FP8 quantisation.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite and the smoke check load this
 * code.  It shares no code, header or table with the CUDA library it checks.
 *
 * 1. Causal convolution with pointer rollback.  The pages give no formula; the
 *    reading taken is the short depthwise causal convolution of the GDN layer
 *    ("Gated Delta Networks", ICLR 2025, which puts one before q, k and v): for
 *    channel c with kernel width W,
 *        y_t[c] = act( bias[c] + sum_{j=0}^{W-1} w[c][j] * x_{t-(W-1)+j}[c] ),
 *    act = identity or SiLU.  Under speculation the inputs x_{-(W-1)} .. x_{-1}
 *    are the last W-1 committed inputs and x_0 .. x_{T-1} the draft block.  The
 *    committed inputs live in a ring of `cap` positions per sequence with a
 *    write position `pos`; verify reads the window before `pos`, emits the T
 *    outputs and stages the draft at positions pos .. pos+T-1 (mod cap), and
 *    accepting p tokens only advances pos by p -- the ReplaySSM treatment
 *    ("Making speculative verification cheaper": rollback moves a pointer, the
 *    accepted prefix is kept) applied to the convolution window.
 *
 * 2. Gated RMSNorm + FP8 (E4M3) quantisation, per row o of d values with gate z:
 *        r = 1 / sqrt(mean(o^2) + eps),  y_i = o_i r w_i silu(z_i),
 *        code_i = E4M3(y_i * inv_scale)
 *    with round-to-nearest-even and saturation to +-448.  The E4M3 format
 *    (1 sign bit, 4 exponent bits, 3 mantissa bits) is the one "Inference
 *    Engineering", chapter 5 (quantisation, number formats) describes; its
 *    exponent bias 7, subnormals and the single NaN encoding per sign are those
 *    of the OCP 8-bit floating point specification.  The scale is static (one
 *    per tensor), the plainest reading of "FP8 quantisation" with no trained
 *    scales.
 *
 * Everything is computed in double.  Parity pins live in the tests.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

typedef struct {
    int B, D, W, T, cap, n_slot, act;   /* act: 0 identity, 1 SiLU */
} orc_conv_dims;

#define ORC_BAD_ACCEPT 1
#define ORC_BAD_POS    4

static double silu(double x) { return x / (1.0 + exp(-x)); }

static int slot_of(const int32_t *state_idx, int b) { return state_idx ? state_idx[b] : b; }

/* Conv verify: ring [n_slot, cap, D], pos [n_slot], x [B, T, D], w [D, W],
 * bias [D] or NULL, y [B, T, D].  Writes y and the staged draft in the ring. */
int orc_conv_verify(const orc_conv_dims *d, double *ring, const int32_t *pos,
                    const int32_t *state_idx, const double *x, const double *w,
                    const double *bias, double *y, int32_t *status)
{
    const int D = d->D, W = d->W, T = d->T, cap = d->cap;
    for (int b = 0; b < d->B; ++b) {
        const int s = slot_of(state_idx, b);
        const int p0 = pos[s];
        if (p0 < 0 || p0 >= cap) { *status |= ORC_BAD_POS; continue; }
        double *rs = ring + (size_t)s * cap * D;
        const double *xb = x + (size_t)b * T * D;
        for (int t = 0; t < T; ++t) {
            for (int c = 0; c < D; ++c) {
                double acc = bias ? bias[c] : 0.0;
                for (int j = 0; j < W; ++j) {
                    const int u = t - (W - 1) + j;         /* input index; < 0: window */
                    double val;
                    if (u >= 0) {
                        val = xb[(size_t)u * D + c];
                    } else {
                        const int r = ((p0 + u) % cap + cap) % cap;
                        val = rs[(size_t)r * D + c];
                    }
                    acc += w[(size_t)c * W + j] * val;
                }
                y[((size_t)b * T + t) * D + c] = d->act ? silu(acc) : acc;
            }
        }
        /* the window was read above; the draft goes after the committed inputs */
        for (int t = 0; t < T; ++t) {
            const int r = (p0 + t) % cap;
            memcpy(rs + (size_t)r * D, xb + (size_t)t * D, (size_t)D * sizeof(double));
        }
    }
    return 0;
}

/* Conv accept: pos[s] = (pos[s] + p) mod cap for 0 <= p <= T. */
int orc_conv_accept(const orc_conv_dims *d, int32_t *pos, const int32_t *state_idx,
                    const int32_t *accepted, int32_t *status)
{
    for (int b = 0; b < d->B; ++b) {
        const int s = slot_of(state_idx, b);
        const int p = accepted[b], p0 = pos[s];
        if (p < 0 || p > d->T) { *status |= ORC_BAD_ACCEPT; continue; }
        if (p0 < 0 || p0 >= d->cap) { *status |= ORC_BAD_POS; continue; }
        pos[s] = (p0 + p) % d->cap;
    }
    return 0;
}

/* E4M3 value of a code (the format definition: bias 7; exponent field 0 is
 * subnormal, 2^-6 * m/8; exponent 15 with mantissa 7 is NaN). */
double orc_e4m3_decode(int code) {
    const int sgn = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* Round x to E4M3, nearest with ties to even, saturating at +-448 (never NaN for
 * finite x).  Exact in double: a is scaled by a power of two and rounded once. */
int orc_e4m3_encode(double x) {
    const int sgn = x < 0 || (x == 0 && signbit(x));
    double a = fabs(x);
    int code;
    if (a >= 448.0) {
        code = 0x7E;                               /* 1.75 * 2^8 */
    } else {
        int e;
        frexp(a, &e);                              /* a = f 2^e, f in [0.5, 1) */
        e -= 1;                                    /* a in [2^e, 2^(e+1)) */
        if (a == 0.0 || e < -6) e = -6;            /* subnormal range shares 2^-6's quantum */
        const double n = rint(ldexp(a, 3 - e));    /* units of the quantum 2^(e-3), ties to even */
        if (n >= 16.0) {                           /* rounded up into the next binade */
            e += 1;
            code = ((e + 7) << 3);                 /* mantissa 0 */
        } else if (n >= 8.0) {
            code = ((e + 7) << 3) | ((int)n - 8);
        } else {                                   /* e == -6, subnormal (or zero) */
            code = (int)n;
        }
        if (code > 0x7E) code = 0x7E;              /* cannot happen below 448; kept for safety */
    }
    return code | (sgn << 7);
}

/* Gated RMSNorm + E4M3 per row: o, z [rows, d], w [d]; q [rows, d] codes; yq the
 * value before rounding (y * inv_scale), for the tests' tie analysis. */
int orc_gated_rmsnorm_fp8(int rows, int d, const double *o, const double *z, const double *w,
                          double eps, double inv_scale, uint8_t *q, double *yq)
{
    for (int r = 0; r < rows; ++r) {
        const double *orow = o + (size_t)r * d, *zrow = z + (size_t)r * d;
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += orow[i] * orow[i];
        const double rinv = 1.0 / sqrt(ss / d + eps);
        for (int i = 0; i < d; ++i) {
            const double y = orow[i] * rinv * w[i] * silu(zrow[i]);
            const double v = y * inv_scale;
            if (yq) yq[(size_t)r * d + i] = v;
            q[(size_t)r * d + i] = (uint8_t)orc_e4m3_encode(v);
        }
    }
    return 0;
}
