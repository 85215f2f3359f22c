/*
 * tf_oracle.c -- plain, slow CPU oracle for the Ulysses sequence<->head relayout
 * and the fused per-head RMSNorm + RoPE (interleaved, or half-split) applied to Q/K.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Sources (web pages this follows):
 *  - TeleFuser docs, "Communication Architecture", section "Sequence Parallel
 *    Communication / Ulysses": the sequence->head all-to-all maps
 *    [B, S_local, H_global, D] to [B, S_global, H_local, D]; the inverse maps back.
 *  - same page, "Shared Collective Primitives / Equal-shape gather": shards are
 *    concatenated in rank order (rank-major), which fixes target row = r*S_local + t.
 *  - flashinfer PR #6332 (QkvNormRopeExchangeOverlap) commit message, section
 *    "Assumptions", items "Exchange algorithm" (each rank ends up with its own band
 *    of heads for the whole sequence) and "Operator math" (fp32 RMSNorm, eps 1e-6, shared
 *    [head_dim] weight per Q / K; RoPE on interleaved element pairs applied in fp32 from a
 *    per-token cos/sin table; order QK-norm -> RoPE; 16-bit operands/outputs);
 *    section "Tests" (RMSNorm with the 16-bit cast before the 16-bit weight scale).
 *
 * Readings where the pages leave a step open (each also listed in the design notes):
 *  - head band g is the contiguous heads [g*Hl, (g+1)*Hl);
 *  - the sum of squares is accumulated in double (exact for ordinary inputs) and
 *    the mean is rounded once to fp32; 1/sqrt is IEEE sqrt then IEEE division;
 *  - rounding to the 16-bit type happens after normalising, after the weight
 *    scale and after the rotation, each time round-to-nearest-even from fp32;
 *  - RoPE pair i of a head uses frequency theta^(-2i/D) at the global token
 *    index p = r*S_local + t; cos and sin are evaluated in double and stored as fp32;
 *  - the half-split variant (not on the pages, which name only the interleaved
 *    form) pairs element i with i + D/2 and uses the same table entry i.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no FMA contraction, so
 * every float expression below is rounded to fp32 after each operation).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#if FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in float (FLT_EVAL_METHOD == 0)"
#endif

/* ------------------------------------------------------------------------- */
/* 16-bit floating-point formats, written from their definitions.             */
/*   fmt 0: IEEE 754 binary16  (1 sign, 5 exponent, 10 fraction bits, bias 15) */
/*   fmt 1: bfloat16           (1 sign, 8 exponent,  7 fraction bits, bias 127) */
/* ------------------------------------------------------------------------- */

typedef struct {
    int frac_bits; /* stored fraction bits */
    int exp_bits;  /* exponent field width */
    int bias;      /* exponent bias */
} fmt16;

static const fmt16 FMT[2] = {
    {10, 5, 15},  /* binary16 */
    {7, 8, 127},  /* bfloat16 */
};

/* Value of a 16-bit pattern, exactly, as a double. */
double tfo_decode16(int fmt, uint16_t bits)
{
    const fmt16 *f = &FMT[fmt];
    uint32_t frac = bits & ((1u << f->frac_bits) - 1u);
    uint32_t e = (bits >> f->frac_bits) & ((1u << f->exp_bits) - 1u);
    double sign = (bits & 0x8000u) ? -1.0 : 1.0;
    int emin = 1 - f->bias;
    if (e == (1u << f->exp_bits) - 1u)
        return frac ? NAN : sign * INFINITY;
    if (e == 0) /* zero or subnormal: frac * 2^(emin - frac_bits) */
        return sign * ldexp((double)frac, emin - f->frac_bits);
    return sign * ldexp((double)(frac + (1u << f->frac_bits)), (int)e - f->bias - f->frac_bits);
}

/* Nearest 16-bit value to x, ties to even, overflow to infinity, gradual underflow. */
uint16_t tfo_encode16(int fmt, double x)
{
    const fmt16 *f = &FMT[fmt];
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    uint16_t exp_all = (uint16_t)(((1u << f->exp_bits) - 1u) << f->frac_bits);
    int emin = 1 - f->bias, emax = f->bias;
    double a = fabs(x);
    if (isnan(x))
        return (uint16_t)(sign | exp_all | (1u << (f->frac_bits - 1))); /* quiet NaN */
    if (isinf(a))
        return (uint16_t)(sign | exp_all);
    if (a == 0.0)
        return sign;
    int E;
    frexp(a, &E);
    E -= 1; /* a lies in [2^E, 2^(E+1)) */
    if (E < emin)
        E = emin; /* subnormal range: fixed quantum 2^(emin - frac_bits) */
    /* a / quantum is exact (power-of-two scaling); nearbyint rounds ties to even
     * under the default rounding mode. */
    double q = nearbyint(ldexp(a, f->frac_bits - E));
    if (q >= ldexp(1.0, f->frac_bits + 1)) { /* rounding carried into the next binade */
        q = ldexp(q, -1);
        E += 1;
    }
    if (E > emax)
        return (uint16_t)(sign | exp_all); /* overflow */
    uint32_t qi = (uint32_t)q;
    if (qi < (1u << f->frac_bits)) /* subnormal (E == emin) */
        return (uint16_t)(sign | qi);
    return (uint16_t)(sign | ((uint32_t)(E + f->bias) << f->frac_bits) | (qi - (1u << f->frac_bits)));
}

/* ------------------------------------------------------------------------- */
/* Ulysses relayout (bit copies of elements of any size).                     */
/* Shard r holds tokens [r*Sl, (r+1)*Sl); head group g holds heads            */
/* [g*Hl, (g+1)*Hl), Hl = H / P.                                              */
/* ------------------------------------------------------------------------- */

/*
 * Sequence->head scatter ("scatter heads / gather sequence"):
 *     T_g[b][r*Sl + t][h][d] = S_r[b][t][g*Hl + h][d]
 * src[r]: shard r, read through element strides (sb, st, sh) with unit d stride.
 * dst[g]: P contiguous targets [B][P*Sl][Hl][D].
 */
void tfo_scatter(int P, int B, int Sl, int H, int D, int esize,
                 const void *const *src, int64_t sb, int64_t st, int64_t sh,
                 void *const *dst)
{
    int Hl = H / P;
    int64_t S = (int64_t)P * Sl;
    for (int g = 0; g < P; ++g)
        for (int b = 0; b < B; ++b)
            for (int r = 0; r < P; ++r)
                for (int t = 0; t < Sl; ++t)
                    for (int h = 0; h < Hl; ++h)
                        for (int d = 0; d < D; ++d) {
                            int64_t si = (int64_t)b * sb + (int64_t)t * st + (int64_t)(g * Hl + h) * sh + d;
                            int64_t ti = (((int64_t)b * S + (int64_t)r * Sl + t) * Hl + h) * D + d;
                            memcpy((uint8_t *)dst[g] + ti * esize,
                                   (const uint8_t *)src[r] + si * esize, (size_t)esize);
                        }
}

/*
 * Head->sequence gather ("gather heads / scatter sequence"), the inverse:
 *     O_r[b][t][g*Hl + h][d] = A_g[b][r*Sl + t][h][d]
 * src[g]: head-group buffer g [B][P*Sl][Hl][D] read through strides (ab, at, ah).
 * dst[r]: P contiguous outputs [B][Sl][H][D].
 */
void tfo_gather(int P, int B, int Sl, int H, int D, int esize,
                const void *const *src, int64_t ab, int64_t at, int64_t ah,
                void *const *dst)
{
    int Hl = H / P;
    for (int r = 0; r < P; ++r)
        for (int b = 0; b < B; ++b)
            for (int t = 0; t < Sl; ++t)
                for (int g = 0; g < P; ++g)
                    for (int h = 0; h < Hl; ++h)
                        for (int d = 0; d < D; ++d) {
                            int64_t si = (int64_t)b * ab + ((int64_t)r * Sl + t) * at + (int64_t)h * ah + d;
                            int64_t oi = (((int64_t)b * Sl + t) * H + g * Hl + h) * D + d;
                            memcpy((uint8_t *)dst[r] + oi * esize,
                                   (const uint8_t *)src[g] + si * esize, (size_t)esize);
                        }
}

/* ------------------------------------------------------------------------- */
/* RoPE table and the fused per-row RMSNorm + interleaved RoPE.               */
/* ------------------------------------------------------------------------- */

/*
 * Per-token cos/sin table, fp32, layout [S][D/2][2]: entry (p, i) holds
 * cos(p * theta^(-2i/D)) and sin(p * theta^(-2i/D)), evaluated in double.
 */
void tfo_rope_table(double theta, int S, int D, float *out)
{
    for (int p = 0; p < S; ++p)
        for (int i = 0; i < D / 2; ++i) {
            double freq = pow(theta, -2.0 * i / D);
            double angle = (double)p * freq;
            out[((int64_t)p * (D / 2) + i) * 2 + 0] = (float)cos(angle);
            out[((int64_t)p * (D / 2) + i) * 2 + 1] = (float)sin(angle);
        }
}

static float round16(int fmt, float v)
{
    return (float)tfo_decode16(fmt, tfo_encode16(fmt, (double)v));
}

/*
 * RMSNorm and weight scale of one head row x[0..D) (16-bit, format fmt):
 *   ms  = mean(x^2)                     (sum in double, mean rounded to fp32)
 *   inv = 1 / sqrt(ms + eps)            (fp32)
 *   y   = round16(x * inv)              (normalised value cast before the scale)
 *   z   = round16(y * w)                (16-bit weight scale, product in fp32)
 */
static void rmsnorm_scale(int fmt, int D, const uint16_t *x, const uint16_t *w, float eps, float *z)
{
    float xf[1024], y[1024];
    double ss = 0.0;
    for (int d = 0; d < D; ++d) {
        xf[d] = (float)tfo_decode16(fmt, x[d]);
        ss += (double)xf[d] * (double)xf[d];
    }
    float ms = (float)(ss / D);
    float inv = 1.0f / sqrtf(ms + eps);
    for (int d = 0; d < D; ++d) {
        float prod = xf[d] * inv;
        y[d] = round16(fmt, prod);
    }
    for (int d = 0; d < D; ++d) {
        float prod = y[d] * (float)tfo_decode16(fmt, w[d]);
        z[d] = round16(fmt, prod);
    }
}

/*
 * One head row at a token whose table row is cs, RoPE on interleaved pairs:
 * z = rmsnorm_scale(x), then for i < D/2
 *   o[2i]   = round16(z[2i]*cos - z[2i+1]*sin)
 *   o[2i+1] = round16(z[2i]*sin + z[2i+1]*cos)
 */
void tfo_rmsnorm_rope_row(int fmt, int D, const uint16_t *x, const uint16_t *w,
                          float eps, const float *cs, uint16_t *out)
{
    float z[1024];
    rmsnorm_scale(fmt, D, x, w, eps, z);
    for (int i = 0; i < D / 2; ++i) {
        float a = z[2 * i], b = z[2 * i + 1];
        float c = cs[2 * i], s = cs[2 * i + 1];
        float ac = a * c, bs = b * s, as = a * s, bc = b * c;
        out[2 * i] = tfo_encode16(fmt, (double)(ac - bs));
        out[2 * i + 1] = tfo_encode16(fmt, (double)(as + bc));
    }
}

/*
 * The same row with half-split RoPE (the GPT-NeoX pairing; RoFormer's rotation
 * of each coordinate pair by p * theta_i): element i pairs with element i + D/2
 * and both use table entry i, for i < D/2:
 *   o[i]       = round16(z[i]*cos_i - z[i + D/2]*sin_i)
 *   o[i + D/2] = round16(z[i]*sin_i + z[i + D/2]*cos_i)
 */
void tfo_rmsnorm_rope_neox_row(int fmt, int D, const uint16_t *x, const uint16_t *w,
                               float eps, const float *cs, uint16_t *out)
{
    float z[1024];
    int half = D / 2;
    rmsnorm_scale(fmt, D, x, w, eps, z);
    for (int i = 0; i < half; ++i) {
        float first = z[i], second = z[i + half];
        float cos_i = cs[2 * i], sin_i = cs[2 * i + 1];
        float fc = first * cos_i, ss_ = second * sin_i, fs = first * sin_i, sc = second * cos_i;
        out[i] = tfo_encode16(fmt, (double)(fc - ss_));
        out[i + half] = tfo_encode16(fmt, (double)(fs + sc));
    }
}

/*
 * Scatter of one tensor (Q or K) with the fused RMSNorm + RoPE: each target row
 * T_g[b][r*Sl + t][h][:] is tfo_rmsnorm_rope_row (neox == 0) or
 * tfo_rmsnorm_rope_neox_row (neox != 0) of source row S_r[b][t][g*Hl + h][:] at
 * global position p = r*Sl + t.  table: [>= P*Sl][D/2][2] fp32.
 */
void tfo_scatter_norm_rope(int fmt, int P, int B, int Sl, int H, int D,
                           const void *const *src, int64_t sb, int64_t st, int64_t sh,
                           const uint16_t *w, float eps, const float *table,
                           void *const *dst, int neox)
{
    int Hl = H / P;
    int64_t S = (int64_t)P * Sl;
    for (int g = 0; g < P; ++g)
        for (int b = 0; b < B; ++b)
            for (int r = 0; r < P; ++r)
                for (int t = 0; t < Sl; ++t)
                    for (int h = 0; h < Hl; ++h) {
                        int64_t p = (int64_t)r * Sl + t;
                        const uint16_t *row = (const uint16_t *)src[r] +
                                              (int64_t)b * sb + (int64_t)t * st + (int64_t)(g * Hl + h) * sh;
                        uint16_t *trow = (uint16_t *)dst[g] + (((int64_t)b * S + p) * Hl + h) * D;
                        if (neox)
                            tfo_rmsnorm_rope_neox_row(fmt, D, row, w, eps, table + p * D, trow);
                        else
                            tfo_rmsnorm_rope_row(fmt, D, row, w, eps, table + p * D, trow);
                    }
}

/* ------------------------------------------------------------------------- */
/* QKV projection (the GEMM in front of the exchange).                        */
/* ------------------------------------------------------------------------- */

/*
 * One row of the projection of flashinfer PR #6332 ("Description": a BF16 QKV
 * projection feeds per-head RMSNorm, RoPE and the head exchange; "Assumptions /
 * Operator math": order projection -> QK-norm -> RoPE, 16-bit operands and
 * outputs).  x[0..K) is one token's hidden vector, w the [N][K] weight in the
 * nn.Linear layout (row n holds output feature n, w_row elements apart); for
 * n in [n0, n1):
 *     out[n - n0] = round16( sum_k x[k] * w[n][k] )
 * with the sum accumulated in double (products of 16-bit values are exact; the
 * sum is exact up to double rounding) and rounded once to the 16-bit type.
 */
void tfo_project_row(int fmt, int K, const uint16_t *x, const uint16_t *w, int64_t w_row, int n0, int n1,
                     uint16_t *out)
{
    double xd[8192];
    for (int k = 0; k < K; ++k)
        xd[k] = tfo_decode16(fmt, x[k]);
    for (int n = n0; n < n1; ++n) {
        const uint16_t *wn = w + (int64_t)n * w_row;
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += xd[k] * tfo_decode16(fmt, wn[k]);
        out[n - n0] = tfo_encode16(fmt, acc);
    }
}

/* All M rows of one shard: x [M][K] with row stride x_row, out [M][N] contiguous. */
void tfo_project(int fmt, int M, int N, int K, const uint16_t *x, int64_t x_row, const uint16_t *w, int64_t w_row,
                 uint16_t *out)
{
    for (int m = 0; m < M; ++m)
        tfo_project_row(fmt, K, x + (int64_t)m * x_row, w, w_row, 0, N, out + (int64_t)m * N);
}
