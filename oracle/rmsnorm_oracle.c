/*
 * rmsnorm_oracle.c -- plain, slow, fp64 CPU reference for the row-wise
 * RMSNorm hot path (fused residual-add forward and the VJP).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file or the library built from it: only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark use it.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * Every function works on double-precision copies of the (already quantised)
 * fp16/bf16 inputs, so the only rounding here is fp64 rounding.  Loops run in
 * the plain order the definitions state: rows ascending, columns ascending.
 * No blocking, fusion or reordering.
 *
 * Sources (web pages; the page title and section are named):
 *  - "Fused residual-add RMSNorm and fused RoPE + KV-append decode kernels"
 *    (lablup/mlxcel issue 905), Background, FusedAddRMSNorm bullet:
 *    residual' = input + residual; out = rmsnorm(residual') * (weight_bias +
 *    weight); weight_bias = 1 is the Gemma (1 + w) convention, 0 the usual one.
 *    Same page, Background, last paragraph: the kernel has two outputs
 *    (normed, new_residual).
 *  - "RMSNormVJP backward writes a full {n_rows, D} gw_temp intermediate"
 *    (ml-explore/mlx pull request 4293), POC section: the eager reference
 *    rsqrt(mean(x^2, last axis) + eps) * x * w, and the gradients (gx, gw) of
 *    sum(rms_norm(x, w, eps) * y) with respect to x and w.  "Proposed changes":
 *    gw is the sum over rows of each row's contribution.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/*
 * Forward.  For every row i (h = x + residual, or h = x when residual is
 * NULL):
 *     ms  = (1/D) * sum_j h_j^2           -- the mean over the last axis
 *     r   = 1 / sqrt(ms + eps)             -- eps inside the root
 *     out_j = h_j * r * (weight_bias + w_j)
 *     new_residual_j = h_j                 -- only when residual is given
 * x, residual, out, new_residual: rows*D, row-major.  w: D.
 */
void rmsnorm_oracle_fwd(const double *x, const double *residual,
                        const double *w, double eps, double weight_bias,
                        double *out, double *new_residual,
                        int64_t rows, int64_t D)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *xi = x + i * D;
        const double *ri = residual ? residual + i * D : NULL;

        double sumsq = 0.0;
        for (int64_t j = 0; j < D; ++j) {
            double h = ri ? xi[j] + ri[j] : xi[j];
            sumsq += h * h;
        }
        double ms = sumsq / (double)D;
        double r = 1.0 / sqrt(ms + eps);

        for (int64_t j = 0; j < D; ++j) {
            double h = ri ? xi[j] + ri[j] : xi[j];
            out[i * D + j] = h * r * (weight_bias + w[j]);
            if (new_residual)
                new_residual[i * D + j] = h;
        }
    }
}

/*
 * VJP of L = sum_ij g_ij * out_ij with respect to the normalised input h
 * (= x here; for the fused op pass new_residual) and to w.  With
 * w'_j = weight_bias + w_j and r, ms as in the forward, per row:
 *     dr/dh_k   = -(r^3 / D) * h_k
 *     dot       = sum_j g_j * w'_j * h_j
 *     gx_k      = r * g_k * w'_k - (r^3 / D) * h_k * dot
 *     gw_k     += g_k * h_k * r            (summed over rows, ascending)
 * gw is overwritten (not accumulated into).
 */
void rmsnorm_oracle_vjp(const double *x, const double *w, const double *g,
                        double eps, double weight_bias, double *gx, double *gw,
                        int64_t rows, int64_t D)
{
    for (int64_t j = 0; j < D; ++j)
        gw[j] = 0.0;

    for (int64_t i = 0; i < rows; ++i) {
        const double *hi = x + i * D;
        const double *gi = g + i * D;

        double sumsq = 0.0;
        for (int64_t j = 0; j < D; ++j)
            sumsq += hi[j] * hi[j];
        double ms = sumsq / (double)D;
        double r = 1.0 / sqrt(ms + eps);

        double dot = 0.0;
        for (int64_t j = 0; j < D; ++j)
            dot += gi[j] * (weight_bias + w[j]) * hi[j];

        double r3_over_d = r * r * r / (double)D;
        for (int64_t j = 0; j < D; ++j) {
            gx[i * D + j] = r * gi[j] * (weight_bias + w[j])
                            - r3_over_d * hi[j] * dot;
            gw[j] += gi[j] * hi[j] * r;
        }
    }
}

/*
 * VJP of the two-output fused op (out, new_residual) = F(x, residual, w).
 * With h = x + residual, out depending on h through the RMSNorm and
 * new_residual = h, the loss L = sum(g_out * out) + sum(g_residual *
 * new_residual) has
 *     dL/dx = dL/dresidual = g_h = (VJP of out at h, g_out) + g_residual
 *     dL/dw = gw of the plain VJP (new_residual does not depend on w).
 * h is the tensor the forward normalised (its new_residual); g_residual may be
 * NULL (no gradient reaches new_residual), which gives the plain VJP.
 */
void rmsnorm_oracle_fused_vjp(const double *h, const double *w, const double *g_out,
                              const double *g_residual, double eps, double weight_bias,
                              double *g_h, double *gw, int64_t rows, int64_t D)
{
    rmsnorm_oracle_vjp(h, w, g_out, eps, weight_bias, g_h, gw, rows, D);
    if (g_residual) {
        for (int64_t i = 0; i < rows * D; ++i)
            g_h[i] = g_h[i] + g_residual[i];
    }
}

/*
 * Gated activation of the decode loop ("Fused residual-add RMSNorm and fused
 * RoPE + KV-append decode kernels", Background, third bullet): for each row
 * of x = [a | b] (2*d values, a = the first d, b = the last d),
 *     out_j = silu(a_j) * b_j,   silu(a) = a * sigmoid(a) = a / (1 + exp(-a)).
 * x: rows * 2d, out: rows * d, row-major.
 */
void rmsnorm_oracle_gated_silu(const double *x, double *out, int64_t rows, int64_t d)
{
    for (int64_t i = 0; i < rows; ++i) {
        const double *a = x + i * 2 * d;
        const double *b = a + d;
        for (int64_t j = 0; j < d; ++j) {
            double silu = a[j] / (1.0 + exp(-a[j]));
            out[i * d + j] = silu * b[j];
        }
    }
}

/*
 * Rotary embedding of q and k plus the KV-cache append of the decode loop
 * ("Fused residual-add RMSNorm and fused RoPE + KV-append decode kernels",
 * Background, second bullet, and Task item 3: rope applied to q and k, k and v
 * written into the cache slab or a paged pool block, cos/sin from a
 * precomputed cache or computed on the fly).
 *
 * For token t at absolute position p = positions[t] and pair index
 * i in [0, Dh/2), the angle is  theta_i = p * base^(-2i/Dh)  (or, when
 * cos_sin is given, cos/sin are read from row p of that table: Dh/2 cosines
 * then Dh/2 sines).  A pair (x_a, x_b) rotates to
 *     (x_a cos - x_b sin,  x_b cos + x_a sin),
 * with (a, b) = (i, i + Dh/2) (rotate-half layout) or (2i, 2i + 1)
 * (interleaved, when interleaved != 0).
 *   q_out[t, h, :]            = rope(q[t, h, :])          for h < Hq
 *   k_cache[slots[t], h, :]   = rope(k[t, h, :])          for h < Hkv
 *   v_cache[slots[t], h, :]   = v[t, h, :]
 * A negative slot writes nothing to the caches.  Shapes: q, q_out
 * [T, Hq, Dh]; k, v [T, Hkv, Dh]; caches [num_slots, Hkv, Dh]; positions and
 * slots [T].  Rows of the caches that no token writes are left as they are.
 */
static void rope_pair_cs(const double *cos_sin, double base, int64_t p, int64_t i, int64_t Dh,
                         double *c, double *s)
{
    if (cos_sin) {
        *c = cos_sin[p * Dh + i];
        *s = cos_sin[p * Dh + Dh / 2 + i];
    } else {
        double theta = (double)p * pow(base, -2.0 * (double)i / (double)Dh);
        *c = cos(theta);
        *s = sin(theta);
    }
}

static void rope_vector(const double *x, double *y, const double *cos_sin, double base,
                        int64_t p, int64_t Dh, int interleaved)
{
    for (int64_t i = 0; i < Dh / 2; ++i) {
        int64_t ia = interleaved ? 2 * i : i;
        int64_t ib = interleaved ? 2 * i + 1 : i + Dh / 2;
        double c, s;
        rope_pair_cs(cos_sin, base, p, i, Dh, &c, &s);
        double xa = x[ia], xb = x[ib];
        y[ia] = xa * c - xb * s;
        y[ib] = xb * c + xa * s;
    }
}

void rmsnorm_oracle_rope_kv_append(const double *q, const double *k, const double *v,
                                   const int64_t *positions, const int64_t *slots,
                                   double *q_out, double *k_cache, double *v_cache,
                                   const double *cos_sin, double base, int interleaved,
                                   int64_t T, int64_t Hq, int64_t Hkv, int64_t Dh)
{
    for (int64_t t = 0; t < T; ++t) {
        int64_t p = positions[t];
        for (int64_t h = 0; h < Hq; ++h)
            rope_vector(q + (t * Hq + h) * Dh, q_out + (t * Hq + h) * Dh, cos_sin, base, p, Dh,
                        interleaved);
        int64_t slot = slots[t];
        if (slot < 0)
            continue;
        for (int64_t h = 0; h < Hkv; ++h) {
            rope_vector(k + (t * Hkv + h) * Dh, k_cache + (slot * Hkv + h) * Dh, cos_sin, base,
                        p, Dh, interleaved);
            for (int64_t j = 0; j < Dh; ++j)
                v_cache[(slot * Hkv + h) * Dh + j] = v[(t * Hkv + h) * Dh + j];
        }
    }
}

/*
 * The per-row scale of the forward on its own ("Fused residual-add RMSNorm
 * and fused RoPE + KV-append decode kernels", Background, FusedAddRMSNorm
 * bullet: the rsqrt of the mean square plus eps; "RMSNormVJP backward writes
 * a full {n_rows, D} gw_temp intermediate", POC section: the same rsqrt factor
 * in the eager reference):
 *     rstd_i = 1 / sqrt((1/D) * sum_j h_j^2 + eps),   h = x + residual, or x.
 * The forward multiplies row i by exactly this value, so a backward pass can
 * take it instead of summing h^2 again.
 */
void rmsnorm_oracle_rstd(const double *x, const double *residual, double eps,
                         double *rstd, int64_t rows, int64_t D)
{
    for (int64_t i = 0; i < rows; ++i) {
        double sq = 0.0;
        for (int64_t j = 0; j < D; ++j) {
            double hv = residual ? x[i * D + j] + residual[i * D + j] : x[i * D + j];
            sq += hv * hv;
        }
        rstd[i] = 1.0 / sqrt(sq / (double)D + eps);
    }
}

/*
 * The VJP with each row's scale supplied (rstd[i], as the forward saved it)
 * instead of recomputed from h.  Per row, with rho = rstd[i] and
 * w'_j = weight_bias + w_j:
 *     dot   = sum_j g_j * w'_j * h_j
 *     gx_k  = rho * g_k * w'_k - (rho^3 / D) * h_k * dot
 *     gw_k += g_k * h_k * rho           (summed over rows, ascending)
 * With rstd[i] = 1 / sqrt(mean(h_i^2) + eps) this is rmsnorm_oracle_vjp; eps
 * enters only through rstd.  gw is overwritten.
 */
void rmsnorm_oracle_vjp_rstd(const double *x, const double *w, const double *g,
                             const double *rstd, double weight_bias, double *gx,
                             double *gw, int64_t rows, int64_t D)
{
    for (int64_t j = 0; j < D; ++j)
        gw[j] = 0.0;

    for (int64_t i = 0; i < rows; ++i) {
        const double rho = rstd[i];
        double dg = 0.0;
        for (int64_t j = 0; j < D; ++j)
            dg += g[i * D + j] * (weight_bias + w[j]) * x[i * D + j];

        const double k3 = rho * rho * rho / (double)D;
        for (int64_t j = 0; j < D; ++j) {
            gx[i * D + j] = rho * g[i * D + j] * (weight_bias + w[j])
                            - k3 * x[i * D + j] * dg;
            gw[j] += g[i * D + j] * x[i * D + j] * rho;
        }
    }
}
