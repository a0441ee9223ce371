/*
 * ln_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU oracle for the fused residual-add + LayerNorm forward and
 * backward (and, at the end of the file, the fused residual-add + RMSNorm ones).  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load it; the CUDA
 * library never links or calls it, and it shares no code with it.
 *
 * Sources (page titles and sections; the pages are course notes and blog posts):
 *  - Forward definition, per row of length m:
 *      xhat_i = (x_i - mu) / sigma,  sigma = sqrt(var + eps),  y_i = gamma_i * xhat_i + beta_i,
 *    with mu and r = 1/sigma saved per row.
 *    ("Accelerating Transformer on GPU (II): Training with LightSeq2", section 2.1.)
 *    The variance is the biased one (divide by m), the way the one-thread-per-row kernel of
 *    "AI infra learning log (2): LayerNorm operator optimisation", section 2.1 (v1), computes it.
 *  - Fused residual: the residual sum s = inp1 + inp2 is written out first and then
 *    normalised ("llm.c: the llmc/ CUDA kernel layer", section 3.2, fused_residual_forward5).
 *    Reading taken here: the STORED residual (s rounded to the I/O precision) is what gets
 *    normalised, so that the backward, which only sees that stored tensor, differentiates
 *    exactly the function the forward evaluated.
 *  - Backward, "HW4 form" ("Training with LightSeq2", section 2.1): with g_i = gamma_i * dy_i,
 *      dx_i = r * [ g_i - (sum_j g_j + xhat_i * sum_j g_j xhat_j) / m ].
 *  - Backward, "slides form" (same section), used only as an independent cross-check:
 *      dx_i = g_i / sigma + alpha_i sum_j g_j + beta_i sum_j g_j x_j,
 *      alpha_i = ((x_i - mu) mu - sigma^2) / (m sigma^3),  beta_i = (mu - x_i) / (m sigma^3).
 *  - Column gradients ("Training with LightSeq2", sections 2.1 and 2.4):
 *      dgamma_j = sum over rows of dy * xhat,   dbeta_j = sum over rows of dy.
 *
 * Precision: every stored input is an exact float64 upcast of an fp32 or bf16 value.  All
 * arithmetic is float64.  Results that the GPU stores in the I/O precision are rounded here
 * to that precision with round-to-nearest-even ("io" = 0: no rounding, 1: fp32, 2: bf16).
 * Mean and rstd are returned unrounded (float64).
 *
 * Threads: rows are independent, so the row loops run in parallel over rows.  The column
 * sums run in parallel over columns, each column summed over rows in row order, which is
 * the definition's order.  Nothing is blocked, fused or reordered beyond that.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define IO_F64 0
#define IO_F32 1
#define IO_BF16 2

/* Largest finite bf16: (2 - 2^-7) * 2^127. */
static const double kBf16Max = 3.3895313892515355e38;

/* Round a float64 value to the nearest bf16 value, ties to even.  bf16 keeps 8 significant
 * bits and the fp32 exponent range; below 2^-126 the spacing is fixed at 2^-133. */
static double round_to_bf16(double v) {
    if (v == 0.0 || isnan(v) || isinf(v)) return v;
    int e;
    (void)frexp(v, &e); /* |v| = f * 2^e with f in [0.5, 1) */
    int qexp = e - 8;   /* spacing of 8-significant-bit numbers in [2^(e-1), 2^e) */
    if (qexp < -133) qexp = -133;
    double q = ldexp(1.0, qexp);
    double r = nearbyint(v / q) * q; /* v/q is exact; nearbyint rounds ties to even */
    if (fabs(r) > kBf16Max) r = copysign(INFINITY, v);
    return r;
}

static double round_io(double v, int io) {
    if (io == IO_F32) return (double)(float)v; /* C conversion: round to nearest even */
    if (io == IO_BF16) return round_to_bf16(v);
    return v;
}

double oracle_round_io(double v, int io) { return round_io(v, io); }

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Forward.  x, res: [rows, cols] (res may be NULL: no residual).  gamma, beta: [cols].
 * Outputs: out, res_out [rows, cols] (either may be NULL), mean, rstd [rows].
 */
void oracle_ln_fwd(const double* x, const double* res, const double* gamma, const double* beta,
                   double eps, int64_t rows, int64_t cols, int io, double* out, double* res_out,
                   double* mean, double* rstd, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * cols;
        const double* rr = res ? res + r * cols : NULL;
        /* The residual sum, rounded to the stored precision (it is what gets normalised). */
        double sum = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double s = rr ? xr[j] + rr[j] : xr[j];
            s = round_io(s, io);
            if (res_out) res_out[r * cols + j] = s;
            sum += s;
        }
        double mu = sum / (double)cols;
        /* Second, dependent pass: the centred sum of squares (two-pass variance). */
        double sq = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double s = rr ? xr[j] + rr[j] : xr[j];
            s = round_io(s, io);
            double d = s - mu;
            sq += d * d;
        }
        double var = sq / (double)cols;
        double rs = 1.0 / sqrt(var + eps);
        mean[r] = mu;
        rstd[r] = rs;
        if (out) {
            for (int64_t j = 0; j < cols; ++j) {
                double s = rr ? xr[j] + rr[j] : xr[j];
                s = round_io(s, io);
                double xhat = (s - mu) * rs;
                out[r * cols + j] = round_io(gamma[j] * xhat + beta[j], io);
            }
        }
    }
}

/*
 * Backward, HW4 form.  dy, xr: [rows, cols] (xr is the tensor the forward normalised);
 * gamma: [cols]; mean, rstd: [rows].  Outputs: dx [rows, cols] (may be NULL),
 * dgamma, dbeta [cols] (either may be NULL).
 */
void oracle_ln_bwd(const double* dy, const double* xr, const double* gamma, const double* mean,
                   const double* rstd, int64_t rows, int64_t cols, int io, double* dx,
                   double* dgamma, double* dbeta, int nthreads) {
    set_threads(nthreads);
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            const double* d = dy + r * cols;
            const double* x = xr + r * cols;
            double mu = mean[r], rs = rstd[r];
            double sum_g = 0.0, sum_gx = 0.0;
            for (int64_t j = 0; j < cols; ++j) {
                double xhat = (x[j] - mu) * rs;
                double g = gamma[j] * d[j];
                sum_g += g;
                sum_gx += g * xhat;
            }
            for (int64_t j = 0; j < cols; ++j) {
                double xhat = (x[j] - mu) * rs;
                double g = gamma[j] * d[j];
                double v = rs * (g - (sum_g + xhat * sum_gx) / (double)cols);
                dx[r * cols + j] = round_io(v, io);
            }
        }
    }
    if (dgamma || dbeta) {
        /* Each thread owns a contiguous slice of columns and walks the rows in order, so
         * every column is summed over rows 0, 1, ..., rows-1 exactly as written above. */
#pragma omp parallel
        {
            int t = 0, nt = 1;
#ifdef _OPENMP
            t = omp_get_thread_num();
            nt = omp_get_num_threads();
#endif
            int64_t j0 = cols * t / nt, j1 = cols * (t + 1) / nt;
            int64_t w = j1 - j0;
            double* acc = w > 0 ? (double*)calloc((size_t)(2 * w), sizeof(double)) : NULL;
            if (w > 0 && acc) {
                double* acc_g = acc;
                double* acc_b = acc + w;
                for (int64_t r = 0; r < rows; ++r) {
                    const double* d = dy + r * cols;
                    const double* x = xr + r * cols;
                    double mu = mean[r], rs = rstd[r];
                    for (int64_t j = j0; j < j1; ++j) {
                        double xhat = (x[j] - mu) * rs;
                        acc_g[j - j0] += d[j] * xhat;
                        acc_b[j - j0] += d[j];
                    }
                }
                for (int64_t j = j0; j < j1; ++j) {
                    if (dgamma) dgamma[j] = round_io(acc_g[j - j0], io);
                    if (dbeta) dbeta[j] = round_io(acc_b[j - j0], io);
                }
            } else if (w > 0) {
                /* Out of memory for the slice: fall back to one column at a time. */
                for (int64_t j = j0; j < j1; ++j) {
                    double ag = 0.0, ab = 0.0;
                    for (int64_t r = 0; r < rows; ++r) {
                        double xhat = (xr[r * cols + j] - mean[r]) * rstd[r];
                        ag += dy[r * cols + j] * xhat;
                        ab += dy[r * cols + j];
                    }
                    if (dgamma) dgamma[j] = round_io(ag, io);
                    if (dbeta) dbeta[j] = round_io(ab, io);
                }
            }
            free(acc);
        }
    }
}

/*
 * Backward dx only, slides form (raw x instead of xhat in the second sum).  Unrounded
 * float64 output; used to cross-check the HW4 form, never as the expected GPU value.
 */
void oracle_ln_bwd_dx_slides(const double* dy, const double* xr, const double* gamma,
                             const double* mean, const double* rstd, int64_t rows, int64_t cols,
                             double* dx, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double* d = dy + r * cols;
        const double* x = xr + r * cols;
        double mu = mean[r];
        double sigma = 1.0 / rstd[r];
        double m = (double)cols;
        double sum_g = 0.0, sum_gx = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double g = gamma[j] * d[j];
            sum_g += g;
            sum_gx += g * x[j];
        }
        double s3 = m * sigma * sigma * sigma;
        for (int64_t j = 0; j < cols; ++j) {
            double g = gamma[j] * d[j];
            double alpha = ((x[j] - mu) * mu - sigma * sigma) / s3;
            double beta = (mu - x[j]) / s3;
            dx[r * cols + j] = g / sigma + alpha * sum_g + beta * sum_gx;
        }
    }
}

/*
 * Fused residual-add + RMSNorm, forward.  "GPU Performance from First Principles", section
 * 6.1 (operator fusion, the "fused add + RMSNorm" item) and exercise 4 of the same page: one
 * kernel reads x and the residual and writes the new residual stream and the normalised
 * result.  The page names the operation without printing its formula; the plainest reading,
 * taken here, is the usual RMSNorm: no mean is subtracted, no shift is added, eps is added to
 * the mean square inside the square root, and a per-column gain gamma scales the result.
 * Per row of length m:
 *    s = x + res (rounded to the stored precision, as for LayerNorm above; it is written
 *    out and it is what gets normalised),  ms = mean(s^2),  r = 1 / sqrt(ms + eps),
 *    out_i = gamma_i * s_i * r.
 * Outputs: out, res_out [rows, cols] (either may be NULL), rrms [rows] (r, unrounded).
 */
void oracle_rms_fwd(const double* x, const double* res, const double* gamma, double eps,
                    int64_t rows, int64_t cols, int io, double* out, double* res_out,
                    double* rrms, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * cols;
        const double* rr = res ? res + r * cols : NULL;
        double sq = 0.0;
        for (int64_t j = 0; j < cols; ++j) {
            double s = round_io(rr ? xr[j] + rr[j] : xr[j], io);
            if (res_out) res_out[r * cols + j] = s;
            sq += s * s;
        }
        double rs = 1.0 / sqrt(sq / (double)cols + eps);
        rrms[r] = rs;
        if (out) {
            for (int64_t j = 0; j < cols; ++j) {
                double s = round_io(rr ? xr[j] + rr[j] : xr[j], io);
                out[r * cols + j] = round_io(gamma[j] * (s * rs), io);
            }
        }
    }
}

/*
 * Fused residual-add + RMSNorm, backward, from the forward above by the chain rule
 * (d r / d s_j = -r^3 s_j / m).  With shat = s * r and g = gamma * dy:
 *    dx_j = r * (g_j - shat_j * sum_i g_i shat_i / m)   (the gradient of s, hence of x and res)
 *    dgamma_j = sum over rows of dy_j * shat_j.
 * xr is the tensor the forward normalised (its res_out, or x without a residual).  Outputs:
 * dx [rows, cols] (may be NULL), dgamma [cols] (may be NULL), rounded to `io`.
 */
void oracle_rms_bwd(const double* dy, const double* xr, const double* gamma, const double* rrms,
                    int64_t rows, int64_t cols, int io, double* dx, double* dgamma,
                    int nthreads) {
    set_threads(nthreads);
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            const double* d = dy + r * cols;
            const double* s = xr + r * cols;
            double rs = rrms[r];
            double sum_gs = 0.0;
            for (int64_t j = 0; j < cols; ++j) sum_gs += gamma[j] * d[j] * (s[j] * rs);
            for (int64_t j = 0; j < cols; ++j) {
                double shat = s[j] * rs;
                double v = rs * (gamma[j] * d[j] - shat * sum_gs / (double)cols);
                dx[r * cols + j] = round_io(v, io);
            }
        }
    }
    if (dgamma) {
        /* Each thread owns a contiguous slice of columns and walks the rows in order. */
#pragma omp parallel
        {
            int t = 0, nt = 1;
#ifdef _OPENMP
            t = omp_get_thread_num();
            nt = omp_get_num_threads();
#endif
            int64_t j0 = cols * t / nt, j1 = cols * (t + 1) / nt;
            int64_t w = j1 - j0;
            /* Running sums of the slice, every column summed over rows 0, 1, ... in order. */
            double* acc = w > 0 ? (double*)calloc((size_t)w, sizeof(double)) : NULL;
            if (acc) {
                for (int64_t r = 0; r < rows; ++r)
                    for (int64_t j = j0; j < j1; ++j)
                        acc[j - j0] += dy[r * cols + j] * (xr[r * cols + j] * rrms[r]);
                for (int64_t j = j0; j < j1; ++j) dgamma[j] = round_io(acc[j - j0], io);
            } else {
                for (int64_t j = j0; j < j1; ++j) {
                    double a = 0.0;
                    for (int64_t r = 0; r < rows; ++r)
                        a += dy[r * cols + j] * (xr[r * cols + j] * rrms[r]);
                    dgamma[j] = round_io(a, io);
                }
            }
            free(acc);
        }
    }
}

/*
 * Fused softmax, forward ("Accelerating Transformer on GPU (I)", section 4.1: scale, add the
 * mask, row maximum, exponentiate the difference, row sum, divide -- one kernel).  Per row r
 * of length m:
 *    z_j = scale * x_j + mask[(r % mask_rows) * m + j]   (no mask term when mask is NULL)
 *    y_j = exp(z_j - max z) / sum_i exp(z_i - max z).
 * The mask is additive (0 keeps an entry, -inf removes it) and its rows repeat every
 * mask_rows rows (an attention mask of [L, L] over rows batch x heads x L).  A row whose
 * entries are all -inf has no defined softmax; the definition gives NaN (0 / 0) there.
 * Output y [rows, cols], rounded to `io`.
 */
void oracle_softmax_fwd(const double* x, const double* mask, int64_t mask_rows, double scale,
                        int64_t rows, int64_t cols, int io, double* y, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * cols;
        const double* mr = mask ? mask + (r % mask_rows) * cols : NULL;
        double mx = -INFINITY;
        for (int64_t j = 0; j < cols; ++j) {
            double z = scale * xr[j] + (mr ? mr[j] : 0.0);
            if (z > mx) mx = z;
        }
        double sum = 0.0;
        for (int64_t j = 0; j < cols; ++j) sum += exp(scale * xr[j] + (mr ? mr[j] : 0.0) - mx);
        for (int64_t j = 0; j < cols; ++j)
            y[r * cols + j] = round_io(exp(scale * xr[j] + (mr ? mr[j] : 0.0) - mx) / sum, io);
    }
}

/*
 * Fused softmax, backward ("Accelerating Transformer on GPU (II)", section 3.1: only y is
 * needed, and one row reduction): with s = sum_i dy_i y_i,
 *    dx_j = scale * y_j * (dy_j - s)
 * (scale: the forward's factor on x; the mask has no gradient).  Output dx, rounded to `io`.
 */
void oracle_softmax_bwd(const double* dy, const double* y, double scale, int64_t rows,
                        int64_t cols, int io, double* dx, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double* d = dy + r * cols;
        const double* yr = y + r * cols;
        double s = 0.0;
        for (int64_t j = 0; j < cols; ++j) s += d[j] * yr[j];
        for (int64_t j = 0; j < cols; ++j) dx[r * cols + j] = round_io(scale * yr[j] * (d[j] - s), io);
    }
}

/*
 * Fused cross-entropy with label smoothing, forward and backward in one pass
 * ("Accelerating Transformer on GPU (I)", section 5.2; the fused classifier of "llm.c: the
 * llmc/ CUDA kernel layer", section 6).  Per row of V logits x with target t:
 *    p = (1 - alpha) onehot(t) + alpha / V,   q = softmax(x),
 *    loss = -sum_i p_i log q_i = log Z + m - [(1 - alpha) x_t + (alpha / V) sum_i x_i]
 * with m = max x and Z = sum exp(x - m), and the gradient of the loss, scaled by dloss,
 *    dx = dloss * (q - p).
 * targets must lie in [0, V).  Outputs: losses [rows] (unrounded float64; may be NULL),
 * dx [rows, V] rounded to `io` (may be NULL).
 */
void oracle_xent(const double* x, const int32_t* targets, int64_t rows, int64_t V, double alpha,
                 double dloss, int io, double* losses, double* dx, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * V;
        const int64_t t = targets[r];
        double m = -INFINITY, sx = 0.0;
        for (int64_t j = 0; j < V; ++j) {
            if (xr[j] > m) m = xr[j];
            sx += xr[j];
        }
        double z = 0.0;
        for (int64_t j = 0; j < V; ++j) z += exp(xr[j] - m);
        if (losses) losses[r] = log(z) + m - ((1.0 - alpha) * xr[t] + alpha / (double)V * sx);
        if (dx) {
            for (int64_t j = 0; j < V; ++j) {
                double p = alpha / (double)V + (j == t ? 1.0 - alpha : 0.0);
                dx[r * V + j] = round_io(dloss * (exp(xr[j] - m) / z - p), io);
            }
        }
    }
}

/*
 * Counter-based random numbers for dropout: Philox-4x32 with 10 rounds (Salmon, Moraes,
 * Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011).  One round maps
 * the counter (c0, c1, c2, c3) under the key (k0, k1) to
 *    (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0))
 * with M0 = 0xD2511F53, M1 = 0xCD9E8D57 (64-bit products split into 32-bit halves); the key
 * is advanced by the Weyl constants (0x9E3779B9, 0xBB67AE85) before every round after the
 * first.  The generator is written here from that definition; the CUDA path has its own.
 */
void oracle_philox4x32(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/*
 * The dropout decision of element i (= row * cols + col) under (seed, offset) with drop
 * probability p: the word i % 4 of Philox-4x32-10 at counter (i / 4 split into low and high
 * 32 bits, offset split likewise) and key (seed split likewise); the element is kept when that
 * word is at least floor(p * 2^32), so it is dropped with probability p (to 2^-32).
 * This is the reading taken for the RNG, which the pages do not specify.
 */
static uint32_t drop_threshold(double p) {
    const double t = floor(p * 4294967296.0);
    return t >= 4294967295.0 ? 4294967295u : (uint32_t)t;
}

static int dropout_keep(uint64_t seed, uint64_t offset, uint32_t thr, uint64_t i) {
    const uint64_t blk = i >> 2;
    const uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)offset,
                             (uint32_t)(offset >> 32)};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32(ctr, key, out);
    return out[i & 3] >= thr;
}

void oracle_dropout_mask(uint64_t seed, uint64_t offset, double p, int64_t rows, int64_t cols,
                         uint8_t* keep, int nthreads) {
    set_threads(nthreads);
    const uint32_t thr = drop_threshold(p);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < cols; ++j)
            keep[r * cols + j] = (uint8_t)dropout_keep(seed, offset, thr, (uint64_t)(r * cols + j));
}

/*
 * Bias + dropout + residual, the prologue fused into the LayerNorm forward ("Accelerating
 * Transformer on GPU (I)", section 2.3: after a linear layer, add the bias, apply dropout,
 * add the residual).  With keep from oracle_dropout_mask:
 *    s = res + keep * (h + bias) / (1 - p)     (rounded to `io`, written as res_out)
 * followed by the LayerNorm of s exactly as oracle_ln_fwd.
 */
void oracle_bdr_ln_fwd(const double* h, const double* bias, const double* res,
                       const double* gamma, const double* beta, double eps, double p,
                       uint64_t seed, uint64_t offset, int64_t rows, int64_t cols, int io,
                       double* out, double* res_out, double* mean, double* rstd, int nthreads) {
    double* s = (double*)malloc((size_t)(rows * cols) * sizeof(double));
    if (!s) return;
    set_threads(nthreads);
    const uint32_t thr = drop_threshold(p);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < cols; ++j) {
            const int64_t i = r * cols + j;
            const double v = dropout_keep(seed, offset, thr, (uint64_t)i) ? (h[i] + bias[j]) / (1.0 - p)
                                                                          : 0.0;
            s[i] = round_io(res[i] + v, io);
        }
    oracle_ln_fwd(s, NULL, gamma, beta, eps, rows, cols, io, out, res_out, mean, rstd, nthreads);
    free(s);
}

/*
 * Backward of the prologue: ds is the gradient with respect to s (the LayerNorm backward's
 * dx); the residual's gradient is ds itself, and
 *    dh = ds * keep / (1 - p),   dbias = sum over rows of dh
 * (dh rounded to `io`; dbias summed unrounded in row order, then rounded).
 */
void oracle_dropout_bwd(const double* ds, double p, uint64_t seed, uint64_t offset, int64_t rows,
                        int64_t cols, int io, double* dh, double* dbias, int nthreads) {
    set_threads(nthreads);
    const uint32_t thr = drop_threshold(p);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < cols; ++j) {
        double acc = 0.0;
        for (int64_t r = 0; r < rows; ++r) {
            const int64_t i = r * cols + j;
            const double v = dropout_keep(seed, offset, thr, (uint64_t)i) ? ds[i] / (1.0 - p) : 0.0;
            if (dh) dh[i] = round_io(v, io);
            acc += v;
        }
        if (dbias) dbias[j] = round_io(acc, io);
    }
}
