/*
 * fp64 CPU oracle for the fused convolution + normalization forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or table with the CUDA path.
 *
 * Every routine is the plain definition of one step, written as loops in
 * double precision with no blocking, fusion or reordering.  Each cites the
 * transcript passage it follows.  Transcripts are named by their problem
 * page: l2_p27 (Conv3d -> HardSwish -> GroupNorm -> mean), l2_p17 (Conv2d
 * -> InstanceNorm2d -> divide), l2_p6 (Conv3d -> Softmax -> MaxPool3d x2),
 * l2_p19 (ConvTranspose2d -> GELU -> GroupNorm).
 *
 * Parallelism: OpenMP over independent outputs only (each output value is
 * produced by exactly one thread in a fixed order), so results do not depend
 * on the thread count.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int ocn_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ocn_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Direct 3-D convolution (cross-correlation), stride 1, no padding, with
 * channel groups.  l2_p27 and l2_p6 state the layer as nn.Conv3d with
 * stride 1 and padding 0; the output extent along each axis is L - k + 1.
 *   y[n,co,d,h,w] = b[co] + sum_{ci in group(co)} sum_{a,p,q}
 *                   x[n,ci,d+a,h+p,w+q] * w[co, ci - g*Cig, a, p, q]
 * A 2-D convolution (l2_p17, nn.Conv2d) is the case D = kd = 1.
 * Layouts: x (N,Ci,D,H,W), w (Co,Ci/groups,kd,kh,kw), y (N,Co,Do,Ho,Wo).
 */
void ocn_conv3d(const double *x, int N, int Ci, int D, int H, int W,
                const double *w, int Co, int kd, int kh, int kw, int groups,
                const double *b, double *y) {
    const int Do = D - kd + 1, Ho = H - kh + 1, Wo = W - kw + 1;
    const int Cig = Ci / groups, Cog = Co / groups;
    long nco = (long)N * Co;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < nco; ++t) {
        const int n = (int)(t / Co), co = (int)(t % Co);
        const int g = co / Cog;
        for (int d = 0; d < Do; ++d)
            for (int h = 0; h < Ho; ++h)
                for (int ww = 0; ww < Wo; ++ww) {
                    double acc = b ? b[co] : 0.0;
                    for (int cl = 0; cl < Cig; ++cl) {
                        const int ci = g * Cig + cl;
                        for (int a = 0; a < kd; ++a)
                            for (int p = 0; p < kh; ++p)
                                for (int q = 0; q < kw; ++q) {
                                    double xv = x[((((long)n * Ci + ci) * D + d + a) * H + h + p) * W + ww + q];
                                    double wv = w[((((long)co * Cig + cl) * kd + a) * kh + p) * kw + q];
                                    acc += xv * wv;
                                }
                    }
                    y[((((long)n * Co + co) * Do + d) * Ho + h) * Wo + ww] = acc;
                }
    }
}

/*
 * 2-D transposed convolution, stride 1, padding 0, output padding 0,
 * dilation 1, with channel groups (l2_p19, nn.ConvTranspose2d).  The
 * transcript derives it as the adjoint of the stride-1 convolution: each
 * output gathers input values at i - kh, j - kw with the stored kernel used
 * unflipped; indices outside the input contribute zero.  Output extent is
 * (L - 1) * 1 - 0 + (k - 1) + 0 + 1 = L + k - 1.  PyTorch's weight layout
 * for the transposed layer is (C_in, C_out/groups, kH, kW).
 *   y[n,co,i,j] = b[co] + sum_{ci in group(co)} sum_{p,q}
 *                 x[n,ci,i-p,j-q] * w[ci, co - g*Cog, p, q]
 */
void ocn_conv_transpose2d(const double *x, int N, int Ci, int H, int W,
                          const double *w, int Co, int k, int groups,
                          const double *b, double *y) {
    const int Ho = H + k - 1, Wo = W + k - 1;
    const int Cig = Ci / groups, Cog = Co / groups;
    long nco = (long)N * Co;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < nco; ++t) {
        const int n = (int)(t / Co), co = (int)(t % Co);
        const int g = co / Cog, col = co - g * Cog;
        for (int i = 0; i < Ho; ++i)
            for (int j = 0; j < Wo; ++j) {
                double acc = b ? b[co] : 0.0;
                for (int cl = 0; cl < Cig; ++cl) {
                    const int ci = g * Cig + cl;
                    for (int p = 0; p < k; ++p) {
                        const int ii = i - p;
                        if (ii < 0 || ii >= H) continue;
                        for (int q = 0; q < k; ++q) {
                            const int jj = j - q;
                            if (jj < 0 || jj >= W) continue;
                            double xv = x[(((long)n * Ci + ci) * H + ii) * W + jj];
                            double wv = w[(((long)ci * Cog + col) * k + p) * k + q];
                            acc += xv * wv;
                        }
                    }
                }
                y[(((long)n * Co + co) * Ho + i) * Wo + j] = acc;
            }
    }
}

/* HardSwish, l2_p27 (checked there at x = -3 -> 0 and x = 3 -> 3):
 *   hardswish(v) = v * min(max(v + 3, 0), 6) / 6 */
void ocn_hardswish(double *v, long n) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) {
        double r = v[i] + 3.0;
        if (r < 0.0) r = 0.0;
        if (r > 6.0) r = 6.0;
        v[i] = v[i] * r / 6.0;
    }
}

/* GELU in its exact (erf) form, l2_p19: PyTorch's nn.GELU default
 * approximate='none':  gelu(v) = 0.5 * v * (1 + erf(v / sqrt(2))) */
void ocn_gelu_erf(double *v, long n) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i)
        v[i] = 0.5 * v[i] * (1.0 + erf(v[i] / sqrt(2.0)));
}

/* Softmax over the channel axis with the maximum subtracted (l2_p6,
 * torch.softmax(x, dim=1)):  s_c = exp(v_c - max) / sum_c' exp(v_c' - max).
 * v is (N, C, S) with S the flattened spatial extent. */
void ocn_softmax_channels(double *v, int N, int C, long S) {
    long ns = (long)N * S;
#pragma omp parallel for schedule(static)
    for (long t = 0; t < ns; ++t) {
        const long n = t / S, s = t % S;
        double m = -INFINITY;
        for (int c = 0; c < C; ++c) {
            double a = v[((long)n * C + c) * S + s];
            if (a > m) m = a;
        }
        double z = 0.0;
        for (int c = 0; c < C; ++c) z += exp(v[((long)n * C + c) * S + s] - m);
        for (int c = 0; c < C; ++c) {
            long i = ((long)n * C + c) * S + s;
            v[i] = exp(v[i] - m) / z;
        }
    }
}

/*
 * GroupNorm (l2_p27, l2_p19): for every sample n and group g the statistics
 * run over the group's C/G channels and all S spatial positions; the
 * variance is the population (biased) one and eps sits inside the root:
 *   mu = mean(y), var = mean((y - mu)^2)   (two passes)
 *   out = (y - mu) / sqrt(var + eps) * gamma[c] + beta[c]
 * gamma/beta may be NULL (no affine transform).  InstanceNorm (l2_p17,
 * nn.InstanceNorm2d with affine=False) is the case G = C without gamma/beta.
 */
void ocn_group_norm(const double *y, int N, int C, long S, int G, double eps,
                    const double *gamma, const double *beta, double *out) {
    const int cpg = C / G;
    long ng = (long)N * G;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < ng; ++t) {
        const long n = t / G, g = t % G;
        const long base = (n * C + g * cpg) * S;
        const long cnt = (long)cpg * S;
        double s = 0.0;
        for (long i = 0; i < cnt; ++i) s += y[base + i];
        const double mu = s / (double)cnt;
        double q = 0.0;
        for (long i = 0; i < cnt; ++i) {
            double d = y[base + i] - mu;
            q += d * d;
        }
        const double var = q / (double)cnt;
        const double inv = 1.0 / sqrt(var + eps);
        for (int cl = 0; cl < cpg; ++cl) {
            const int c = (int)g * cpg + cl;
            const double ga = gamma ? gamma[c] : 1.0;
            const double be = beta ? beta[c] : 0.0;
            for (long i = 0; i < S; ++i) {
                long idx = base + (long)cl * S + i;
                out[idx] = (y[idx] - mu) * inv * ga + be;
            }
        }
    }
}

/* Multiply every value by a constant (l2_p17 divides by 2.0; the workload
 * states it as a multiplication by 0.5, the same in binary floating point). */
void ocn_scale(double *v, long n, double s) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) v[i] *= s;
}

/* Mean over all spatial positions (l2_p27: torch.mean over D, H, W):
 * v is (N, C, S) -> out (N, C). */
void ocn_mean_spatial(const double *v, int N, int C, long S, double *out) {
    long nc = (long)N * C;
#pragma omp parallel for schedule(static)
    for (long t = 0; t < nc; ++t) {
        double s = 0.0;
        for (long i = 0; i < S; ++i) s += v[t * S + i];
        out[t] = s / (double)S;
    }
}

/* MaxPool3d(kernel 2, stride 2, padding 0, floor mode) (l2_p6): output
 * extent floor(L / 2) per axis; a trailing odd slice is dropped.
 * v (N, C, D, H, W) -> out (N, C, D/2, H/2, W/2). */
void ocn_maxpool3d_2(const double *v, int N, int C, int D, int H, int W,
                     double *out) {
    const int Dp = D / 2, Hp = H / 2, Wp = W / 2;
    long nc = (long)N * C;
#pragma omp parallel for schedule(static)
    for (long t = 0; t < nc; ++t) {
        for (int d = 0; d < Dp; ++d)
            for (int h = 0; h < Hp; ++h)
                for (int w = 0; w < Wp; ++w) {
                    double m = -INFINITY;
                    for (int a = 0; a < 2; ++a)
                        for (int p = 0; p < 2; ++p)
                            for (int q = 0; q < 2; ++q) {
                                double e = v[((t * D + 2 * d + a) * (long)H + 2 * h + p) * W + 2 * w + q];
                                if (e > m) m = e;
                            }
                    out[((t * Dp + d) * (long)Hp + h) * Wp + w] = m;
                }
    }
}

/* ---------------------------------------------------------------------------
 * Backward pass (the gradient of a scalar loss L through the same layers).
 * The pages treat only the forward; each routine below is the derivative of
 * the forward routine it names, written out as plain loops, with dy the
 * gradient of L with respect to that routine's output.
 * ------------------------------------------------------------------------- */

/* Gradient of ocn_conv3d with respect to its input:
 *   dx[n,ci,z,h,w] = sum_{co in group(ci)} sum_{a,p,q} dy[n,co,z-a,h-p,w-q] * w[co, ci - g*Cig, a, p, q]
 * over the output positions that exist (0 <= z-a < Do, ...). */
void ocn_conv3d_grad_input(const double *dy, int N, int Co, int Do, int Ho, int Wo,
                           const double *w, int Ci, int kd, int kh, int kw, int groups,
                           double *dx) {
    const int D = Do + kd - 1, H = Ho + kh - 1, W = Wo + kw - 1;
    const int Cig = Ci / groups, Cog = Co / groups;
    long nci = (long)N * Ci;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < nci; ++t) {
        const int n = (int)(t / Ci), ci = (int)(t % Ci);
        const int g = ci / Cig, cl = ci - g * Cig;
        for (int z = 0; z < D; ++z)
            for (int h = 0; h < H; ++h)
                for (int x = 0; x < W; ++x) {
                    double acc = 0.0;
                    for (int j = 0; j < Cog; ++j) {
                        const int co = g * Cog + j;
                        for (int a = 0; a < kd; ++a) {
                            const int zo = z - a;
                            if (zo < 0 || zo >= Do) continue;
                            for (int p = 0; p < kh; ++p) {
                                const int ho = h - p;
                                if (ho < 0 || ho >= Ho) continue;
                                for (int q = 0; q < kw; ++q) {
                                    const int xo = x - q;
                                    if (xo < 0 || xo >= Wo) continue;
                                    acc += dy[((((long)n * Co + co) * Do + zo) * Ho + ho) * Wo + xo] *
                                           w[((((long)co * Cig + cl) * kd + a) * kh + p) * kw + q];
                                }
                            }
                        }
                    }
                    dx[((((long)n * Ci + ci) * D + z) * H + h) * W + x] = acc;
                }
    }
}

/* Gradient of ocn_conv3d with respect to its weight and bias:
 *   dw[co, cl, a, p, q] = sum_{n, z, h, x} dy[n,co,z,h,x] * x[n, g*Cig + cl, z+a, h+p, x+q]
 *   db[co] = sum_{n, z, h, x} dy[n,co,z,h,x]            (db may be NULL) */
void ocn_conv3d_grad_weight(const double *x, int N, int Ci, int D, int H, int W,
                            const double *dy, int Co, int kd, int kh, int kw, int groups,
                            double *dw, double *db) {
    const int Do = D - kd + 1, Ho = H - kh + 1, Wo = W - kw + 1;
    const int Cig = Ci / groups, Cog = Co / groups;
#pragma omp parallel for schedule(dynamic, 1)
    for (int co = 0; co < Co; ++co) {
        const int g = co / Cog;
        for (int cl = 0; cl < Cig; ++cl) {
            const int ci = g * Cig + cl;
            for (int a = 0; a < kd; ++a)
                for (int p = 0; p < kh; ++p)
                    for (int q = 0; q < kw; ++q) {
                        double acc = 0.0;
                        for (int n = 0; n < N; ++n)
                            for (int z = 0; z < Do; ++z)
                                for (int h = 0; h < Ho; ++h)
                                    for (int xo = 0; xo < Wo; ++xo)
                                        acc += dy[((((long)n * Co + co) * Do + z) * Ho + h) * Wo + xo] *
                                               x[((((long)n * Ci + ci) * D + z + a) * H + h + p) * W + xo + q];
                        dw[((((long)co * Cig + cl) * kd + a) * kh + p) * kw + q] = acc;
                    }
        }
        if (db) {
            double s = 0.0;
            for (int n = 0; n < N; ++n)
                for (long i = 0; i < (long)Do * Ho * Wo; ++i) s += dy[((long)n * Co + co) * Do * Ho * Wo + i];
            db[co] = s;
        }
    }
}

/* Gradient of ocn_conv_transpose2d with respect to its input:
 *   dx[n,ci,ii,jj] = sum_{co in group(ci)} sum_{p,q} dy[n,co,ii+p,jj+q] * w[ci, co - g*Cog, p, q] */
void ocn_conv_transpose2d_grad_input(const double *dy, int N, int Co, int H, int W,
                                     const double *w, int Ci, int k, int groups, double *dx) {
    const int Ho = H + k - 1, Wo = W + k - 1;
    const int Cig = Ci / groups, Cog = Co / groups;
    long nci = (long)N * Ci;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < nci; ++t) {
        const int n = (int)(t / Ci), ci = (int)(t % Ci);
        const int g = ci / Cig;
        for (int ii = 0; ii < H; ++ii)
            for (int jj = 0; jj < W; ++jj) {
                double acc = 0.0;
                for (int col = 0; col < Cog; ++col) {
                    const int co = g * Cog + col;
                    for (int p = 0; p < k; ++p)
                        for (int q = 0; q < k; ++q)
                            acc += dy[(((long)n * Co + co) * Ho + ii + p) * Wo + jj + q] *
                                   w[(((long)ci * Cog + col) * k + p) * k + q];
                }
                dx[(((long)n * Ci + ci) * H + ii) * W + jj] = acc;
            }
    }
}

/* Gradient of ocn_conv_transpose2d with respect to its weight and bias:
 *   dw[ci, col, p, q] = sum_{n, ii, jj} x[n,ci,ii,jj] * dy[n, g*Cog + col, ii+p, jj+q]
 *   db[co] = sum_{n, i, j} dy[n,co,i,j]                  (db may be NULL) */
void ocn_conv_transpose2d_grad_weight(const double *x, int N, int Ci, int H, int W,
                                      const double *dy, int Co, int k, int groups,
                                      double *dw, double *db) {
    const int Ho = H + k - 1, Wo = W + k - 1;
    const int Cig = Ci / groups, Cog = Co / groups;
#pragma omp parallel for schedule(dynamic, 1)
    for (int ci = 0; ci < Ci; ++ci) {
        const int g = ci / Cig;
        for (int col = 0; col < Cog; ++col) {
            const int co = g * Cog + col;
            for (int p = 0; p < k; ++p)
                for (int q = 0; q < k; ++q) {
                    double acc = 0.0;
                    for (int n = 0; n < N; ++n)
                        for (int ii = 0; ii < H; ++ii)
                            for (int jj = 0; jj < W; ++jj)
                                acc += x[(((long)n * Ci + ci) * H + ii) * W + jj] *
                                       dy[(((long)n * Co + co) * Ho + ii + p) * Wo + jj + q];
                    dw[(((long)ci * Cog + col) * k + p) * k + q] = acc;
                }
        }
    }
    if (db) {
#pragma omp parallel for schedule(static)
        for (int co = 0; co < Co; ++co) {
            double s = 0.0;
            for (int n = 0; n < N; ++n)
                for (long i = 0; i < (long)Ho * Wo; ++i) s += dy[((long)n * Co + co) * Ho * Wo + i];
            db[co] = s;
        }
    }
}

/* g *= hardswish'(v): 0 below -3, v/3 + 1/2 on [-3, 3], 1 above (the
 * one-sided values PyTorch uses at the two kinks). */
void ocn_hardswish_grad(const double *v, double *g, long n) {
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) {
        const double a = v[i];
        const double d = a < -3.0 ? 0.0 : (a <= 3.0 ? a / 3.0 + 0.5 : 1.0);
        g[i] *= d;
    }
}

/* g *= gelu'(v) for the erf form: Phi(v) + v * phi(v), with Phi the normal
 * CDF 0.5 (1 + erf(v / sqrt(2))) and phi its density exp(-v^2/2)/sqrt(2 pi). */
void ocn_gelu_erf_grad(const double *v, double *g, long n) {
    const double inv_sqrt2pi = 0.39894228040143267794;
#pragma omp parallel for schedule(static)
    for (long i = 0; i < n; ++i) {
        const double a = v[i];
        g[i] *= 0.5 * (1.0 + erf(a / sqrt(2.0))) + a * inv_sqrt2pi * exp(-0.5 * a * a);
    }
}

/*
 * Gradient of ocn_group_norm.  Per (n, g), with M = (C/G) S values, mu and
 * var as in the forward (two passes), r = 1/sqrt(var + eps), xh = (y - mu) r
 * and dxh = dout * gamma[c]:
 *   dy = r (dxh - mean(dxh) - xh mean(dxh xh))
 *   dgamma[c] = sum_{n, s} dout xh,   dbeta[c] = sum_{n, s} dout
 * gamma NULL means 1; dgamma and dbeta may be NULL.
 */
void ocn_group_norm_grad(const double *y, int N, int C, long S, int G, double eps,
                         const double *gamma, const double *dout, double *dy,
                         double *dgamma, double *dbeta) {
    const int cpg = C / G;
    const long cnt = (long)cpg * S;
    double *xh_all = (double *)malloc(sizeof(double) * (size_t)N * C * S);
    long ng = (long)N * G;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < ng; ++t) {
        const long n = t / G, g = t % G;
        const long base = (n * C + g * cpg) * S;
        double s = 0.0;
        for (long i = 0; i < cnt; ++i) s += y[base + i];
        const double mu = s / (double)cnt;
        double q = 0.0;
        for (long i = 0; i < cnt; ++i) {
            const double d = y[base + i] - mu;
            q += d * d;
        }
        const double r = 1.0 / sqrt(q / (double)cnt + eps);
        double m1 = 0.0, m2 = 0.0;
        for (int cl = 0; cl < cpg; ++cl) {
            const double ga = gamma ? gamma[g * cpg + cl] : 1.0;
            for (long i = 0; i < S; ++i) {
                const long idx = base + (long)cl * S + i;
                const double xh = (y[idx] - mu) * r;
                xh_all[idx] = xh;
                m1 += dout[idx] * ga;
                m2 += dout[idx] * ga * xh;
            }
        }
        m1 /= (double)cnt;
        m2 /= (double)cnt;
        for (int cl = 0; cl < cpg; ++cl) {
            const double ga = gamma ? gamma[g * cpg + cl] : 1.0;
            for (long i = 0; i < S; ++i) {
                const long idx = base + (long)cl * S + i;
                dy[idx] = r * (dout[idx] * ga - m1 - xh_all[idx] * m2);
            }
        }
    }
    if (dgamma || dbeta) {
#pragma omp parallel for schedule(static)
        for (int c = 0; c < C; ++c) {
            double sg = 0.0, sb = 0.0;
            for (int n = 0; n < N; ++n)
                for (long i = 0; i < S; ++i) {
                    const long idx = ((long)n * C + c) * S + i;
                    sg += dout[idx] * xh_all[idx];
                    sb += dout[idx];
                }
            if (dgamma) dgamma[c] = sg;
            if (dbeta) dbeta[c] = sb;
        }
    }
    free(xh_all);
}
