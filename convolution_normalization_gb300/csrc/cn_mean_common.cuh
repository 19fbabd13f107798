// Per-sample finish of the spatial-mean variant, shared by its CUDA-core and
// tensor-core kernels: the last CTA to finish a chunk of sample n merges the
// chunks' per-channel moments (fixed chunk order, fp64) and writes the
// sample's (C_out) result.
//
// Method (l2_p27, Conv3d -> HardSwish -> GroupNorm -> mean): the spatial mean
// of a GroupNorm output of channel c is
//   gamma_c * (m_c - mu_g) / sqrt(var_g + eps) + beta_c,
// m_c the channel's spatial mean, mu_g and var_g the population mean and
// variance over the group's channels and positions.
#pragma once
#include "cn_common.cuh"
#include "cn_internal.h"

namespace cn {

// Moments of channel c of sample n, merged over its nchunks chunks in chunk
// order (partial[N][nchunks][Co][3]).
template <class Args>
CN_DEV Moments<double> mean_chunks_merged(const Args &a, int nchunks, int n, int c) {
    Moments<double> m{0.0, 0.0, 0.0};
    for (int ch = 0; ch < nchunks; ++ch) {
        const double *p = a.partial + (((size_t)n * nchunks + ch) * a.Co + c) * 3;
        m = merge(m, Moments<double>{ldcg_f64(p), ldcg_f64(p + 1), ldcg_f64(p + 2)});
    }
    return m;
}

// Output of channel c of sample n from every channel's merged moments,
// sch[Co][3] = (count, mean, M2).
template <class Args>
CN_DEV void mean_write_output(const Args &a, int n, int c, const double *sch) {
    const double mc = sch[c * 3 + 1];
    double val;
    if (a.norm == CN_NORM_NONE) {
        val = mc;
    } else {
        const int cpg = a.Co / a.G, g = c / cpg;
        Moments<double> mg{0.0, 0.0, 0.0};
        for (int u = 0; u < cpg; ++u) {
            const int cc = g * cpg + u;
            mg = merge(mg, Moments<double>{sch[cc * 3], sch[cc * 3 + 1], sch[cc * 3 + 2]});
        }
        const double var = mg.m2 / mg.n;
        const double rstd = 1.0 / sqrt(var + (double)a.eps);
        const double ga = a.affine ? (double)a.gamma[c] : 1.0;
        const double be = a.affine ? (double)a.beta[c] : 0.0;
        val = ga * (mc - mg.mean) * rstd + be;
    }
    if (CN_CHECK(n < a.N && c < a.Co, a.err)) a.out[(size_t)n * a.Co + c] = (float)(val * (double)a.post_scale);
}

}  // namespace cn
