// Variant 0, small problems: Conv3d -> activation -> GroupNorm / InstanceNorm
// / none -> spatial mean for batches too small to fill the persistent
// kernels.
//
// Method (l2_p27): the mean over D, H, W of a normalized channel c is
//   gamma_c (m_c - mu_g) / sqrt(var_g + eps) + beta_c,
// m_c the channel's spatial mean, mu_g and var_g the mean and population
// variance over the group's channels and positions; the conv output is never
// written.  The persistent kernels pay a ramp of tens of microseconds (the
// first item's copy, conversion and MMAs in series) that a small batch never
// amortizes.  Here the work of each (sample, normalization group) is split by
// output rows over `nsplit` CTAs, so the grid spreads over the SMs: a CTA
// stages the input planes its rows need and the group's filter in shared
// memory, computes the group's channels at its positions, and keeps
// per-channel sums about values of its own data (each thread's first one,
// then the warp's and the CTA's, moved by the identities below).  Its partial (count,
// K, S1, S2) goes to a slot; the CTA that takes the group's last ticket
// (acquire-release) moves every partial to the first one's shift by the exact
// identities
// S1' = S1 + n d, S2' = S2 + d (2 S1 + n d) (d = K - K0), adds them in split
// order and writes the group's results.  Deterministic; fp32 throughout.
#include "cn_common.cuh"
#include "cn_internal.h"

#include <algorithm>
#include <cstdlib>

namespace cn {
namespace {

constexpr int kSmallThreads = 128;

CN_DEV int small_ticket(int *p) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;\n" : "=r"(old) : "l"(p) : "memory");
    return old;
}

template <int K, int CPG>
__global__ void __launch_bounds__(kSmallThreads) k_conv3d_mean_small(const __grid_constant__ Mean3dArgs a) {
    extern __shared__ __align__(16) float sm[];
    __shared__ float4 s_red[kSmallThreads / 32][CPG];  // per warp (count, K, S1, S2)
    __shared__ int s_last;
    constexpr int T = K * K * K;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ns = a.sm_nsplit;
    const int split = blockIdx.x % ns, ng = blockIdx.x / ns;  // ng = n * ngroups + group
    const int n = ng / a.sm_ngrp, grp = ng - n * a.sm_ngrp;
    const int c0 = grp * CPG;
    // this CTA's output rows (od, oh) and the input planes they read
    const int rows = a.Do * a.Ho;
    const int r0 = (int)((long long)rows * split / ns), r1 = (int)((long long)rows * (split + 1) / ns);
    const int pl0 = r0 / a.Ho, pl1 = (r1 - 1) / a.Ho + K;  // input planes [pl0, pl1)
    const int plane = a.H * a.W, np = pl1 - pl0;
    float *xs = sm;                                               // [Ci][np][H][W]
    float *ws = xs + (((size_t)a.Ci * np * plane + 3) & ~(size_t)3);  // [Ci * T][CPG]

    // ---- stage the planes and the group's filter ----
    // the planes of an input channel are one contiguous run: one bulk async
    // copy each (16-byte multiples), plain loads otherwise
    __shared__ __align__(8) uint64_t s_bar;
    const bool bulk = (plane & 3) == 0 && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
    if (bulk && tid == 0) {
        mbar_init(&s_bar, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(&s_bar, (uint32_t)(a.Ci * np * plane * 4));
        for (int ci = 0; ci < a.Ci; ++ci)
            bulk_load(xs + (size_t)ci * np * plane, a.x + (((size_t)n * a.Ci + ci) * a.D + pl0) * plane,
                      (uint32_t)(np * plane * 4), &s_bar);
    }
    if (!bulk) {
        for (int ci = 0; ci < a.Ci; ++ci) {
            const float *src = a.x + (((size_t)n * a.Ci + ci) * a.D + pl0) * plane;
            float *dst = xs + (size_t)ci * np * plane;
            for (int i = tid; i < np * plane; i += blockDim.x) dst[i] = __ldg(src + i);
        }
    }
    for (int e = tid; e < a.Ci * T * CPG; e += blockDim.x) {
        const int c = e % CPG, ct = e / CPG;  // ct = ci * T + tap
        ws[e] = __ldg(a.w + (size_t)(c0 + c) * a.Ci * T + ct);
    }
    __syncthreads();  // (also: the barrier is initialised before anyone waits on it)
    if (bulk && !mbar_wait_bounded(&s_bar, 0, kWaitLimitNs)) {
        flag_error(a.err, ERR_TIMEOUT);
        mbar_wait_bounded(&s_bar, 0, kWaitLimitNs);  // the copy lands before the CTA moves on
    }

    float bias[CPG];
#pragma unroll
    for (int c = 0; c < CPG; ++c) bias[c] = a.b ? __ldg(a.b + c0 + c) : 0.0f;
    const int P0 = r0 * a.Wo, P1 = r1 * a.Wo;  // this CTA's positions
    // Two threads per position (lanes 2i and 2i + 1 of a warp): thread h
    // takes the (input channel, kd) slices h, h + 2, ... of the taps, so each
    // chain of dependent multiply-adds is half as long; the halves are added
    // by one shuffle.
    auto conv_half = [&](int p, int h, float (&acc)[CPG]) {
        const int ow = p % a.Wo, t = p / a.Wo, oh = t % a.Ho, od = t / a.Ho;
#pragma unroll
        for (int c = 0; c < CPG; ++c) acc[c] = 0.0f;
        for (int j = h; j < a.Ci * K; j += 2) {
            const int ci = j / K, kd = j - ci * K;
            const float *xb = xs + ((size_t)ci * np + (od - pl0 + kd)) * plane + oh * a.W + ow;
            const float *wb = ws + ((size_t)ci * T + kd * K * K) * CPG;
#pragma unroll
            for (int kh = 0; kh < K; ++kh)
#pragma unroll
                for (int kw = 0; kw < K; ++kw) {
                    const float xv = xb[kh * a.W + kw];
#pragma unroll
                    for (int c = 0; c < CPG; ++c) acc[c] = fmaf(xv, wb[(kh * K + kw) * CPG + c], acc[c]);
                }
        }
    };
    // Each thread sums about its own first value (a value of the data, so
    // nothing cancels); the sums then move to the warp's shift (its lowest
    // lane with values) and the CTA's (its first warp with values) by the
    // exact identities S1' = S1 + n d, S2' = S2 + d (2 S1 + n d), d = K - K'.
    float kt[CPG], s1[CPG], s2[CPG];
#pragma unroll
    for (int c = 0; c < CPG; ++c) {
        kt[c] = 0.0f;
        s1[c] = 0.0f;
        s2[c] = 0.0f;
    }
    int nt = 0;
    const int h = tid & 1;
    for (int pb = P0; pb < P1; pb += (int)(blockDim.x >> 1)) {  // uniform: every lane shuffles
        const int p = pb + (tid >> 1);
        float acc[CPG];
        if (p < P1) {
            conv_half(p, h, acc);
        } else {
#pragma unroll
            for (int c = 0; c < CPG; ++c) acc[c] = 0.0f;
        }
#pragma unroll
        for (int c = 0; c < CPG; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 1);
        if (p < P1 && h == 0) {
#pragma unroll
            for (int c = 0; c < CPG; ++c) acc[c] = apply_act(a.act, acc[c] + bias[c]);
            if (nt == 0)
#pragma unroll
                for (int c = 0; c < CPG; ++c) kt[c] = acc[c];
            ++nt;
#pragma unroll
            for (int c = 0; c < CPG; ++c) {
                const float d = acc[c] - kt[c];
                s1[c] += d;
                s2[c] = fmaf(d, d, s2[c]);
            }
        }
    }
    const unsigned has = __ballot_sync(0xffffffffu, nt > 0);
    const int src = has ? __ffs(has) - 1 : 0;
#pragma unroll
    for (int c = 0; c < CPG; ++c) {
        const float kw = __shfl_sync(0xffffffffu, kt[c], src);
        const float d = nt > 0 ? kt[c] - kw : 0.0f;
        s2[c] += d * fmaf((float)nt, d, 2.0f * s1[c]);
        s1[c] = fmaf((float)nt, d, s1[c]);
        kt[c] = kw;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nt += __shfl_xor_sync(0xffffffffu, nt, o);
#pragma unroll
    for (int c = 0; c < CPG; ++c)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            s1[c] += __shfl_xor_sync(0xffffffffu, s1[c], o);
            s2[c] += __shfl_xor_sync(0xffffffffu, s2[c], o);
        }
    if (lane == 0)
#pragma unroll
        for (int c = 0; c < CPG; ++c) s_red[warp][c] = make_float4((float)nt, kt[c], s1[c], s2[c]);
    __syncthreads();
    // the CTA's partial per channel (warps added in order), then its ticket
    float4 *part = reinterpret_cast<float4 *>(a.partial) + (size_t)ng * ns * CPG;
    if (tid < CPG) {
        float Kc = 0.0f, S1 = 0.0f, S2 = 0.0f;
        bool have = false;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            const float4 t = s_red[w][tid];
            if (!(t.x > 0.0f)) continue;
            if (!have) Kc = t.y;
            have = true;
            const float d = t.y - Kc;
            S2 += t.w + d * fmaf(t.x, d, 2.0f * t.z);
            S1 += fmaf(t.x, d, t.z);
        }
        if (CN_CHECK(ng < a.N * a.sm_ngrp, a.err))
            part[(size_t)split * CPG + tid] = make_float4((float)(P1 - P0), Kc, S1, S2);
    }
    __syncthreads();
    // the acquire-release ticket publishes the partial (ordered before it by
    // the barrier) and, for the last CTA, makes every other partial visible
    if (tid == 0) s_last = small_ticket(a.tickets + ng) == ns - 1;
    __syncthreads();
    if (!s_last) return;
    // ---- the group's last CTA: merge the splits, write the results ----
    // every partial to shared memory at once (the input planes are done with)
    float4 *sp = reinterpret_cast<float4 *>(sm);
    for (int i = tid; i < ns * CPG; i += blockDim.x) sp[i] = __ldcg(part + i);
    if (tid == 0) a.tickets[ng] = 0;  // ready for the next launch
    __syncthreads();
    // fp32 throughout: every partial is a sum about a value of its own data,
    // so the merge has no cancellation to guard against, and this GPU's FP64
    // pipe would make the few divisions and the square root of the finish
    // cost tens of microseconds
    float *smc = reinterpret_cast<float *>(sp + ns * CPG);  // [CPG] means, [CPG] M2
    const float cnt = (float)rows * (float)a.Wo;
    if (tid < CPG) {
        const float k0 = sp[tid].y;
        float S1 = 0.0f, S2 = 0.0f;
        for (int s = 0; s < ns; ++s) {
            const float4 q = sp[s * CPG + tid];
            const float d = q.y - k0;
            S1 += fmaf(q.x, d, q.z);
            S2 += fmaf(d, fmaf(q.x, d, 2.0f * q.z), q.w);
        }
        const float mu_s = S1 / cnt;
        smc[tid] = k0 + mu_s;
        smc[CPG + tid] = fmaxf(S2 - S1 * mu_s, 0.0f);
    }
    __syncthreads();
    if (tid >= CPG) return;
    float mu = 0.0f, rstd = 1.0f;
    if (a.norm != CN_NORM_NONE) {
#pragma unroll
        for (int c = 0; c < CPG; ++c) mu += smc[c];
        mu /= (float)CPG;
        float m2 = 0.0f;
#pragma unroll
        for (int c = 0; c < CPG; ++c) m2 += smc[CPG + c] + cnt * (smc[c] - mu) * (smc[c] - mu);
        rstd = rsqrtf(m2 / (cnt * CPG) + a.eps);
    }
    float val = smc[tid];
    if (a.norm != CN_NORM_NONE) {
        const float ga = a.affine ? a.gamma[c0 + tid] : 1.0f;
        const float be = a.affine ? a.beta[c0 + tid] : 0.0f;
        val = ga * (smc[tid] - mu) * rstd + be;
    }
    if (CN_CHECK(n < a.N && c0 + tid < a.Co, a.err)) a.out[(size_t)n * a.Co + c0 + tid] = val * a.post_scale;
}

struct SmallInst {
    int K, CPG;
    Mean3dKernel fn;
    const char *name;
};
#define CN_SMALL(K, C) {K, C, k_conv3d_mean_small<K, C>, "k_conv3d_mean_small<" #K "," #C ">"}
const SmallInst kSmall[] = {CN_SMALL(1, 1), CN_SMALL(2, 1), CN_SMALL(3, 1), CN_SMALL(4, 1),
                            CN_SMALL(1, 2), CN_SMALL(2, 2), CN_SMALL(3, 2), CN_SMALL(4, 2),
                            CN_SMALL(1, 4), CN_SMALL(2, 4), CN_SMALL(3, 4), CN_SMALL(4, 4),
                            CN_SMALL(1, 8), CN_SMALL(2, 8), CN_SMALL(3, 8), CN_SMALL(4, 8)};
#undef CN_SMALL

}  // namespace

// Plans the small-problem kernel: Conv3d (groups 1) -> mean with 1, 2, 4 or 8
// channels per normalization group (InstanceNorm and no norm: one channel per
// CTA), up to ~16 M multiply-adds in all (beyond that the persistent kernels
// are faster).  The splits give each CTA at most 64 positions where the rows
// allow (one pass of its 64 thread pairs), and the grid at most about two
// CTAs per SM.
int small3d_plan(const conv_norm_desc &d, Mean3dArgs &a, Mean3dConfig &cfg) {
    if (d.conv != CN_CONV3D || d.groups != 1 || d.red != CN_RED_MEAN_SPATIAL || d.act == CN_ACT_SOFTMAX_C)
        return CN_ERR_UNSUPPORTED;
    if (d.k < 1 || d.k > 4) return CN_ERR_UNSUPPORTED;
    const char *e = getenv("CN_NO_SMALL");
    if (e && atoi(e)) return CN_ERR_UNSUPPORTED;
    const int K = d.k;
    const int Do = d.D - K + 1, Ho = d.H - K + 1, Wo = d.W - K + 1;
    const int cpg = d.norm == CN_NORM_GROUP ? d.C_out / d.num_groups : 1;
    const SmallInst *inst = nullptr;
    for (const SmallInst &in : kSmall)
        if (in.K == K && in.CPG == cpg) inst = &in;
    if (!inst) return CN_ERR_UNSUPPORTED;
    const double macs = (double)d.N * d.C_out * Do * Ho * Wo * d.C_in * K * K * K;
    if (macs > 16.0e6) return CN_ERR_UNSUPPORTED;
    const long long groups = (long long)d.N * (d.C_out / cpg);
    const int rows = Do * Ho;
    // at most 64 positions a CTA where rows allow (one pass of 64 thread pairs)
    const int rows_per = std::max(1, 64 / Wo);
    const long long by_pos = (rows + rows_per - 1) / rows_per;
    // about two CTAs per SM of a 152-SM GPU (a heuristic fixed at plan time,
    // since the workspace depends on it)
    const long long by_grid = std::max(1LL, (2LL * 152 + groups - 1) / std::max(1LL, groups));
    const int nsplit = (int)std::max(1LL, std::min({(long long)rows, by_pos, by_grid}));
    // shared memory: the most input planes one split reads, and the filter
    const int rows_max = (rows + nsplit - 1) / nsplit;
    const int np_max = std::min(d.D, (rows_max + Ho - 1) / Ho + 1 + K - 1);
    const long long smem = std::max((((long long)d.C_in * np_max * d.H * d.W + 3) & ~3LL) * 4 +
                                        (long long)d.C_in * K * K * K * cpg * 4,
                                    (long long)nsplit * cpg * 16 + 2LL * cpg * 4);
    if (smem > 200 * 1024) return CN_ERR_UNSUPPORTED;
    const long long grid = groups * nsplit;
    if (grid > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;
    a.tc = 0;
    a.small = 1;
    a.sm_cpg = cpg;
    a.sm_ngrp = d.C_out / cpg;
    a.sm_nsplit = nsplit;
    a.N = d.N;
    a.Ci = d.C_in;
    a.Co = d.C_out;
    a.D = d.D;
    a.H = d.H;
    a.W = d.W;
    a.Do = Do;
    a.Ho = Ho;
    a.Wo = Wo;
    a.items = (int)grid;
    a.act = d.act;
    a.norm = d.norm;
    a.G = d.norm == CN_NORM_GROUP ? d.num_groups : d.C_out;
    a.affine = d.affine && d.norm != CN_NORM_NONE;
    a.eps = d.eps;
    a.post_scale = d.post_scale;
    cfg.kern = inst->fn;
    cfg.name = inst->name;
    cfg.K = K;
    cfg.RW = 0;
    cfg.COT = cpg;
    cfg.threads = kSmallThreads;
    cfg.smem = (int)smem;
    cfg.grid = (int)grid;
    return CN_OK;
}

// Partial slots [N][groups][nsplit][channels per group] float4; the per-group
// tickets follow them in the plan's workspace.
size_t small3d_partial_bytes(const Mean3dArgs &a) {
    return (size_t)a.N * a.sm_ngrp * a.sm_nsplit * a.sm_cpg * sizeof(float4);
}

}  // namespace cn
