// Backward pass of the full-output 2-D block: Conv2d or ConvTranspose2d
// (groups) -> activation (none, HardSwish, GELU) -> GroupNorm / InstanceNorm
// / none -> post scale.  The pages state only the forward; the gradients are
// the derivatives of that forward (the chain rule through each layer).
//
// Given dout = dL/d(out), with A the conv output (pre-activation), y = act(A),
// per (n, group) mu, r = 1/sqrt(var + eps), xh = (y - mu) r, and s the post
// scale:
//   dxh   = s gamma_c dout
//   dy    = r (dxh - mean(dxh) - xh mean(dxh xh))        (mean over the group)
//   dA    = dy act'(A)
//   dgamma_c = s sum_{n,p} dout xh,  dbeta_c = s sum_{n,p} dout,  db_co = sum dA
//   dx    = the adjoint conv of dA with the same weights (a transposed conv for
//           Conv2d, a conv for ConvTranspose2d)
//   dw    = the correlation of dA with x over every sample and position.
//
// Steps (one stream, all deterministic):
//   1. A: the forward plan of the conv alone (no activation, norm or scale);
//   2. k_bwd_plane_sums: per (n, c) plane, sums about the plane's first value
//      y0: count, sum(y - y0), sum (y - y0)^2, sum dout, sum dout (y - y0);
//   3. k_bwd_group: per (n, group) the planes merge at one shift (exact
//      identities), giving mu, r and the two group means above; per (n, c)
//      the coefficients of dy = a dout + b + c (y - mu) and the plane's
//      dgamma / dbeta terms;
//   4. k_bwd_dA: dA in place of A, and per-plane-slice sums for db;
//   5. dx: the forward plan of the adjoint conv on dA; for Conv2d the
//      tensor-core Conv2d plan of the zero-padded dA with the turned filter
//      (k_bwd_pad, k_bwd_wadj, then k_bwd_crop); k_bwd_dx_g8 for a
//      ConvTranspose2d with 8 channels a group;
//   6. k_bwd_weight: dw as a GEMM over all positions (split over the
//      positions), or k_bwd_weight_win for groups of 8 channels (the k x k
//      window slid along rows); fixed-order sum of the splits in
//      k_bwd_weight_sum;
//   7. k_bwd_channel_sums: dgamma, dbeta and db, summed over n in order.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>

#include "cn_common.cuh"
#include "cn_internal.h"

namespace cn {
namespace {

constexpr int kBwdThreads = 256;

// Copies 8 bytes global -> shared; when !pred the destination is zero-filled
// and the source is not read.
CN_DEV void cp_async8(void *smem, const void *gmem, bool pred) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
                 "r"(pred ? 8 : 0));
}

// act'(a): HardSwish 0 below -3, a/3 + 1/2 on [-3, 3], 1 above; GELU (erf
// form) Phi(a) + a phi(a), erf by Abramowitz & Stegun 7.1.26 as in the
// forward (|error| <= 1.5e-7).
CN_DEV float act_grad(int act, float a) {
    if (act == ACT_HARDSWISH) return a < -3.0f ? 0.0f : (a <= 3.0f ? fmaf(a, 1.0f / 3.0f, 0.5f) : 1.0f);
    if (act == ACT_GELU) {
        const float z = fabsf(a) * 0.70710678118654752f;
        const float t = 1.0f / fmaf(CN_AS_P, z, 1.0f);
        float y = fmaf(t, CN_AS_A5, CN_AS_A4);
        y = fmaf(t, y, CN_AS_A3);
        y = fmaf(t, y, CN_AS_A2);
        y = fmaf(t, y, CN_AS_A1);
        const float e = expf(-0.5f * a * a);
        const float q = y * t * e;  // erfc(|a| / sqrt 2)
        const float Phi = a >= 0.0f ? 1.0f - 0.5f * q : 0.5f * q;
        return fmaf(a * 0.39894228040143268f, e, Phi);
    }
    return 1.0f;
}

// Block sum of kBwdThreads values in a fixed order (warp butterflies, then
// the warps' results in warp order); every thread gets the result.
template <int NV>
CN_DEV void block_sum(float (&v)[NV]) {
    __shared__ float red[kBwdThreads / 32][NV];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v[j] += __shfl_xor_sync(0xffffffffu, v[j], o);
    if (lane == 0)
#pragma unroll
        for (int j = 0; j < NV; ++j) red[warp][j] = v[j];
    __syncthreads();
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        float s = 0.0f;
        for (int w = 0; w < kBwdThreads / 32; ++w) s += red[w][j];
        v[j] = s;
    }
    __syncthreads();
}

// Step 2: one block per (n, c) plane.
__global__ void __launch_bounds__(kBwdThreads) k_bwd_plane_sums(const float *A, const float *dout, long long S,
                                                                int act, float4 *ps) {
    const long long plane = blockIdx.x;
    const float *ap = A + plane * S, *gp = dout + plane * S;
    const float K = apply_act(act, ap[0]);
    float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // sum d, sum d^2, sum g, sum g d
    auto add = [&](float a, float g) {
        const float d = apply_act(act, a) - K;
        v[0] += d;
        v[1] = fmaf(d, d, v[1]);
        v[2] += g;
        v[3] = fmaf(g, d, v[3]);
    };
    if ((S & 3) == 0) {  // planes start on 16 bytes: four values a load
        const float4 *a4 = reinterpret_cast<const float4 *>(ap), *g4 = reinterpret_cast<const float4 *>(gp);
        for (long long i = threadIdx.x; i < S / 4; i += kBwdThreads) {
            const float4 a = a4[i], g = g4[i];
            add(a.x, g.x);
            add(a.y, g.y);
            add(a.z, g.z);
            add(a.w, g.w);
        }
    } else {
        for (long long i = threadIdx.x; i < S; i += kBwdThreads) add(ap[i], gp[i]);
    }
    block_sum<4>(v);
    if (threadIdx.x == 0) {
        ps[2 * plane] = make_float4((float)S, K, v[0], v[1]);
        ps[2 * plane + 1] = make_float4(v[2], v[3], 0.0f, 0.0f);
    }
}

// Step 3: one thread per (n, group), planes in channel order.
__global__ void k_bwd_group(const float4 *ps, int N, int C, int G, int norm, float eps, float scale,
                            const float *gamma, float4 *coef, float2 *gpart) {
    const int ng = blockIdx.x * blockDim.x + threadIdx.x;
    if (ng >= N * G) return;
    const int n = ng / G, g = ng - n * G, cpg = C / G;
    const int c0 = g * cpg;
    if (norm == CN_NORM_NONE) {
        for (int cl = 0; cl < cpg; ++cl) {
            coef[(size_t)n * C + c0 + cl] = make_float4(scale, 0.0f, 0.0f, 0.0f);
            gpart[(size_t)n * C + c0 + cl] = make_float2(0.0f, 0.0f);
        }
        return;
    }
    // (count, K, S1, S2) of the planes moved to the first plane's shift K0
    const float K0 = ps[2 * ((size_t)n * C + c0)].y;
    float M = 0.0f, S1 = 0.0f, S2 = 0.0f;
    for (int cl = 0; cl < cpg; ++cl) {
        const float4 p = ps[2 * ((size_t)n * C + c0 + cl)];
        const float d = p.y - K0;
        S2 += p.w + d * fmaf(p.x, d, 2.0f * p.z);
        S1 += fmaf(p.x, d, p.z);
        M += p.x;
    }
    const float mu_s = S1 / M;  // mu - K0
    const float r = 1.0f / sqrtf(fmaxf(fmaf(-S1, mu_s, S2), 0.0f) / M + eps);
    const float mu = K0 + mu_s;
    // T1 = sum dxh, T2 = sum dxh (y - mu); a plane's sum dout (y - mu) is
    // sum dout (y - K_c) + (K_c - mu) sum dout
    float T1 = 0.0f, T2 = 0.0f;
    for (int cl = 0; cl < cpg; ++cl) {
        const size_t pl = (size_t)n * C + c0 + cl;
        const float4 p0 = ps[2 * pl], p1 = ps[2 * pl + 1];
        const float ga = gamma ? gamma[c0 + cl] : 1.0f;
        const float gy = fmaf(p0.y - mu, p1.x, p1.y);
        T1 = fmaf(scale * ga, p1.x, T1);
        T2 = fmaf(scale * ga, gy, T2);
        gpart[pl] = make_float2(scale * r * gy, scale * p1.x);  // this plane's dgamma, dbeta terms
    }
    const float m1 = T1 / M, m2 = r * T2 / M;  // mean(dxh), mean(dxh xh)
    for (int cl = 0; cl < cpg; ++cl) {
        const float ga = gamma ? gamma[c0 + cl] : 1.0f;
        // dy = r dxh - r m1 - r^2 m2 (y - mu)
        coef[(size_t)n * C + c0 + cl] = make_float4(r * scale * ga, -r * m1, -r * r * m2, mu);
    }
}

// Step 4: dA in place of A over `slices` blocks per plane; each block's sum of dA.
__global__ void __launch_bounds__(kBwdThreads) k_bwd_dA(float *A, const float *dout, const float4 *coef,
                                                        long long S, int act, int slices, float *dbpart) {
    const long long plane = blockIdx.x / slices;
    const int slice = (int)(blockIdx.x - plane * slices);
    const float4 cf = coef[plane];
    // slice bounds on multiples of 4 (the last one ends at S)
    const long long i0 = (S * slice / slices) & ~3LL, i1 = slice + 1 == slices ? S : (S * (slice + 1) / slices) & ~3LL;
    float *ap = A + plane * S;
    const float *gp = dout + plane * S;
    float v[1] = {0.0f};
    auto grad = [&](float a, float g) {
        const float y = act == ACT_NONE ? a : apply_act(act, a);
        const float dy = fmaf(cf.x, g, fmaf(cf.z, y - cf.w, cf.y));
        const float da = act == ACT_NONE ? dy : dy * act_grad(act, a);
        v[0] += da;
        return da;
    };
    if ((S & 3) == 0 && (i0 & 3) == 0 && (i1 & 3) == 0) {  // four values a load
        float4 *a4 = reinterpret_cast<float4 *>(ap);
        const float4 *g4 = reinterpret_cast<const float4 *>(gp);
        for (long long i = i0 / 4 + threadIdx.x; i < i1 / 4; i += kBwdThreads) {
            float4 a = a4[i];
            const float4 g = g4[i];
            a.x = grad(a.x, g.x);
            a.y = grad(a.y, g.y);
            a.z = grad(a.z, g.z);
            a.w = grad(a.w, g.w);
            a4[i] = a;
        }
    } else {
        for (long long i = i0 + threadIdx.x; i < i1; i += kBwdThreads) ap[i] = grad(ap[i], gp[i]);
    }
    block_sum<1>(v);
    if (threadIdx.x == 0) dbpart[plane * slices + slice] = v[0];
}

// Step 6: R[g][m][nn] over positions pos = (n, i, j) of U's planes:
//   R = sum_pos U[n][g CUg + m][i][j] * V[n][g CVg + c][i + p][j + q],  nn = (c, p, q)
// (Conv2d: U = dA, V = x, R = dw[co][ci][p][q]; ConvTranspose2d: U = x, V = dA,
// R = dw[ci][co][p][q]).  A block takes a BM x BN tile of (m, nn) and one
// split of the positions; BK positions per step staged in shared memory; a
// thread owns TM x TN outputs (128 x 128 tiles of 8 x 8 for at least 96
// channels a group, 64 x 64 tiles of 4 x 4 below that, 8 x 128 tiles of
// 1 x 4 for groups of at most 8 channels).  Its split's
// sums go to part[split][g][m][nn].
template <int BM, int BN, int TM, int TN, int BK>
__global__ void __launch_bounds__(kBwdThreads) k_bwd_weight(const float *U, const float *V, int N, int CU, int CV,
                                                            int PH, int PW, int k, int groups, long long kchunk,
                                                            float *part) {
    static_assert((BM / TM) * (BN / TN) == kBwdThreads, "one output tile per thread");
    constexpr int RU = (BM * BK + kBwdThreads - 1) / kBwdThreads;  // U rows a thread loads
    constexpr int RV = BN * BK / kBwdThreads;                      // V rows a thread loads
    constexpr int RS = kBwdThreads / BK;                           // rows a load step covers
    static_assert(kBwdThreads % BK == 0 && (BN * BK) % kBwdThreads == 0, "load mapping");
    __shared__ __align__(16) float Us[BK][BM + 4];
    __shared__ __align__(16) float Vs[BK][BN + 4];
    const int tid = threadIdx.x;
    const int CUg = CU / groups, CVg = CV / groups, kk2 = k * k, NN = CVg * kk2;
    const int mtiles = (CUg + BM - 1) / BM, ntiles = (NN + BN - 1) / BN;
    int bx = blockIdx.x;
    const int mt = bx % mtiles;
    bx /= mtiles;
    const int nt = bx % ntiles;
    const int g = bx / ntiles;
    const long long P = (long long)PH * PW, Ktot = (long long)N * P;
    const long long kbeg = (long long)blockIdx.y * kchunk, kend = Ktot < kbeg + kchunk ? Ktot : kbeg + kchunk;
    const int VH = PH + k - 1, VW = PW + k - 1;
    // this thread's loads: position lane kk, tile rows tid / BK + RS t
    const int kk = tid % BK, r0 = tid / BK;
    long long ub[RU], vb[RV];
    bool uok[RU], vok[RV];
#pragma unroll
    for (int t = 0; t < RU; ++t) {
        const int ml = r0 + RS * t, m = mt * BM + ml;
        uok[t] = ml < BM && m < CUg;
        ub[t] = (long long)(g * CUg + (uok[t] ? m : 0)) * P;
    }
#pragma unroll
    for (int t = 0; t < RV; ++t) {
        const int nn = nt * BN + r0 + RS * t;
        vok[t] = nn < NN;
        const int c = vok[t] ? nn / kk2 : 0, pq = vok[t] ? nn - c * kk2 : 0;
        const int p = pq / k, q = pq - p * k;
        vb[t] = ((long long)(g * CVg + c) * VH + p) * VW + q;
    }
    // the thread's position k0 + kk as (n, i, j), advanced by BK each step
    long long pos = kbeg + kk;
    int n = (int)(pos / P);
    long long rr = pos - (long long)n * P;
    int i = (int)(rr / PW), j = (int)(rr - (long long)i * PW);
    const int ty = tid / (BN / TN), tx = tid % (BN / TN);
    float acc[TM][TN] = {};
    for (long long k0 = kbeg; k0 < kend; k0 += BK) {
        const bool pok = pos < kend;
        const long long uo = (long long)n * CU * P + (long long)i * PW + j;
        const long long vo = (long long)n * CV * VH * VW + (long long)i * VW + j;
#pragma unroll
        for (int t = 0; t < RU; ++t)
            if (r0 + RS * t < BM) Us[kk][r0 + RS * t] = pok && uok[t] ? __ldg(U + ub[t] + uo) : 0.0f;
#pragma unroll
        for (int t = 0; t < RV; ++t) Vs[kk][r0 + RS * t] = pok && vok[t] ? __ldg(V + vb[t] + vo) : 0.0f;
        __syncthreads();
#pragma unroll
        for (int s = 0; s < BK; ++s) {
            float av[TM], bv[TN];
            if (TM % 4 == 0) {
#pragma unroll
                for (int x = 0; x < TM; x += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(&Us[s][ty * TM + x]);
                    av[x] = a4.x;
                    av[x + 1] = a4.y;
                    av[x + 2] = a4.z;
                    av[x + 3] = a4.w;
                }
            } else {
#pragma unroll
                for (int x = 0; x < TM; ++x) av[x] = Us[s][ty * TM + x];
            }
#pragma unroll
            for (int y = 0; y < TN; y += 4) {
                const float4 b4 = *reinterpret_cast<const float4 *>(&Vs[s][tx * TN + y]);
                bv[y] = b4.x;
                bv[y + 1] = b4.y;
                bv[y + 2] = b4.z;
                bv[y + 3] = b4.w;
            }
#pragma unroll
            for (int x = 0; x < TM; ++x)
#pragma unroll
                for (int y = 0; y < TN; ++y) acc[x][y] = fmaf(av[x], bv[y], acc[x][y]);
        }
        __syncthreads();
        pos += BK;
        j += BK;
        while (j >= PW) {
            j -= PW;
            if (++i == PH) {
                i = 0;
                ++n;
            }
        }
    }
    float *pp = part + ((size_t)blockIdx.y * groups + g) * (size_t)CUg * NN;
#pragma unroll
    for (int x = 0; x < TM; ++x) {
        const int m = mt * BM + ty * TM + x;
        if (m >= CUg) continue;
#pragma unroll
        for (int y = 0; y < TN; ++y) {
            const int nn = nt * BN + tx * TN + y;
            if (nn < NN) pp[(size_t)m * NN + nn] = acc[x][y];
        }
    }
}

// positions a step (measured on the l2_p19 and l2_p17 blocks: 16 and 32)
constexpr int kWBKSmall = 16, kWBKWide = 32;

// Step 6 for narrow groups (8 V channels and at most 8 U channels a group,
// k <= 3; the l2_p19 block's ConvTranspose2d: U = x, V = dA): the same R,
// computed with the window slid along the rows instead of as a GEMM.  A
// block takes one (group, sample) and a run of bands of kWinRB U rows; per
// band it stages the band's U rows and the V rows they reach in shared
// memory.  Lane (c, r) of a warp owns the CUG x k x k outputs of V channel c
// for the positions of band row r in the warp's 32-column segments, four
// positions at a time: 16-byte loads of the four positions' U values (the
// same for the warp's 8 channels) and of the k x k V window's four new
// columns feed 4 CUG k^2 multiply-adds.  V rows start k - 1 columns before a
// 16-byte boundary, so those loads are aligned; the pitches put the 16-byte
// loads of every quarter warp on distinct banks (U rows 1 bank group apart,
// V rows 2 and V channels an odd number of groups apart).  Columns the
// staging never writes are zeroed once, so the positions past a row's end
// add zeros.  At the end the block sums its threads' outputs per channel in
// a fixed order and writes them to part[(n, run)][w numel].
constexpr int kWinRB = 4, kWinSeg = 32;
CN_DEV int win_upitch(int PW) { return (PW + 31) / 32 * 32 + 4; }
CN_DEV int win_vpitch(int VW) { return (VW + 31) / 32 * 32 + 8; }
CN_DEV int win_vpad(int K) { return (4 - (K - 1) % 4) % 4; }  // zero columns before a V row

template <int K, int CUG>
__global__ void __launch_bounds__(kBwdThreads, 2) k_bwd_weight_win(const float *U, const float *V, int N, int CU,
                                                                   int CV, int PH, int PW, int nrun, int bpr,
                                                                   float *part) {
    constexpr int CVG = 8, KK = K * K, NO = CUG * KK, RP = NO + 1, NW = kBwdThreads / 32;
    extern __shared__ __align__(16) float wsm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = lane >> 2, r = lane & 3;
    const int VH = PH + K - 1, VW = PW + K - 1, VR = kWinRB + K - 1;
    const int up = win_upitch(PW), vp = win_vpitch(VW), vcs = VR * vp + 4, vpad = win_vpad(K);
    float *us = wsm;                       // [CUG][kWinRB][up]
    float *vs = wsm + CUG * kWinRB * up;   // [CVG][vcs]: rows vp apart, column j at vpad + j
    int bx = blockIdx.x;
    const int run = bx % nrun;
    bx /= nrun;
    const int n = bx % N, g = bx / N;
    const int nband = (PH + kWinRB - 1) / kWinRB;
    const int band0 = run * bpr, band1 = min(band0 + bpr, nband);
    const float *Ub = U + ((size_t)n * CU + (size_t)g * CUG) * PH * PW;
    const float *Vb = V + ((size_t)n * CV + (size_t)g * CVG) * VH * VW;
    const int nseg = (PW + kWinSeg - 1) / kWinSeg;
    const bool u4 = (PW & 3) == 0 && (reinterpret_cast<uintptr_t>(U) & 15) == 0;
    // V rows in 8-byte copies where every row and its shared-memory place start on 8 bytes
    const bool v8 = (VW & 1) == 0 && (vpad & 1) == 0 && (reinterpret_cast<uintptr_t>(V) & 7) == 0;
    float acc[CUG][KK];
#pragma unroll
    for (int m = 0; m < CUG; ++m)
#pragma unroll
        for (int e = 0; e < KK; ++e) acc[m][e] = 0.0f;
    // the columns no staging writes: U past PW, V before vpad and past vpad + VW
    for (int row = warp; row < CUG * kWinRB; row += NW)
        for (int j = PW + lane; j < up; j += 32) us[(size_t)row * up + j] = 0.0f;
    for (int row = warp; row < CVG * VR; row += NW) {
        float *dst = vs + (size_t)(row / VR) * vcs + (size_t)(row % VR) * vp;
        for (int j = lane; j < vp; j += 32)
            if (j < vpad || j >= vpad + VW) dst[j] = 0.0f;
    }
    for (int band = band0; band < band1; ++band) {
        const int i0 = band * kWinRB;
        // stage with asynchronous copies (all in flight at once; zero fill
        // past the edges): rows spread over the warps, coalesced
        for (int row = warp; row < CUG * kWinRB; row += NW) {
            const int m = row / kWinRB, rr = row - m * kWinRB;
            float *dst = us + (size_t)row * up;
            const bool ok = i0 + rr < PH;
            const float *src = Ub + ((size_t)m * PH + (ok ? i0 + rr : 0)) * PW;
            if (u4) {
                for (int j = 4 * lane; j < PW; j += 128) cp_async16(dst + j, src + j, ok);
            } else {
                for (int j = lane; j < PW; j += 32) cp_async4(dst + j, src + j, ok);
            }
        }
        for (int row = warp; row < CVG * VR; row += NW) {
            const int cc = row / VR, rr = row - cc * VR;
            float *dst = vs + (size_t)cc * vcs + (size_t)rr * vp + vpad;
            const bool ok = i0 + rr < VH;
            const float *src = Vb + ((size_t)cc * VH + (ok ? i0 + rr : 0)) * VW;
            if (v8) {
                for (int j = 2 * lane; j < VW; j += 64) cp_async8(dst + j, src + j, ok);
            } else {
                for (int j = lane; j < VW; j += 32) cp_async4(dst + j, src + j, ok);
            }
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();
        if (i0 + r < PH) {
            for (int seg = warp; seg < nseg; seg += NW) {
                const int j0 = seg * kWinSeg, jn = min(kWinSeg, PW - j0);
                const float *ur = us + (size_t)r * up + j0;
                const float *vr = vs + (size_t)c * vcs + (size_t)r * vp + vpad + j0;
                // W[p][e]: V row r + p, columns t + e, e < k + 3
                float W[K][K + 3];
#pragma unroll
                for (int p = 0; p < K; ++p)
#pragma unroll
                    for (int q = 0; q + 1 < K; ++q) W[p][q] = vr[p * vp + q];
                for (int t = 0; t < jn; t += 4) {
#pragma unroll
                    for (int p = 0; p < K; ++p) {
                        const float4 v4 = *reinterpret_cast<const float4 *>(vr + p * vp + t + K - 1);
                        W[p][K - 1] = v4.x;
                        W[p][K] = v4.y;
                        W[p][K + 1] = v4.z;
                        W[p][K + 2] = v4.w;
                    }
#pragma unroll
                    for (int m = 0; m < CUG; ++m) {
                        const float4 u4 = *reinterpret_cast<const float4 *>(ur + (size_t)m * kWinRB * up + t);
                        const float uu[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                        for (int tt = 0; tt < 4; ++tt)
#pragma unroll
                            for (int p = 0; p < K; ++p)
#pragma unroll
                                for (int q = 0; q < K; ++q)
                                    acc[m][p * K + q] = fmaf(uu[tt], W[p][tt + q], acc[m][p * K + q]);
                    }
#pragma unroll
                    for (int p = 0; p < K; ++p)
#pragma unroll
                        for (int q = 0; q + 1 < K; ++q) W[p][q] = W[p][q + 4];
                }
            }
        }
        __syncthreads();
    }
    // the block's sums per (m, c, p, q): threads of channel c in warp, then
    // band-row order
    float *red = wsm;  // [kBwdThreads][RP]
#pragma unroll
    for (int m = 0; m < CUG; ++m)
#pragma unroll
        for (int e = 0; e < KK; ++e) red[(size_t)tid * RP + m * KK + e] = acc[m][e];
    __syncthreads();
    float *pp = part + ((size_t)n * nrun + run) * ((size_t)CU * CVG * KK) + (size_t)g * CUG * CVG * KK;
    for (int e = tid; e < CUG * CVG * KK; e += kBwdThreads) {
        const int m = e / (CVG * KK), rem = e - m * (CVG * KK), cc = rem / KK, pq = rem - cc * KK;
        float sum = 0.0f;
        for (int w = 0; w < NW; ++w)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) sum += red[(size_t)(w * 32 + cc * 4 + rr) * RP + m * KK + pq];
        pp[e] = sum;
    }
}

// Step 5 for the ConvTranspose2d block with 8 input and 8 output channels a
// group (the l2_p19 block; k <= 3, W a multiple of 4): dx is the valid
// correlation of dA with the filter,
//   dx[n][g 8 + ci][i][j] = sum_{co, ky, kx} dA[n][g 8 + co][i + ky][j + kx] w[g 8 + ci][co][ky][kx].
// A block takes one (group, sample) and a band of kWinRB output rows; it
// stages the band's dA rows (cp.async, zero past the edges) and the group's
// filter as [co][ky][kx][ci].  Thread (r, quad) computes the 8 channels of
// output row r at 4 consecutive columns: per dA channel, 16-byte loads of
// its k x (k + 3) window and of the taps' 8 filter values (the same for the
// whole block: broadcast) feed 8 x k^2 x 4 multiply-adds.  Each output is
// one sum in a fixed order; the stores are 16 bytes a thread, coalesced.
constexpr int kDxQuads = 64;  // column quads a band row takes per pass
template <int K>
__global__ void __launch_bounds__(kBwdThreads, 2) k_bwd_dx_g8(const float *dA, const float *w, int N, int C_in,
                                                              int C_out, int H, int W, float *dx) {
    constexpr int KK = K * K;
    extern __shared__ __align__(16) float dsm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int VH = H + K - 1, VW = W + K - 1, VR = kWinRB + K - 1;
    const int vp = (VW + 3) / 4 * 4 + 8;  // the window's 16-byte loads reach 4 columns past W + k - 2
    float *vs = dsm;                        // [8][VR][vp]
    float *ws = dsm + 8 * VR * vp;          // [co][ky][kx][ci]
    const int nband = (H + kWinRB - 1) / kWinRB;
    int bx = blockIdx.x;
    const int band = bx % nband;
    bx /= nband;
    const int n = bx % N, g = bx / N;
    const int i0 = band * kWinRB;
    const float *Vb = dA + ((size_t)n * C_out + (size_t)g * 8) * VH * VW;
    // rows in 8-byte copies where every row starts on 8 bytes
    const bool v8 = (VW & 1) == 0 && (reinterpret_cast<uintptr_t>(dA) & 7) == 0;
    for (int row = warp; row < 8 * VR; row += kBwdThreads / 32) {
        const int cc = row / VR, rr = row - cc * VR;
        float *dst = vs + (size_t)row * vp;
        const bool ok = i0 + rr < VH;
        const float *src = Vb + ((size_t)cc * VH + (ok ? i0 + rr : 0)) * VW;
        if (v8) {
            for (int j = 2 * lane; j < VW; j += 64) cp_async8(dst + j, src + j, ok);
        } else {
            for (int j = lane; j < VW; j += 32) cp_async4(dst + j, src + j, ok);
        }
        for (int j = VW + lane; j < vp; j += 32) dst[j] = 0.0f;
    }
    cp_async_commit();
    // the group's filter w[g 8 + ci][co][ky][kx] as [co][tap][ci]
    for (int e = tid; e < 8 * 8 * KK; e += kBwdThreads) {
        const int ci = e / (8 * KK), rem = e - ci * (8 * KK), co = rem / KK, tap = rem - co * KK;
        ws[(co * KK + tap) * 8 + ci] = __ldg(w + ((size_t)(g * 8 + ci) * 8 + co) * KK + tap);
    }
    cp_async_wait_all();
    __syncthreads();
    const int r = tid / kDxQuads, i = i0 + r;
    if (i < H) {
        for (int qd = tid % kDxQuads; 4 * qd < W; qd += kDxQuads) {
            const int j = 4 * qd;
            float acc[8][4];
#pragma unroll
            for (int ci = 0; ci < 8; ++ci)
#pragma unroll
                for (int t = 0; t < 4; ++t) acc[ci][t] = 0.0f;
#pragma unroll 1
            for (int co = 0; co < 8; ++co) {
                const float *vr = vs + ((size_t)co * VR + r) * vp + j;
#pragma unroll
                for (int ky = 0; ky < K; ++ky) {
                    const float4 a = *reinterpret_cast<const float4 *>(vr + ky * vp);
                    const float4 b = *reinterpret_cast<const float4 *>(vr + ky * vp + 4);
                    const float win[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int kx = 0; kx < K; ++kx) {
                        const float4 w0 = *reinterpret_cast<const float4 *>(ws + (co * KK + ky * K + kx) * 8);
                        const float4 w1 = *reinterpret_cast<const float4 *>(ws + (co * KK + ky * K + kx) * 8 + 4);
                        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                        for (int ci = 0; ci < 8; ++ci)
#pragma unroll
                            for (int t = 0; t < 4; ++t) acc[ci][t] = fmaf(wv[ci], win[t + kx], acc[ci][t]);
                    }
                }
            }
#pragma unroll
            for (int ci = 0; ci < 8; ++ci) {
                float *o = dx + (((size_t)n * C_in + g * 8 + ci) * H + i) * W + j;
                *reinterpret_cast<float4 *>(o) = make_float4(acc[ci][0], acc[ci][1], acc[ci][2], acc[ci][3]);
            }
        }
    }
}
size_t dx_g8_smem_bytes(int K, int W) {
    const int vp = (W + K - 1 + 3) / 4 * 4 + 8;
    return 4 * ((size_t)8 * (kWinRB + K - 1) * vp + (size_t)64 * K * K);
}
typedef void (*DxKernel)(const float *, const float *, int, int, int, int, int, float *);
DxKernel dx_g8_kernel(int K) {
    return K == 1 ? k_bwd_dx_g8<1> : (K == 2 ? k_bwd_dx_g8<2> : (K == 3 ? k_bwd_dx_g8<3> : nullptr));
}

// Step 5 for Conv2d on the tensor cores: dx is the full correlation of dA
// with the filter turned by 180 degrees and its channel axes swapped,
//   dx[n][ci][i][j] = sum_{co, p, q} dAp[n][co][i + p][j + q] w[co][ci][k - 1 - p][k - 1 - q],
// dAp being dA with k - 1 zero rows and columns before and after, i.e. a
// valid Conv2d of dAp with w'[ci][co][p][q] = w[co][ci][k - 1 - p][k - 1 - q].
// The library's tensor-core Conv2d plan runs it; its output channels are
// padded to a multiple of 128 (zero filters) and its input rows to a
// multiple of 4 columns (zeros), and k_bwd_crop copies the valid part to dx.
// One warp per padded row (rows of all planes in order), lanes along it.
// Rows of dA inside the padding also go to dAq, rows of pitch Pq with
// zeros past Wo (the tensor-core dw's operand), when dAq is given.
__global__ void __launch_bounds__(kBwdThreads) k_bwd_pad(const float *dA, int Ho, int Wo, int k, int Hp, int Wp,
                                                         long long rows, float *dAp, float *dAq, int Pq) {
    const long long row = (long long)blockIdx.x * (kBwdThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const long long pl = row / Hp;
    const int i = (int)(row - pl * Hp) - (k - 1);
    float *dst = dAp + row * Wp;
    if (i < 0 || i >= Ho) {
        for (int c = lane; c < Wp; c += 32) dst[c] = 0.0f;
        return;
    }
    const float *src = dA + (pl * Ho + i) * Wo;
    for (int c = lane; c < Wp; c += 32) {
        const int j = c - (k - 1);
        dst[c] = (j >= 0 && j < Wo) ? __ldg(src + j) : 0.0f;
    }
    if (dAq) {
        float *q = dAq + (pl * Ho + i) * Pq;
        for (int j = lane; j < Pq; j += 32) q[j] = j < Wo ? __ldg(src + j) : 0.0f;
    }
}
__global__ void k_bwd_wadj(const float *w, int Co, int Ci, int Cip, int k, float *wa) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x, kk = k * k;
    if (e >= Cip * Co * kk) return;
    const int ci = e / (Co * kk), rem = e - ci * Co * kk, co = rem / kk, t = rem - co * kk;
    wa[e] = ci < Ci ? __ldg(w + ((size_t)co * Ci + ci) * kk + (kk - 1 - t)) : 0.0f;
}
// One warp per dx row, lanes along it.
__global__ void __launch_bounds__(kBwdThreads) k_bwd_crop(const float *src, int Cs, int Hs, int Ws, int C, int H,
                                                          int W, long long rows, float *dx) {
    const long long row = (long long)blockIdx.x * (kBwdThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const long long pl = row / H;  // n * C + c
    const int i = (int)(row - pl * H);
    const long long n = pl / C;
    const int c = (int)(pl - n * C);
    const float *s = src + (((size_t)n * Cs + c) * Hs + i) * Ws;
    float *d = dx + row * W;
    for (int j = lane; j < W; j += 32) d[j] = __ldg(s + j);
}

// Dynamic shared memory of k_bwd_weight_win: the staged rows, or the
// threads' sums at the end, whichever is larger.
size_t win_smem_bytes(int CUG, int K, int PW) {
    const int up = (PW + 31) / 32 * 32 + 4, vp = (PW + K - 1 + 31) / 32 * 32 + 8;
    const size_t tiles = (size_t)CUG * kWinRB * up + (size_t)8 * ((kWinRB + K - 1) * vp + 4);
    const size_t red = (size_t)kBwdThreads * (CUG * K * K + 1);
    return 4 * std::max(tiles, red);
}
typedef void (*WinKernel)(const float *, const float *, int, int, int, int, int, int, int, float *);
WinKernel win_kernel(int CUG, int K) {
#define CN_WIN(KK_, CC_) \
    if (K == KK_ && CUG == CC_) return k_bwd_weight_win<KK_, CC_>;
    CN_WIN(1, 1) CN_WIN(1, 2) CN_WIN(1, 4) CN_WIN(1, 8)
    CN_WIN(2, 1) CN_WIN(2, 2) CN_WIN(2, 4) CN_WIN(2, 8)
    CN_WIN(3, 1) CN_WIN(3, 2) CN_WIN(3, 4) CN_WIN(3, 8)
#undef CN_WIN
    return nullptr;
}

// dw[e] = sum over the splits of part[split][e], in split order.
__global__ void k_bwd_weight_sum(const float *part, int splits, long long total, float *dw) {
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= total) return;
    float s = 0.0f;
    for (int q = 0; q < splits; ++q) s += part[(size_t)q * total + e];
    dw[e] = s;
}

// Step 7: per channel, sums over n (and the db slices) in order.
__global__ void k_bwd_channel_sums(const float2 *gpart, const float *dbpart, int N, int C, int slices,
                                   float *dgamma, float *dbeta, float *db) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    float sg = 0.0f, sb = 0.0f, sd = 0.0f;
    for (int n = 0; n < N; ++n) {
        const size_t pl = (size_t)n * C + c;
        sg += gpart[pl].x;
        sb += gpart[pl].y;
        for (int s = 0; s < slices; ++s) sd += dbpart[pl * slices + s];
    }
    if (dgamma) dgamma[c] = sg;
    if (dbeta) dbeta[c] = sb;
    if (db) db[c] = sd;
}

}  // namespace
}  // namespace cn

using namespace cn;

struct conv_norm_bwd_plan_s {
    conv_norm_desc d;
    int device = -1;
    conv_norm_plan conv_fwd = nullptr;  // A = conv(x) + b
    conv_norm_plan conv_adj = nullptr;  // dx = the adjoint conv of dA
    int Ho = 0, Wo = 0;
    long long S = 0, planes = 0;
    int slices = 1;
    int wsplits = 1;
    long long wchunk = 0, wtotal = 0;
    int wgrid = 0;
    int wtile = 1;  // dw: 0 = 8 x 128 tiles (groups of at most 8 channels), 1 = 64 x 64, 2 = 128 x 128, 3 = sliding window
    int wrun = 1, wbpr = 1;  // sliding window: runs of bands per (group, sample), bands a run
    size_t wsmem = 0;
    int dxg8 = 0;            // dx by k_bwd_dx_g8 (else the adjoint conv's forward plan)
    size_t dxsmem = 0;
    conv_norm_plan adj_tc = nullptr;  // Conv2d: dx as a tensor-core Conv2d of the padded dA
    BwdWtState *wt = nullptr;         // Conv2d: dw on the tensor cores (with adj_tc)
    int wt_nrun = 0, wt_pitch = 0, wsplits_gemm = 1;
    float *dAq = nullptr;             // dA rows of pitch wt_pitch
    int *werr = nullptr;              // device error flag of the tensor-core dw
    int Cip = 0, Hp = 0, Wp = 0, Hs = 0, Ws = 0;
    float *dAp = nullptr, *wadj = nullptr, *adjout = nullptr;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    float *A = nullptr;      // [N][C_out][S]: A, then dA
    float4 *ps = nullptr;    // [planes][2]
    float4 *coef = nullptr;  // [planes]
    float2 *gpart = nullptr; // [planes]
    float *dbpart = nullptr; // [planes][slices]
    float *wpart = nullptr;  // [wsplits][w numel]
};

namespace {

size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace

extern "C" {

int conv_norm_bwd_plan_create(const conv_norm_desc *d, conv_norm_bwd_plan *out) {
    if (!d || !out) return CN_ERR_INVALID_ARG;
    *out = nullptr;
    int st = conv_norm_desc_validate(d);
    if (st != CN_OK) return st;
    if ((d->conv != CN_CONV2D && d->conv != CN_CONVT2D) || d->red != CN_RED_NONE ||
        d->act == CN_ACT_SOFTMAX_C || d->N < 1)
        return CN_ERR_UNSUPPORTED;
    conv_norm_bwd_plan_s *p = new (std::nothrow) conv_norm_bwd_plan_s();
    if (!p) return CN_ERR_ALLOC;
    p->d = *d;
    auto fail = [&](int s) {
        conv_norm_bwd_plan_destroy(p);
        return s;
    };
    if (cudaGetDevice(&p->device) != cudaSuccess) {
        cudaGetLastError();
        return fail(CN_ERR_CUDA);
    }
    const bool T = d->conv == CN_CONVT2D;
    p->Ho = T ? d->H + d->k - 1 : d->H - d->k + 1;
    p->Wo = T ? d->W + d->k - 1 : d->W - d->k + 1;
    p->S = (long long)p->Ho * p->Wo;
    p->planes = (long long)d->N * d->C_out;
    // the conv alone, and its adjoint (C_in and C_out swapped, dA's extent in)
    conv_norm_desc f = *d;
    f.act = CN_ACT_NONE;
    f.norm = CN_NORM_NONE;
    f.affine = 0;
    f.post_scale = 1.0f;
    f.red = CN_RED_NONE;
    if ((st = conv_norm_plan_create(&f, &p->conv_fwd)) != CN_OK) return fail(st);
    conv_norm_desc j = f;
    j.conv = T ? CN_CONV2D : CN_CONVT2D;
    j.C_in = d->C_out;
    j.C_out = d->C_in;
    j.H = p->Ho;
    j.W = p->Wo;
    j.has_bias = 0;
    if ((st = conv_norm_plan_create(&j, &p->conv_adj)) != CN_OK) return fail(st);
    // Conv2d: the adjoint as a valid Conv2d of the zero-padded dA, on the
    // tensor-core kernel where the padded shape takes it
    const char *notc = getenv("CN_NO_TC");
    if (!T && d->groups == 1 && !(notc && atoi(notc))) {
        conv_norm_desc a = f;
        a.C_in = d->C_out;
        a.C_out = (d->C_in + 127) / 128 * 128;
        a.H = p->Ho + 2 * (d->k - 1);
        a.W = (p->Wo + 2 * (d->k - 1) + 3) / 4 * 4;
        a.has_bias = 0;
        conv_norm_plan q = nullptr;
        conv_norm_info qi;
        if (conv_norm_plan_create(&a, &q) == CN_OK && conv_norm_plan_info(q, &qi) == CN_OK && qi.kernel_names &&
            strstr(qi.kernel_names, "k_conv2d_tc")) {
            p->adj_tc = q;
            p->Cip = a.C_out;
            p->Hp = a.H;
            p->Wp = a.W;
            p->Hs = a.H - d->k + 1;
            p->Ws = a.W - d->k + 1;
        } else {
            conv_norm_plan_destroy(q);
        }
    }
    // db slices: about 16 K values per block
    p->slices = (int)std::max(1LL, std::min(64LL, p->S / 16384));
    // dw: enough position splits for ~4 blocks per SM
    int sms = 152;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    const int G = d->groups;
    const int CU = T ? d->C_in : d->C_out, CV = T ? d->C_out : d->C_in;
    const int CUg = CU / G, NN = (CV / G) * d->k * d->k;
    p->wtile = CUg <= 8 ? 0 : (CUg < 96 ? 1 : 2);
    const int PHw = T ? d->H : p->Ho, PWw = T ? d->W : p->Wo;
    p->wtotal = (long long)CU * NN;
    const char *nowin = getenv("CN_NO_WIN");
    if (CV / G == 8 && d->k <= 3 && win_kernel(CUg, d->k) && !(nowin && atoi(nowin))) {
        // sliding window: about four blocks' worth per SM slot (two a SM)
        p->wtile = 3;
        const int nband = (PHw + kWinRB - 1) / kWinRB;
        const long long gn = (long long)G * d->N;
        p->wrun = (int)std::max(1LL, std::min((long long)nband, (8LL * sms + gn - 1) / gn));
        p->wbpr = (nband + p->wrun - 1) / p->wrun;
        p->wrun = (nband + p->wbpr - 1) / p->wbpr;
        p->wgrid = (int)(gn * p->wrun);
        p->wsplits = d->N * p->wrun;
        p->wsmem = win_smem_bytes(CUg, d->k, PWw);
        if (gn * p->wrun > 0x7fffffffLL || p->wsmem > 200 * 1024 ||
            raise_dyn_smem(reinterpret_cast<const void *>(win_kernel(CUg, d->k)), (int)p->wsmem) != cudaSuccess) {
            cudaGetLastError();
            p->wtile = 0;
        }
    }
    // dx of a ConvTranspose2d with 8 channels a group on both sides
    if (T && d->C_in / G == 8 && d->C_out / G == 8 && d->k <= 3 && d->W % 4 == 0 && !(nowin && atoi(nowin))) {
        p->dxsmem = dx_g8_smem_bytes(d->k, d->W);
        const long long blocks = (long long)G * d->N * ((d->H + kWinRB - 1) / kWinRB);
        if (p->dxsmem <= 100 * 1024 && blocks <= 0x7fffffffLL &&
            raise_dyn_smem(reinterpret_cast<const void *>(dx_g8_kernel(d->k)), (int)p->dxsmem) == cudaSuccess)
            p->dxg8 = 1;
        else
            cudaGetLastError();
    }
    if (p->wtile != 3) {
        const int BM = p->wtile == 0 ? 8 : (p->wtile == 1 ? 64 : 128), BN = p->wtile == 1 ? 64 : 128;
        const int tiles = ((CUg + BM - 1) / BM) * ((NN + BN - 1) / BN) * G;
        const long long Ktot = (long long)d->N * (T ? (long long)d->H * d->W : p->S);
        p->wsplits = (int)std::max(1LL, std::min((long long)(4 * sms + tiles - 1) / tiles, (Ktot + 4095) / 4096));
        p->wchunk = ((Ktot + p->wsplits - 1) / p->wsplits + 63) / 64 * 64;
        p->wsplits = (int)((Ktot + p->wchunk - 1) / p->wchunk);
        p->wgrid = tiles;
        if (p->wsplits > 65535) return fail(CN_ERR_UNSUPPORTED);
    }
    p->wsplits_gemm = p->wsplits;
    // dense Conv2d: dw on the tensor cores, fed by the padded-row copy of dA
    // that the tensor-core adjoint's pad pass writes beside its own
    if (p->adj_tc && p->wtile != 3 &&
        bwd_wt_plan(d->N, d->C_out, d->C_in, d->H, d->W, d->k, sms, nullptr, &p->wt, &p->wt_nrun, &p->wt_pitch) !=
            CN_OK) {
        p->wt = nullptr;
    }
    const size_t bA = al256((size_t)p->planes * p->S * 4), bps = al256((size_t)p->planes * 32),
                 bcoef = al256((size_t)p->planes * 16), bg = al256((size_t)p->planes * 8),
                 bdb = al256((size_t)p->planes * p->slices * 4);
    size_t bw = al256((size_t)p->wsplits * p->wtotal * 4);
    const size_t bwt = p->wt ? al256((size_t)std::max(p->wt_nrun, p->wsplits_gemm) * p->wtotal * 4) : 0,
                 bdaq = p->wt ? al256((size_t)d->N * d->C_out * p->Ho * p->wt_pitch * 4) + 256 : 0;
    if (p->wt) bw = bwt;
    const size_t bdap = p->adj_tc ? al256((size_t)d->N * d->C_out * p->Hp * p->Wp * 4) : 0,
                 bwa = p->adj_tc ? al256((size_t)p->Cip * d->C_out * d->k * d->k * 4) : 0,
                 bout = p->adj_tc ? al256((size_t)d->N * p->Cip * p->Hs * p->Ws * 4) : 0;
    p->ws_bytes = bA + bps + bcoef + bg + bdb + bw + bdap + bwa + bout + bdaq;
    if (cudaMalloc(&p->ws, p->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        return fail(CN_ERR_ALLOC);
    }
    char *b = static_cast<char *>(p->ws);
    p->A = reinterpret_cast<float *>(b);
    p->ps = reinterpret_cast<float4 *>(b + bA);
    p->coef = reinterpret_cast<float4 *>(b + bA + bps);
    p->gpart = reinterpret_cast<float2 *>(b + bA + bps + bcoef);
    p->dbpart = reinterpret_cast<float *>(b + bA + bps + bcoef + bg);
    p->wpart = reinterpret_cast<float *>(b + bA + bps + bcoef + bg + bdb);
    if (p->adj_tc) {
        p->dAp = reinterpret_cast<float *>(b + bA + bps + bcoef + bg + bdb + bw);
        p->wadj = reinterpret_cast<float *>(b + bA + bps + bcoef + bg + bdb + bw + bdap);
        p->adjout = reinterpret_cast<float *>(b + bA + bps + bcoef + bg + bdb + bw + bdap + bwa);
    }
    if (p->wt) {
        char *q = b + bA + bps + bcoef + bg + bdb + bw + bdap + bwa + bout;
        p->werr = reinterpret_cast<int *>(q);
        p->dAq = reinterpret_cast<float *>(q + 256);
        if (cudaMemset(p->werr, 0, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return fail(CN_ERR_CUDA);
        }
        bwd_wt_set_err(p->wt, p->werr);
    }
    *out = p;
    return CN_OK;
}

void conv_norm_bwd_plan_destroy(conv_norm_bwd_plan p) {
    if (!p) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (p->device >= 0 && cur != p->device) cudaSetDevice(p->device);
    conv_norm_plan_destroy(p->conv_fwd);
    conv_norm_plan_destroy(p->conv_adj);
    conv_norm_plan_destroy(p->adj_tc);
    bwd_wt_destroy(p->wt);
    cudaFree(p->ws);
    if (cur >= 0 && p->device >= 0 && cur != p->device) cudaSetDevice(cur);
    cudaGetLastError();
    delete p;
}

size_t conv_norm_bwd_workspace_bytes(conv_norm_bwd_plan p) {
    if (!p) return 0;
    return p->ws_bytes + conv_norm_workspace_bytes(p->conv_fwd) + conv_norm_workspace_bytes(p->conv_adj) +
           (p->adj_tc ? conv_norm_workspace_bytes(p->adj_tc) : 0);
}

int conv_norm_backward(conv_norm_bwd_plan p, const float *x, const float *w, const float *b,
                       const float *gamma, const float *beta, const float *dout, float *dx, float *dw,
                       float *db, float *dgamma, float *dbeta, void *stream) {
    if (!p) return CN_ERR_INVALID_ARG;
    const conv_norm_desc &d = p->d;
    const bool aff = d.affine && d.norm != CN_NORM_NONE;
    (void)beta;  // the gradients do not depend on beta
    if (!x || !w || !dout || !dx || !dw) return CN_ERR_INVALID_ARG;
    if ((b != nullptr) != (d.has_bias == 1) || (db != nullptr) != (d.has_bias == 1)) return CN_ERR_INVALID_ARG;
    if (aff && (!gamma || !dgamma || !dbeta)) return CN_ERR_INVALID_ARG;
    if (!aff && (dgamma || dbeta)) return CN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dout) % 16 || reinterpret_cast<uintptr_t>(dx) % 16) return CN_ERR_INVALID_ARG;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    if (cur != p->device && cudaSetDevice(p->device) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = conv_norm_forward(p->conv_fwd, x, w, b, nullptr, nullptr, p->A, stream);
    if (st == CN_OK) {
        const int act = d.act == CN_ACT_HARDSWISH ? ACT_HARDSWISH : (d.act == CN_ACT_GELU_ERF ? ACT_GELU : ACT_NONE);
        const int G = d.norm == CN_NORM_GROUP ? d.num_groups : (d.norm == CN_NORM_INSTANCE ? d.C_out : 1);
        if (d.norm != CN_NORM_NONE)
            k_bwd_plane_sums<<<(unsigned)p->planes, kBwdThreads, 0, s>>>(p->A, dout, p->S, act, p->ps);
        const int ng = d.N * G;
        k_bwd_group<<<(ng + 127) / 128, 128, 0, s>>>(p->ps, d.N, d.C_out, G, d.norm, d.eps, d.post_scale,
                                                     aff ? gamma : nullptr, p->coef, p->gpart);
        k_bwd_dA<<<(unsigned)(p->planes * p->slices), kBwdThreads, 0, s>>>(p->A, dout, p->coef, p->S, act,
                                                                           p->slices, p->dbpart);
        if (cudaGetLastError() != cudaSuccess) st = CN_ERR_CUDA;
    }
    if (st == CN_OK) {
        if (p->dxg8) {
            const unsigned blocks = (unsigned)((long long)d.groups * d.N * ((d.H + kWinRB - 1) / kWinRB));
            dx_g8_kernel(d.k)<<<blocks, kBwdThreads, p->dxsmem, s>>>(p->A, w, d.N, d.C_in, d.C_out, d.H, d.W, dx);
            if (cudaGetLastError() != cudaSuccess) st = CN_ERR_CUDA;
        } else if (p->adj_tc) {
            const long long prow = (long long)d.N * d.C_out * p->Hp, rpb = kBwdThreads / 32;
            k_bwd_pad<<<(unsigned)((prow + rpb - 1) / rpb), kBwdThreads, 0, s>>>(
                p->A, p->Ho, p->Wo, d.k, p->Hp, p->Wp, prow, p->dAp, p->wt ? p->dAq : nullptr, p->wt_pitch);
            const int nw = p->Cip * d.C_out * d.k * d.k;
            k_bwd_wadj<<<(nw + 255) / 256, 256, 0, s>>>(w, d.C_out, d.C_in, p->Cip, d.k, p->wadj);
            st = cudaGetLastError() == cudaSuccess ? CN_OK : CN_ERR_CUDA;
            if (st == CN_OK)
                st = conv_norm_forward(p->adj_tc, p->dAp, p->wadj, nullptr, nullptr, nullptr, p->adjout, stream);
            if (st == CN_OK) {
                const long long xrow = (long long)d.N * d.C_in * d.H, rpb = kBwdThreads / 32;
                k_bwd_crop<<<(unsigned)((xrow + rpb - 1) / rpb), kBwdThreads, 0, s>>>(
                    p->adjout, p->Cip, p->Hs, p->Ws, d.C_in, d.H, d.W, xrow, dx);
                if (cudaGetLastError() != cudaSuccess) st = CN_ERR_CUDA;
            }
        } else {
            st = conv_norm_forward(p->conv_adj, p->A, w, nullptr, nullptr, nullptr, dx, stream);
        }
    }
    if (st == CN_OK) {
        const bool T = d.conv == CN_CONVT2D;
        const float *U = T ? x : p->A, *V = T ? p->A : x;
        const int CU = T ? d.C_in : d.C_out, CV = T ? d.C_out : d.C_in;
        const int PH = T ? d.H : p->Ho, PW = T ? d.W : p->Wo;
        const dim3 grid((unsigned)p->wgrid, (unsigned)p->wsplits_gemm);
        const bool wt = p->wt && p->adj_tc && reinterpret_cast<uintptr_t>(x) % 16 == 0;
        p->wsplits = wt ? p->wt_nrun : p->wsplits_gemm;
        if (wt) {
            st = bwd_wt_launch(p->wt, p->dAq, x, p->wpart, s);
        } else if (p->wtile == 3)
            win_kernel(CU / d.groups, d.k)<<<(unsigned)p->wgrid, kBwdThreads, p->wsmem, s>>>(
                U, V, d.N, CU, CV, PH, PW, p->wrun, p->wbpr, p->wpart);
        else if (p->wtile == 0)
            k_bwd_weight<8, 128, 1, 4, kWBKSmall><<<grid, kBwdThreads, 0, s>>>(U, V, d.N, CU, CV, PH, PW, d.k,
                                                                              d.groups, p->wchunk, p->wpart);
        else if (p->wtile == 1)
            k_bwd_weight<64, 64, 4, 4, kWBKWide><<<grid, kBwdThreads, 0, s>>>(U, V, d.N, CU, CV, PH, PW, d.k,
                                                                             d.groups, p->wchunk, p->wpart);
        else
            k_bwd_weight<128, 128, 8, 8, kWBKSmall><<<grid, kBwdThreads, 0, s>>>(U, V, d.N, CU, CV, PH, PW, d.k,
                                                                                d.groups, p->wchunk, p->wpart);
        k_bwd_weight_sum<<<(unsigned)((p->wtotal + 255) / 256), 256, 0, s>>>(p->wpart, p->wsplits, p->wtotal, dw);
        k_bwd_channel_sums<<<(d.C_out + 127) / 128, 128, 0, s>>>(p->gpart, p->dbpart, d.N, d.C_out, p->slices,
                                                                 aff ? dgamma : nullptr, aff ? dbeta : nullptr, db);
        if (cudaGetLastError() != cudaSuccess) st = CN_ERR_CUDA;
    }
    if (st != CN_OK) cudaGetLastError();
    if (cur != p->device) cudaSetDevice(cur);
    return st;
}

int conv_norm_bwd_check_device(conv_norm_bwd_plan p, void *stream) {
    if (!p) return CN_ERR_INVALID_ARG;
    const int a = conv_norm_plan_check_device(p->conv_fwd, stream);
    const int c = conv_norm_plan_check_device(p->conv_adj, stream);
    const int t = p->adj_tc ? conv_norm_plan_check_device(p->adj_tc, stream) : CN_OK;
    int w = CN_OK;
    if (p->werr) {
        int flag = 0;
        if (cudaMemcpy(&flag, p->werr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            w = CN_ERR_CUDA;
        } else if (flag != 0) {
            const int zero = 0;
            cudaMemcpy(p->werr, &zero, sizeof(int), cudaMemcpyHostToDevice);
            w = flag == 1 ? CN_ERR_TIMEOUT : CN_ERR_DEVICE_CHECK;
        }
    }
    return a != CN_OK ? a : (c != CN_OK ? c : (t != CN_OK ? t : w));
}

}  // extern "C"
