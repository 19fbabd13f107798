// Variant 1: Conv3d -> Softmax over channels -> MaxPool3d(2,2) -> MaxPool3d(2,2)
// in one launch; only the pooled tensor is written.
//
// Method (l2_p6, Conv3d -> Softmax -> MaxPool3d x2):
//  * two stacked 2x2x2 stride-2 floor-mode pools equal one 4x4x4 stride-4
//    pool, since floor(floor(L/2)/2) = floor(L/4) and max is associative;
//  * only the conv outputs inside the kept 4*floor(L/4) region are needed,
//    so the dropped tail is never computed;
//  * softmax is taken per voxel over the channels BEFORE the max (the two do
//    not commute).
// Mapping: 16 threads per pooled voxel, one per (dz, dy) row of the 4x4x4
// window; each thread computes all CO channels x the 4 w positions of its
// row (4*CO accumulators), applies bias + softmax per position in registers,
// takes the max over its 4 positions, then a 4-step xor-shuffle max over the
// voxel's 16 lanes.  Each CTA stages the (4+K-1)^3 x C_in input patch of each
// of its 16 voxels with one TMA tensor copy per voxel, and the whole filter.
#include "cn_common.cuh"
#include "cn_internal.h"

#include <algorithm>
#include <cstdlib>

namespace cn {
namespace {

template <int K, int CO>
__global__ void __launch_bounds__(256) k_conv3d_softmax_pool4(const __grid_constant__ Pool3dArgs a) {
    extern __shared__ __align__(128) float smem[];
    __shared__ __align__(8) uint64_t bar;
    constexpr int P = 4 + K - 1;      // patch extent per axis
    constexpr int PX = (P + 3) & ~3;  // patch row pitch
    constexpr int KKK = K * K * K;
    const int tid = threadIdx.x;
    const int v = tid >> 4, l16 = tid & 15;
    const int dz = l16 >> 2, dy = l16 & 3;
    float *sx = smem;
    float *sw = smem + (size_t)a.vox_per_cta * a.vox_stride;
    const long long vbase = (long long)blockIdx.x * a.vox_per_cta;
    const int nv = (int)min((long long)a.vox_per_cta, a.nvox - vbase);

    // ---- stage each voxel's (P x P x P) x C_in input patch ----
    if (a.use_tma) {
        if (tid == 0) {
            mbar_init(&bar, 1);
            fence_barrier_init();
            fence_proxy_async();
            mbar_arrive_expect_tx(&bar, (uint32_t)(nv * a.Ci * P * P * PX * 4));
        }
        __syncthreads();
        if (tid < nv) {
            long long gv = vbase + tid;
            const int pw = (int)(gv % a.Pw);
            gv /= a.Pw;
            const int ph = (int)(gv % a.Ph);
            gv /= a.Ph;
            const int pd = (int)(gv % a.Pd);
            const int n = (int)(gv / a.Pd);
            tma_load_4d(sx + (size_t)tid * a.vox_stride, &a.tmap, 4 * pw, 4 * ph, 4 * pd, n * a.Ci,
                        &bar);
        }
    } else {
        const int rows = nv * a.Ci * P * P;
        for (int rI = tid; rI < rows; rI += blockDim.x) {
            int t = rI;
            const int yy = t % P;
            t /= P;
            const int zz = t % P;
            t /= P;
            const int ci = t % a.Ci;
            const int vv = t / a.Ci;
            long long gv = vbase + vv;
            const int pw = (int)(gv % a.Pw);
            gv /= a.Pw;
            const int ph = (int)(gv % a.Ph);
            gv /= a.Ph;
            const int pd = (int)(gv % a.Pd);
            const int n = (int)(gv / a.Pd);
            const float *src = a.x + ((((size_t)n * a.Ci + ci) * a.D + 4 * pd + zz) * a.H + 4 * ph + yy) *
                                         (size_t)a.W + 4 * pw;
            float *dst = sx + (size_t)vv * a.vox_stride + ((ci * P + zz) * P + yy) * PX;
#pragma unroll
            for (int c = 0; c < P; ++c) cp_async4(dst + c, src + c, true);
        }
        cp_async_commit();
    }
    // ---- the filter, transposed to [ci][tap][co], and the bias ----
    // Every load of a round is issued before any store, so a CTA waits for
    // one global round trip per 8 values a thread stages, not one per value.
    {
        const int total = a.Ci * KKK * CO;
        for (int base = tid; base < total + CO; base += 8 * (int)blockDim.x) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = base + u * (int)blockDim.x;
                float t = 0.0f;
                if (e < total) {
                    const int co = e % CO, tap = e / CO;  // e = tap * CO + co
                    t = __ldg(a.w + (size_t)co * a.Ci * KKK + tap);
                } else if (e < total + CO && a.b) {
                    t = __ldg(a.b + (e - total));
                }
                v[u] = t;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = base + u * (int)blockDim.x;
                if (e < total + CO) sw[e] = v[u];
            }
        }
    }
    const float *sbias = sw + (size_t)a.Ci * KKK * CO;
    bool staged = true;
    if (a.use_tma) {
        staged = mbar_wait_bounded(&bar, 0, kWaitLimitNs);
        if (!staged) {
            flag_error(a.err, ERR_TIMEOUT);
            mbar_wait_bounded(&bar, 0, kWaitLimitNs);
        }
    } else {
        cp_async_wait_all();
    }
    __syncthreads();

    const long long gvox = vbase + v;
    const bool valid = v < nv;

    float acc[CO][4];
#pragma unroll
    for (int c = 0; c < CO; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[c][i] = 0.0f;

    const float *xv = sx + (size_t)(valid ? v : 0) * a.vox_stride;
    // Loop bounds depend only on kernel parameters (warp-uniform); after a
    // staging timeout the flagged forward computes on stale shared memory.
    (void)staged;
    for (int ci = 0; ci < a.Ci; ++ci) {
        CN_UNROLL(CN_TAP_UNROLL)
        for (int kd = 0; kd < K; ++kd) {
            CN_UNROLL(CN_TAP_UNROLL)
            for (int kh = 0; kh < K; ++kh) {
                const float *row = xv + ((ci * P + dz + kd) * P + dy + kh) * PX;
                float xr[PX];
#pragma unroll
                for (int j = 0; j < PX / 4; ++j) {
                    const float4 t = *reinterpret_cast<const float4 *>(row + 4 * j);
                    xr[4 * j + 0] = t.x;
                    xr[4 * j + 1] = t.y;
                    xr[4 * j + 2] = t.z;
                    xr[4 * j + 3] = t.w;
                }
#pragma unroll
                for (int kw = 0; kw < K; ++kw) {
                    const float4 *wp =
                        reinterpret_cast<const float4 *>(sw + ((size_t)ci * KKK + (kd * K + kh) * K + kw) * CO);
#pragma unroll
                    for (int c4 = 0; c4 < CO / 4; ++c4) {
                        const float4 wv = wp[c4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            acc[4 * c4 + 0][i] = fmaf(xr[i + kw], wv.x, acc[4 * c4 + 0][i]);
                            acc[4 * c4 + 1][i] = fmaf(xr[i + kw], wv.y, acc[4 * c4 + 1][i]);
                            acc[4 * c4 + 2][i] = fmaf(xr[i + kw], wv.z, acc[4 * c4 + 2][i]);
                            acc[4 * c4 + 3][i] = fmaf(xr[i + kw], wv.w, acc[4 * c4 + 3][i]);
                        }
                    }
                }
            }
        }
    }

    // ---- bias + softmax over channels per position, then max ----
    float best[CO];
#pragma unroll
    for (int c = 0; c < CO; ++c) best[c] = 0.0f;  // softmax values are > 0
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float m = -INFINITY;
#pragma unroll
        for (int c = 0; c < CO; ++c) {
            acc[c][i] += sbias[c];
            m = fmaxf(m, acc[c][i]);
        }
        float s = 0.0f;
#pragma unroll
        for (int c = 0; c < CO; ++c) {
            acc[c][i] = __expf(acc[c][i] - m);
            s += acc[c][i];
        }
        const float inv = 1.0f / s;
#pragma unroll
        for (int c = 0; c < CO; ++c) best[c] = fmaxf(best[c], acc[c][i] * inv);
    }
#pragma unroll
    for (int off = 1; off < 16; off <<= 1)
#pragma unroll
        for (int c = 0; c < CO; ++c) best[c] = fmaxf(best[c], __shfl_xor_sync(0xffffffffu, best[c], off));

    if (valid) {
        long long g = gvox;
        const int pw = (int)(g % a.Pw);
        g /= a.Pw;
        const int ph = (int)(g % a.Ph);
        g /= a.Ph;
        const int pd = (int)(g % a.Pd);
        const int n = (int)(g / a.Pd);
#pragma unroll
        for (int c = 0; c < CO; ++c) {
            if ((c % 16) == l16 && CN_CHECK(n < a.N, a.err)) {
                a.out[((((size_t)n * CO + c) * a.Pd + pd) * a.Ph + ph) * a.Pw + pw] = best[c] * a.post_scale;
            }
        }
    }
}

struct Inst {
    int K, CO;
    Pool3dKernel fn;
    const char *name;
};
#define CN_POOL_INST(K, CO) {K, CO, k_conv3d_softmax_pool4<K, CO>, "k_conv3d_softmax_pool4<" #K "," #CO ">"}
const Inst kInst[] = {CN_POOL_INST(1, 16), CN_POOL_INST(2, 16), CN_POOL_INST(3, 16),
                      CN_POOL_INST(4, 16)};
#undef CN_POOL_INST

int env_int(const char *name, int dflt) {
    const char *v = getenv(name);
    return v ? atoi(v) : dflt;
}
}  // namespace

int pool3d_plan(const conv_norm_desc &d, Pool3dArgs &a, Pool3dConfig &cfg) {
    const Inst *in = nullptr;
    for (const Inst &i : kInst)
        if (i.K == d.k && i.CO == d.C_out) in = &i;
    if (!in || d.groups != 1) return CN_ERR_UNSUPPORTED;
    const int K = d.k, P = 4 + K - 1, PX = (P + 3) & ~3;
    a.post_scale = d.post_scale;  // > 0 (checked by the caller): commutes with the max
    // the tensor-core kernel where the problem fits it
    if (tc3_plan(d, a.t, cfg.tc3) == CN_OK) {
        a.tc = 1;
        a.N = d.N;
        cfg.name = cfg.tc3.name;
        cfg.threads = cfg.tc3.threads;
        cfg.smem = cfg.tc3.smem;
        cfg.grid = cfg.tc3.grid;
        return CN_OK;
    }
    a.tc = 0;
    a.N = d.N;
    a.Ci = d.C_in;
    a.D = d.D;
    a.H = d.H;
    a.W = d.W;
    a.Do = d.D - K + 1;
    a.Ho = d.H - K + 1;
    a.Wo = d.W - K + 1;
    a.Pd = a.Do / 4;
    a.Ph = a.Ho / 4;
    a.Pw = a.Wo / 4;
    a.nvox = (long long)d.N * a.Pd * a.Ph * a.Pw;
    a.vox_per_cta = 16;
    a.pw_pitch = PX;
    // each voxel patch starts 128-byte aligned (TMA destination)
    a.vox_stride = (d.C_in * P * P * PX + 31) & ~31;
    a.use_tma = (d.W % 4 == 0) && d.C_in <= 256 && env_int("CN_NO_TMA", 0) == 0;
    a.tmap_base = nullptr;
    const size_t smem = ((size_t)a.vox_per_cta * a.vox_stride + (size_t)d.C_in * K * K * K * in->CO + in->CO) * 4;
    if (smem > 227 * 1024) return CN_ERR_UNSUPPORTED;
    const long long grid = (a.nvox + a.vox_per_cta - 1) / a.vox_per_cta;
    if (grid > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;
    cfg.kern = in->fn;
    cfg.name = in->name;
    cfg.threads = 16 * a.vox_per_cta;
    cfg.smem = (int)smem;
    cfg.grid = (int)grid;
    return CN_OK;
}

size_t pool3d_workspace(const Pool3dArgs &a) { return a.tc ? 2 * sizeof(int) : 0; }

int pool3d_prepare(Pool3dConfig &cfg, const Pool3dArgs &a) {
    if (a.tc) {
        const int st = tc3_prepare(cfg.tc3, a.t);
        cfg.grid = cfg.tc3.grid;
        return st;
    }
    if (raise_dyn_smem(reinterpret_cast<const void *>(cfg.kern), cfg.smem) !=
        cudaSuccess)
        return CN_ERR_CUDA;
    return CN_OK;
}

int pool3d_launch(const Pool3dConfig &cfg, Pool3dArgs &a, cudaStream_t s, const LaunchEvents *ev) {
    if (cfg.grid == 0) return CN_OK;
    if (a.tc) {
        Tc3Args &t = a.t;
        t.x = a.x;
        t.w = a.w;
        t.b = a.b;
        t.out = a.out;
        t.err = a.err;
        return tc3_launch(cfg.tc3, t, s, ev);
    }
    if (a.use_tma && a.tmap_base != a.x) {
        const int K = a.D - a.Do + 1, P = 4 + K - 1, PX = (P + 3) & ~3;
        const uint64_t dims[4] = {(uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.D, (uint64_t)a.N * a.Ci};
        const uint64_t strides[3] = {(uint64_t)a.W * 4, (uint64_t)a.H * a.W * 4,
                                     (uint64_t)a.D * a.H * a.W * 4};
        const uint32_t box[4] = {(uint32_t)PX, (uint32_t)P, (uint32_t)P, (uint32_t)a.Ci};
        const int st = encode_tmap_f32_4d(&a.tmap, a.x, dims, strides, box);
        if (st != CN_OK) return st;
        a.tmap_base = a.x;
    }
    record_launch(ev, 0, s);
    cfg.kern<<<cfg.grid, cfg.threads, cfg.smem, s>>>(a);
    record_launch(ev, 1, s);
    return cudaGetLastError() == cudaSuccess ? CN_OK : CN_ERR_CUDA;
}

}  // namespace cn
