// Variant 2: Conv2d or ConvTranspose2d (stride 1, padding 0, channel groups)
// -> activation -> GroupNorm / InstanceNorm / none -> post scale, with the
// full normalized tensor as the output.
//
// Method (l2_p17, Conv2d -> InstanceNorm2d -> divide; l2_p19,
// ConvTranspose2d -> GELU -> GroupNorm): the statistics of a normalization
// group span a whole (C/G) x H x W block of one sample, so nothing can be
// normalized before the whole block is computed.  The transcripts' answer is
// a pass that computes the conv, a statistics step and a normalize pass; here
// that is two launches:
//   A. conv + bias + activation for a tile, the pre-norm value written to
//      out, and per-(n, c, tile) moments (count, mean, M2); the last CTA of
//      each sample merges the moments in a fixed order (fp64) into
//      per-channel coefficients (mu_g, a = gamma*rstd*scale, bb = beta*scale);
//   B. a single read-modify-write of out: (y - mu) * a + bb.
// The transposed conv is handled as the adjoint of the stride-1 conv
// (l2_p19 derivation): output (i, j) gathers x[i - p][j - q] * w[ci][co][p][q]
// with out-of-range x read as zero; the tile origin is shifted by K-1 and
// the filter taps are reversed while staging, so both kinds share one
// mainloop.
//
// Mapping of kernel A: a thread owns COT=8 output channels x RW consecutive
// outputs of one output row; the lanes of a warp own (row, segment) items of
// the CTA tile, rows fastest (conflict-free shared loads with a row pitch
// of 4 mod 8 floats); warps split into channel slices x spatial groups.
// Input channels stream through a two-stage cp.async pipeline holding the
// haloed input tile and the tile's filter slice.
#include "cn_common.cuh"
#include "cn_internal.h"

#include <algorithm>

namespace cn {
namespace {
constexpr int COT = 8;

template <int K, int RW, bool TRANSPOSED>
__global__ void __launch_bounds__(256) k_conv2d_act_stats(Full2dArgs a) {
    extern __shared__ __align__(16) float smem[];
    constexpr int XW = RW + K - 1;
    constexpr bool VEC = (RW % 4) == 0;
    constexpr int LOADW = VEC ? ((XW + 3) & ~3) : XW;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int cs = warp % a.wco;
    const int sg = warp / a.wco;
    const int COB = COT * a.wco;
    int bid = blockIdx.x;
    const int ct = bid % a.col_tiles;
    bid /= a.col_tiles;
    const int rt = bid % a.row_tiles;
    bid /= a.row_tiles;
    const int cob = bid % a.ncob;
    const int n = bid / a.ncob;
    const int co0 = cob * COB;
    const int g = co0 / a.Cog;
    const int ci0 = g * a.Cig;
    const int r0 = rt * a.TR;
    const int c0 = ct * a.NT * RW;
    const int ir0 = TRANSPOSED ? r0 - (K - 1) : r0;
    const int ic0 = TRANSPOSED ? c0 - (K - 1) : c0;

    const int item = sg * 32 + lane;
    const int il = item % a.TR;
    const int sl_raw = item / a.TR;
    const bool item_ok = sl_raw < a.NT;
    const int sl = item_ok ? sl_raw : 0;
    const int orow = r0 + il;
    const int ocol0 = c0 + sl * RW;

    const int xstage = a.cib * a.rows_in * a.pitch;

    auto load_stage = [&](int chunk, int buf) {
        float *sxb = smem + (size_t)buf * a.stage_floats;
        float *swb = sxb + xstage;
        const int cbase = chunk * a.cib;
        const int nrows = a.cib * a.rows_in;
        for (int rI = warp; rI < nrows; rI += nwarps) {
            const int cl = rI / a.rows_in, rr = rI - cl * a.rows_in;
            const int gr = ir0 + rr;
            const bool rok = (cbase + cl < a.Cig) && gr >= 0 && gr < a.H;
            const float *src =
                a.x + (((size_t)n * a.Ci + ci0 + (rok ? cbase + cl : 0)) * a.H + (rok ? gr : 0)) * a.W;
            float *dst = sxb + (size_t)rI * a.pitch;
            for (int cc = lane; cc < a.cols_in; cc += 32) {
                const int gc = ic0 + cc;
                const bool ok = rok && gc >= 0 && gc < a.W;
                cp_async4(dst + cc, ok ? (const void *)(src + gc) : (const void *)a.x, ok);
            }
        }
        const int totw = a.cib * K * K * COB;
        for (int i = tid; i < totw; i += blockDim.x) {
            const int col = i % COB;
            const int t = i / COB;
            const int tap = t % (K * K), cl = t / (K * K);
            const int kh = tap / K, kw = tap - kh * K;
            const int cil = cbase + cl;
            float v = 0.0f;
            if (cil < a.Cig) {
                if (TRANSPOSED) {
                    const int col_g = co0 - g * a.Cog + col;
                    v = __ldg(a.w + (((size_t)(ci0 + cil) * a.Cog + col_g) * K + (K - 1 - kh)) * K +
                              (K - 1 - kw));
                } else {
                    v = __ldg(a.w + (((size_t)(co0 + col) * a.Cig + cil) * K + kh) * K + kw);
                }
            }
            swb[i] = v;
        }
    };

    float acc[COT][RW];
#pragma unroll
    for (int c = 0; c < COT; ++c)
#pragma unroll
        for (int i = 0; i < RW; ++i) acc[c][i] = 0.0f;

    load_stage(0, 0);
    cp_async_commit();
    for (int chunk = 0; chunk < a.nchunk; ++chunk) {
        if (chunk + 1 < a.nchunk) load_stage(chunk + 1, (chunk + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const float *sxb = smem + (size_t)(chunk & 1) * a.stage_floats;
        const float *swb = sxb + xstage;
        const int ncl = min(a.cib, a.Cig - chunk * a.cib);
        for (int cl = 0; cl < ncl; ++cl) {
            CN_UNROLL(CN_TAP_UNROLL)
            for (int kh = 0; kh < K; ++kh) {
                const float *xp = sxb + (size_t)(cl * a.rows_in + il + kh) * a.pitch + sl * RW;
                float xr[LOADW];
                if constexpr (VEC) {
#pragma unroll
                    for (int j = 0; j < LOADW / 4; ++j) {
                        const float4 v = *reinterpret_cast<const float4 *>(xp + 4 * j);
                        xr[4 * j + 0] = v.x;
                        xr[4 * j + 1] = v.y;
                        xr[4 * j + 2] = v.z;
                        xr[4 * j + 3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < LOADW; ++j) xr[j] = xp[j];
                }
#pragma unroll
                for (int kw = 0; kw < K; ++kw) {
                    const float4 *wp = reinterpret_cast<const float4 *>(
                        swb + (size_t)((cl * K + kh) * K + kw) * COB + cs * COT);
                    const float4 w0 = wp[0], w1 = wp[1];
#pragma unroll
                    for (int i = 0; i < RW; ++i) {
                        const float xv = xr[i + kw];
                        acc[0][i] = fmaf(xv, w0.x, acc[0][i]);
                        acc[1][i] = fmaf(xv, w0.y, acc[1][i]);
                        acc[2][i] = fmaf(xv, w0.z, acc[2][i]);
                        acc[3][i] = fmaf(xv, w0.w, acc[3][i]);
                        acc[4][i] = fmaf(xv, w1.x, acc[4][i]);
                        acc[5][i] = fmaf(xv, w1.y, acc[5][i]);
                        acc[6][i] = fmaf(xv, w1.z, acc[6][i]);
                        acc[7][i] = fmaf(xv, w1.w, acc[7][i]);
                    }
                }
            }
        }
        __syncthreads();
    }

    // ---- epilogue: bias + activation, store the pre-norm value, moments ----
    double *sred = reinterpret_cast<double *>(smem + 2 * (size_t)a.stage_floats);
    const bool row_ok = item_ok && orow < a.Ho;
#pragma unroll
    for (int c = 0; c < COT; ++c) {
        const int co = co0 + cs * COT + c;
        const float bias = a.b ? __ldg(a.b + co) : 0.0f;
        float s = 0.0f, cnt = 0.0f;
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const float v = apply_act(a.act, acc[c][i] + bias);
            acc[c][i] = v;
            if (row_ok && ocol0 + i < a.Wo) {
                s += v;
                cnt += 1.0f;
            }
        }
        const float mean = cnt > 0.0f ? s / cnt : 0.0f;
        float m2 = 0.0f;
        float *op = a.out + (((size_t)n * a.Co + co) * a.Ho + (row_ok ? orow : 0)) * a.Wo + ocol0;
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            if (row_ok && ocol0 + i < a.Wo) {
                const float dv = acc[c][i] - mean;
                m2 = fmaf(dv, dv, m2);
                op[i] = acc[c][i];
            }
        }
        Moments<float> m{cnt, mean, m2};
        m = warp_merge(m);
        if (lane == 0) {
            double *o = sred + ((size_t)sg * COB + cs * COT + c) * 3;
            o[0] = m.n;
            o[1] = m.mean;
            o[2] = m.m2;
        }
    }
    __syncthreads();
    const int tile = rt * a.col_tiles + ct;
    for (int c = tid; c < COB; c += blockDim.x) {
        Moments<double> m{0.0, 0.0, 0.0};
        for (int q = 0; q < a.wsp; ++q) {
            const double *o = sred + ((size_t)q * COB + c) * 3;
            m = merge(m, Moments<double>{o[0], o[1], o[2]});
        }
        double *p = a.partial + (((size_t)n * a.Co + co0 + c) * a.ntiles + tile) * 3;
        p[0] = m.n;
        p[1] = m.mean;
        p[2] = m.m2;
    }

    // ---- the last CTA of sample n turns the moments into coefficients ----
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int prev = atomicAdd(a.tickets + n, 1);
        s_last = (prev == a.ncob * a.ntiles - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    double *sch = reinterpret_cast<double *>(smem);
    for (int c = tid; c < a.Co; c += blockDim.x) {
        Moments<double> m{0.0, 0.0, 0.0};
        const double *p = a.partial + ((size_t)n * a.Co + c) * a.ntiles * 3;
        for (int t = 0; t < a.ntiles; ++t)
            m = merge(m, Moments<double>{ldcg_f64(p + 3 * t), ldcg_f64(p + 3 * t + 1),
                                         ldcg_f64(p + 3 * t + 2)});
        sch[c * 3 + 0] = m.n;
        sch[c * 3 + 1] = m.mean;
        sch[c * 3 + 2] = m.m2;
    }
    __syncthreads();
    for (int c = tid; c < a.Co; c += blockDim.x) {
        float4 cf;
        if (a.norm == CN_NORM_NONE) {
            cf = make_float4(0.0f, a.post_scale, 0.0f, 0.0f);
        } else {
            const int cpg = a.Co / a.NG, gg = c / cpg;
            Moments<double> mg{0.0, 0.0, 0.0};
            for (int j = 0; j < cpg; ++j) {
                const int cc = gg * cpg + j;
                mg = merge(mg, Moments<double>{sch[cc * 3], sch[cc * 3 + 1], sch[cc * 3 + 2]});
            }
            const double rstd = 1.0 / sqrt(mg.m2 / mg.n + (double)a.eps);
            const double ga = a.affine ? (double)a.gamma[c] : 1.0;
            const double be = a.affine ? (double)a.beta[c] : 0.0;
            cf = make_float4((float)mg.mean, (float)(rstd * ga * a.post_scale),
                             (float)(be * a.post_scale), 0.0f);
        }
        a.coef[(size_t)n * a.Co + c] = cf;
    }
    if (tid == 0) a.tickets[n] = 0;
}

// Normalize pass: out = (y - mu) * a + bb per (n, c) plane, in place.
__global__ void __launch_bounds__(256) k_norm_apply(float *out, const float4 *coef, long long S,
                                                    int vec4) {
    const size_t plane = blockIdx.x;
    const float4 cf = coef[plane];
    float *p = out + plane * (size_t)S;
    const long long step = (long long)gridDim.y * blockDim.x;
    if (vec4) {
        float4 *p4 = reinterpret_cast<float4 *>(p);
        const long long n4 = S >> 2;
        for (long long i = (long long)blockIdx.y * blockDim.x + threadIdx.x; i < n4; i += step) {
            float4 v = p4[i];
            v.x = (v.x - cf.x) * cf.y + cf.z;
            v.y = (v.y - cf.x) * cf.y + cf.z;
            v.z = (v.z - cf.x) * cf.y + cf.z;
            v.w = (v.w - cf.x) * cf.y + cf.z;
            p4[i] = v;
        }
    } else {
        for (long long i = (long long)blockIdx.y * blockDim.x + threadIdx.x; i < S; i += step)
            p[i] = (p[i] - cf.x) * cf.y + cf.z;
    }
}

struct Inst {
    int K, RW, T;
    Full2dKernel fn;
    const char *name;
};
#define CN_FULL_INST(K, RW, T)                                       \
    {K, RW, T, k_conv2d_act_stats<K, RW, (T != 0)>,                  \
     "k_conv2d_act_stats<" #K "," #RW "," #T ">,k_norm_apply"}
const Inst kInst[] = {
    CN_FULL_INST(1, 16, 0), CN_FULL_INST(2, 16, 0), CN_FULL_INST(3, 16, 0), CN_FULL_INST(3, 13, 0),
    CN_FULL_INST(4, 16, 0), CN_FULL_INST(1, 16, 1), CN_FULL_INST(2, 16, 1), CN_FULL_INST(3, 16, 1),
    CN_FULL_INST(3, 13, 1), CN_FULL_INST(4, 16, 1),
};
#undef CN_FULL_INST

struct Tiling {
    int wsp, TR, NT;
    double cost;
};

Tiling choose_tiling(int Ho, int Wo, int RW, int max_wsp) {
    Tiling best{1, 1, 1, 1e30};
    const int nseg = (Wo + RW - 1) / RW;
    for (int wsp = 1; wsp <= max_wsp; ++wsp) {
        const int lanes = 32 * wsp;
        int NT, TR;
        if (nseg <= lanes) {
            NT = nseg;
            TR = lanes / nseg;
        } else {
            NT = lanes;
            TR = 1;
        }
        TR = std::min(TR, std::max(1, Ho));
        const int rtiles = (Ho + TR - 1) / TR, ctiles = (nseg + NT - 1) / NT;
        const double row_w = (double)rtiles * TR / Ho;
        const double col_w = (double)ctiles * NT * RW / Wo;
        const double lane_w = (double)lanes / (TR * NT);
        const double cost = row_w * col_w * lane_w * (1.0 + 0.02 * (1.0 / wsp));
        if (cost < best.cost - 1e-9) best = Tiling{wsp, TR, NT, cost};
    }
    return best;
}

int pick_wco(int units) {
    for (int c = 8; c >= 1; --c)
        if (units % c == 0) return c;
    return 1;
}
}  // namespace

int full2d_plan(const conv_norm_desc &d, Full2dArgs &a, Full2dConfig &cfg) {
    const int T = d.conv == CN_CONVT2D ? 1 : 0;
    const int K = d.k;
    const int Ho = T ? d.H + K - 1 : d.H - K + 1;
    const int Wo = T ? d.W + K - 1 : d.W - K + 1;
    const int Cig = d.C_in / d.groups, Cog = d.C_out / d.groups;
    if (Cog % COT != 0) return CN_ERR_UNSUPPORTED;
    const int wco = pick_wco(Cog / COT);
    const int max_wsp = std::max(1, 8 / wco);
    const Inst *best = nullptr;
    Tiling bt{};
    double best_cost = 1e30;
    for (const Inst &in : kInst) {
        if (in.K != K || in.T != T) continue;
        const Tiling t = choose_tiling(Ho, Wo, in.RW, max_wsp);
        const int XW = in.RW + K - 1;
        const double loads = (in.RW % 4 == 0) ? (XW + 3) / 4 : XW;
        const double ratio = 1.0 + (loads + 2.0 * K) / (8.0 * K * in.RW);
        const double cost = t.cost * ratio;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = &in;
            bt = t;
        }
    }
    if (!best) return CN_ERR_UNSUPPORTED;
    const int RW = best->RW;
    const int XW = RW + K - 1;
    const int LOADW = (RW % 4 == 0) ? ((XW + 3) & ~3) : XW;
    a.N = d.N;
    a.Ci = d.C_in;
    a.Co = d.C_out;
    a.H = d.H;
    a.W = d.W;
    a.Ho = Ho;
    a.Wo = Wo;
    a.Cig = Cig;
    a.Cog = Cog;
    a.wco = wco;
    a.wsp = bt.wsp;
    a.TR = bt.TR;
    a.NT = bt.NT;
    const int nseg = (Wo + RW - 1) / RW;
    a.row_tiles = (Ho + a.TR - 1) / a.TR;
    a.col_tiles = (nseg + a.NT - 1) / a.NT;
    a.ncob = d.C_out / (COT * wco);
    a.ntiles = a.row_tiles * a.col_tiles;
    a.rows_in = a.TR + K - 1;
    a.cols_in = a.NT * RW + K - 1;
    int pitch = std::max((a.NT - 1) * RW + LOADW, a.cols_in);
    pitch = (pitch + 3) & ~3;
    if (((pitch / 4) & 1) == 0) pitch += 4;
    a.pitch = pitch;
    const int COB = COT * wco;
    const int per_ci = a.rows_in * pitch + K * K * COB;
    int cib = std::min(Cig, 8);
    while (cib > 1 && 2 * (size_t)cib * per_ci * 4 > 100 * 1024) --cib;
    a.cib = cib;
    a.nchunk = (Cig + cib - 1) / cib;
    a.stage_floats = ((cib * per_ci) + 3) & ~3;
    a.act = d.act;
    a.norm = d.norm;
    a.NG = d.norm == CN_NORM_GROUP ? d.num_groups : d.C_out;
    a.affine = d.affine && d.norm != CN_NORM_NONE;
    a.eps = d.eps;
    a.post_scale = d.post_scale;
    a.S = (long long)Ho * Wo;
    a.apply_needed = !(d.norm == CN_NORM_NONE && d.post_scale == 1.0f);
    a.vec4 = (a.S % 4) == 0;
    const int threads = 32 * wco * a.wsp;
    size_t smem = (size_t)2 * a.stage_floats * 4 + (size_t)a.wsp * COB * 3 * 8;
    smem = std::max(smem, (size_t)d.C_out * 3 * 8);
    if (smem > 227 * 1024) return CN_ERR_UNSUPPORTED;
    const long long grid = (long long)d.N * a.ncob * a.ntiles;
    if (grid > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;
    cfg.kern = best->fn;
    cfg.names = best->name;
    cfg.K = K;
    cfg.RW = RW;
    cfg.transposed = T;
    cfg.threads = threads;
    cfg.smem = (int)smem;
    cfg.grid = (int)grid;
    cfg.apply_threads = 256;
    const long long units = a.vec4 ? a.S / 4 : a.S;
    long long gy = (units + 256 * 4 - 1) / (256 * 4);
    cfg.apply_grid_y = (int)std::max(1LL, std::min(gy, 65535LL));
    const long long gx = (long long)d.N * d.C_out;
    if (gx > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;
    cfg.apply_grid_x = (int)gx;
    return CN_OK;
}

size_t full2d_workspace(const Full2dArgs &a) {
    const size_t part = (size_t)a.N * a.Co * a.ntiles * 3 * sizeof(double);
    const size_t coef = (size_t)a.N * a.Co * sizeof(float4);
    return ((part + 255) & ~(size_t)255) + ((coef + 255) & ~(size_t)255) + (size_t)a.N * sizeof(int);
}

void full2d_bind_workspace(Full2dArgs &a, char *base, int *err_flag) {
    const size_t part = (size_t)a.N * a.Co * a.ntiles * 3 * sizeof(double);
    const size_t coef = (size_t)a.N * a.Co * sizeof(float4);
    a.partial = reinterpret_cast<double *>(base);
    a.coef = reinterpret_cast<float4 *>(base + ((part + 255) & ~(size_t)255));
    a.tickets = reinterpret_cast<int *>(base + ((part + 255) & ~(size_t)255) +
                                        ((coef + 255) & ~(size_t)255));
    a.err = err_flag;
}

int full2d_prepare(const Full2dConfig &cfg) {
    if (cudaFuncSetAttribute(cfg.kern, cudaFuncAttributeMaxDynamicSharedMemorySize, cfg.smem) !=
        cudaSuccess)
        return CN_ERR_CUDA;
    return CN_OK;
}

int full2d_launches(const Full2dConfig &cfg, const Full2dArgs &a) {
    if (cfg.grid == 0) return 0;
    return 1 + (a.apply_needed ? 1 : 0);
}

int full2d_launch(const Full2dConfig &cfg, const Full2dArgs &a, cudaStream_t s) {
    if (cfg.grid == 0) return CN_OK;
    cfg.kern<<<cfg.grid, cfg.threads, cfg.smem, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return CN_ERR_CUDA;
    if (a.apply_needed) {
        dim3 grid(cfg.apply_grid_x, cfg.apply_grid_y);
        k_norm_apply<<<grid, cfg.apply_threads, 0, s>>>(a.out, a.coef, a.S, a.vec4);
        if (cudaGetLastError() != cudaSuccess) return CN_ERR_CUDA;
    }
    return CN_OK;
}

}  // namespace cn
