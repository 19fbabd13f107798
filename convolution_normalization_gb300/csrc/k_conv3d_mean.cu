// Variant 0: Conv3d -> activation -> GroupNorm/InstanceNorm -> mean over D,H,W
// in ONE launch, without writing the conv tensor.
//
// Method (l2_p27, Conv3d -> HardSwish -> GroupNorm -> mean): the mean over
// space of a GroupNorm output only needs, per channel c of sample n, the
// spatial mean m_c and the spread of the activated conv values:
//   out[n,c] = gamma_c * (m_c - mu_g) / sqrt(var_g + eps) + beta_c,
// with mu_g, var_g the (population) mean and variance over the group's
// channels and all positions.  So the kernel computes the conv + activation
// in registers, reduces each channel to (count, mean, M2) moments, and the
// last CTA of each sample merges the moments (fixed order, fp64) and writes
// the (N, C_out) result.
//
// Mapping: work items are chunks of 32*wrows consecutive rows of a sample's
// flattened (d, h, w-segment) output-row list; one persistent CTA per SM
// walks them.  Each thread owns COT output channels x RW consecutive outputs
// of one row; the lanes of a warp own 32 consecutive rows; warps split the
// channel block and the row groups.  A chunk's input depth planes, for all
// input channels, arrive in shared memory with ONE TMA tensor copy (box =
// pitch x H x planes x C_in; columns past W arrive zero-filled) into one of
// two buffers, so the next chunk loads while this one computes; and
// the filter of its channel block regrouped so that the K*COT weights a
// thread needs for one tap row (ci, kd, kh) are contiguous.  The inner loop
// per tap row loads one input row segment and those weights into registers
// (vector loads, broadcast across the warp) and issues COT*K*RW FFMAs.
#include "cn_common.cuh"
#include "cn_internal.h"
#include "cn_mean_common.cuh"

#include <algorithm>
#include <cstdlib>

namespace cn {

namespace {

// Bias + activation of RW values in place, then their moments (the first
// nvalid values are valid; all are when nvalid == RW).
template <int RW, int ACT>
CN_DEV Moments<float> row_moments(float (&v)[RW], float bias, int nvalid) {
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        float t = v[i] + bias;
        if (ACT == ACT_HARDSWISH) t = hardswish(t);
        if (ACT == ACT_GELU) t = gelu_erf(t);
        v[i] = t;
    }
    float s = 0.0f, m2 = 0.0f;
    if (nvalid == RW) {
#pragma unroll
        for (int i = 0; i < RW; ++i) s += v[i];
        const float mean = s * (1.0f / RW);
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const float d = v[i] - mean;
            m2 = fmaf(d, d, m2);
        }
        return Moments<float>{(float)RW, mean, m2};
    }
#pragma unroll
    for (int i = 0; i < RW; ++i) s += (i < nvalid) ? v[i] : 0.0f;
    const float mean = nvalid > 0 ? s / (float)nvalid : 0.0f;
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        const float d = (i < nvalid) ? v[i] - mean : 0.0f;
        m2 = fmaf(d, d, m2);
    }
    return Moments<float>{(float)nvalid, mean, m2};
}

// Threads per CTA this instantiation allows (register budget of one SM).
constexpr int mean_max_threads(int COT, int RW) { return COT * RW <= 64 ? 512 : 256; }

template <int K, int RW, int COT>
__global__ void __launch_bounds__(mean_max_threads(COT, RW), 1)
    k_conv3d_act_mean(const __grid_constant__ Mean3dArgs a) {
    extern __shared__ __align__(128) float smem[];
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int s_last, s_next;
    constexpr int KKK = K * K * K;
    constexpr int LOADW = (RW + K - 1 + 3) & ~3;
    constexpr int WS = COT * K;  // weights of one tap row for one thread's slice
    const int COB = COT * a.wco;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cs = warp % a.wco;
    const int rg = warp / a.wco;
    const int HP = a.H * a.pitch;
    float *sw = smem + (size_t)a.nbuf * a.buf_stride;
    double *sred = reinterpret_cast<double *>(sw + (size_t)a.Ci * KKK * COB);
    double *sch = sred + (size_t)a.wrows * COB * 3;
    const int wrow = COB * K;  // floats per tap row of the staged filter

    // work item q -> (channel block, sample, chunk of 32*wrows rows)
    auto decode = [&](int q, int &cob, int &n, int &chunk) {
        chunk = q % a.nchunks;
        q /= a.nchunks;
        n = q % a.N;
        cob = q / a.N;
    };
    auto plane_range = [&](int chunk, int &d_lo, int &np) {
        const int r_begin = chunk * a.rows_per_cta;
        const int r_end = min(a.rows, r_begin + a.rows_per_cta);
        d_lo = (r_begin / a.nseg) / a.Ho;
        np = ((r_end - 1) / a.nseg) / a.Ho - d_lo + K;
    };
    // one TMA tensor copy brings a chunk's input planes (all channels)
    auto issue = [&](int q, int b) {
        int cob, n, chunk, d_lo, np;
        decode(q, cob, n, chunk);
        plane_range(chunk, d_lo, np);
        fence_proxy_async();
        mbar_arrive_expect_tx(&bars[b], (uint32_t)(a.Ci * a.planes_max * HP * 4));
        tma_load_4d(smem + (size_t)b * a.buf_stride, &a.tmap, 0, 0, d_lo, n * a.Ci, &bars[b]);
    };

    if (a.use_tma && tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    __syncthreads();
    int q = blockIdx.x;
    if (a.use_tma && tid == 0 && q < a.items) issue(q, 0);
    int cur_cob = -1;
    for (int j = 0; q < a.items; ++j) {
        const int b = (a.nbuf == 2) ? (j & 1) : 0;
        int cob, n, chunk, d_lo, np;
        decode(q, cob, n, chunk);
        plane_range(chunk, d_lo, np);
        const int co0 = cob * COB;
        float *sx = smem + (size_t)b * a.buf_stride;

        if (a.use_tma) {
            // two buffers: prefetch the next item (static stride) into the
            // other buffer, freed by the barrier that ended the previous
            // iteration.  One buffer: the next item is claimed and issued once
            // this item's mainloop is done (below).
            if (tid == 0 && a.nbuf == 2 && q + (int)gridDim.x < a.items) issue(q + gridDim.x, b ^ 1);
        } else {
            const float *xn = a.x + (size_t)n * a.Ci * a.D * a.H * a.W;
            const int nrows = a.Ci * np * a.H;
            const int nwarps = blockDim.x >> 5;
            for (int row = warp; row < nrows; row += nwarps) {
                const int h = row % a.H, t = row / a.H;
                const int p = t % np, ci = t / np;
                const float *src = xn + (((size_t)ci * a.D + d_lo + p) * a.H + h) * a.W;
                float *dst = sx + ((size_t)(ci * a.planes_max + p) * a.H + h) * a.pitch;
                for (int c = lane; c < a.W; c += 32) cp_async4(dst + c, src + c, true);
                for (int c = a.W + lane; c < a.pitch; c += 32) dst[c] = 0.0f;
            }
            cp_async_commit();
        }
        // filter of this channel block, staged when the block changes: for
        // each tap row (ci, kd, kh) and each COT-channel slice the K*COT
        // weights [kw][c] sit together.  Coalesced reads, four in flight.
        if (a.nbuf == 2 && tid == 0) s_next = q + gridDim.x;
        if (cob != cur_cob) {
            const int ckkk = a.Ci * KKK, total = COB * ckkk;
            const float *wg = a.w + (size_t)co0 * ckkk;
            for (int base = tid; base < total; base += 4 * blockDim.x) {
                float v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = base + u * blockDim.x;
                    v[u] = e < total ? __ldg(wg + e) : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = base + u * blockDim.x;
                    if (e < total) {
                        const int col = e / ckkk, t = e - col * ckkk;
                        const int kw = t % K, trow = t / K;
                        sw[trow * wrow + (col / COT) * WS + kw * COT + col % COT] = v[u];
                    }
                }
            }
            cur_cob = cob;
        }
        if (a.use_tma) {
            const uint32_t parity = (a.nbuf == 2) ? ((j >> 1) & 1) : (j & 1);
            if (!mbar_wait_bounded(&bars[b], parity, kWaitLimitNs)) {
                flag_error(a.err, ERR_TIMEOUT);
                // let a late copy land before the buffer is reused
                mbar_wait_bounded(&bars[b], parity, kWaitLimitNs);
            }
        } else {
            cp_async_wait_all();
        }
        __syncthreads();

        // ---- mainloop ----
        const int r_begin = chunk * a.rows_per_cta;
        const int r_end = min(a.rows, r_begin + a.rows_per_cta);
        int r = r_begin + rg * 32 + lane;
        const bool rvalid = r < r_end;
        if (!rvalid) r = r_end - 1;
        const int seg = r % a.nseg;
        const int t0 = r / a.nseg;
        const int h = t0 % a.Ho, d = t0 / a.Ho;

        float acc[COT][RW];
#pragma unroll
        for (int c = 0; c < COT; ++c)
#pragma unroll
            for (int i = 0; i < RW; ++i) acc[c][i] = 0.0f;

        const float *xbase = sx + ((size_t)(d - d_lo) * a.H + h) * a.pitch + seg * RW;
        const float *wbase = sw + cs * WS;
        // Loop bounds depend only on kernel parameters (warp-uniform).  After a
        // staging timeout the loop still runs on whatever shared memory holds;
        // the error flag marks that forward's output as invalid.
        for (int ci = 0; ci < a.Ci; ++ci) {
            const float *xc = xbase + (size_t)ci * a.planes_max * HP;
            const float *wc = wbase + (size_t)ci * K * K * wrow;
            CN_UNROLL(CN_TAP_UNROLL)
            for (int kd = 0; kd < K; ++kd) {
                CN_UNROLL(CN_KH_UNROLL)
                for (int kh = 0; kh < K; ++kh) {
                    const float *xp = xc + kd * HP + kh * a.pitch;
                    float xr[LOADW];
#pragma unroll
                    for (int u = 0; u < LOADW / 4; ++u) {
                        const float4 v = *reinterpret_cast<const float4 *>(xp + 4 * u);
                        xr[4 * u + 0] = v.x;
                        xr[4 * u + 1] = v.y;
                        xr[4 * u + 2] = v.z;
                        xr[4 * u + 3] = v.w;
                    }
                    const float *wt = wc + (kd * K + kh) * wrow;
                    float wr[WS];
                    if constexpr (WS % 4 == 0) {
#pragma unroll
                        for (int u = 0; u < WS / 4; ++u) {
                            const float4 v = *reinterpret_cast<const float4 *>(wt + 4 * u);
                            wr[4 * u + 0] = v.x;
                            wr[4 * u + 1] = v.y;
                            wr[4 * u + 2] = v.z;
                            wr[4 * u + 3] = v.w;
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < WS / 2; ++u) {
                            const float2 v = *reinterpret_cast<const float2 *>(wt + 2 * u);
                            wr[2 * u + 0] = v.x;
                            wr[2 * u + 1] = v.y;
                        }
                    }
#pragma unroll
                    for (int kw = 0; kw < K; ++kw) {
#pragma unroll
                        for (int i = 0; i < RW; ++i) {
                            const float xv = xr[i + kw];
#pragma unroll
                            for (int c = 0; c < COT; ++c)
                                acc[c][i] = fmaf(xv, wr[kw * COT + c], acc[c][i]);
                        }
                    }
                }
            }
        }

        // ---- epilogue: bias + activation, per-channel moments ----
        const int nvalid = rvalid ? max(0, min(RW, a.Wo - seg * RW)) : 0;
#pragma unroll
        for (int c = 0; c < COT; ++c) {
            const int co = co0 + cs * COT + c;
            const float bias = a.b ? __ldg(a.b + co) : 0.0f;
            Moments<float> m;
            if (a.act == ACT_HARDSWISH)
                m = row_moments<RW, ACT_HARDSWISH>(acc[c], bias, nvalid);
            else if (a.act == ACT_GELU)
                m = row_moments<RW, ACT_GELU>(acc[c], bias, nvalid);
            else
                m = row_moments<RW, ACT_NONE>(acc[c], bias, nvalid);
            m = warp_merge(m);
            if (lane == 0) {
                double *o = sred + ((size_t)rg * COB + cs * COT + c) * 3;
                o[0] = m.n;
                o[1] = m.mean;
                o[2] = m.m2;
            }
        }
        __syncthreads();
        // Every warp is past its mainloop.  With one buffer, claim the next
        // item now (from the shared work counter, so faster SMs take more
        // items) and let its planes arrive while this epilogue finishes.
        if (a.nbuf == 1 && tid == 0) {
            s_next = (int)gridDim.x + atomicAdd(a.tickets + a.N, 1);
            if (a.use_tma && s_next < a.items) issue(s_next, 0);
        }
        for (int c = tid; c < COB; c += blockDim.x) {
            Moments<double> m{0.0, 0.0, 0.0};
            for (int g = 0; g < a.wrows; ++g) {
                const double *o = sred + ((size_t)g * COB + c) * 3;
                m = merge(m, Moments<double>{o[0], o[1], o[2]});
            }
            if (!CN_CHECK(n < a.N && chunk < a.nchunks && co0 + c < a.Co, a.err)) continue;
            double *p = a.partial + (((size_t)n * a.nchunks + chunk) * a.Co + co0 + c) * 3;
            p[0] = m.n;
            p[1] = m.mean;
            p[2] = m.m2;
        }

        // ---- the last CTA to finish a chunk of sample n merges its moments ----
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int prev = atomicAdd(a.tickets + n, 1);
            s_last = (prev == a.nchunks * a.ncob - 1);
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            for (int c = tid; c < a.Co; c += blockDim.x) {
                const Moments<double> m = mean_chunks_merged(a, a.nchunks, n, c);
                sch[c * 3 + 0] = m.n;
                sch[c * 3 + 1] = m.mean;
                sch[c * 3 + 2] = m.m2;
            }
            __syncthreads();
            for (int c = tid; c < a.Co; c += blockDim.x) mean_write_output(a, n, c, sch);
            if (tid == 0) a.tickets[n] = 0;
        }
        __syncthreads();  // buffer b, sred and sch are free for the next item
        q = s_next;
    }
    // the last CTA to leave resets the work counters for the next launch
    if (a.nbuf == 1 && tid == 0 && atomicAdd(a.tickets + a.N + 1, 1) == (int)gridDim.x - 1) {
        a.tickets[a.N] = 0;
        a.tickets[a.N + 1] = 0;
    }
}

struct Inst {
    int K, RW, COT;
    Mean3dKernel fn;
    const char *name;
    int max_threads() const { return mean_max_threads(COT, RW); }
};
#define CN_MEAN_INST(K, RW, C) \
    {K, RW, C, k_conv3d_act_mean<K, RW, C>, "k_conv3d_act_mean<" #K "," #RW "," #C ">"}
const Inst kInst[] = {
    CN_MEAN_INST(1, 8, 4),  CN_MEAN_INST(1, 16, 4), CN_MEAN_INST(2, 8, 4),  CN_MEAN_INST(2, 16, 4),
    CN_MEAN_INST(3, 8, 4),  CN_MEAN_INST(3, 16, 4), CN_MEAN_INST(3, 14, 4), CN_MEAN_INST(3, 29, 4),
    CN_MEAN_INST(4, 8, 4),  CN_MEAN_INST(4, 16, 4), CN_MEAN_INST(4, 14, 4), CN_MEAN_INST(4, 29, 4),
    CN_MEAN_INST(4, 29, 2), CN_MEAN_INST(3, 29, 2), CN_MEAN_INST(3, 14, 2),
};
#undef CN_MEAN_INST

int env_int(const char *name, int dflt) {
    const char *v = getenv(name);
    return v ? atoi(v) : dflt;
}
}  // namespace

int mean3d_plan(const conv_norm_desc &d, Mean3dArgs &a, Mean3dConfig &cfg) {
    // small batches: one CTA per (sample, normalization group)
    if (small3d_plan(d, a, cfg) == CN_OK) return CN_OK;
    a.small = 0;
    // the tensor-core kernel where the problem fits it
    if (tc3_plan(d, a.t, cfg.tc3) == CN_OK) {
        a.tc = 1;
        a.N = d.N;  // the fields the workspace and the plan's callers read
        a.Co = d.C_out;
        a.nchunks = a.t.ngroups * a.t.nsplit;
        a.items = a.t.items;
        cfg.name = cfg.tc3.name;
        cfg.threads = cfg.tc3.threads;
        cfg.smem = cfg.tc3.smem;
        cfg.grid = cfg.tc3.grid;
        return CN_OK;
    }
    a.tc = 0;
    const int K = d.k;
    const int Do = d.D - K + 1, Ho = d.H - K + 1, Wo = d.W - K + 1;
    if (d.groups != 1 || d.C_out % 4 != 0) return CN_ERR_UNSUPPORTED;
    // Channel slice per thread: 2 lets two 256-thread CTAs share an SM
    // (about 110 registers); 4 halves shared-memory traffic per FFMA but
    // needs about 190.  Measured on the k=4 workload: 0.80 ms vs 0.93 ms.
    const int want_cot = env_int("CN_MEAN3D_COT", 2);
    // pick the row width: an exact instantiation if there is one, else the
    // segmented width with the least padding.
    const Inst *best = nullptr;
    double best_cost = 1e30;
    for (const Inst &in : kInst) {
        if (in.K != K) continue;
        const int nseg = (Wo + in.RW - 1) / in.RW;
        if (nseg > 1 && (in.RW % 4) != 0) continue;  // float4 row loads need aligned segments
        const double waste = (double)nseg * in.RW / Wo;
        const double load = 1.0 + (double)(((in.RW + K - 1 + 3) / 4) + K) / (4.0 * K * in.RW);
        const double cost = waste * load * (in.COT == want_cot ? 1.0 : 1.001);
        if (cost < best_cost - 1e-12) {
            best_cost = cost;
            best = &in;
        }
    }
    if (!best) return CN_ERR_UNSUPPORTED;
    const int RW = best->RW, COT = best->COT;
    const int LOADW = (RW + K - 1 + 3) & ~3;
    a.N = d.N;
    a.Ci = d.C_in;
    a.Co = d.C_out;
    a.D = d.D;
    a.H = d.H;
    a.W = d.W;
    a.Do = Do;
    a.Ho = Ho;
    a.Wo = Wo;
    a.nseg = (Wo + RW - 1) / RW;
    a.rows = Do * Ho * a.nseg;
    int wco = 1;
    for (int c = 8; c >= 1; --c)
        if ((d.C_out / COT) % c == 0) {
            wco = c;
            break;
        }
    a.wco = wco;
    a.ncob = d.C_out / (COT * wco);
    const int COB = COT * wco;
    // Rows per chunk: as many 32-row groups as the thread budget allows (one
    // persistent CTA per SM keeps 16 warps resident when it is 512 threads).
    // Default: 256-thread CTAs with one staging buffer, so two persistent
    // CTAs share an SM and one's epilogue overlaps the other's mainloop (a
    // single 512-thread CTA with two buffers measured 0.90 vs 0.71 ms).
    const int max_wrows = std::max(1, best->max_threads() / (32 * wco));
    const int dflt_wrows = std::max(1, std::min(max_wrows, 8 / wco));
    int wrows = std::max(1, std::min(env_int("CN_MEAN3D_WROWS", dflt_wrows), max_wrows));
    int need = 0, pitch = 0, pm = 0;
    size_t smem = 0;
    for (;; --wrows) {
        a.wrows = wrows;
        a.rows_per_cta = 32 * wrows;
        a.nchunks = (a.rows + a.rows_per_cta - 1) / a.rows_per_cta;
        pm = 0;
        for (int ch = 0; ch < a.nchunks; ++ch) {
            const int rb = ch * a.rows_per_cta;
            const int re = std::min(a.rows, rb + a.rows_per_cta);
            const int dl = (rb / a.nseg) / Ho, dh = ((re - 1) / a.nseg) / Ho;
            pm = std::max(pm, dh - dl + K);
        }
        need = std::max((a.nseg - 1) * RW + LOADW, d.W);
        pitch = (need + 3) & ~3;
        if (((pitch / 4) & 1) == 0) pitch += 4;  // pitch = 4 (mod 8): conflict-free row loads
        const size_t buf = (((size_t)d.C_in * pm * d.H * pitch) + 31) & ~(size_t)31;
        const size_t rest = (size_t)d.C_in * K * K * K * COB * 4 + (size_t)wrows * COB * 3 * 8 +
                            (size_t)d.C_out * 3 * 8;
        a.buf_stride = (int)buf;
        if (2 * buf * 4 + rest <= 227 * 1024 && env_int("CN_MEAN3D_NBUF", 1) == 2) {
            a.nbuf = 2;
            smem = 2 * buf * 4 + rest;
            break;
        }
        if (buf * 4 + rest <= 227 * 1024) {
            a.nbuf = 1;
            smem = buf * 4 + rest;
            break;
        }
        if (wrows == 1) return CN_ERR_UNSUPPORTED;
    }
    a.planes_max = pm;
    a.pitch = pitch;
    a.vec16 = (d.W % 4 == 0);
    a.items = 0;
    // One TMA box covers a chunk's planes: every box extent must be <= 256
    // and the row stride a multiple of 16 bytes.
    a.use_tma = (d.W % 4 == 0) && pitch <= 256 && d.H <= 256 && pm <= 256 && d.C_in <= 256 &&
                env_int("CN_NO_TMA", 0) == 0;
    a.tmap_base = nullptr;
    a.act = d.act;
    a.norm = d.norm;
    a.G = d.norm == CN_NORM_GROUP ? d.num_groups : d.C_out;
    a.affine = d.affine && d.norm != CN_NORM_NONE;
    a.eps = d.eps;
    a.post_scale = d.post_scale;
    const long long items = (long long)d.N * a.ncob * a.nchunks;
    if (items > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;
    a.items = (int)items;
    cfg.kern = best->fn;
    cfg.name = best->name;
    cfg.K = K;
    cfg.RW = RW;
    cfg.COT = COT;
    cfg.threads = 32 * wco * wrows;
    cfg.smem = (int)smem;
    cfg.grid = std::min(a.items, 148);  // refined from the device in mean3d_prepare
    return CN_OK;
}

int mean3d_launches(const Mean3dConfig &cfg, const Mean3dArgs &a) {
    if (a.N == 0) return 0;
    return a.tc ? tc3_launches(cfg.tc3) : 1;
}

size_t mean3d_partial_bytes(const Mean3dArgs &a) {
    if (a.small) return small3d_partial_bytes(a);
    return (size_t)a.N * a.nchunks * a.Co * (a.tc ? sizeof(float4) : 3 * sizeof(double));
}

size_t mean3d_tickets(const Mean3dArgs &a) {
    return (a.small ? (size_t)a.N * a.sm_ngrp : (size_t)a.N) + 2;
}

size_t mean3d_workspace(const Mean3dArgs &a) {
    const size_t part = mean3d_partial_bytes(a);
    return ((part + 255) & ~(size_t)255) + mean3d_tickets(a) * sizeof(int);
}

int mean3d_prepare(Mean3dConfig &cfg, const Mean3dArgs &a) {
    if (a.small)  // the grid is one CTA per (sample, normalization group)
        return raise_dyn_smem(reinterpret_cast<const void *>(cfg.kern), cfg.smem) ==
                       cudaSuccess
                   ? CN_OK
                   : CN_ERR_CUDA;
    if (a.tc) {
        const int st = tc3_prepare(cfg.tc3, a.t);
        cfg.grid = cfg.tc3.grid;
        return st;
    }
    if (raise_dyn_smem(reinterpret_cast<const void *>(cfg.kern), cfg.smem) !=
        cudaSuccess)
        return CN_ERR_CUDA;
    // persistent grid: every CTA slot of the device, capped by the work items
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cfg.kern, cfg.threads, cfg.smem) !=
            cudaSuccess)
        return CN_ERR_CUDA;
    if (per_sm < 1) return CN_ERR_UNSUPPORTED;
    cfg.grid = (int)std::min<long long>((long long)sms * per_sm, (long long)a.items);
    if (env_int("CN_MEAN3D_ONE_ITEM_PER_CTA", 0)) cfg.grid = a.items;
    return CN_OK;
}

int mean3d_launch(const Mean3dConfig &cfg, Mean3dArgs &a, cudaStream_t s, const LaunchEvents *ev) {
    if (cfg.grid == 0) return CN_OK;
    if (a.small) {
        record_launch(ev, 0, s);
        cfg.kern<<<cfg.grid, cfg.threads, cfg.smem, s>>>(a);
        record_launch(ev, 1, s);
        return cudaGetLastError() == cudaSuccess ? CN_OK : CN_ERR_CUDA;
    }
    if (a.tc) {
        Tc3Args &t = a.t;
        t.x = a.x;
        t.w = a.w;
        t.b = a.b;
        t.gamma = a.gamma;
        t.beta = a.beta;
        t.out = a.out;
        t.err = a.err;
        t.partial = reinterpret_cast<float4 *>(a.partial);
        t.tickets = a.tickets;
        t.work = a.tickets + a.N;
        return tc3_launch(cfg.tc3, t, s, ev);
    }
    if (a.use_tma && a.tmap_base != a.x) {
        const uint64_t dims[4] = {(uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.D,
                                  (uint64_t)a.N * a.Ci};
        const uint64_t strides[3] = {(uint64_t)a.W * 4, (uint64_t)a.H * a.W * 4,
                                     (uint64_t)a.D * a.H * a.W * 4};
        const uint32_t box[4] = {(uint32_t)a.pitch, (uint32_t)a.H, (uint32_t)a.planes_max,
                                 (uint32_t)a.Ci};
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
