// Variant 2: Conv2d or ConvTranspose2d (stride 1, padding 0, channel groups)
// -> activation -> GroupNorm / InstanceNorm / none -> post scale, with the
// full normalized tensor as the output.
//
// Method (l2_p17, Conv2d -> InstanceNorm2d -> divide; l2_p19,
// ConvTranspose2d -> GELU -> GroupNorm): the statistics of a normalization
// group span a whole (C/G) x H x W block of one sample, so nothing can be
// normalized before the whole block is computed.  The transcripts' answer is
// a pass that computes the conv, a statistics step and a normalize pass; here
// that is three launches (after a tiny filter pre-pass):
//   A. conv + bias + activation for a tile, the pre-norm value written to
//      out, and per-(n, c, tile, warp) shifted power sums;
//   B. a small pass merging each normalization group's sums in a fixed order
//      (fp64) into per-channel coefficients (mu_g, a = gamma*rstd*scale,
//      bb = beta*scale);
//   C. a single read-modify-write of out: (y - mu) * a + bb.
// The transposed conv is handled as the adjoint of the stride-1 conv
// (l2_p19 derivation): output (i, j) gathers x[i - p][j - q] * w[ci][co][p][q]
// with out-of-range x read as zero; the tile origin is shifted by K-1 and
// the filter taps are reversed while staging, so both kinds share one
// mainloop.
//
// Mapping of kernel A: a thread owns COT output channels x RW consecutive
// outputs of one output row; the lanes of a warp own (row, segment) items of
// the CTA tile, rows fastest (conflict-free shared loads with a row pitch of
// 4 mod 8 floats); warps split into channel slices x spatial groups.  Input
// channels stream through a two-stage pipeline: each in-image input row of a
// stage arrives with one bulk async copy (TMA engine, completion on an
// mbarrier), out-of-image halo cells are zeroed once per kernel; the tile's
// filter slice is transposed into shared memory by the threads.
#include "cn_common.cuh"
#include "cn_internal.h"

#include <algorithm>
#include <cstdlib>

namespace cn {
namespace {

template <int ACT>
CN_DEV float act_value(float t) {
    if (ACT == ACT_HARDSWISH) return hardswish(t);
    if (ACT == ACT_GELU) return gelu_erf(t);
    return t;
}

// Bias + activation of RW values in place.
template <int RW, int ACT>
CN_DEV void bias_act(float (&v)[RW], float bias) {
#pragma unroll
    for (int i = 0; i < RW; ++i) v[i] = act_value<ACT>(v[i] + bias);
}
// Shifted sums (count, S1 = sum(v - K), S2 = sum((v - K)^2)) of the first
// nvalid of RW values (all on the common path).
template <int RW>
CN_DEV float3 shifted_sums(const float (&v)[RW], float K, int nvalid) {
    float s1 = 0.0f, s2 = 0.0f;
    if (nvalid == RW) {
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const float d = v[i] - K;
            s1 += d;
            s2 = fmaf(d, d, s2);
        }
    } else {
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const float d = (i < nvalid) ? v[i] - K : 0.0f;
            s1 += d;
            s2 = fmaf(d, d, s2);
        }
    }
    return make_float3((float)nvalid, s1, s2);
}

// Filter pre-pass: writes, for every (channel block, input-channel chunk)
// stage, the block's filter slice exactly as the conv kernel reads it from
// shared memory: [cl][kh][kw][col], taps reversed for the transposed conv,
// zero past the group's input channels.  One contiguous bulk copy per stage.
__global__ void __launch_bounds__(256) k_prep_weights(const float *__restrict__ w, float *wprep,
                                                      int K, int transposed, int Cig, int Cog,
                                                      int COB, int cib, int nchunk, int total) {
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
        int t = e;
        const int col = t % COB;
        t /= COB;
        const int tap = t % (K * K);
        t /= K * K;
        const int cl = t % cib;
        t /= cib;
        const int chunk = t % nchunk;
        const int cob = t / nchunk;
        const int kh = tap / K, kw = tap - kh * K;
        const int cil = chunk * cib + cl;
        const int co = cob * COB + col;
        float v = 0.0f;
        if (cil < Cig) {
            if (transposed) {
                const int g = co / Cog, col_g = co - g * Cog;
                v = w[(((size_t)(g * Cig + cil) * Cog + col_g) * K + (K - 1 - kh)) * K + (K - 1 - kw)];
            } else {
                v = w[(((size_t)co * Cig + cil) * K + kh) * K + kw];
            }
        }
        wprep[e] = v;
    }
}

// CTAs per SM an instantiation is compiled for: two with the small
// 4-channel x 16-output thread tile (at most 128 registers), else one.
constexpr int full_min_ctas(int COT, int RW) { return COT * RW <= 64 ? 2 : 1; }
constexpr int kMaxStages = 4;  // deepest input pipeline the kernel supports

// ACTT >= 0 compiles the epilogue for that one activation; -1 switches at
// run time (three copies of the unrolled epilogue, more instruction cache).
// OFF (with VECW = 4): the tile's first input column sits OFF floats past a
// 16-byte boundary of the row buffer (2 for the transposed k = 3 conv, whose
// tile origin moves left by k - 1); rows are then read as aligned float4
// windows starting OFF floats early, which keeps the loads conflict-free.
template <int K, int RW, int COT, int VECW, bool TRANSPOSED, int ACTT, int OFF = 0>
__global__ void __launch_bounds__(256, full_min_ctas(COT, RW))
    k_conv2d_act_stats(const __grid_constant__ Full2dArgs a) {
    extern __shared__ __align__(128) float smem[];
    // full[b]: stage data in buffer b has landed; empty[b]: every warp is done
    // reading buffer b
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages];
    __shared__ int s_tile[kMaxStages], s_chunk[kMaxStages];
    static_assert(COT == 4 || COT == 8, "channel slice of 4 or 8");
    static_assert(OFF == 0 || VECW == 4, "an input offset needs float4 row loads");
    constexpr int XW = RW + K - 1;
    constexpr int LOADW = (OFF + XW + VECW - 1) / VECW * VECW;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int cs = warp % a.wco;
    const int sg = warp / a.wco;
    const int COB = COT * a.wco;

    // tile t -> geometry
    struct Geo {
        int n, d, cob, rt, ct, co0, ci0, r0, c0, ir0, ic0, xs, off, gc_lo, gc_hi;
    };
    // tiles are ordered (sample, channel block, row tile, col tile); a
    // sample is (n, output depth d) of a Conv3d, or n of a 2-D conv
    auto geo = [&](int t) {
        Geo G;
        G.ct = t % a.col_tiles;
        t /= a.col_tiles;
        G.rt = t % a.row_tiles;
        t /= a.row_tiles;
        G.cob = t % a.ncob;
        const int smp = t / a.ncob;
        G.n = smp / a.Dv;
        G.d = smp - G.n * a.Dv;
        G.co0 = G.cob * COB;
        G.ci0 = (G.co0 / a.Cog) * a.Cig;
        G.r0 = G.rt * a.TR;
        G.c0 = G.ct * a.NT * RW;
        G.ir0 = TRANSPOSED ? G.r0 - (K - 1) : G.r0;
        G.ic0 = TRANSPOSED ? G.c0 - (K - 1) : G.c0;
        // Shared row buffers start at global column xs (a multiple of 4 when
        // rows arrive by bulk copy); the tile's first column sits at offset off.
        G.xs = a.use_bulk ? (G.ic0 & ~3) : G.ic0;
        G.off = G.ic0 - G.xs;
        G.gc_lo = max(G.ic0, 0) & ~3;
        G.gc_hi = min((G.ic0 + a.cols_in + 3) & ~3, a.W);
        return G;
    };

    // Input row gr of stacked channel cs (channel cs / KD, depth tap cs % KD)
    // for output depth d of sample n.
    auto x_row = [&](int n, int d, int cs, int gr) {
        const int ci = cs / a.KD, kd = cs - ci * a.KD;
        return a.x + ((((size_t)n * a.Ci + ci) * a.Din + d + kd) * a.H + gr) * a.W;
    };

    // ---- producer (warp 0): one stage = (tile, chunk of cib input channels) ----
    // Zeroes the stage's out-of-image rows (and, with several column tiles,
    // its out-of-image columns), then brings the in-image part of each input
    // row with one bulk copy and the prepared filter slice with another.  A
    // tile of -1 marks the end of this CTA's work.
    Geo PG{};          // producer's decoded current tile
    int pg_tile = -1;
    auto produce = [&](int tile, int chunk, int buf) {
        float *sxb = smem + (size_t)buf * a.stage_floats;
        if (tile < 0) {
            if (lane == 0) {
                s_tile[buf] = -1;
                s_chunk[buf] = 0;
                mbar_arrive_expect_tx(&full[buf], 0);
            }
            __syncwarp();
            return;
        }
        if (tile != pg_tile) {
            PG = geo(tile);
            pg_tile = tile;
        }
        const Geo &G = PG;
        const int cbase = chunk * a.cib;
        if (a.use_tma) {
            // one tensor copy of the stage's rows x columns x channels; the
            // parts outside the image (and past the group's channels at the
            // end of the tensor) arrive as zeros
            if (lane == 0) {
                s_tile[buf] = tile;
                s_chunk[buf] = chunk;
                mbar_arrive_expect_tx(&full[buf], (uint32_t)(a.xstage + a.wstage) * 4u);
                if (a.Din > 1)  // (cib / KD channels) x (KD depth taps) from plane d on
                    tma_load_5d(sxb, &a.xmap, G.xs, G.ir0, G.d, (G.ci0 + cbase) / a.KD, G.n, &full[buf]);
                else
                    tma_load_4d(sxb, &a.xmap, G.xs, G.ir0, G.ci0 + cbase, G.n, &full[buf]);
                bulk_load(sxb + a.xstage, a.wprep + ((size_t)G.cob * a.nchunk + chunk) * a.wstage,
                          (uint32_t)a.wstage * 4u, &full[buf]);
            }
            __syncwarp();
            return;
        }
        const int ncl = min(a.cib, a.Cig - cbase);
        const int gr_lo = max(G.ir0, 0), gr_hi = min(G.ir0 + a.rows_in, a.H);
        const int top = gr_lo - G.ir0, bot = gr_hi - G.ir0;  // in-image rows are [top, bot)
        for (int cl = 0; cl < ncl; ++cl) {
            float *rows = sxb + (size_t)cl * a.rows_in * a.pitch;
            for (int i = lane; i < top * a.pitch; i += 32) rows[i] = 0.0f;
            for (int i = bot * a.pitch + lane; i < a.rows_in * a.pitch; i += 32) rows[i] = 0.0f;
            if (a.col_tiles > 1) {
                for (int rr = top; rr < bot; ++rr) {
                    float *row = rows + (size_t)rr * a.pitch;
                    for (int c = lane; c < G.gc_lo - G.xs; c += 32) row[c] = 0.0f;
                    for (int c = G.gc_hi - G.xs + lane; c < a.pitch; c += 32) row[c] = 0.0f;
                }
            }
        }
        const int nr = gr_hi - gr_lo;
        const uint32_t row_bytes = (uint32_t)(G.gc_hi - G.gc_lo) * 4u;
        fence_proxy_async();
        if (lane == 0) {
            s_tile[buf] = tile;
            s_chunk[buf] = chunk;
            mbar_arrive_expect_tx(&full[buf],
                                  (uint32_t)(ncl * nr) * row_bytes + (uint32_t)a.wstage * 4u);
            bulk_load(sxb + a.xstage, a.wprep + ((size_t)G.cob * a.nchunk + chunk) * a.wstage,
                      (uint32_t)a.wstage * 4u, &full[buf]);
        }
        __syncwarp();
        for (int q = lane; q < ncl * nr; q += 32) {
            const int cl = q / nr, gr = gr_lo + q % nr;
            const float *src = x_row(G.n, G.d, G.ci0 + cbase + cl, gr) + G.gc_lo;
            float *dst = sxb + (size_t)(cl * a.rows_in + gr - G.ir0) * a.pitch + (G.gc_lo - G.xs);
            bulk_load(dst, src, row_bytes, &full[buf]);
        }
    };
    // Work claims (warp 0): the first tile is blockIdx.x; later tiles come
    // from the work counter, one claim kept in flight so its latency hides
    // behind a whole tile of work.  A claimed tile is always processed.
    int pending = 0;
    auto claim = [&]() {
        int t = __shfl_sync(0xffffffffu, pending, 0);
        if (lane == 0 && t < a.items) pending = (int)gridDim.x + atomicAdd(a.tickets + a.N, 1);
        return t < a.items ? t : -1;
    };

    // Both buffers start all zero: cells outside the image stay zero unless a
    // stage of another column tile writes them (then the producer re-zeroes).
    for (int i = tid; i < a.nstage * a.stage_floats; i += blockDim.x) smem[i] = 0.0f;
    if (tid == 0) {
        for (int b = 0; b < a.nstage; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&empty[b], nwarps);
        }
        fence_barrier_init();
    }
    fence_proxy_async();
    __syncthreads();

    // Producer state (warp 0): the last stage issued.  Stages run
    // (tile, chunk 0 .. nchunk-1) per claimed tile; nstage-1 stages are kept
    // in flight ahead of the consumers.
    int p_tile = -1, p_chunk = 0;
    bool p_done = false;
    auto advance = [&]() {
        if (p_chunk + 1 < a.nchunk) {
            ++p_chunk;
        } else {
            p_tile = claim();
            p_chunk = 0;
        }
    };
    if (warp == 0) {
        pending = (int)blockIdx.x;
        p_tile = claim();
        p_chunk = 0;
        if (a.use_bulk) {
            produce(p_tile, 0, 0);
            p_done = p_tile < 0;
            for (int b = 1; b < a.nstage - 1 && !p_done; ++b) {
                advance();
                produce(p_tile, p_chunk, b);
                p_done = p_tile < 0;
            }
        }
    }

    float acc[COT][RW];
    Geo G{};
    int il = 0, sl = 0;
    bool item_ok = false;
    for (int s = 0;; ++s) {
        int buf = 0;
        if (a.use_bulk) {
            buf = s % a.nstage;
            // issue stage s+nstage-1 into the buffer stage s-1 used, once
            // every warp has finished reading it
            if (warp == 0 && !p_done) {
                const int tb = (s + a.nstage - 1) % a.nstage;
                advance();
                if (s >= 1 && !mbar_wait_bounded(&empty[tb], ((s - 1) / a.nstage) & 1, kWaitLimitNs))
                    flag_error(a.err, ERR_TIMEOUT);
                produce(p_tile, p_chunk, tb);
                p_done = p_tile < 0;
            }
            const uint32_t par = (uint32_t)(s / a.nstage) & 1u;
            if (!mbar_wait_bounded(&full[buf], par, kWaitLimitNs)) {
                flag_error(a.err, ERR_TIMEOUT);
                mbar_wait_bounded(&full[buf], par, kWaitLimitNs);
            }
        } else {
            // synchronous staging with cp.async (rows not 16-byte multiples)
            __syncthreads();  // everyone is done with the buffer and s_tile
            if (warp == 0) {
                if (s > 0) advance();
                if (lane == 0) {
                    s_tile[0] = p_tile;
                    s_chunk[0] = p_chunk;
                }
            }
            __syncthreads();
            const int t = s_tile[0], ch = s_chunk[0];
            if (t >= 0) {
                const Geo H = geo(t);
                float *sxb = smem;
                const int cbase = ch * a.cib;
                for (int rI = warp; rI < a.cib * a.rows_in; rI += nwarps) {
                    const int cl = rI / a.rows_in, rr = rI - cl * a.rows_in;
                    const int gr = H.ir0 + rr;
                    const bool rok = (cbase + cl < a.Cig) && gr >= 0 && gr < a.H;
                    const float *src = x_row(H.n, H.d, H.ci0 + (rok ? cbase + cl : 0), rok ? gr : 0);
                    float *dst = sxb + (size_t)rI * a.pitch;
                    for (int cc = lane; cc < a.cols_in; cc += 32) {
                        const int gc = H.ic0 + cc;
                        const bool okc = rok && gc >= 0 && gc < a.W;
                        cp_async4(dst + cc, okc ? (const void *)(src + gc) : (const void *)a.x, okc);
                    }
                }
                cp_async_commit();
                const float *wsrc = a.wprep + ((size_t)H.cob * a.nchunk + ch) * a.wstage;
                for (int i = tid; i < a.wstage; i += blockDim.x) sxb[a.xstage + i] = __ldg(wsrc + i);
                cp_async_wait_all();
            }
            __syncthreads();
        }
        const int tile = s_tile[buf], chunk = s_chunk[buf];
        if (tile < 0) break;
        if (chunk == 0) {
            G = geo(tile);
            const int it = sg * 32 + lane;
            il = it % a.TR;
            const int sl_raw = it / a.TR;
            item_ok = sl_raw < a.NT;
            sl = item_ok ? sl_raw : 0;
#pragma unroll
            for (int c = 0; c < COT; ++c)
#pragma unroll
                for (int i = 0; i < RW; ++i) acc[c][i] = 0.0f;
        }
        const float *sxb = smem + (size_t)buf * a.stage_floats;
        const float *swb = sxb + a.xstage;
        const int ncl = min(a.cib, a.Cig - chunk * a.cib);
        for (int cl = 0; cl < ncl; ++cl) {
            CN_UNROLL(CN_TAP_UNROLL)
            for (int kh = 0; kh < K; ++kh) {
                const float *xp =
                    sxb + (size_t)(cl * a.rows_in + il + kh) * a.pitch + (G.off - OFF) + sl * RW;
                float xr[LOADW];
                if constexpr (VECW == 4) {
#pragma unroll
                    for (int j = 0; j < LOADW / 4; ++j) {
                        const float4 v = *reinterpret_cast<const float4 *>(xp + 4 * j);
                        xr[4 * j + 0] = v.x;
                        xr[4 * j + 1] = v.y;
                        xr[4 * j + 2] = v.z;
                        xr[4 * j + 3] = v.w;
                    }
                } else if constexpr (VECW == 2) {
#pragma unroll
                    for (int j = 0; j < LOADW / 2; ++j) {
                        const float2 v = *reinterpret_cast<const float2 *>(xp + 2 * j);
                        xr[2 * j + 0] = v.x;
                        xr[2 * j + 1] = v.y;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < LOADW; ++j) xr[j] = xp[j];
                }
#pragma unroll
                for (int kw = 0; kw < K; ++kw) {
                    const float4 *wp = reinterpret_cast<const float4 *>(
                        swb + (size_t)((cl * K + kh) * K + kw) * COB + cs * COT);
                    float wv[COT];
#pragma unroll
                    for (int q = 0; q < COT / 4; ++q) {
                        const float4 t = wp[q];
                        wv[4 * q + 0] = t.x;
                        wv[4 * q + 1] = t.y;
                        wv[4 * q + 2] = t.z;
                        wv[4 * q + 3] = t.w;
                    }
#pragma unroll
                    for (int i = 0; i < RW; ++i) {
                        const float xv = xr[OFF + i + kw];
#pragma unroll
                        for (int c = 0; c < COT; ++c) acc[c][i] = fmaf(xv, wv[c], acc[c][i]);
                    }
                }
            }
        }
        // this warp is done reading the buffer
        if (a.use_bulk) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[buf]);
        }

        if (chunk == a.nchunk - 1) {
            // ---- epilogue: bias + activation, pre-norm store, per-warp moments ----
            const int orow = G.r0 + il;
            const int ocol0 = G.c0 + sl * RW;
            const bool row_ok = item_ok && orow < a.Ho;
            const int nvalid = row_ok ? max(0, min(RW, a.Wo - ocol0)) : 0;
            const int tin = G.rt * a.col_tiles + G.ct;
            // The shift of a (warp, channel) partial is one of its own values:
            // the first output of the lowest lane that has a valid one.  The
            // shifted values then stay within a few standard deviations of 0,
            // whatever the channel's mean (no cancellation in S2 - S1^2 / n).
            const unsigned vlanes = __ballot_sync(0xffffffffu, nvalid > 0);
            const int klane = vlanes ? __ffs(vlanes) - 1 : 0;
#pragma unroll
            for (int c = 0; c < COT; ++c) {
                const int co = G.co0 + cs * COT + c;
                const float bias = a.b ? __ldg(a.b + co) : 0.0f;
                if constexpr (ACTT >= 0) {
                    bias_act<RW, ACTT>(acc[c], bias);
                } else {
                    if (a.act == ACT_HARDSWISH)
                        bias_act<RW, ACT_HARDSWISH>(acc[c], bias);
                    else if (a.act == ACT_GELU)
                        bias_act<RW, ACT_GELU>(acc[c], bias);
                    else
                        bias_act<RW, ACT_NONE>(acc[c], bias);
                }
                const float K = __shfl_sync(0xffffffffu, acc[c][0], klane);
                float3 m = shifted_sums<RW>(acc[c], K, nvalid);
                float *op = a.out +
                            ((((size_t)G.n * a.Co + co) * a.Dv + G.d) * a.Ho + (row_ok ? orow : 0)) * a.Wo +
                            ocol0;
                const size_t o0 = (size_t)(op - a.out);
                if (!CN_CHECK(nvalid == 0 || o0 + nvalid <= (size_t)a.N * a.Co * a.S, a.err)) {
                    // (checked build) skip the row
                } else if (nvalid == RW) {
                    if ((RW % 2) == 0 && (reinterpret_cast<uintptr_t>(op) & 7) == 0) {
#pragma unroll
                        for (int i = 0; i < RW - 1; i += 2)
                            *reinterpret_cast<float2 *>(op + i) = make_float2(acc[c][i], acc[c][i + 1]);
                    } else {
#pragma unroll
                        for (int i = 0; i < RW; ++i) op[i] = acc[c][i];
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < RW; ++i)
                        if (i < nvalid) op[i] = acc[c][i];
                }
                m = warp_sum3(m);
                const size_t pi = ((((size_t)G.n * a.Co + co) * a.Dv + G.d) * a.ntiles + tin) * a.wsp + sg;
                if (lane == 0 && CN_CHECK(pi < (size_t)a.N * a.Co * a.Dv * a.ntiles * a.wsp, a.err))
                    a.partial[pi] = make_float4(m.x, K, m.y, m.z);
            }
        }
    }
    // the last CTA to leave resets the work counters for the next launch
    __syncthreads();
    if (tid == 0 && atomicAdd(a.tickets + a.N + 1, 1) == (int)gridDim.x - 1) {
        a.tickets[a.N] = 0;
        a.tickets[a.N + 1] = 0;
    }
}

// Statistics of the normalization groups.  A group of one channel
// (InstanceNorm) gets one warp, eight per block; a wider group gets a block
// of min(channels, 8) x parts warps (below).
// Every partial (count, K, S1, S2) is a sum about its own shift K, one of
// its own values.  A channel's partials are moved to one common shift K0,
// the shift of the channel's first non-empty partial (a value of the
// channel's data), by the exact identities
//   S1' = S1 + n d,  S2' = S2 + d (2 S1 + n d),  d = K - K0,
// which stay well conditioned because every K and K0 lie within a few
// standard deviations of the data; then lanes add them in a fixed order and a
// butterfly of commutative adds gives every lane the same bits, and the
// channel's (count, mean = K0 + S1'/n, M2 = S2' - S1'^2/n) follows with one
// division.  Channel moments are merged (Chan et al.) within a warp in
// channel order, then the warps' results in warp order, so the result is
// deterministic.  The group's coefficients (mu, a = gamma * rstd * scale,
// bb = beta * scale) go to every channel.  Arithmetic is fp32: its ~1e-6
// relative error in mean and variance is far inside the 1e-4 output bound.
// With parts > 1 (wide groups with many partials) each channel's partials
// are split into `parts` contiguous ranges, one warp each: warp w takes
// range w % parts of channels w / parts, w / parts + warps / parts, ...;
// the warps' results still merge in warp order.
// channel_moments with each lane's partials (at most 8) all loaded before
// the first is used, so the loads overlap instead of following one another;
// the same shift, order of additions and result.  Longer ranges take
// channel_moments.
constexpr int kStatsBatch = 8;
CN_DEV Moments<float> channel_moments_batched(const float4 *p, int n, int lane) {
    if (n > 32 * kStatsBatch) return channel_moments(p, n, lane);
    float4 q[kStatsBatch];
#pragma unroll
    for (int j = 0; j < kStatsBatch; ++j)
        q[j] = lane + 32 * j < n ? p[lane + 32 * j] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    // common shift: the first non-empty partial's (lowest index)
    float K0 = 0.0f;
    bool found = false;
#pragma unroll
    for (int j = 0; j < kStatsBatch; ++j) {
        const unsigned has = __ballot_sync(0xffffffffu, q[j].x > 0.0f);
        if (!found && has) {
            K0 = __shfl_sync(0xffffffffu, q[j].y, __ffs(has) - 1);
            found = true;
        }
    }
    if (!found) return Moments<float>{0.0f, 0.0f, 0.0f};
    float3 v = make_float3(0.0f, 0.0f, 0.0f);  // (count, S1', S2') about K0
#pragma unroll
    for (int j = 0; j < kStatsBatch; ++j) {
        if (lane + 32 * j >= n) break;
        const float d = q[j].y - K0;
        v.x += q[j].x;
        v.y += fmaf(q[j].x, d, q[j].z);
        v.z += fmaf(d, fmaf(q[j].x, d, 2.0f * q[j].z), q[j].w);
    }
    v = warp_sum3(v);
    if (!(v.x > 0.0f)) return Moments<float>{0.0f, 0.0f, 0.0f};
    const float mu_s = v.y / v.x;  // mean - K0
    return Moments<float>{v.x, K0 + mu_s, fmaxf(v.z - v.y * mu_s, 0.0f)};
}

constexpr int kStatsWarps = 16;  // most warps of a statistics block
constexpr int kStatsGroupsPerBlock = 8;  // one-channel groups: one warp each
__global__ void __launch_bounds__(32 * kStatsWarps) k_group_stats(const __grid_constant__ Full2dArgs a, int parts) {
    __shared__ float sm[kStatsWarps][3];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int cpg = a.Co / a.NG;
    const int per_c = a.Dv * a.ntiles * a.wsp;  // a channel's partials: depth planes x tiles x warps
    const bool wide = cpg > 1;
    const int ng = wide ? (int)blockIdx.x : (int)blockIdx.x * nw + w;  // (n, group)
    if (ng >= a.N * a.NG) return;  // uniform per block when wide
    const int n = ng / a.NG, g = ng % a.NG;
    const float4 *p0 = a.partial + ((size_t)n * a.Co + (size_t)g * cpg) * per_c;
    Moments<float> m{0.0f, 0.0f, 0.0f};
    if (wide) {
        const int slot = w / parts, part = w - slot * parts;
        const int lo = (int)((long long)per_c * part / parts);
        const int hi = (int)((long long)per_c * (part + 1) / parts);
        for (int cl = slot; cl < cpg; cl += nw / parts)
            m = merge(m, channel_moments_batched(p0 + (size_t)cl * per_c + lo, hi - lo, lane));
    } else {
        m = channel_moments_batched(p0, per_c, lane);
    }
    if (wide) {
        if (lane == 0) {
            sm[w][0] = m.n;
            sm[w][1] = m.mean;
            sm[w][2] = m.m2;
        }
        __syncthreads();
        if (w != 0) return;
        m = Moments<float>{sm[0][0], sm[0][1], sm[0][2]};
        for (int j = 1; j < nw; ++j) m = merge(m, Moments<float>{sm[j][0], sm[j][1], sm[j][2]});
    }
    const float var = m.n > 0.0f ? m.m2 / m.n : 0.0f;
    const float rstd = 1.0f / sqrtf(var + a.eps);
    for (int cl = lane; cl < cpg; cl += 32) {
        const int c = g * cpg + cl;
        if (!CN_CHECK(c < a.Co, a.err)) break;
        const float ga = a.affine ? a.gamma[c] : 1.0f;
        const float be = a.affine ? a.beta[c] : 0.0f;
        a.coef[(size_t)n * a.Co + c] =
            make_float4(m.mean, rstd * ga * a.post_scale, be * a.post_scale, 0.0f);
    }
}

// Coefficients of a pure post scale (no normalization): (0, scale, 0).
__global__ void k_fill_scale(float4 *coef, int n, float scale) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) coef[i] = make_float4(0.0f, scale, 0.0f, 0.0f);
}

// Normalize pass: out = (y - mu) * a + bb per (n, c) plane, in place.
// Block b takes slice b % slices of plane planes - 1 - b / slices: the
// planes run last-written first and whole (the conv pass wrote samples
// roughly in order, so the newest planes are the ones still in L2).  A
// thread loads all its kApplyVec values before it stores any, which keeps
// enough reads in flight to run near the memory bandwidth.
constexpr int kApplyThreads = 256, kApplyVec = 4;
__global__ void __launch_bounds__(kApplyThreads) k_norm_apply(float *out, const float4 *coef, long long S,
                                                              int vec4, int *err, long long planes, int slices) {
    const long long pb = (long long)blockIdx.x / slices;
    const int slice = (int)((long long)blockIdx.x - pb * slices);
    const long long plane = planes - 1 - pb;
    if (!CN_CHECK(plane >= 0 && plane < planes, err)) return;
    const float4 cf = coef[plane];
    const long long i0 = (long long)slice * (kApplyThreads * kApplyVec) + threadIdx.x;
    if (vec4) {
        float4 *p4 = reinterpret_cast<float4 *>(out + plane * S);
        const long long n4 = S >> 2;
        float4 v[kApplyVec];
#pragma unroll
        for (int j = 0; j < kApplyVec; ++j)
            if (i0 + j * kApplyThreads < n4) v[j] = p4[i0 + j * kApplyThreads];
#pragma unroll
        for (int j = 0; j < kApplyVec; ++j)
            if (i0 + j * kApplyThreads < n4) {
                v[j].x = (v[j].x - cf.x) * cf.y + cf.z;
                v[j].y = (v[j].y - cf.x) * cf.y + cf.z;
                v[j].z = (v[j].z - cf.x) * cf.y + cf.z;
                v[j].w = (v[j].w - cf.x) * cf.y + cf.z;
                p4[i0 + j * kApplyThreads] = v[j];
            }
    } else {
        float *p = out + plane * S;
        float v[kApplyVec];
#pragma unroll
        for (int j = 0; j < kApplyVec; ++j)
            if (i0 + j * kApplyThreads < S) v[j] = p[i0 + j * kApplyThreads];
#pragma unroll
        for (int j = 0; j < kApplyVec; ++j)
            if (i0 + j * kApplyThreads < S) p[i0 + j * kApplyThreads] = (v[j] - cf.x) * cf.y + cf.z;
    }
}

struct Inst {
    int K, RW, COT, VECW, T, ACT;  // ACT -1: activation chosen at run time
    int OFF;                       // fixed input-column offset (float4 windows), 0: none
    Full2dKernel fn;
    const char *name;
};
#define CN_FULL_INST(K, RW, C, V, T, A)                               \
    {K, RW, C, V, T, A, 0, k_conv2d_act_stats<K, RW, C, V, (T != 0), A>, \
     "k_prep_weights,k_conv2d_act_stats<" #K "," #RW "," #C "," #V "," #T "," #A ">,k_group_stats,k_norm_apply"}
#define CN_FULL_INST_OFF(K, RW, C, T, A, O)                                    \
    {K, RW, C, 4, T, A, O, k_conv2d_act_stats<K, RW, C, 4, (T != 0), A, O>,      \
     "k_prep_weights,k_conv2d_act_stats<" #K "," #RW "," #C ",4," #T "," #A "," #O \
     ">,k_group_stats,k_norm_apply"}
const Inst kInst[] = {
    // activation-specialised: the 64->128 conv (none), the grouped transposed conv (GELU)
    CN_FULL_INST(3, 16, 4, 4, 0, 0), CN_FULL_INST(3, 16, 4, 2, 1, 2), CN_FULL_INST(3, 13, 4, 1, 1, 2),
    CN_FULL_INST_OFF(3, 12, 4, 1, 2, 2), CN_FULL_INST_OFF(3, 12, 4, 1, -1, 2),
    // run-time activation
    CN_FULL_INST(3, 16, 8, 4, 0, -1), CN_FULL_INST(3, 16, 4, 4, 0, -1), CN_FULL_INST(1, 16, 8, 4, 0, -1),
    CN_FULL_INST(2, 16, 8, 4, 0, -1), CN_FULL_INST(4, 16, 8, 4, 0, -1), CN_FULL_INST(3, 13, 4, 1, 1, -1),
    CN_FULL_INST(3, 16, 4, 2, 1, -1), CN_FULL_INST(1, 16, 8, 4, 1, -1), CN_FULL_INST(2, 16, 8, 1, 1, -1),
    CN_FULL_INST(4, 16, 8, 1, 1, -1),
    // four output channels a conv group (C_out / groups % 8 == 4) at the other extents
    CN_FULL_INST(1, 16, 4, 4, 0, -1), CN_FULL_INST(2, 16, 4, 4, 0, -1), CN_FULL_INST(4, 16, 4, 4, 0, -1),
    CN_FULL_INST(1, 16, 4, 4, 1, -1), CN_FULL_INST(2, 16, 4, 1, 1, -1), CN_FULL_INST(4, 16, 4, 1, 1, -1),
};
#undef CN_FULL_INST
#undef CN_FULL_INST_OFF

int env_int(const char *name, int dflt) {
    const char *v = getenv(name);
    return v ? atoi(v) : dflt;
}

struct Choice {
    const Inst *in = nullptr;
    int wco = 1, wsp = 1, TR = 1, NT = 1;
    double cost = 1e30;
};

// Row pitch (floats) of the staged input, at least min_pitch and a multiple
// of 4 (16-byte rows for TMA and bulk copies).  Lane l of a warp reads row
// l % TR, segment l / TR, so a float4 load's bank group is
// (pitch/4 * row + RW/4 * segment) mod 8.  With pitch/4 = p (mod 8), p odd,
// and RW/4 = p * TR (mod 8) that is p * l: the 8 lanes of every quarter
// warp hit 8 distinct bank groups.  For odd TR, p = RW/4 * TR (odd numbers
// are their own inverse mod 8).  Otherwise p only needs to be odd (distinct
// rows of one segment).
int row_pitch(int min_pitch, int VECW, int RW, int TR) {
    int pitch = (min_pitch + 3) & ~3;
    int want = -1;
    if (VECW == 4 && RW % 4 == 0 && (TR & 1)) {
        const int pw = ((RW / 4) * TR) & 7;
        if (pw & 1) want = pw;
    }
    while (want >= 0 ? ((pitch / 4) & 7) != want : ((pitch / 4) & 1) == 0) pitch += 4;
    return pitch;
}

int pick_wco(int units) {
    for (int c = 8; c >= 1; --c)
        if (units % c == 0) return c;
    return 1;
}
}  // namespace

int full2d_plan(const conv_norm_desc &d, Full2dArgs &a, Full2dConfig &cfg) {
    // dense Conv2d shapes and grouped transposed convs that fit them go to
    // the tensor cores
    a.tct = 0;
    if (tc2d_plan(d, a, cfg) == CN_OK) return CN_OK;
    a.tc = 0;
    if (tct_plan(d, a, cfg) == CN_OK) return CN_OK;
    a.tct = 0;
    const int T = d.conv == CN_CONVT2D ? 1 : 0;
    const int K = d.k;
    const int Ho = T ? d.H + K - 1 : d.H - K + 1;
    const int Wo = T ? d.W + K - 1 : d.W - K + 1;
    // A Conv3d runs as 2-D samples (n, d_out) over depth-stacked channels
    // (ci, kd): the filter [co][ci][kd][kh][kw] already is [co][ci*K + kd][kh][kw].
    const bool d3 = d.conv == CN_CONV3D;
    if (d3 && d.groups != 1) return CN_ERR_UNSUPPORTED;
    const int KD = d3 ? K : 1;
    const int Dv = d3 ? d.D - K + 1 : 1;
    const int Cig = d.C_in / d.groups * KD, Cog = d.C_out / d.groups;
    const bool bulk = (d.W % 4 == 0) && env_int("CN_NO_TMA", 0) == 0;
    const bool tma2d = bulk && tma_available() && env_int("CN_NO_TMA2D", 0) == 0;
    const int f_cot = env_int("CN_FULL2D_COT", 0), f_rw = env_int("CN_FULL2D_RW", 0),
              f_wsp = env_int("CN_FULL2D_WSP", 0);
    const int off = bulk ? (((-(K - 1) * T) % 4) + 4) % 4 : 0;
    Choice best;
    for (const Inst &in : kInst) {
        if (in.K != K || in.T != T || Cog % in.COT != 0) continue;
        if (in.ACT >= 0 && in.ACT != d.act) continue;
        if ((f_cot && in.COT != f_cot) || (f_rw && in.RW != f_rw)) continue;
        if (in.OFF ? in.OFF != off : off % in.VECW != 0) continue;
        const int wco = pick_wco(Cog / in.COT);
        const int nseg = (Wo + in.RW - 1) / in.RW;
        const int XW = in.RW + K - 1;
        const int loadw = (in.OFF + XW + in.VECW - 1) / in.VECW * in.VECW;
        const int regs = std::min(255, in.COT * in.RW + loadw + in.COT + 40);
        for (int cand = 0; cand < 8 * 3; ++cand) {
            const int wsp = 1 + cand / 3, split = 1 + cand % 3;
            if (wco * wsp > 8) break;
            if (f_wsp && wsp != f_wsp) continue;
            const int lanes = 32 * wsp;
            // segments per column tile: all that fit the lanes, or the row
            // split in two or three column tiles (narrower row buffers)
            const int NT = std::min((nseg + split - 1) / split, lanes);
            if (split > 1 && NT == std::min((nseg + split - 2) / (split - 1), lanes)) continue;
            const int TR = std::max(1, std::min(lanes / NT, Ho));
            // segments of every column tile must keep the load alignment
            const int ctiles = (nseg + NT - 1) / NT;
            if (ctiles > 1 && ((NT * in.RW) % 4 != 0)) continue;
            if (NT > 1 && (in.RW % in.VECW) != 0) continue;
            const int rtiles = (Ho + TR - 1) / TR;
            const double waste = ((double)rtiles * TR / Ho) * ((double)ctiles * NT * in.RW / Wo) *
                                 ((double)lanes / (TR * NT));
            // scalar row loads count double: more instructions in flight and
            // bank conflicts (measured: 16-wide float2 rows beat 13-wide scalar)
            const double loads = (double)loadw / in.VECW * (in.VECW == 1 ? 2.0 : 1.0) + 3.0 * in.COT / 4.0;
            const double ratio = 1.0 + loads / ((double)in.COT * K * in.RW);
            const int threads = 32 * wco * wsp;
            const int ctas = std::max(1, std::min(65536 / (threads * ((regs + 7) & ~7)), 2));
            const int warps_sm = ctas * wco * wsp;
            // scheduler balance (warps spread over 4 SM sub-partitions) and
            // latency hiding (fewer than 16 warps measured slower)
            const double balance =
                (warps_sm % 4 == 0) ? 1.0 : (double)((warps_sm + 3) / 4 * 4) / warps_sm;
            const double occ = warps_sm >= 16 ? 1.0 : 1.0 + 0.025 * (16 - warps_sm);
            // a specialised epilogue is smaller and cheaper than the run-time switch
            const double spec = in.ACT >= 0 ? 0.97 : 1.0;
            // staging: one tensor copy per stage when the row buffer fits a TMA
            // box; otherwise one bulk copy per row plus zeroing of the halo,
            // measured at ~15% of the conv time on the 64-channel transposed conv
            const int cols_in_c = NT * in.RW + K - 1;
            const int pitch_c = row_pitch(
                std::max(off - in.OFF + (NT - 1) * in.RW + loadw, off + cols_in_c + 3), in.VECW,
                in.RW, TR);
            const bool tma_c = tma2d && pitch_c <= 256 && TR + K - 1 <= 256;
            const double stage = tma_c ? 1.0 : 1.15;
            const double cost = waste * ratio * balance * occ * spec * stage;
            if (cost < best.cost - 1e-9) {
                best.in = &in;
                best.wco = wco;
                best.wsp = wsp;
                best.TR = TR;
                best.NT = NT;
                best.cost = cost;
            }
        }
    }
    if (!best.in) return CN_ERR_UNSUPPORTED;
    const Inst &in = *best.in;
    const int RW = in.RW, COT = in.COT;
    const int XW = RW + K - 1;
    const int LOADW = (in.OFF + XW + in.VECW - 1) / in.VECW * in.VECW;
    a.use_bulk = bulk ? 1 : 0;
    a.N = d.N;
    a.Ci = d.C_in;
    a.Co = d.C_out;
    a.H = d.H;
    a.W = d.W;
    a.Ho = Ho;
    a.Wo = Wo;
    a.Cig = Cig;
    a.Cog = Cog;
    a.KD = KD;
    a.Din = d3 ? d.D : 1;
    a.Dv = Dv;
    a.wco = best.wco;
    a.wsp = best.wsp;
    a.TR = best.TR;
    a.NT = best.NT;
    const int nseg = (Wo + RW - 1) / RW;
    a.row_tiles = (Ho + a.TR - 1) / a.TR;
    a.col_tiles = (nseg + a.NT - 1) / a.NT;
    a.ncob = d.C_out / (COT * a.wco);
    a.ntiles = a.row_tiles * a.col_tiles;
    a.rows_in = a.TR + K - 1;
    a.cols_in = a.NT * RW + K - 1;
    // row buffer: the tile's reads reach off - OFF + (NT-1)*RW + LOADW; bulk
    // copies of whole 16-byte groups reach at most off + cols_in + 3.
    const int pitch = row_pitch(std::max(off - in.OFF + (a.NT - 1) * RW + LOADW, off + a.cols_in + 3),
                                in.VECW, RW, a.TR);
    a.pitch = pitch;
    // the whole stage as one tensor copy: box (pitch, rows_in, cib, 1)
    a.use_tma = (tma2d && pitch <= 256 && a.rows_in <= 256) ? 1 : 0;  // (box extents; KD <= 4)
    a.xmap_base = nullptr;
    const int COB = COT * a.wco;
    const int per_ci = a.rows_in * pitch + K * K * COB;
    // Pipeline: 3 stages (measured best of 2..4 on both 2-D workloads) when
    // they fit the shared-memory budget with chunks of at least 2 input
    // channels, fewer otherwise.
    const size_t budget = (in.COT * in.RW <= 64 ? 108 : 216) * 1024;
    int nstage = std::max(2, std::min(kMaxStages, env_int("CN_FULL2D_NSTAGE", 3)));
    // stages hold whole input channels: cib is a multiple of the depth taps
    int cib = 1;
    for (;; --nstage) {
        cib = std::min(Cig, std::max(1, env_int("CN_FULL2D_CIB", 8)));
        cib = std::max(KD, cib / KD * KD);
        while (cib > KD && (size_t)nstage * cib * per_ci * 4 > budget) cib -= KD;
        if (cib >= std::min(Cig, 2) || nstage == 2) break;
    }
    a.nstage = nstage;
    a.cib = cib;
    a.nchunk = (Cig + cib - 1) / cib;
    a.xstage = cib * a.rows_in * pitch;
    a.wstage = cib * K * K * COB;
    a.stage_floats = ((a.xstage + a.wstage) + 31) & ~31;  // 128-byte aligned stages
    a.act = d.act;
    a.norm = d.norm;
    a.NG = d.norm == CN_NORM_GROUP ? d.num_groups : d.C_out;
    a.affine = d.affine && d.norm != CN_NORM_NONE;
    a.eps = d.eps;
    a.post_scale = d.post_scale;
    a.S = (long long)Dv * Ho * Wo;
    a.apply_needed = !(d.norm == CN_NORM_NONE && d.post_scale == 1.0f);
    a.vec4 = (a.S % 4) == 0;
    const int threads = 32 * a.wco * a.wsp;
    const size_t smem = (size_t)a.nstage * a.stage_floats * 4;
    if (smem > 227 * 1024) return CN_ERR_UNSUPPORTED;
    const long long items = (long long)d.N * Dv * a.ncob * a.ntiles;
    if (items > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;
    a.items = (int)items;
    a.wprep = nullptr;
    cfg.kern = in.fn;
    cfg.names = in.name;
    cfg.K = K;
    cfg.RW = RW;
    cfg.COT = COT;
    cfg.VECW = in.VECW;
    cfg.transposed = T;
    cfg.threads = threads;
    cfg.smem = (int)smem;
    cfg.grid = (int)std::min<long long>(items, 148);  // refined from the device in full2d_prepare
    const long long wtotal = (long long)a.ncob * a.nchunk * a.wstage;
    cfg.prep_grid = (int)std::max(1LL, std::min((wtotal + 255) / 256, 1024LL));
    return apply_config(d, a, cfg);
}

int apply_config(const conv_norm_desc &d, const Full2dArgs &a, Full2dConfig &cfg) {
    cfg.apply_threads = kApplyThreads;
    const long long units = a.vec4 ? a.S / 4 : a.S;
    const long long slices = std::max(1LL, (units + kApplyThreads * kApplyVec - 1) / (kApplyThreads * kApplyVec));
    const long long blocks = (long long)d.N * d.C_out * slices;
    if (blocks > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;
    cfg.apply_slices = (int)slices;
    cfg.apply_grid = (int)blocks;
    return CN_OK;
}

// Work counters after the N per-sample tickets: claim + exit, or one claim
// counter per group + exit for the tensor-core transposed conv.
static size_t full2d_tickets(const Full2dArgs &a) { return (size_t)(a.N + 2 + (a.tct ? a.tct_G : 0)); }
size_t full2d_counter_bytes(const Full2dArgs &a) { return full2d_tickets(a) * sizeof(int); }

size_t full2d_workspace(const Full2dArgs &a) {
    const size_t part = (size_t)a.N * a.Co * a.Dv * a.ntiles * a.wsp * sizeof(float4);
    const size_t coef = (size_t)a.N * a.Co * sizeof(float4);
    const size_t tick = full2d_tickets(a) * sizeof(int);
    const size_t wprep =
        a.tc ? tc2d_wprep_bytes(a) : (size_t)a.ncob * a.nchunk * a.wstage * sizeof(float);
    auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
    return al(part) + al(coef) + al(tick) + al(wprep);
}

void full2d_bind_workspace(Full2dArgs &a, char *base, int *err_flag) {
    const size_t part = (size_t)a.N * a.Co * a.Dv * a.ntiles * a.wsp * sizeof(float4);
    const size_t coef = (size_t)a.N * a.Co * sizeof(float4);
    const size_t tick = full2d_tickets(a) * sizeof(int);
    auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
    a.partial = reinterpret_cast<float4 *>(base);
    a.coef = reinterpret_cast<float4 *>(base + al(part));
    a.tickets = reinterpret_cast<int *>(base + al(part) + al(coef));
    a.wprep = reinterpret_cast<float *>(base + al(part) + al(coef) + al(tick));
    a.err = err_flag;
}

int full2d_prepare(Full2dConfig &cfg, Full2dArgs &a) {
    if (raise_dyn_smem(reinterpret_cast<const void *>(cfg.kern), cfg.smem) !=
        cudaSuccess)
        return CN_ERR_CUDA;
    // persistent grid: every CTA slot of the device, capped by the tiles
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cfg.kern, cfg.threads, cfg.smem) !=
            cudaSuccess)
        return CN_ERR_CUDA;
    if (per_sm < 1) return CN_ERR_UNSUPPORTED;
    if (a.tct) return tct_prepare(cfg, a, sms);
    cfg.grid = (int)std::min<long long>((long long)sms * per_sm, (long long)a.items);
    return CN_OK;
}

int full2d_launches(const Full2dConfig &cfg, const Full2dArgs &a) {
    if (cfg.grid == 0 || a.items == 0) return 0;
    // the tensor-core transposed conv builds its filter operand itself (no pre-pass)
    return (a.tct ? 1 : 2) + (a.apply_needed ? 2 : 0);
}

int full2d_launch(const Full2dConfig &cfg, Full2dArgs &a, cudaStream_t s, const LaunchEvents *ev) {
    if (cfg.grid == 0 || a.items == 0) return CN_OK;
    int li = 0;  // launch index (timing events)
    if (a.tct) {
        const int st = tct_bind_x(a);
        if (st != CN_OK) return st;
    } else if (a.tc) {
        const int st = tc2d_bind_x(a);
        if (st != CN_OK) return st;
    } else if (a.use_tma && a.xmap_base != a.x) {
        int st;
        if (a.Din > 1) {  // x as (W, H, D, C_in, N), box (pitch, rows_in, KD, cib / KD, 1)
            const uint64_t plane = (uint64_t)a.H * a.W * 4;
            const uint64_t dims[5] = {(uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.Din, (uint64_t)a.Ci,
                                      (uint64_t)a.N};
            const uint64_t strides[4] = {(uint64_t)a.W * 4, plane, plane * a.Din, plane * a.Din * a.Ci};
            const uint32_t box[5] = {(uint32_t)a.pitch, (uint32_t)a.rows_in, (uint32_t)a.KD,
                                     (uint32_t)(a.cib / a.KD), 1u};
            st = encode_tmap_f32_5d(&a.xmap, a.x, dims, strides, box);
        } else {
            const uint64_t dims[4] = {(uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.Ci, (uint64_t)a.N};
            const uint64_t strides[3] = {(uint64_t)a.W * 4, (uint64_t)a.H * a.W * 4,
                                         (uint64_t)a.Ci * a.H * a.W * 4};
            const uint32_t box[4] = {(uint32_t)a.pitch, (uint32_t)a.rows_in, (uint32_t)a.cib, 1u};
            st = encode_tmap_f32_4d(&a.xmap, a.x, dims, strides, box);
        }
        if (st != CN_OK) return st;
        a.xmap_base = a.x;
    }
    record_launch(ev, li++, s);
    if (a.tct) {
        // no filter pre-pass: each CTA builds its group's operand
    } else if (a.tc) {
        const int st = tc2d_prep_launch(cfg, a, s);
        if (st != CN_OK) return st;
        record_launch(ev, li++, s);
    } else {
        const int wtotal = a.ncob * a.nchunk * a.wstage;
        k_prep_weights<<<cfg.prep_grid, 256, 0, s>>>(a.w, a.wprep, cfg.K, cfg.transposed, a.Cig,
                                                      a.Cog, cfg.COT * a.wco, a.cib, a.nchunk, wtotal);
        if (cudaGetLastError() != cudaSuccess) return CN_ERR_CUDA;
        record_launch(ev, li++, s);
    }
    cfg.kern<<<cfg.grid, cfg.threads, cfg.smem, s>>>(a);
    record_launch(ev, li++, s);
    if (cudaGetLastError() != cudaSuccess) return CN_ERR_CUDA;
    if (a.apply_needed) {
        if (a.norm == CN_NORM_NONE) {
            k_fill_scale<<<(a.N * a.Co + 255) / 256, 256, 0, s>>>(a.coef, a.N * a.Co, a.post_scale);
        } else {
            const int cpg = a.Co / a.NG;
            const int per_c = a.Dv * a.ntiles * a.wsp;
            const int parts = (cpg > 1 && per_c >= 128) ? 2 : 1;
            const int nw = cpg > 1 ? std::min(cpg, kStatsWarps / 2) * parts : kStatsGroupsPerBlock;
            const int blocks = cpg > 1 ? a.N * a.NG : (a.N * a.NG + nw - 1) / nw;
            k_group_stats<<<blocks, 32 * nw, 0, s>>>(a, parts);
        }
        if (cudaGetLastError() != cudaSuccess) return CN_ERR_CUDA;
        record_launch(ev, li++, s);
        k_norm_apply<<<cfg.apply_grid, cfg.apply_threads, 0, s>>>(a.out, a.coef, a.S, a.vec4, a.err,
                                                                   (long long)a.N * a.Co, cfg.apply_slices);
        record_launch(ev, li++, s);
        if (cudaGetLastError() != cudaSuccess) return CN_ERR_CUDA;
    }
    return CN_OK;
}

}  // namespace cn
