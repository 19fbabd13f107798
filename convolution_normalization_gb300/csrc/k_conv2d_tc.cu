// Variant 2, tensor-core conv: dense Conv2d (groups 1) as an implicit GEMM on
// the 5th-generation tensor cores, for the l2_p17 problem shape (Conv2d
// 64 -> 128, k = 3, then InstanceNorm and a division by 2).
//
// The convolution is a contraction over K = C_in * k * k, so it maps onto
// tcgen05.mma: D[co][p] += sum_k W[co][k] * X[k][p], M = 128 output channels,
// N = up to 256 output positions, D in tensor memory (TMEM).  fp32 inputs
// with fp32 accuracy come from the split-TF32 scheme: the tensor cores read a
// tf32 operand by dropping the low 13 mantissa bits of an fp32 word, so with
// v = hi(v) + lo(v), hi = truncation, lo = the exact remainder,
//   W * X ~= Wh*Xh + Wl*Xh + Wh*Xl        (Wl*Xl, about 2^-22 relative, dropped)
// where the raw fp32 words serve as Wh and Xh.  That keeps every product to
// about fp32 accuracy; the conv then matches an fp32 conv to ~1e-6 relative.
//
// Operands (K-major, no swizzle): a K step of 8 is two 4-channel "core
// matrices" whose rows are 16 bytes apart.  The input part of a stage holds
// one 4-channel group of R + k - 1 input rows, position-major:
// [row * W + col][4 channels].  Output position p of the tile (row p / W,
// column p % W of the R-row block) reads input position p + kh * W + kw for
// tap (kh, kw), so every tap is the same buffer with its start address moved
// by (kh * W + kw) rows: no im2col copy.  Positions whose column is >= the
// output width read into the next row and are discarded.  The second core
// matrix of a K step is any 16-byte-multiple offset away, which lets one MMA
// take two taps (hi*hi products) or a hi/lo pair of one tap (the cross
// terms): 14 MMAs of K = 8 per group for k = 3 (27 tap products, one padded
// with a zero filter block).
//
// Warp roles (one CTA per SM, persistent, tiles claimed from a counter):
//   warp 0      producer: TMA of the raw input rows of a 4-channel group into
//               a landing buffer, bulk copy of the group's pre-split filter
//               block (lo | hi) into the stage;
//   warps 2-5   converters: landing [c][row][col] -> interleaved hi and lo
//               operand buffers of the stage;
//   warp 1      MMA issuer (one thread): 14 tcgen05.mma per stage into one of
//               two TMEM accumulators (double buffered across tiles);
//   warps 6-9   epilogue: tcgen05.ld of the accumulator (thread = channel),
//               bias + activation, per-channel sums (count, S1, S2) about
//               the tile's first value, in registers, then a 32x32
//               transpose through shared memory so the pre-norm output is
//               stored with coalesced rows.
// The statistics and normalize passes that follow are the ones of the CUDA
// core path (k_group_stats, k_norm_apply).
#include "cn_common.cuh"
#include "cn_internal.h"
#include "cn_tcgen05.cuh"

#include <algorithm>
#include <cstdlib>

namespace cn {
namespace {

constexpr int kTcThreads = 320;
constexpr int kTcM = 128;                 // output channels per tile
constexpr int kTapBytes = kTcM * 16;      // filter slice of one tap: 128 rows x 4 channels
constexpr int kTcMaxStages = 3;
constexpr int kTcLand = 2;
constexpr int kScratchFloats = 4 * 32 * 33;  // epilogue transpose, 4 warps
constexpr int kMaxMmas = 14;                   // MMAs per stage for k <= 3: k*k + ceil(k*k / 2)

// Filter pre-pass: per (channel block of 128, 4-channel group) one block of
// [lo | hi] x [tap][128 rows][4 channels], the A operands of that group's
// MMAs in core-matrix order.
__global__ void __launch_bounds__(256) k_prep_weights_tc(const float *__restrict__ w,
                                                         float *wprep, int Ci, int K, int ngrp,
                                                         long long total) {
    const int T = K * K;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        long long r = e;
        const int j = (int)(r % 4);
        r /= 4;
        const int row = (int)(r % kTcM);
        r /= kTcM;
        const int t = (int)(r % T);
        r /= T;
        const int hi = (int)(r % 2);
        r /= 2;
        const int g = (int)(r % ngrp);
        const int cob = (int)(r / ngrp);
        const int co = cob * kTcM + row, c = 4 * g + j;
        const float v = w[((size_t)co * Ci + c) * T + t];
        wprep[e] = hi ? v : tf32_rest(v);
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) k_conv2d_tc(const __grid_constant__ Full2dArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t land_full[kTcLand], land_empty[kTcLand];
    // full[b]: the stage's filter block landed (tx bytes) and the four
    // converter warps wrote its input operands; st_empty[b]: its MMAs are done
    __shared__ __align__(8) uint64_t full[kTcMaxStages], st_empty[kTcMaxStages];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], fin_bar;
    __shared__ int s_land_tile[kTcLand], s_st_tile[kTcMaxStages], s_acc_tile[2];
    __shared__ uint32_t s_tmem;
    __shared__ uint64_t s_desc[kTcMaxStages][kMaxMmas][2];  // (A, B) descriptors per stage slot
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NS = a.tc_stages;
    const int T = a.tc_K * a.tc_K;
    const int rows_in = a.tc_R + a.tc_K - 1;
    unsigned char *smem = smem_raw;
    auto stage = [&](int b) { return smem + (size_t)b * a.tc_stage_bytes; };
    unsigned char *land0 = smem + (size_t)NS * a.tc_stage_bytes;
    const int land_stride = (a.tc_land_bytes + 127) & ~127;
    auto land = [&](int b) { return land0 + (size_t)b * land_stride; };
    unsigned char *zero_blk = land0 + (size_t)kTcLand * land_stride;
    float *scratch = reinterpret_cast<float *>(zero_blk + kTapBytes);
    const int acc_cols = a.tc_acc_cols;

    // ---- setup: zero the operand tails and the zero block, barriers, TMEM ----
    {
        const int tail0 = rows_in * a.W;  // first position never written by the converters
        const int npos_buf = a.tc_xbuf_bytes / 16;
        for (int b = 0; b < NS; ++b) {
            float4 *xh = reinterpret_cast<float4 *>(stage(b));
            float4 *xl = reinterpret_cast<float4 *>(stage(b) + a.tc_xbuf_bytes);
            for (int i = tail0 + tid; i < npos_buf; i += blockDim.x) {
                xh[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                xl[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float4 *z = reinterpret_cast<float4 *>(zero_blk);
        for (int i = tid; i < kTapBytes / 16; i += blockDim.x) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid == 0) {
        for (int i = 0; i < kTcLand; ++i) {
            mbar_init(&land_full[i], 1);
            mbar_init(&land_empty[i], 4);
        }
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1 + 4);
            mbar_init(&st_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 2);
            mbar_init(&acc_empty[i], 4);
        }
        mbar_init(&fin_bar, 1);
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(2 * acc_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    int *abort_p = const_cast<int *>(&s_abort);
    auto wait = [&](uint64_t *bar, uint32_t par) {
        return tc_wait(bar, par, abort_p, a.err, a.wait_ns);
    };

    const int per_sample = a.row_tiles * a.ncob;

    if (warp == 0) {
        // ---------------- producer ----------------
        // Stage k uses landing buffer k % kTcLand and stage slot k % NS;
        // slot indices and phase parities advance incrementally.
        if (lane == 0) {
            int kl = 0, kw = 0;  // landing / filter stages armed so far
            // failure-path test hook: CTA 0 never arms its first landing stage,
            // a barrier phase nothing completes, so the waits on it run out
            const bool stall = a.stall && blockIdx.x == 0;
            int lb = 0, b = 0;
            uint32_t lph = 0, sph = 0;  // parity of the current pass over each ring
            int next = (int)blockIdx.x;
            bool live = true;
            while (live) {
                const int tile = next < a.items ? next : -1;
                if (tile >= 0) next = (int)gridDim.x + atomicAdd(a.tickets + a.N, 1);
                int n = 0, rt = 0, cob = 0;
                if (tile >= 0) {
                    n = tile / per_sample;
                    const int rem = tile - n * per_sample;
                    cob = rem / a.row_tiles;
                    rt = rem - cob * a.row_tiles;
                }
                const int ng = tile >= 0 ? a.tc_ngrp : 1;  // a stop marker is one stage
                for (int g = 0; g < ng; ++g) {
                    // landing buffer lb was last used kTcLand stages ago
                    if (kl >= kTcLand && !wait(&land_empty[lb], lph ^ 1u)) {
                        live = false;
                        break;
                    }
                    s_land_tile[lb] = tile;
                    if (stall && kl == 0) {
                        // left unarmed (never drained below)
                    } else if (tile >= 0) {
                        mbar_arrive_expect_tx(&land_full[lb], (uint32_t)a.tc_land_bytes);
                        tma_load_4d(land(lb), &a.tc_xmap, 0, rt * a.tc_R, 4 * g, n, &land_full[lb]);
                    } else {
                        mbar_arrive(&land_full[lb]);
                    }
                    ++kl;
                    if (++lb == kTcLand) {
                        lb = 0;
                        lph ^= 1u;
                    }
                    if (kw >= NS && !wait(&st_empty[b], sph ^ 1u)) {
                        live = false;
                        break;
                    }
                    s_st_tile[b] = tile;
                    if (tile >= 0) {
                        mbar_arrive_expect_tx(&full[b], (uint32_t)a.tc_wblk_bytes);
                        bulk_load(stage(b) + 2 * (size_t)a.tc_xbuf_bytes,
                                  reinterpret_cast<const unsigned char *>(a.wprep) +
                                      ((size_t)cob * a.tc_ngrp + g) * a.tc_wblk_bytes,
                                  (uint32_t)a.tc_wblk_bytes, &full[b]);
                    } else {
                        mbar_arrive(&full[b]);
                    }
                    ++kw;
                    if (++b == NS) {
                        b = 0;
                        sph ^= 1u;
                    }
                }
                if (tile < 0) live = false;
            }
            // copies still in flight (only after an abort) land before the CTA
            // exits; in a normal run these phases are long complete
            for (int j = std::max(0, kl - kTcLand); j < kl; ++j)
                if (!(stall && j == 0))
                    mbar_wait_bounded(&land_full[j % kTcLand], (j / kTcLand) & 1, kWaitLimitNs);
            for (int j = std::max(0, kw - NS); j < kw; ++j)
                mbar_wait_bounded(&full[j % NS], (j / NS) & 1, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // Between two stages this thread only waits for one barrier and
        // commits: the tensor pipe's queue holds a few MMAs (under ~1000
        // cycles of work), so per-stage overhead shows up as idle time.
        if (lane == 0) {
            const uint32_t idesc = idesc_tf32(kTcM, a.tc_npos);
            // The operand descriptors of a stage depend only on its slot:
            // built once here.
            const uint32_t zaddr = smem_u32(zero_blk);
            int nm = 0;
            for (int sb_i = 0; sb_i < NS; ++sb_i) {
                const uint32_t sb = smem_u32(stage(sb_i));
                const uint32_t xh = sb;
                const uint32_t wl = sb + 2u * (uint32_t)a.tc_xbuf_bytes;
                const uint32_t wh = wl + (uint32_t)(T * kTapBytes);
                auto off = [&](int tp) { return (tp / a.tc_K) * a.W + tp % a.tc_K; };
                nm = 0;
                // cross terms: Wl(t) Xh(t) + Wh(t) Xl(t)
                for (int tp = 0; tp < T; ++tp, ++nm) {
                    s_desc[sb_i][nm][0] = umma_desc(wl + tp * kTapBytes, (uint32_t)(T * kTapBytes), 128);
                    s_desc[sb_i][nm][1] = umma_desc(xh + off(tp) * 16, (uint32_t)a.tc_xbuf_bytes, 128);
                }
                // hi * hi, two taps per MMA
                int tp = 0;
                for (; tp + 1 < T; tp += 2, ++nm) {
                    s_desc[sb_i][nm][0] = umma_desc(wh + tp * kTapBytes, kTapBytes, 128);
                    s_desc[sb_i][nm][1] =
                        umma_desc(xh + off(tp) * 16, (uint32_t)((off(tp + 1) - off(tp)) * 16), 128);
                }
                if (tp < T) {  // odd tap count: the last tap with the zero block
                    const uint32_t wa = wh + tp * kTapBytes;
                    s_desc[sb_i][nm][0] = umma_desc(wa, zaddr - wa, 128);
                    s_desc[sb_i][nm][1] = umma_desc(xh + off(tp) * 16, 16, 128);
                    ++nm;
                }
            }
            int b = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = 0; ok; ++t) {
                const int as = t & 1;
                // first stage of a tile: its id (or the stop marker)
                if (!wait(&full[b], ph)) break;
                const int tile = s_st_tile[b];
                if (t >= 2 && !wait(&acc_empty[as], ((t >> 1) - 1) & 1)) break;
                tc_fence_after();  // the epilogue's reads of this accumulator are done
                s_acc_tile[as] = tile;
                mbar_arrive(&acc_full[as]);  // publishes the tile id (1 of 2 arrivals)
                if (tile < 0) {
                    mbar_arrive(&acc_full[as]);
                    break;
                }
                const uint32_t d = tmem + (uint32_t)(as * acc_cols);
                for (int g = 0;;) {
                    uint64_t da[kMaxMmas], db[kMaxMmas];
#pragma unroll
                    for (int i = 0; i < kMaxMmas; ++i) {
                        if (i < nm) {
                            da[i] = s_desc[b][i][0];
                            db[i] = s_desc[b][i][1];
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kMaxMmas; ++i)
                        if (i < nm) umma_tf32(d, da[i], db[i], idesc, (g | i) ? 1u : 0u);
                    umma_commit(&st_empty[b]);
                    if (++b == NS) {
                        b = 0;
                        ph ^= 1u;
                    }
                    if (++g == a.tc_ngrp) break;
                    if (!wait(&full[b], ph)) {
                        ok = false;
                        break;
                    }
                }
                if (ok) umma_commit(&acc_full[as]);  // the tile's MMAs are done (2 of 2)
            }
            // every MMA issued by this thread completes before TMEM is freed
            umma_commit(&fin_bar);
            mbar_wait_bounded(&fin_bar, 0, kWaitLimitNs);
        }
    } else if (warp < 6) {
        // ---------------- converters ----------------
        const int ct = tid - 64;
        const int npix = rows_in * a.W;
        int lb = 0, b = 0;
        uint32_t lph = 0, sph = 0;
        for (int k = 0;; ++k) {
            if (!wait(&land_full[lb], lph)) break;
            const int tile = s_land_tile[lb];
            if (k >= NS && !wait(&st_empty[b], sph ^ 1u)) break;
            if (tile >= 0) {
                const float *src = reinterpret_cast<const float *>(land(lb));
                float4 *xh = reinterpret_cast<float4 *>(stage(b));
                float4 *xl = reinterpret_cast<float4 *>(stage(b) + a.tc_xbuf_bytes);
                for (int p = ct; p < npix; p += 128) {
                    if (!CN_CHECK(p < a.tc_xbuf_bytes / 16, a.err)) break;
                    const float v0 = src[p], v1 = src[npix + p], v2 = src[2 * npix + p],
                                v3 = src[3 * npix + p];
                    xh[p] = make_float4(v0, v1, v2, v3);
                    xl[p] = make_float4(tf32_rest(v0), tf32_rest(v1), tf32_rest(v2), tf32_rest(v3));
                }
                fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&land_empty[lb]);
                mbar_arrive(&full[b]);
            }
            if (tile < 0) break;
            if (++lb == kTcLand) {
                lb = 0;
                lph ^= 1u;
            }
            if (++b == NS) {
                b = 0;
                sph ^= 1u;
            }
        }
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        float *scr = scratch + (warp - 6) * 32 * 33;
        const long long S = a.S;
        for (int t = 0;; ++t) {
            const int as = t & 1;
            if (!wait(&acc_full[as], (t >> 1) & 1)) break;
            const int tile = s_acc_tile[as];
            if (tile < 0) break;
            tc_fence_after();
            const int n = tile / per_sample;
            const int rem = tile - n * per_sample;
            const int cob = rem / a.row_tiles;
            const int rt = rem - cob * a.row_tiles;
            const int r0 = rt * a.tc_R;
            const int co = cob * kTcM + q * 32 + lane;
            const float bias = a.b ? __ldg(a.b + co) : 0.0f;
            // shift of the channel's sums: its first value of the tile
            // (position 0, always valid), so the shifted values stay within a
            // few standard deviations of 0 whatever the channel's mean
            float Ksh = 0.0f;
            const int rows_ok = min(a.tc_R, a.Ho - r0);
            float s1 = 0.0f, s2 = 0.0f;
            float *obase = a.out + ((size_t)n * a.Co + cob * kTcM + q * 32) * (size_t)S;
            for (int i = 0; i < a.tc_npos / 32; ++i) {
                uint32_t v[32];
                tmem_ld32(tmem + (uint32_t)(as * acc_cols + 32 * i) + ((uint32_t)(q * 32) << 16), v);
                // lane l owns position 32i + l for the stores; the warp's
                // validity mask serves the per-channel sums over j
                const int p = 32 * i + lane;
                const int rr = p / a.W;
                const int col = p - rr * a.W;
                const bool vl = rr < rows_ok && col < a.Wo;
                const unsigned vmask = __ballot_sync(0xffffffffu, vl);
                if (i == 0) Ksh = apply_act(a.act, __uint_as_float(v[0]) + bias);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float y = apply_act(a.act, __uint_as_float(v[j]) + bias);
                    if ((vmask >> j) & 1u) {
                        const float dlt = y - Ksh;
                        s1 += dlt;
                        s2 = fmaf(dlt, dlt, s2);
                    }
                    scr[lane * 33 + j] = y;
                }
                __syncwarp();
                if (vl && CN_CHECK((size_t)(obase - a.out) + (size_t)(r0 + rr) * a.Wo + col +
                                           31 * (size_t)S < (size_t)a.N * a.Co * S,
                                       a.err)) {
                    float *op = obase + (size_t)(r0 + rr) * a.Wo + col;
#pragma unroll 8
                    for (int c = 0; c < 32; ++c) op[(size_t)c * S] = scr[c * 33 + lane];
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[as]);
            const float cnt = (float)(rows_ok * a.Wo);
            if (CN_CHECK(((size_t)n * a.Co + co) * a.ntiles + rt < (size_t)a.N * a.Co * a.ntiles, a.err))
                a.partial[((size_t)n * a.Co + co) * a.ntiles + rt] = make_float4(cnt, Ksh, s1, s2);
        }
    }

    // ---- teardown ----
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(2 * acc_cols)
                     : "memory");
    if (tid == 0 && atomicAdd(a.tickets + a.N + 1, 1) == (int)gridDim.x - 1) {
        a.tickets[a.N] = 0;
        a.tickets[a.N + 1] = 0;
    }
}

}  // namespace

// Plans the tensor-core path; CN_ERR_UNSUPPORTED when the problem does not
// fit it (the CUDA-core kernels then take it).
int tc2d_plan(const conv_norm_desc &d, Full2dArgs &a, Full2dConfig &cfg) {
    if (d.conv != CN_CONV2D || d.groups != 1) return CN_ERR_UNSUPPORTED;
    if (d.C_in % 4 != 0 || d.C_out % kTcM != 0 || d.W % 4 != 0 || d.k > 3) return CN_ERR_UNSUPPORTED;
    if (!tma_available()) return CN_ERR_UNSUPPORTED;
    const char *e = getenv("CN_NO_TC");
    if (e && atoi(e)) return CN_ERR_UNSUPPORTED;
    const int K = d.k, W = d.W, H = d.H;
    const int Ho = H - K + 1, Wo = W - K + 1;
    if (W > 256 || Wo > 256) return CN_ERR_UNSUPPORTED;
    int R = 1 + (256 - Wo) / W;
    R = std::max(1, std::min(R, Ho));
    // MMA N: the tile's positions, a multiple of 32 (the epilogue reads TMEM
    // in 32-column pieces)
    const int npos = (((R - 1) * W + Wo) + 31) / 32 * 32;
    if (npos > 256) return CN_ERR_UNSUPPORTED;
    const int rows_in = R + K - 1;
    if (rows_in > 256) return CN_ERR_UNSUPPORTED;
    // operand buffer: rows_in * W positions, plus a zeroed tail covering the
    // farthest read (last tap, last position, +1 for the padded pair)
    const int need = (K - 1) * W + (K - 1) + npos + 1;
    const int pos_buf = std::max(rows_in * W, need) + 8;
    const int xbuf = (pos_buf * 16 + 127) / 128 * 128;
    const int T = K * K;
    const int wblk = 2 * T * kTapBytes;
    const int stage_bytes = 2 * xbuf + wblk;
    const int land_bytes = 4 * rows_in * W * 4;  // buffers 128-byte aligned apart
    const int fixed = kTcLand * ((land_bytes + 127) & ~127) + kTapBytes + kScratchFloats * 4;
    int ns = kTcMaxStages;
    while (ns > 2 && ns * stage_bytes + fixed > 225 * 1024) --ns;
    if (ns * stage_bytes + fixed > 225 * 1024) return CN_ERR_UNSUPPORTED;
    const int row_tiles = (Ho + R - 1) / R;
    const long long items = (long long)d.N * row_tiles * (d.C_out / kTcM);
    if (items > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;

    a.tc = 1;
    a.tc_xmap_base = nullptr;
    a.wait_ns = kWaitLimitNs;
    a.tc_K = K;
    a.tc_R = R;
    a.tc_npos = npos;
    a.tc_ngrp = d.C_in / 4;
    a.tc_xbuf_bytes = xbuf;
    a.tc_wblk_bytes = wblk;
    a.tc_stage_bytes = stage_bytes;
    a.tc_land_bytes = land_bytes;
    a.tc_stages = ns;
    a.tc_acc_cols = npos <= 32 ? 32 : npos <= 64 ? 64 : npos <= 128 ? 128 : 256;
    a.use_bulk = 1;
    a.N = d.N;
    a.Ci = d.C_in;
    a.Co = d.C_out;
    a.H = H;
    a.W = W;
    a.Ho = Ho;
    a.Wo = Wo;
    a.Cig = d.C_in;
    a.Cog = d.C_out;
    a.KD = 1;
    a.Din = 1;
    a.Dv = 1;
    a.row_tiles = row_tiles;
    a.col_tiles = 1;
    a.ncob = d.C_out / kTcM;
    a.ntiles = row_tiles;
    a.wsp = 1;
    a.items = (int)items;
    a.wprep = nullptr;
    a.act = d.act;
    a.norm = d.norm;
    a.NG = d.norm == CN_NORM_GROUP ? d.num_groups : d.C_out;
    a.affine = d.affine && d.norm != CN_NORM_NONE;
    a.eps = d.eps;
    a.post_scale = d.post_scale;
    a.S = (long long)Ho * Wo;
    a.apply_needed = !(d.norm == CN_NORM_NONE && d.post_scale == 1.0f);
    a.vec4 = (a.S % 4) == 0;

    cfg.kern = k_conv2d_tc;
    cfg.names = "k_prep_weights_tc,k_conv2d_tc,k_group_stats,k_norm_apply";
    cfg.K = K;
    cfg.RW = 0;
    cfg.COT = kTcM;
    cfg.VECW = 0;
    cfg.transposed = 0;
    cfg.threads = kTcThreads;
    cfg.smem = ns * stage_bytes + fixed;
    cfg.grid = (int)std::min<long long>(items, 148);
    const long long wtotal = (long long)a.ncob * a.tc_ngrp * wblk / 4;
    cfg.prep_grid = (int)std::max(1LL, std::min((wtotal + 255) / 256, 1024LL));
    return apply_config(d, a, cfg);
}

size_t tc2d_wprep_bytes(const Full2dArgs &a) { return (size_t)a.ncob * a.tc_ngrp * a.tc_wblk_bytes; }

// Encodes the input tensor map for this x (cached while x stays the same).
int tc2d_bind_x(Full2dArgs &a) {
    if (a.tc_xmap_base == a.x) return CN_OK;
    const uint64_t dims[4] = {(uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.Ci, (uint64_t)a.N};
    const uint64_t strides[3] = {(uint64_t)a.W * 4, (uint64_t)a.H * a.W * 4,
                                 (uint64_t)a.Ci * a.H * a.W * 4};
    const uint32_t box[4] = {(uint32_t)a.W, (uint32_t)(a.tc_R + a.tc_K - 1), 4u, 1u};
    const int st = encode_tmap_f32_4d(&a.tc_xmap, a.x, dims, strides, box);
    if (st != CN_OK) return st;
    a.tc_xmap_base = a.x;
    return CN_OK;
}

int tc2d_prep_launch(const Full2dConfig &cfg, const Full2dArgs &a, cudaStream_t s) {
    const long long total = (long long)a.ncob * a.tc_ngrp * a.tc_wblk_bytes / 4;
    k_prep_weights_tc<<<cfg.prep_grid, 256, 0, s>>>(a.w, a.wprep, a.Ci, a.tc_K, a.tc_ngrp, total);
    return cudaGetLastError() == cudaSuccess ? CN_OK : CN_ERR_CUDA;
}

}  // namespace cn
