// Tensor-core Conv3d with up to 4 input channels, as an implicit GEMM on the
// 5th-generation tensor cores, for two of the fused problems:
//   mean: Conv3d (16 or 32 output channels) -> activation -> GroupNorm /
//         InstanceNorm / none -> mean over D, H, W (l2_p27: Conv3d 3 -> 16,
//         k = 4, HardSwish, GroupNorm(4), mean);
//   pool: Conv3d (16 output channels) -> softmax over channels -> MaxPool3d(2)
//         twice = one 4x4x4 stride-4 max (l2_p6: Conv3d 3 -> 16, k = 3).
//
// GEMM.  A stage covers one band of RB = 128 / W output rows (M = 128
// positions p = row * W + x, TMEM lanes) of a group of ZG consecutive output
// depth planes z0 .. z0 + ZG - 1, and N = (zg, co, kx) columns:
//   Dacc[p][(zg, co, kx)] = sum_{u, ky, c} X[c][z0 + u][p + ky * W] * w[co][c][u - zg][ky][kx]
// over the stage's ZG + k - 1 input planes u (w = 0 where u - zg is not a
// tap), and the conv output is the kx-shifted sum of accumulator rows,
//   conv[co][z0 + zg][p] = sum_kx Dacc[p + kx][(zg, co, kx)],
// done by the epilogue with warp shuffles.  Tiles are whole rows, so a shift
// never reaches a row's next row for a valid output (x + kx < W); where W
// divides 32 the 32-lane quadrants also hold whole rows, otherwise the k - 1
// rows past a quadrant come from a small shared halo (mean only).
//
// Why this shape: a tcgen05.mma with M = 128 and K = 8 costs about the same
// up to N = 128 (measured ~144 cycles at N = 64, ~162 at N = 128 on this
// GPU, ~185 at N = 256, the full rate), so N is made as wide as it goes: the
// kx taps and ZG output planes (16 * 4 * 4 = 256 for C_out = 16, k = 4),
// which reads each staged input plane once for the ZG output planes it
// feeds.  For input plane u the filter operand rows (zg, co, kx) hold taps
// kz = u - zg: consecutive blocks of one sequence stored with kz descending
// and zero blocks at both ends, so B for every u is a window of that
// sequence (no copies per u).  Where a plane's columns are a multiple of
// 32, an input plane's MMAs span only the planes it feeds (narrower N).
// With ZG = 4 a plane group and a band of 4 * (32 / W) rows are exactly
// whole 4x4x4 pooling windows.
//
// Precision: split TF32 as in the 2-D tensor-core kernel (the tensor cores
// read tf32 by dropping 13 mantissa bits; with v = hi + lo,
// W * X ~= Wl*Xh + Wh*Xl + Wh*Xh), so the conv matches an fp32 conv to
// ~1e-6 relative.  Per (u, ky) one MMA takes both cross terms (A = [Xh |
// Xl], B = [Wl | Wh]); the hi*hi terms pair two ky taps per MMA (A = Xh at
// rows ky and ky + 1, B = [Wh(ky) | Wh(ky + 1)]; an odd k pairs its last tap
// with a zero filter block).  MMAs per stage: (ZG + k - 1) (k + ceil(k/2)),
// plus one per newly started plane where the MMAs are narrowed.
//
// Operands (K-major, no swizzle): a staged input plane is [position][4
// channels] fp32, hi part then lo part; a K step of 8 is two 4-channel core
// matrices, 16 bytes a row.  Tap offsets move the start address only.
//
// Warp roles (one persistent CTA per SM, items claimed from a counter: an
// item is some bands of one group of ZG output planes of one sample: half
// the group's bands for the mean, one band for the pool):
//   warp 0      producer: one TMA tensor copy per stage (W x (RB + k - 1)
//               rows x (ZG + k - 1) planes x C_in, zero fill outside x) into
//               a ring of up to four landing buffers (as many as fit); for
//               the mean also the finisher below;
//   warps 2-3   converters: landing [c][u][row][x] -> operand stage hi / lo;
//   warp 1      MMA issuer (one thread): the stage's MMAs into one of two
//               TMEM accumulators;
//   warps 4-19  epilogue, four warps per TMEM lane quadrant, thread =
//               position:
//     mean: a warp takes C_out / 4 channels of all ZG planes: the kx sum,
//           bias + activation, per-channel shifted sums in registers; at the
//           end of an item the sums are posted through a shared-memory ring
//           to warp 0, which writes them to the item's slot, takes the
//           sample's ticket and, for the sample's last item, merges the
//           slots and writes the output;
//     pool: a warp takes the 16 channels of one plane zg: the kx sum, bias,
//           softmax over the channels in registers, the max over the
//           window's 4 columns (and rows inside the quadrant) by shuffles,
//           then across quadrants and planes by shared-memory atomic max
//           (softmax values are positive, so their bits order as integers);
//           the stage's pooled values are scaled and stored.
#include "cn_common.cuh"
#include "cn_internal.h"
#include "cn_tcgen05.cuh"

#include <algorithm>
#include <cstdlib>
#include <type_traits>

namespace cn {
namespace {

constexpr int kT3Threads = 640;    // 20 warps: 5 per SM sub-partition, up to 96 registers each
constexpr int kConvWarps = 2;      // warps 2-3
constexpr int kEpiWarp0 = 4;       // epilogue: warps 4-19
constexpr int kEpiWarps = 16;
constexpr int kT3SmemLimit = 227 * 1024 - 1024;  // dynamic part (static barriers beside it)
constexpr int kPoolCells = 8;      // pooled outputs per channel per stage: (RB / 4) (W / 4)
constexpr int kPosts = 4;          // mean: item sums in flight from the epilogue to warp 0
constexpr int kMaxLand = 4;        // landing buffers, where they fit

enum { MODE_MEAN = 0, MODE_POOL = 1 };

// Ticket increment with acquire-release semantics at GPU scope: it publishes
// the writes the calling thread has observed (the warp's, after __syncwarp)
// and orders its later reads after the other CTAs' published writes.
CN_DEV int atomic_add_acq_rel(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

template <int K, int CO>
struct T3 {
    static constexpr int ZG = CO * K * 4 <= 256 ? 4 : 2;  // output planes per stage
    static constexpr int N = ZG * CO * K;                 // MMA N: (zg, co, kx) columns
    static constexpr int NU = ZG + K - 1;                 // staged input planes
    static constexpr int NPAIR = (K + 1) / 2;             // hi*hi MMAs per input plane
    // Narrow MMAs (a plane's columns a multiple of 32, see the MMA issuer)
    // read only the K nonzero blocks of a kz sequence; the others also read
    // the ZG - 1 zero blocks at each end.
    static constexpr bool NARROW = (CO * K) % 32 == 0;
    static constexpr int NB = NARROW ? K : K + 2 * (ZG - 1);  // stored blocks of one kz sequence
    static constexpr int B0 = NARROW ? ZG - 1 : 0;            // leading zero blocks not stored
    static constexpr int BLK = CO * K * 16;               // one kz block: (co, kx) rows x 4 channels
    static constexpr int SLEN = NB * BLK;                 // one (ky, lo | hi) kz sequence
    static constexpr int ZBYTES = (K & 1) ? N * 16 : 0;   // zero block for an odd k
    static constexpr int WBYTES = K * 2 * SLEN + ZBYTES;
    static constexpr int ACC = N <= 128 ? 128 : 256;      // TMEM columns per accumulator
    static constexpr int HALO = 2 * 4 * (K - 1) * N;      // floats: [parity][quadrant][row][N]
    static constexpr int RED = kPosts * 4 * CO * 4;       // floats: mean post ring [slot][quadrant][CO] float4 / pool cells
    static_assert(N % 16 == 0 && N <= 256, "MMA N");
    static_assert(RED >= CO * kPoolCells, "pool cells");
};

// The epilogue warps agree on a flag (barrier 1 with an AND reduction), so
// none of them goes on to a later barrier that another has left.
CN_DEV bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 1, 512, q;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}
CN_DEV void epi_sync() { asm volatile("bar.sync 1, 512;\n" ::: "memory"); }

// NC consecutive TMEM columns of this warp's lane quadrant into v (no wait).
template <int NC>
CN_DEV void tmem_ld_cols(uint32_t taddr, uint32_t *v) {
#pragma unroll
    for (int i = 0; i < NC / 16; ++i) tmem_ld16(taddr + 16 * i, v + 16 * i);
    constexpr int R = NC % 16, B8 = NC / 16 * 16;
    if (R >= 8) tmem_ld8(taddr + B8, v + B8);
    if (R % 8 >= 4) tmem_ld4(taddr + B8 + (R >= 8 ? 8 : 0), v + B8 + (R >= 8 ? 8 : 0));
}

// Finish of one sample of the mean, by one warp (lane = channel).  Slot i of
// a channel holds an item's (count n_i, K_i, S1_i, S2_i): sums about K_i, a
// value of the item's data.  The slots move to one shift K0 (slot 0's) by
// the exact identities
//   S1 += S1_i + n_i d,  S2 += S2_i + d (2 S1_i + n_i d),  d = K_i - K0,
// summed in a fixed tree, and with one reciprocal 1/n of the sample's count
//   m_c = K0 + S1 / n,  M2_c = S2 - S1^2 / n,
//   mu_g = mean of the group's m_c,  M2_g = sum (M2_c + n (m_c - mu_g)^2),
// and out = gamma (m_c - mu_g) / sqrt(M2_g / (n C/G) + eps) + beta, times the
// post scale.  All in fp32: every shift is within a few standard deviations
// of the data, so nothing cancels (and this GPU's FP64 pipe is slow enough
// that fp64 here cost the kernel ~8%).
CN_DEV void tc3_finish_sample(const Tc3Args &a, int n, int c) {
    const int nchunks = a.ngroups * a.nsplit;
    const bool on = c < a.Co;
    float S1 = 0.0f, S2 = 0.0f, K0 = 0.0f;
    if (on) {
        // sixteen slot loads in flight (other CTAs' slots: not through L1),
        // summed pairwise in a fixed tree, blocks of 16 in slot order
        const float4 *pc = a.partial + (size_t)n * nchunks * a.Co + c;
        K0 = __ldcg(pc).y;  // slot 0 (the first bands of the first planes) is never empty
        for (int ch0 = 0; ch0 < nchunks; ch0 += 16) {
            float v1[16], v2[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float4 v = ch0 + j < nchunks ? __ldcg(pc + (size_t)(ch0 + j) * a.Co)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                const float d = v.x > 0.0f ? v.y - K0 : 0.0f;
                v1[j] = fmaf(v.x, d, v.z);
                v2[j] = fmaf(d, fmaf(v.x, d, 2.0f * v.z), v.w);
            }
#pragma unroll
            for (int w = 8; w > 0; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) {
                    v1[j] += v1[j + w];
                    v2[j] += v2[j + w];
                }
            S1 += v1[0];
            S2 += v2[0];
        }
    }
    const float cnt = (float)a.Do * a.Ho * a.Wo;
    const float inv_n = (float)a.inv_cnt;  // 1 / cnt and 1 / cpg come from the host
    const float mc = fmaf(S1, inv_n, K0);
    const float m2c = fmaxf(fmaf(-S1, S1 * inv_n, S2), 0.0f);
    float val = mc;
    if (a.norm != CN_NORM_NONE) {
        // the group's lanes: cpg consecutive channels (a power of two or not)
        const int cpg = a.Co / a.G, g0 = (c / cpg) * cpg;
        const float inv_cpg = (float)a.inv_cpg;
        float sm = 0.0f;
        for (int u = 0; u < cpg; ++u) sm += __shfl_sync(0xffffffffu, mc, g0 + u);
        const float mu = sm * inv_cpg;
        float m2 = 0.0f;
        for (int u = 0; u < cpg; ++u) {
            const float dm = __shfl_sync(0xffffffffu, mc, g0 + u) - mu;
            m2 += fmaf(cnt * dm, dm, __shfl_sync(0xffffffffu, m2c, g0 + u));
        }
        const float rstd = rsqrtf(m2 * inv_n * inv_cpg + a.eps);
        const float ga = a.affine && on ? a.gamma[c] : 1.0f;
        const float be = a.affine && on ? a.beta[c] : 0.0f;
        val = fmaf(ga * (mc - mu), rstd, be);
    }
    if (on && CN_CHECK(n < a.N, a.err)) a.out[(size_t)n * a.Co + c] = val * a.post_scale;
}

template <int K, int CO, int MODE>
CN_DEV void tc3_body(const Tc3Args &a) {
    using P = T3<K, CO>;
    constexpr int N = P::N, ZG = P::ZG, NU = P::NU;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t land_full[kMaxLand], land_empty[kMaxLand];
    // st_full[b]: the converters wrote stage b; st_empty[b]: its MMAs are done
    __shared__ __align__(8) uint64_t st_full[2], st_empty[2];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], fin_bar;
    // stage info: (item or -1 to stop, band, 1 if the item's last band, valid planes)
    __shared__ int4 s_land_info[kMaxLand], s_st_info[2], s_acc_info[2];
    // mean: item sums posted by the epilogue to warp 0 (ring of kPosts)
    __shared__ __align__(8) uint64_t post_full[kPosts], post_empty[kPosts];
    __shared__ int s_post_item[kPosts];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int PP = a.pp, PPU = a.ppu;
    // position p of a staged plane -> its 16-byte unit (a gap after every 8
    // positions with pad: the converters' strided stores then miss no bank)
    auto unit = [&](int p) { return a.pad ? p + (p >> 3) : p; };
    unsigned char *stages = smem_raw;
    auto stage = [&](int b) { return stages + (size_t)b * a.stage; };
    const int land_stride = (a.land + 127) & ~127;
    unsigned char *land0 = stages + 2 * (size_t)a.stage;
    auto land = [&](int lb) { return land0 + (size_t)lb * land_stride; };
    unsigned char *wts = land0 + (size_t)a.nland * land_stride;
    float *halo = reinterpret_cast<float *>(wts + P::WBYTES);
    float *red = halo + (a.halo ? P::HALO : 0);  // mean post ring [slot][quadrant][CO] (n, K, S1, S2) / pool cells
    const int rows_in = a.rb + K - 1;
    const int P0 = rows_in * a.W;  // staged positions per plane

    // item -> (sample n, plane group g, split s of the group's bands: bands
    // s * bpi .. s * bpi + bpi - 1).  The groups with ZG output planes of
    // every sample come first, the depth's last, partial groups (fewer
    // MMAs: cheaper items) at the end of the queue, so the CTAs finish
    // closer together.
    const int bpi = (a.nband + a.nsplit - 1) / a.nsplit;
    const int nfull = (MODE == MODE_POOL || a.Do % ZG == 0) ? a.ngroups : a.ngroups - 1;
    auto item_group = [&](int item, int &n, int &g, int &z0, int &nzv) {
        const int grp = item / a.nsplit;
        if (grp < a.N * nfull) {
            n = grp / nfull;
            g = grp - n * nfull;
        } else {
            n = grp - a.N * nfull;
            g = a.ngroups - 1;
        }
        z0 = g * ZG;
        nzv = min(ZG, a.Do - z0);
    };

    // ---- setup: filter sequences, zeroed operand tails, barriers, TMEM ----
    {
        // the raw filter (C_out x C_in x k^3 floats) lands in the stage
        // buffers with coalesced loads (they are free until the first stage),
        // and the blocks are built from there: no dependent global loads
        float *wraw = reinterpret_cast<float *>(stages);
        const int nraw = CO * a.Ci * K * K * K;
#pragma unroll 4
        for (int e = tid; e < nraw; e += blockDim.x) wraw[e] = __ldg(a.w + e);
        __syncthreads();
        // [ky][lo | hi][block i: kz = K + ZG - 2 - B0 - i][(co, kx) rows][4 channels], zero block
        float *wf = reinterpret_cast<float *>(wts);
        constexpr int ROWS = CO * K;
        constexpr int NW = K * 2 * P::NB * ROWS * 4;
        for (int e = tid; e < P::WBYTES / 4; e += blockDim.x) {
            float v = 0.0f;
            if (e < NW) {
                const int c = e & 3;
                int r = e >> 2;
                const int row = r % ROWS;
                r /= ROWS;
                const int i = r % P::NB;
                r /= P::NB;
                const int hi = r & 1, ky = r >> 1;
                const int kz = K + ZG - 2 - P::B0 - i;
                const int co = row / K, kx = row - co * K;
                if (c < a.Ci && kz >= 0 && kz < K) {
                    const float x = wraw[((((size_t)co * a.Ci + c) * K + kz) * K + ky) * K + kx];
                    v = hi ? x : tf32_rest(x);
                }
            }
            wf[e] = v;
        }
        if (MODE == MODE_POOL)
            for (int e = tid; e < P::RED; e += blockDim.x) red[e] = 0.0f;  // pool cells
        __syncthreads();  // the raw filter is read before the tails below are zeroed
        for (int b = 0; b < 2; ++b) {
            float4 *xs = reinterpret_cast<float4 *>(stage(b));
            const int tail = PP - P0;
            for (int i = tid; i < 2 * NU * tail; i += blockDim.x) {
                const int pl = i / tail, r = i - pl * tail;
                xs[(size_t)pl * PPU + unit(P0 + r)] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
    if (tid == 0) {
        for (int i = 0; i < kMaxLand; ++i) {
            mbar_init(&land_full[i], 1);
            mbar_init(&land_empty[i], kConvWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&st_full[i], kConvWarps);
            mbar_init(&st_empty[i], 1);
            mbar_init(&acc_full[i], 2);
            mbar_init(&acc_empty[i], kEpiWarps);
        }
        for (int i = 0; i < kPosts; ++i) {
            mbar_init(&post_full[i], 1);
            mbar_init(&post_empty[i], 1);
        }
        mbar_init(&fin_bar, 1);
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(2 * P::ACC));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    fence_proxy_async();  // the filter sequences and zeroed tails are MMA operands
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    int *abort_p = const_cast<int *>(&s_abort);
    auto wait = [&](uint64_t *bar, uint32_t par) {
        return tc_wait(bar, par, abort_p, a.err, a.wait_ns);
    };

    if (warp == 0) {
        // ---------------- producer (+ mean finisher) ----------------
        // Lane 0 arms the stages' TMA copies.  For the mean the whole warp
        // also takes the items the epilogue posts: it publishes the item's
        // sums to its global slot, takes the sample's ticket, and on the
        // sample's last item merges the slots and writes the output.  Both
        // are polled, so the work of a merge only delays copies that are
        // already up to two stages ahead, and never the epilogue.
        int k = 0, lb = 0;           // stages armed; stage k lands in buffer lb = k % nland
        uint32_t lph = 0;            // parity of the current pass over the landing buffers
        int next = (int)blockIdx.x;  // lane 0: the next item to claim
        int item = 0, band = 0, bend = 0, n = 0, g = 0, z0 = 0, nzv = 0;  // lane 0: current item
        bool prod_live = true, fin_live = MODE == MODE_MEAN;
        int pr = 0;
        uint32_t pph = 0;
        uint64_t t_idle = 0;
        for (uint32_t it = 0; prod_live || fin_live; ++it) {
            bool progress = false;
            if (prod_live) {
                bool ready = k < a.nland || mbar_test_wait(&land_empty[lb], lph ^ 1u);
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (ready) {
                    int stop = 0;
                    if (lane == 0) {
                        if (band == bend) {  // claim the next item (a stop marker is one stage)
                            item = next < a.items ? next : -1;
                            if (item >= 0) {
                                next = (int)gridDim.x + atomicAdd(a.work, 1);
                                item_group(item, n, g, z0, nzv);
                                band = (item % a.nsplit) * bpi;
                                bend = min(band + bpi, a.nband);
                            } else {
                                band = 0;
                                bend = 1;
                            }
                        }
                        s_land_info[lb] = make_int4(item, band, band == bend - 1, nzv);
                        if (a.stall && blockIdx.x == 0 && k == 0) {
                            // failure-path test hook: the first landing stage of
                            // CTA 0 stays unarmed, a phase nothing completes
                        } else if (item >= 0) {
                            mbar_arrive_expect_tx(&land_full[lb], (uint32_t)a.land);
                            tma_load_4d(land(lb), &a.xmap, 0, band * a.rb, z0, n * a.Ci, &land_full[lb]);
                        } else {
                            mbar_arrive(&land_full[lb]);
                            stop = 1;
                        }
                        ++band;
                    }
                    if (__shfl_sync(0xffffffffu, stop, 0)) prod_live = false;
                    ++k;
                    if (++lb == a.nland) {
                        lb = 0;
                        lph ^= 1u;
                    }
                    progress = true;
                }
            }
            if (MODE == MODE_MEAN && fin_live) {
                bool got = mbar_test_wait(&post_full[pr], pph);
                got = __shfl_sync(0xffffffffu, got, 0);
                if (got) {
                    const int pitem = s_post_item[pr];
                    if (pitem < 0) {
                        fin_live = false;  // the epilogue is done
                    } else {
                        int pn, pg, pz0, pnzv;
                        item_group(pitem, pn, pg, pz0, pnzv);
                        const int nchunks = a.ngroups * a.nsplit;
                        const int chunk = pg * a.nsplit + pitem % a.nsplit;
                        // the quadrants' sums moved to the first non-empty
                        // quadrant's shift, in fixed quadrant order
                        float K0 = 0.0f, S1 = 0.0f, S2 = 0.0f;
                        if (lane < CO) {
                            bool have = false;
                            const float4 *ring = reinterpret_cast<const float4 *>(red) + (size_t)pr * 4 * CO + lane;
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq) {
                                const float4 t = ring[qq * CO];
                                if (!(t.x > 0.0f)) continue;
                                if (!have) K0 = t.y;
                                have = true;
                                const float d = t.y - K0;
                                S2 += t.w + d * fmaf(t.x, d, 2.0f * t.z);
                                S1 += fmaf(t.x, d, t.z);
                            }
                        }
                        float4 sums = make_float4(0.0f, K0, S1, S2);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&post_empty[pr]);  // the ring entry is read
                        // the item's count: its valid rows x Wo x valid planes
                        const int b0 = (pitem % a.nsplit) * bpi, b1 = min(b0 + bpi, a.nband);
                        sums.x = (float)((min(b1 * a.rb, a.Ho) - b0 * a.rb) * a.Wo * pnzv);
                        if (lane < CO && CN_CHECK(pn < a.N && chunk < nchunks, a.err))
                            a.partial[((size_t)pn * nchunks + chunk) * a.Co + lane] = sums;
                        __syncwarp();
                        // the ticket publishes the warp's slot writes; the last
                        // item of the sample sees every other item's slot
                        int last = 0;
                        if (lane == 0) last = atomic_add_acq_rel(a.tickets + pn, 1) == nchunks - 1;
                        if (__shfl_sync(0xffffffffu, last, 0)) {
                            tc3_finish_sample(a, pn, lane);
                            if (lane == 0) a.tickets[pn] = 0;
                        }
                    }
                    if (++pr == kPosts) {
                        pr = 0;
                        pph ^= 1u;
                    }
                    progress = true;
                }
            }
            // bounded idling: stop at another role's abort or after the wait limit
            if (progress) {
                t_idle = 0;
            } else {
                __nanosleep(64);  // leave the issue slots to this sub-partition's epilogue warps
            }
            if (!progress && (it & 255u) == 255u) {
                int quit = 0;
                if (lane == 0) {
                    const uint64_t now = globaltimer_ns();
                    if (*abort_p) {
                        quit = 1;
                    } else if (t_idle == 0) {
                        t_idle = now;
                    } else if (now - t_idle > a.wait_ns) {
                        flag_error(a.err, ERR_TIMEOUT);
                        *abort_p = 1;
                        quit = 1;
                    }
                }
                if (__shfl_sync(0xffffffffu, quit, 0)) break;
            }
        }
        // a copy still in flight (only after an abort) lands before the CTA exits
        if (lane == 0)
            for (int j = max(0, k - a.nland); j < k; ++j)
                if (!(a.stall && blockIdx.x == 0 && j == 0))
                    mbar_wait_bounded(&land_full[j % a.nland], (j / a.nland) & 1, kWaitLimitNs);
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t wbase = smem_u32(wts);
            const uint32_t zaddr = wbase + K * 2 * P::SLEN;
            // descriptors are linear in the start address (units of 16 bytes)
            const uint64_t bc0 = umma_desc(wbase, P::SLEN, 128);                 // [Wl | Wh](ky)
            const uint64_t bp0 = umma_desc(wbase + P::SLEN, 2 * P::SLEN, 128);  // [Wh(ky) | Wh(ky+1)]
            const uint32_t xl_off = (uint32_t)(NU * PPU * 16);
            const uint32_t sbo = a.pad ? 144u : 128u;  // bytes between 8-position groups
            const int WU = unit(a.W);                  // units per input row (W % 8 == 0 with pad)
            for (int k = 0;; ++k) {
                const int b = k & 1;
                if (!wait(&st_full[b], (k >> 1) & 1)) break;
                const int4 info = s_st_info[b];
                if (k >= 2 && !wait(&acc_empty[b], ((k >> 1) - 1) & 1)) break;
                tc_fence_after();  // the epilogue's reads of this accumulator are done
                s_acc_info[b] = info;
                mbar_arrive(&acc_full[b]);  // publishes the stage (1 of 2 arrivals)
                if (info.x < 0) {
                    mbar_arrive(&acc_full[b]);
                    break;
                }
                const uint32_t d = tmem + (uint32_t)(b * P::ACC);
                const uint32_t sb = smem_u32(stage(b));
                const uint64_t ac0 = umma_desc(sb, xl_off, sbo);                // [Xh | Xl]
                const uint64_t ap0 = umma_desc(sb, (uint32_t)(WU * 16), sbo);   // [Xh(ky) | Xh(ky+1)]
                // Input plane u feeds output planes zg in [zlo, zhi] (taps
                // kz = u - zg in [0, k)): its MMAs cover only those columns
                // (N = their count x C_out x k, D moved to zlo's first column,
                // B's window moved past the zero blocks).  A plane's columns
                // are first written at u = zg, by a cross MMA of its own that
                // does not accumulate.  Only where a plane's columns are a
                // multiple of 32 (the TMEM allocation granule), so every D
                // starts on one; otherwise every MMA spans all ZG planes.
                // With narrow MMAs, a group with fewer than ZG output planes
                // left (the depth's last) gets MMAs only for its planes: the
                // same code with the window's end and the fresh planes taken
                // at run time.
                constexpr int NZ = CO * K;  // columns of one output plane
                constexpr bool NARROW = P::NARROW;
                auto stage_mmas = [&](auto partial_tag) {
                constexpr bool PARTIAL = decltype(partial_tag)::value;
                const int nzv = info.w;  // valid output planes of the group
#pragma unroll
                for (int u = 0; u < NU; ++u) {
                    const int zlo = NARROW ? (u - (K - 1) > 0 ? u - (K - 1) : 0) : 0;
                    const int zhi_g = NARROW ? (u < ZG - 1 ? u : ZG - 1) : ZG - 1;
                    const int zhi = PARTIAL ? min(zhi_g, nzv - 1) : zhi_g;
                    if (PARTIAL && zhi < zlo) continue;  // feeds no valid plane
                    const bool fresh = NARROW ? (u < ZG && (!PARTIAL || u < nzv)) : u == 0;  // plane zg = u starts here
                    const uint32_t id_all = idesc_tf32(128, (zhi - zlo + 1) * NZ);
                    const uint32_t id_one = idesc_tf32(128, NZ);
                    const uint32_t id_old = idesc_tf32(128, (u - zlo > 0 ? u - zlo : 1) * NZ);
                    const uint64_t au = (uint64_t)(u * PPU);
                    const int blk = K + ZG - 2 - u + zlo - P::B0;  // first valid block of the kz sequences
                    const uint32_t dz = d + (uint32_t)(zlo * NZ);
#pragma unroll
                    for (int ky = 0; ky < K; ++ky) {
                        const uint64_t ad = ac0 + au + (uint64_t)(ky * WU);
                        const uint64_t bd = bc0 + (uint64_t)((ky * 2 * P::SLEN + blk * P::BLK) >> 4);
                        if (ky == 0 && fresh && !NARROW) {
                            umma_tf32(dz, ad, bd, id_all, 0u);  // u = 0 initialises every plane
                        } else if (ky == 0 && fresh) {
                            // the new plane u alone (its B rows: u - zlo blocks on), then the others
                            umma_tf32(d + (uint32_t)(u * NZ), ad,
                                      bd + (uint64_t)(((u - zlo) * P::BLK) >> 4), id_one, 0u);
                            if (u > zlo) umma_tf32(dz, ad, bd, id_old, 1u);
                        } else {
                            umma_tf32(dz, ad, bd, id_all, 1u);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < P::NPAIR; ++j) {
                        const int ky = 2 * j;
                        uint64_t bd;
                        if (ky + 1 < K) {
                            bd = bp0 + (uint64_t)((ky * 2 * P::SLEN + blk * P::BLK) >> 4);
                        } else {  // odd k: the last tap pairs with the zero block
                            const uint32_t ad = wbase + (uint32_t)((ky * 2 + 1) * P::SLEN + blk * P::BLK);
                            bd = umma_desc(ad, zaddr - ad, 128);
                        }
                        umma_tf32(dz, ap0 + au + (uint64_t)(ky * WU), bd, id_all, 1u);
                    }
                }
                };
                if (NARROW && info.w < ZG)
                    stage_mmas(std::true_type{});
                else
                    stage_mmas(std::false_type{});
                umma_commit(&st_empty[b]);
                umma_commit(&acc_full[b]);  // the stage's MMAs are done (2 of 2)
            }
            // every MMA issued by this thread completes before TMEM is freed
            umma_commit(&fin_bar);
            mbar_wait_bounded(&fin_bar, 0, kWaitLimitNs);
        }
    } else if (warp < kEpiWarp0) {
        // ---------------- converters ----------------
        const int ct = tid - 64;
        int lb = 0;
        uint32_t lph = 0;
        for (int k = 0;; ++k) {
            if (!wait(&land_full[lb], lph)) break;
            const int4 info = s_land_info[lb];
            const int b = k & 1;
            if (k >= 2 && !wait(&st_empty[b], ((k >> 1) - 1) & 1)) break;
            if (info.x >= 0) {
                const float *src = reinterpret_cast<const float *>(land(lb));
                float4 *xh = reinterpret_cast<float4 *>(stage(b));
                float4 *xl = xh + (size_t)NU * PPU;
                constexpr int CT = 32 * kConvWarps;  // converter threads
                // narrow MMAs of a partial group read only the planes that
                // feed its valid output planes
                const int nuc = P::NARROW ? min(NU, info.w + K - 1) : NU;
                if (a.pad) {
                    // a thread takes 4 consecutive positions of a plane: one
                    // 16-byte load per channel; its i-th stores of a warp land
                    // 64 bytes apart, on distinct banks thanks to the gaps
                    const int nq = P0 >> 2;
#pragma unroll 1
                    for (int u = 0; u < nuc; ++u) {
                        for (int q = ct; q < nq; q += CT) {
                            float4 cv[4];
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                cv[c] = c < a.Ci ? *reinterpret_cast<const float4 *>(
                                                       src + ((size_t)c * NU + u) * P0 + 4 * q)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                            const int o = u * PPU + unit(4 * q);  // 4q % 8 is 0 or 4: one group
                            if (!CN_CHECK(4 * q + 3 < PP, a.err)) continue;
                            xh[o + 0] = make_float4(cv[0].x, cv[1].x, cv[2].x, cv[3].x);
                            xh[o + 1] = make_float4(cv[0].y, cv[1].y, cv[2].y, cv[3].y);
                            xh[o + 2] = make_float4(cv[0].z, cv[1].z, cv[2].z, cv[3].z);
                            xh[o + 3] = make_float4(cv[0].w, cv[1].w, cv[2].w, cv[3].w);
                            xl[o + 0] = make_float4(tf32_rest(cv[0].x), tf32_rest(cv[1].x), tf32_rest(cv[2].x),
                                                    tf32_rest(cv[3].x));
                            xl[o + 1] = make_float4(tf32_rest(cv[0].y), tf32_rest(cv[1].y), tf32_rest(cv[2].y),
                                                    tf32_rest(cv[3].y));
                            xl[o + 2] = make_float4(tf32_rest(cv[0].z), tf32_rest(cv[1].z), tf32_rest(cv[2].z),
                                                    tf32_rest(cv[3].z));
                            xl[o + 3] = make_float4(tf32_rest(cv[0].w), tf32_rest(cv[1].w), tf32_rest(cv[2].w),
                                                    tf32_rest(cv[3].w));
                        }
                    }
                } else
#pragma unroll 1
                for (int u = 0; u < nuc; ++u) {
                    const float *su = src + (size_t)u * P0;
                    // four positions per thread per pass, their loads in flight together
                    for (int p0 = ct; p0 < P0; p0 += 4 * CT) {
                        float v[4][4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                v[j][c] = (c < a.Ci && p0 + j * CT < P0)
                                              ? su[(size_t)c * NU * P0 + p0 + j * CT] : 0.0f;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int p = p0 + j * CT;
                            if (p < P0 && CN_CHECK(P0 <= PP, a.err)) {
                                xh[(size_t)u * PP + p] = make_float4(v[j][0], v[j][1], v[j][2], v[j][3]);
                                xl[(size_t)u * PP + p] =
                                    make_float4(tf32_rest(v[j][0]), tf32_rest(v[j][1]),
                                                tf32_rest(v[j][2]), tf32_rest(v[j][3]));
                            }
                        }
                    }
                }
                fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) {
                if (warp == 2) s_st_info[b] = info;
                mbar_arrive(&land_empty[lb]);
                mbar_arrive(&st_full[b]);
            }
            if (info.x < 0) break;
            if (++lb == a.nland) {
                lb = 0;
                lph ^= 1u;
            }
        }
    } else if (MODE == MODE_MEAN) {
        // ---------------- epilogue: activation, moments, mean ----------------
        constexpr int CQ = CO / 4, NC = CQ * K;  // a warp's channels; its columns of one plane
        const int q = warp & 3;                 // TMEM lane quadrant this warp may read
        const int h = (warp - kEpiWarp0) >> 2;  // channel quarter
        const int r = 32 * q + lane;  // tile row: this thread's position in the band
        const int ry = (int)__umulhi((uint32_t)r, a.wmagic);
        const int rx = r - ry * a.W;
        float bias[CQ], ksh[CQ], s1[CQ], s2[CQ];
#pragma unroll
        for (int c = 0; c < CQ; ++c) {
            bias[c] = a.b ? __ldg(a.b + h * CQ + c) : 0.0f;
            ksh[c] = apply_act(a.act, bias[c]);
            s1[c] = 0.0f;
            s2[c] = 0.0f;
        }
        int pr = 0, pk = 0;  // post ring: slot, items posted (every epilogue warp keeps them)
        uint32_t pph = 0;
        bool post_ok = true, stop_seen = false;
        // A thread's sums of an item are taken about its own first value of
        // the item (plane 0 of the item's first stage: every thread with any
        // valid value of the item has that one), so they never cancel; at the
        // item's end they move to one shift per warp and then per item.
        bool item_first = true;
        int cnt_t = 0;  // the thread's values of the item (per channel)
        for (int k = 0;; ++k) {
            const int b = k & 1;
            const bool got = wait(&acc_full[b], (k >> 1) & 1);
            int4 info = make_int4(-1, 0, 0, 0);
            if (got) info = s_acc_info[b];
            const uint32_t tq = tmem + (uint32_t)(b * P::ACC) + ((uint32_t)(q * 32) << 16);
            float *hb = halo + (size_t)(k & 1) * 4 * (K - 1) * N;
            if (got && info.x >= 0 && a.halo) {
                // rows 0 .. k-2 of this quadrant are the shift halo of the one below
                tc_fence_after();
#pragma unroll 1
                for (int zg = 0; zg < info.w; ++zg) {
                    uint32_t v[NC];
                    const int col0 = (zg * CO + h * CQ) * K;
                    tmem_ld_cols<NC>(tq + (uint32_t)col0, v);
                    tmem_wait_ld();
                    if (q > 0 && lane < K - 1) {
#pragma unroll
                        for (int j = 0; j < NC; ++j)
                            hb[(q * (K - 1) + lane) * N + col0 + j] = __uint_as_float(v[j]);
                    }
                }
            }
            // every epilogue warp got the stage and could post (else all
            // stop), and the halo is written
            if (!epi_all(got && post_ok)) break;
            if (info.x < 0) {
                stop_seen = true;
                break;
            }
            tc_fence_after();
            const bool pos_ok = r < a.rb * a.W && info.y * a.rb + ry < a.Ho && rx < a.Wo;
            if (pos_ok) cnt_t += info.w;
            const float *hq = hb + (size_t)(min(q + 1, 3) * (K - 1)) * N;
#pragma unroll 1
            for (int zg = 0; zg < info.w; ++zg) {
                uint32_t v[NC];
                const int col0 = (zg * CO + h * CQ) * K;
                tmem_ld_cols<NC>(tq + (uint32_t)col0, v);
                tmem_wait_ld();
                const bool valid = pos_ok;  // planes past the group's valid ones are not computed
#pragma unroll
                for (int c = 0; c < CQ; ++c) {
                    float acc = __uint_as_float(v[c * K]);
#pragma unroll
                    for (int kx = 1; kx < K; ++kx) {
                        const float o = __shfl_down_sync(0xffffffffu, __uint_as_float(v[c * K + kx]), kx);
                        // lanes past the quadrant: the halo (W not dividing
                        // 32), else they are columns x >= Wo and unused
                        float hv = 0.0f;
                        if (a.halo && q < 3) hv = hq[max(lane + kx - 32, 0) * N + col0 + c * K + kx];
                        acc += lane + kx < 32 ? o : hv;
                    }
                    const float y = apply_act(a.act, acc + bias[c]);
                    if (item_first && zg == 0) ksh[c] = valid ? y : 0.0f;
                    const float dl = valid ? y - ksh[c] : 0.0f;
                    s1[c] += dl;
                    s2[c] = fmaf(dl, dl, s2[c]);
                }
            }
            item_first = false;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
            if (!info.z) continue;

            // ---- end of the item: its per-channel shifted sums ----
            // Each thread's sums move from its shift to the warp's (that of
            // its lowest lane with values) by the exact identities
            //   S1' = S1 + n d,  S2' = S2 + d (2 S1 + n d),  d = K_t - K_w,
            // then plain adds over the warp.
            item_first = true;
            {
                const unsigned has = __ballot_sync(0xffffffffu, cnt_t > 0);
                const int src = has ? __ffs(has) - 1 : 0;
                const float nt = (float)cnt_t;
#pragma unroll
                for (int c = 0; c < CQ; ++c) {
                    const float kw = __shfl_sync(0xffffffffu, ksh[c], src);
                    const float d = cnt_t > 0 ? ksh[c] - kw : 0.0f;
                    s2[c] += d * fmaf(nt, d, 2.0f * s1[c]);
                    s1[c] = fmaf(nt, d, s1[c]);
                    ksh[c] = kw;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) cnt_t += __shfl_xor_sync(0xffffffffu, cnt_t, off);
#pragma unroll
            for (int c = 0; c < CQ; ++c) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    s1[c] += __shfl_xor_sync(0xffffffffu, s1[c], off);
                    s2[c] += __shfl_xor_sync(0xffffffffu, s2[c], off);
                }
            }
            // straight into the post ring's slot pr (free: the posting warp
            // saw it consumed before the stage's first barrier)
            if (lane == 0) {
#pragma unroll
                for (int c = 0; c < CQ; ++c)
                    reinterpret_cast<float4 *>(red)[((size_t)pr * 4 + q) * CO + h * CQ + c] =
                        make_float4((float)cnt_t, ksh[c], s1[c], s2[c]);
            }
#pragma unroll
            for (int c = 0; c < CQ; ++c) {
                s1[c] = 0.0f;
                s2[c] = 0.0f;
            }
            cnt_t = 0;
            epi_sync();
            // one warp posts the item (its quadrants' sums are in ring slot
            // pr) to warp 0, which merges, publishes and finishes the sample:
            // the epilogue never waits on global memory
            if (warp == kEpiWarp0 && lane == 0) {
                s_post_item[pr] = info.x;
                mbar_arrive(&post_full[pr]);
            }
            ++pk;
            if (++pr == kPosts) {
                pr = 0;
                pph ^= 1u;
            }
            // the next slot must be consumed before any warp writes it: the
            // posting warp checks before the next stage's barrier
            if (warp == kEpiWarp0) post_ok = pk < kPosts || wait(&post_empty[pr], pph ^ 1u);
        }
        // the stop marker reaches warp 0 too
        if (warp == kEpiWarp0 && stop_seen && (pk < kPosts || wait(&post_empty[pr], pph ^ 1u))) {
            if (lane == 0) {
                s_post_item[pr] = -1;
                mbar_arrive(&post_full[pr]);
            }
        }
    } else {
        // ---------------- epilogue: softmax, 4x4x4 max ----------------
        constexpr int CH = 4;                    // channels per TMEM load
        const int q = warp & 3;                  // TMEM lane quadrant this warp may read
        const int zg = (warp - kEpiWarp0) >> 2;  // this warp's output plane of the group
        const int et = tid - 32 * kEpiWarp0;
        const int rq = 32 / a.W;                 // rows per quadrant (W divides 32 here)
        const int row_q = lane / a.W, x = lane - row_q * a.W;
        const int br = q * rq + row_q;           // row in the band
        const bool rep = (x & 3) == 0 && (row_q & (min(rq, 4) - 1)) == 0;  // holds its window's max
        const int cell = (br >> 2) * (a.W >> 2) + (x >> 2);  // pooled (row, column) in the band
        unsigned *cells = reinterpret_cast<unsigned *>(red);  // [CO][kPoolCells]
        float bias[CO];
#pragma unroll
        for (int c = 0; c < CO; ++c) bias[c] = a.b ? __ldg(a.b + c) : 0.0f;
        for (int k = 0;; ++k) {
            const int b = k & 1;
            const bool got = wait(&acc_full[b], (k >> 1) & 1);
            int4 info = make_int4(-1, 0, 0, 0);
            if (got) info = s_acc_info[b];
            // every epilogue warp got the stage (else all stop); the previous
            // stage's cells are stored and cleared
            if (!epi_all(got)) break;
            if (info.x < 0) break;
            tc_fence_after();
            const uint32_t tq = tmem + (uint32_t)(b * P::ACC) + ((uint32_t)(q * 32) << 16);
            float cv[CO];
#pragma unroll
            for (int c0 = 0; c0 < CO; c0 += CH) {
                uint32_t v[CH * K];
                tmem_ld_cols<CH * K>(tq + (uint32_t)((zg * CO + c0) * K), v);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    float acc = __uint_as_float(v[c * K]);
                    // lanes past the quadrant are columns x >= W - kx, in no
                    // window that is stored
#pragma unroll
                    for (int kx = 1; kx < K; ++kx)
                        acc += __shfl_down_sync(0xffffffffu, __uint_as_float(v[c * K + kx]), kx);
                    cv[c0 + c] = acc + bias[c0 + c];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
            float m = cv[0];
#pragma unroll
            for (int c = 1; c < CO; ++c) m = fmaxf(m, cv[c]);
            float s = 0.0f;
#pragma unroll
            for (int c = 0; c < CO; ++c) {
                cv[c] = __expf(cv[c] - m);
                s += cv[c];
            }
            const float inv = 1.0f / s;
#pragma unroll
            for (int c = 0; c < CO; ++c) {
                float p = cv[c] * inv;
                p = fmaxf(p, __shfl_xor_sync(0xffffffffu, p, 1));  // the window's 4 columns
                p = fmaxf(p, __shfl_xor_sync(0xffffffffu, p, 2));
                if (rq >= 2) p = fmaxf(p, __shfl_xor_sync(0xffffffffu, p, a.W));  // rows in the quadrant
                if (rq >= 4) p = fmaxf(p, __shfl_xor_sync(0xffffffffu, p, 2 * a.W));
                if (rep) atomicMax(&cells[c * kPoolCells + cell], __float_as_uint(p));
            }
            epi_sync();
            if (et < CO * kPoolCells) {
                const int c = et / kPoolCells, e = et - c * kPoolCells;
                const int prow = e / (a.W >> 2), pcol = e - prow * (a.W >> 2);
                const int ph = info.y * (a.rb >> 2) + prow;
                if (ph < a.Ph && pcol < a.Pw) {
                    int n, g, z0, nzv;
                    item_group(info.x, n, g, z0, nzv);
                    if (CN_CHECK(n < a.N && g < a.Pd, a.err))
                    a.out[((((size_t)n * CO + c) * a.Pd + g) * a.Ph + ph) * a.Pw + pcol] =
                        a.post_scale * __uint_as_float(cells[et]);
                }
                cells[et] = 0u;
            }
        }
    }

    // ---- teardown ----
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(2 * P::ACC)
                     : "memory");
    if (tid == 0 && atomicAdd(a.work + 1, 1) == (int)gridDim.x - 1) {
        a.work[0] = 0;
        a.work[1] = 0;
    }
}

template <int K, int CO>
__global__ void __launch_bounds__(kT3Threads, 1) k_conv3d_tc_mean(const __grid_constant__ Tc3Args a) {
    tc3_body<K, CO, MODE_MEAN>(a);
}
// The pool kernel capped at 80 registers a thread (it needs no more than
// 77): measured 1% faster on the n128 pool than with the 96 the launch
// bound allows.
template <int K>
__global__ void __maxnreg__(80) k_conv3d_tc_pool(const __grid_constant__ Tc3Args a) {
    tc3_body<K, 16, MODE_POOL>(a);
}

struct T3Inst {
    int mode, K, CO, ZG, WBYTES, HALO, RED;
    Tc3Kernel fn;
    const char *name;
};
#define CN_T3_MEAN(K, CO)                                                                       \
    {MODE_MEAN, K, CO, T3<K, CO>::ZG, T3<K, CO>::WBYTES, T3<K, CO>::HALO, T3<K, CO>::RED, \
     k_conv3d_tc_mean<K, CO>, "k_conv3d_tc_mean<" #K "," #CO ">"}
#define CN_T3_POOL(K)                                                                           \
    {MODE_POOL, K, 16, T3<K, 16>::ZG, T3<K, 16>::WBYTES, T3<K, 16>::HALO, T3<K, 16>::RED, \
     k_conv3d_tc_pool<K>, "k_conv3d_tc_pool<" #K ">"}
const T3Inst kT3Inst[] = {CN_T3_MEAN(3, 16), CN_T3_MEAN(4, 16), CN_T3_MEAN(3, 32),
                          CN_T3_MEAN(4, 32), CN_T3_POOL(3),     CN_T3_POOL(4)};
#undef CN_T3_MEAN
#undef CN_T3_POOL

}  // namespace

int tc3_plan(const conv_norm_desc &d, Tc3Args &a, Tc3Config &cfg) {
    int mode;
    if (d.red == CN_RED_MEAN_SPATIAL && d.act != CN_ACT_SOFTMAX_C)
        mode = MODE_MEAN;
    else if (d.red == CN_RED_MAXPOOL2_X2 && d.act == CN_ACT_SOFTMAX_C && d.norm == CN_NORM_NONE &&
             d.post_scale > 0.0f)
        mode = MODE_POOL;
    else
        return CN_ERR_UNSUPPORTED;
    if (d.conv != CN_CONV3D || d.groups != 1 || d.C_in < 1 || d.C_in > 4) return CN_ERR_UNSUPPORTED;
    const T3Inst *inst = nullptr;
    for (const T3Inst &in : kT3Inst)
        if (in.mode == mode && in.K == d.k && in.CO == d.C_out) inst = &in;
    if (!inst) return CN_ERR_UNSUPPORTED;
    // whole-row tiles of up to 128 positions; the TMA box is a whole row wide;
    // pooling windows need quadrants of whole rows
    if (d.W % 4 != 0 || d.W > 128 || !tma_available()) return CN_ERR_UNSUPPORTED;
    if (mode == MODE_POOL && 32 % d.W != 0) return CN_ERR_UNSUPPORTED;
    const char *e = getenv("CN_NO_TC");
    if (e && atoi(e)) return CN_ERR_UNSUPPORTED;
    const int K = d.k, ZG = inst->ZG, NU = ZG + K - 1;
    const int Do = d.D - K + 1, Ho = d.H - K + 1, Wo = d.W - K + 1;
    if (Do < 1 || Ho < 1 || Wo < 1) return CN_ERR_UNSUPPORTED;
    const int Pd = Do / 4, Ph = Ho / 4, Pw = Wo / 4;
    if (mode == MODE_POOL && (Pd < 1 || Ph < 1 || Pw < 1)) return CN_ERR_UNSUPPORTED;
    const int rb = 128 / d.W;
    const int rows_in = rb + K - 1;
    // farthest operand row an MMA reads: tile row 127 + the largest ky offset
    // (+1 row for the zero-padded pair of an odd k)
    const int far = 127 + (K - 1 + (K & 1)) * d.W;
    const int pp = (std::max(rows_in * d.W, far + 1) + 7) & ~7;
    const int pad = d.W % 8 == 0;
    const int ppu = pad ? pp / 8 * 9 : pp;
    // stage buffers and the landing buffers after them start on 128 bytes
    // (TMA destinations): the padded planes are only 32-byte multiples
    const int stage_bytes = (2 * NU * ppu * 16 + 127) & ~127;
    // the raw filter passes through the two stage buffers at setup
    if ((long long)d.C_out * d.C_in * K * K * K * 4 > 2LL * stage_bytes) return CN_ERR_UNSUPPORTED;
    const int land = d.C_in * NU * rows_in * d.W * 4;
    const int halo = mode == MODE_MEAN && (32 % d.W) != 0;
    // up to four landing buffers (the next stages' copies in flight while
    // this one is converted: n512 0.2600 -> 0.2570 ms with three, 0.2561
    // with four), as many as fit
    const int fixed = 2 * stage_bytes + inst->WBYTES + (halo ? inst->HALO * 4 : 0) + inst->RED * 4;
    int nland = kMaxLand;
    while (nland > 1 && fixed + nland * ((land + 127) & ~127) > kT3SmemLimit) --nland;
    const int smem = fixed + nland * ((land + 127) & ~127);
    if (smem > kT3SmemLimit) return CN_ERR_UNSUPPORTED;
    // one item = some bands of one group of ZG output planes of one sample
    // (the mean keeps one partial-sum slot per item).  A function of the
    // sample's shape only, so a sample's result (its items' merge order) does
    // not depend on the batch it is part of.  The pool needs only the planes
    // and rows its windows cover.
    const int ngroups = mode == MODE_MEAN ? (Do + ZG - 1) / ZG : Pd;
    const int rows = mode == MODE_MEAN ? Ho : 4 * Ph;
    const int nband = (rows + rb - 1) / rb;
    // pool: one band per item; mean: half the group's bands (n512: 0.2567 ms
    // with a quarter, 0.2443 with half, 0.2465 with all, 0.320 with one:
    // every item ends with its sums' round trip through the finisher)
    const int bpi = mode == MODE_POOL ? 1 : std::max(1, nband / 2);
    const int nsplit = (nband + bpi - 1) / bpi;
    const long long items = (long long)d.N * ngroups * nsplit;
    if (items > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;

    a.xmap_base = nullptr;
    a.wait_ns = kWaitLimitNs;
    a.N = d.N;
    a.Ci = d.C_in;
    a.Co = d.C_out;
    a.D = d.D;
    a.H = d.H;
    a.W = d.W;
    a.Do = Do;
    a.Ho = Ho;
    a.Wo = Wo;
    a.k = K;
    a.nu = NU;
    a.rb = rb;
    a.nband = nband;
    a.nsplit = nsplit;
    a.pp = pp;
    a.pad = pad;
    a.ppu = ppu;
    a.stage = stage_bytes;
    a.land = land;
    a.nland = nland;
    a.halo = halo;
    a.wmagic = (uint32_t)(((1ull << 32) + (uint64_t)d.W - 1) / (uint64_t)d.W);
    a.ngroups = ngroups;
    a.items = (int)items;
    a.act = d.act;
    a.norm = d.norm;
    a.G = d.norm == CN_NORM_GROUP ? d.num_groups : d.C_out;
    a.affine = d.affine && d.norm != CN_NORM_NONE;
    a.eps = d.eps;
    a.post_scale = d.post_scale;
    a.Pd = Pd;
    a.Ph = Ph;
    a.Pw = Pw;
    a.inv_cnt = 1.0 / ((double)Do * Ho * Wo);
    a.inv_cpg = 1.0 / (double)(d.C_out / a.G);
    cfg.kern = inst->fn;
    cfg.name = inst->name;
    cfg.threads = kT3Threads;
    cfg.smem = smem;
    cfg.grid = (int)std::min<long long>(items, 148);  // refined from the device in tc3_prepare
    return CN_OK;
}

int tc3_prepare(Tc3Config &cfg, const Tc3Args &a) {
    if (raise_dyn_smem(reinterpret_cast<const void *>(cfg.kern), cfg.smem) !=
        cudaSuccess)
        return CN_ERR_CUDA;
    // persistent grid: one CTA per SM, capped by the work items
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cfg.kern, cfg.threads, cfg.smem) !=
            cudaSuccess)
        return CN_ERR_CUDA;
    if (per_sm < 1) return CN_ERR_UNSUPPORTED;
    cfg.grid = (int)std::min<long long>((long long)sms, (long long)a.items);
    return CN_OK;
}

// Encodes the input tensor map for this x (cached while x stays the same):
// x as (W, H, D, N * C_in), box (W, rb + k - 1 rows, ZG + k - 1 planes,
// C_in); then launches.
int tc3_launch(const Tc3Config &cfg, Tc3Args &a, cudaStream_t s, const LaunchEvents *ev) {
    if (cfg.grid == 0) return CN_OK;
    if (a.xmap_base != a.x) {
        const uint64_t dims[4] = {(uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.D, (uint64_t)a.N * a.Ci};
        const uint64_t strides[3] = {(uint64_t)a.W * 4, (uint64_t)a.H * a.W * 4,
                                     (uint64_t)a.D * a.H * a.W * 4};
        const uint32_t box[4] = {(uint32_t)a.W, (uint32_t)(a.rb + a.k - 1), (uint32_t)a.nu,
                                 (uint32_t)a.Ci};
        const int st = encode_tmap_f32_4d(&a.xmap, a.x, dims, strides, box);
        if (st != CN_OK) return st;
        a.xmap_base = a.x;
    }
    record_launch(ev, 0, s);
    cfg.kern<<<cfg.grid, cfg.threads, cfg.smem, s>>>(a);
    record_launch(ev, 1, s);
    return cudaGetLastError() == cudaSuccess ? CN_OK : CN_ERR_CUDA;
}

int tc3_launches(const Tc3Config &cfg) { return cfg.grid == 0 ? 0 : 1; }

}  // namespace cn
