// Variant 0, tensor-core conv: Conv3d with up to 4 input channels and 16
// or 32 output channels -> activation -> GroupNorm / InstanceNorm / none ->
// mean over D, H, W, as an implicit GEMM on the 5th-generation tensor cores
// (the l2_p27 problem: Conv3d 3 -> 16, k = 4, HardSwish, GroupNorm(4), mean).
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
// rows past a quadrant come from a small shared halo.
//
// Why this shape: a tcgen05.mma with M = 128 and K = 8 costs about the same
// up to N = 128 (measured ~130 cycles at N = 64 and N = 128 on this GPU,
// ~185 at N = 256, the full rate), so N is made as wide as it goes: the kx
// taps and ZG output planes (16 * 4 * 4 = 256 for C_out = 16, k = 4), which
// reads each staged input plane once for the ZG output planes it feeds.
// For input plane u the filter operand rows (zg, co, kx) hold taps
// kz = u - zg: consecutive blocks of one sequence stored with kz descending
// and zero blocks at both ends, so B for every u is a window of that
// sequence (no copies per u).
//
// Precision: split TF32 as in the 2-D tensor-core kernel (the tensor cores
// read tf32 by dropping 13 mantissa bits; with v = hi + lo,
// W * X ~= Wl*Xh + Wh*Xl + Wh*Xh), so the conv matches an fp32 conv to
// ~1e-6 relative.  Per (u, ky) one MMA takes both cross terms (A = [Xh |
// Xl], B = [Wl | Wh]); the hi*hi terms pair two ky taps per MMA (A = Xh at
// rows ky and ky + 1, B = [Wh(ky) | Wh(ky + 1)]; an odd k pairs its last tap
// with a zero filter block).  MMAs per stage: (ZG + k - 1) (k + ceil(k/2)).
//
// Operands (K-major, no swizzle): a staged input plane is [position][4
// channels] fp32, hi part then lo part; a K step of 8 is two 4-channel core
// matrices, 16 bytes a row.  Tap offsets move the start address only.
//
// Warp roles (one persistent CTA per SM, items = (sample, group of ZG
// output planes) claimed from a counter, each item nband stages):
//   warp 0      producer: one TMA tensor copy per stage (W x (RB + k - 1)
//               rows x (ZG + k - 1) planes x C_in, zero fill outside x);
//   warps 2-3   converters: landing [c][u][row][x] -> operand stage hi / lo;
//   warp 1      MMA issuer (one thread): the stage's MMAs into one of two
//               TMEM accumulators;
//   warps 4-19  epilogue, four warps per TMEM lane quadrant (C_out / 4
//               channels each, all ZG planes): tcgen05.ld of the accumulator
//               (thread = position), the kx sum, bias + activation,
//               per-channel shifted sums in registers; at the end of an item
//               its per-channel moments, then the sample's ticket: the last
//               item of a sample merges its items and writes the output (the
//               CUDA-core mean kernel's finish).
#include "cn_common.cuh"
#include "cn_internal.h"
#include "cn_mean_common.cuh"
#include "cn_tcgen05.cuh"

#include <algorithm>
#include <cstdlib>

namespace cn {
namespace {

constexpr int kT3Threads = 640;    // 20 warps: 5 per SM sub-partition, up to 96 registers each
constexpr int kConvWarps = 2;      // warps 2-3
constexpr int kEpiWarp0 = 4;       // epilogue: warps 4-19
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kT3SmemLimit = 227 * 1024 - 1024;  // dynamic part (static barriers beside it)

template <int K, int CO>
struct T3 {
    static constexpr int ZG = CO * K * 4 <= 256 ? 4 : 2;  // output planes per stage
    static constexpr int N = ZG * CO * K;                 // MMA N: (zg, co, kx) columns
    static constexpr int NU = ZG + K - 1;                 // staged input planes
    static constexpr int NPAIR = (K + 1) / 2;             // hi*hi MMAs per input plane
    static constexpr int NB = K + 2 * (ZG - 1);           // blocks of one kz sequence
    static constexpr int BLK = CO * K * 16;               // one kz block: (co, kx) rows x 4 channels
    static constexpr int SLEN = NB * BLK;                 // one (ky, lo | hi) kz sequence
    static constexpr int ZBYTES = (K & 1) ? N * 16 : 0;   // zero block for an odd k
    static constexpr int WBYTES = K * 2 * SLEN + ZBYTES;
    static constexpr int ACC = N <= 128 ? 128 : 256;      // TMEM columns per accumulator
    static constexpr int CQ = CO / 4;                     // channels per epilogue warp
    static constexpr int NC = CQ * K;                     // its columns of one plane zg
    static constexpr int HALO = 2 * 4 * (K - 1) * N;      // floats: [parity][quadrant][row][N]
    static_assert(N % 16 == 0 && N <= 256, "MMA N");
    static_assert(NC % 4 == 0 && NC <= 32, "epilogue columns");
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

template <int K, int CO>
__global__ void __launch_bounds__(kT3Threads, 1) k_conv3d_tc_mean(const __grid_constant__ Mean3dArgs a) {
    using P = T3<K, CO>;
    constexpr int N = P::N, ZG = P::ZG, NU = P::NU;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t land_full, land_empty;
    // st_full[b]: the converters wrote stage b; st_empty[b]: its MMAs are done
    __shared__ __align__(8) uint64_t st_full[2], st_empty[2];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], fin_bar;
    // stage info: (item or -1 to stop, band, 1 if the item's last band, valid planes)
    __shared__ int4 s_land_info, s_st_info[2], s_acc_info[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_last;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int PP = a.tc_pp;
    unsigned char *stages = smem_raw;
    auto stage = [&](int b) { return stages + (size_t)b * a.tc_stage; };
    unsigned char *land = stages + 2 * (size_t)a.tc_stage;
    unsigned char *wts = land + ((a.tc_land + 127) & ~127);
    float *halo = reinterpret_cast<float *>(wts + P::WBYTES);
    float *red = halo + (a.tc_halo ? P::HALO : 0);               // [4 quadrants][CO][2]
    double *sch = reinterpret_cast<double *>(red + 4 * CO * 2);  // [CO][3]
    const int rows_in = a.tc_rb + K - 1;
    const int P0 = rows_in * a.W;  // staged positions per plane

    auto item_group = [&](int item, int &n, int &g, int &z0, int &nzv) {
        n = item / a.nchunks;
        g = item - n * a.nchunks;
        z0 = g * ZG;
        nzv = min(ZG, a.Do - z0);
    };

    // ---- setup: zero the operand tails, filter sequences, barriers, TMEM ----
    for (int b = 0; b < 2; ++b) {
        float4 *xs = reinterpret_cast<float4 *>(stage(b));
        const int tail = PP - P0;
        for (int i = tid; i < 2 * NU * tail; i += blockDim.x) {
            const int pl = i / tail, r = i - pl * tail;
            xs[(size_t)pl * PP + P0 + r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    {
        // [ky][lo | hi][block i: kz = K + ZG - 2 - i][(co, kx) rows][4 channels], zero block
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
                const int kz = K + ZG - 2 - i;
                const int co = row / K, kx = row - co * K;
                if (c < a.Ci && kz >= 0 && kz < K) {
                    const float x = __ldg(a.w + ((((size_t)co * a.Ci + c) * K + kz) * K + ky) * K + kx);
                    v = hi ? x : tf32_rest(x);
                }
            }
            wf[e] = v;
        }
    }
    if (tid == 0) {
        mbar_init(&land_full, 1);
        mbar_init(&land_empty, kConvWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&st_full[i], kConvWarps);
            mbar_init(&st_empty[i], 1);
            mbar_init(&acc_full[i], 2);
            mbar_init(&acc_empty[i], kEpiWarps);
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
    auto wait = [&](uint64_t *bar, uint32_t par) { return tc_wait(bar, par, abort_p, a.err); };

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int k = 0;  // stages armed so far (one landing buffer)
            int next = (int)blockIdx.x;
            bool live = true;
            while (live) {
                const int item = next < a.items ? next : -1;
                if (item >= 0) next = (int)gridDim.x + atomicAdd(a.tickets + a.N, 1);
                int n = 0, g = 0, z0 = 0, nzv = 0;
                if (item >= 0) item_group(item, n, g, z0, nzv);
                const int nb = item >= 0 ? a.tc_nband : 1;  // a stop marker is one stage
                for (int band = 0; band < nb; ++band) {
                    if (k >= 1 && !wait(&land_empty, (k - 1) & 1)) {
                        live = false;
                        break;
                    }
                    s_land_info = make_int4(item, band, band == nb - 1, nzv);
                    if (item >= 0) {
                        mbar_arrive_expect_tx(&land_full, (uint32_t)a.tc_land);
                        tma_load_4d(land, &a.tc_xmap, 0, band * a.tc_rb, z0, n * a.Ci, &land_full);
                    } else {
                        mbar_arrive(&land_full);
                    }
                    ++k;
                }
                if (item < 0) live = false;
            }
            // a copy still in flight (only after an abort) lands before the CTA exits
            if (k >= 1) mbar_wait_bounded(&land_full, (k - 1) & 1, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_tf32(128, N);
            const uint32_t wbase = smem_u32(wts);
            const uint32_t zaddr = wbase + K * 2 * P::SLEN;
            // descriptors are linear in the start address (units of 16 bytes)
            const uint64_t bc0 = umma_desc(wbase, P::SLEN, 128);                 // [Wl | Wh](ky)
            const uint64_t bp0 = umma_desc(wbase + P::SLEN, 2 * P::SLEN, 128);  // [Wh(ky) | Wh(ky+1)]
            const uint32_t xl_off = (uint32_t)(NU * PP * 16);
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
                const uint64_t ac0 = umma_desc(sb, xl_off, 128);                // [Xh | Xl]
                const uint64_t ap0 = umma_desc(sb, (uint32_t)(a.W * 16), 128);  // [Xh(ky) | Xh(ky+1)]
#pragma unroll
                for (int u = 0; u < NU; ++u) {
                    const uint64_t au = (uint64_t)(u * PP);
                    const int blk = K + ZG - 2 - u;  // window start in the kz sequences
#pragma unroll
                    for (int ky = 0; ky < K; ++ky)
                        umma_tf32(d, ac0 + au + (uint64_t)(ky * a.W),
                                  bc0 + (uint64_t)((ky * 2 * P::SLEN + blk * P::BLK) >> 4), idesc,
                                  (u | ky) ? 1u : 0u);
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
                        umma_tf32(d, ap0 + au + (uint64_t)(ky * a.W), bd, idesc, 1u);
                    }
                }
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
        for (int k = 0;; ++k) {
            if (!wait(&land_full, k & 1)) break;
            const int4 info = s_land_info;
            const int b = k & 1;
            if (k >= 2 && !wait(&st_empty[b], ((k >> 1) - 1) & 1)) break;
            if (info.x >= 0) {
                const float *src = reinterpret_cast<const float *>(land);
                float4 *xh = reinterpret_cast<float4 *>(stage(b));
                float4 *xl = xh + (size_t)NU * PP;
#pragma unroll 1
                for (int u = 0; u < NU; ++u) {
                    const float *su = src + (size_t)u * P0;
                    for (int p = ct; p < P0; p += 32 * kConvWarps) {
                        float v[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) v[c] = c < a.Ci ? su[(size_t)c * NU * P0 + p] : 0.0f;
                        xh[(size_t)u * PP + p] = make_float4(v[0], v[1], v[2], v[3]);
                        xl[(size_t)u * PP + p] = make_float4(tf32_rest(v[0]), tf32_rest(v[1]),
                                                             tf32_rest(v[2]), tf32_rest(v[3]));
                    }
                }
                fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) {
                if (warp == 2) s_st_info[b] = info;
                mbar_arrive(&land_empty);
                mbar_arrive(&st_full[b]);
            }
            if (info.x < 0) break;
        }
    } else {
        // ---------------- epilogue ----------------
        constexpr int CQ = P::CQ, NC = P::NC;
        const int q = warp & 3;                 // TMEM lane quadrant this warp may read
        const int h = (warp - kEpiWarp0) >> 2;  // channel quarter
        const int et = tid - 32 * kEpiWarp0;
        const int r = 32 * q + lane;  // tile row: this thread's position in the band
        const int ry = (int)__umulhi((uint32_t)r, a.tc_wmagic);
        const int rx = r - ry * a.W;
        float bias[CQ], ksh[CQ], s1[CQ], s2[CQ];
#pragma unroll
        for (int c = 0; c < CQ; ++c) {
            bias[c] = a.b ? __ldg(a.b + h * CQ + c) : 0.0f;
            ksh[c] = apply_act(a.act, bias[c]);
            s1[c] = 0.0f;
            s2[c] = 0.0f;
        }
        for (int k = 0;; ++k) {
            const int b = k & 1;
            const bool got = wait(&acc_full[b], (k >> 1) & 1);
            int4 info = make_int4(-1, 0, 0, 0);
            if (got) info = s_acc_info[b];
            const uint32_t tq = tmem + (uint32_t)(b * P::ACC) + ((uint32_t)(q * 32) << 16);
            float *hb = halo + (size_t)(k & 1) * 4 * (K - 1) * N;
            if (got && info.x >= 0 && a.tc_halo) {
                // rows 0 .. k-2 of this quadrant are the shift halo of the one below
                tc_fence_after();
#pragma unroll 1
                for (int zg = 0; zg < ZG; ++zg) {
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
            // every epilogue warp got the stage (else all stop), and the halo is written
            if (!epi_all(got)) break;
            if (info.x < 0) break;
            tc_fence_after();
            const bool pos_ok = r < a.tc_rb * a.W && info.y * a.tc_rb + ry < a.Ho && rx < a.Wo;
            const float *hq = hb + (size_t)(min(q + 1, 3) * (K - 1)) * N;
#pragma unroll 1
            for (int zg = 0; zg < ZG; ++zg) {
                uint32_t v[NC];
                const int col0 = (zg * CO + h * CQ) * K;
                tmem_ld_cols<NC>(tq + (uint32_t)col0, v);
                tmem_wait_ld();
                const bool valid = pos_ok && zg < info.w;
#pragma unroll
                for (int c = 0; c < CQ; ++c) {
                    float acc = __uint_as_float(v[c * K]);
#pragma unroll
                    for (int kx = 1; kx < K; ++kx) {
                        const float o = __shfl_down_sync(0xffffffffu, __uint_as_float(v[c * K + kx]), kx);
                        // lanes past the quadrant: the halo (W not dividing
                        // 32), else they are columns x >= Wo and unused
                        float hv = 0.0f;
                        if (a.tc_halo && q < 3) hv = hq[max(lane + kx - 32, 0) * N + col0 + c * K + kx];
                        acc += lane + kx < 32 ? o : hv;
                    }
                    const float y = apply_act(a.act, acc + bias[c]);
                    const float dl = valid ? y - ksh[c] : 0.0f;
                    s1[c] += dl;
                    s2[c] = fmaf(dl, dl, s2[c]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
            if (!info.z) continue;

            // ---- end of the item: its per-channel moments, then the ticket ----
            int n, g, z0, nzv;
            item_group(info.x, n, g, z0, nzv);
#pragma unroll
            for (int c = 0; c < CQ; ++c) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    s1[c] += __shfl_xor_sync(0xffffffffu, s1[c], off);
                    s2[c] += __shfl_xor_sync(0xffffffffu, s2[c], off);
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int c = 0; c < CQ; ++c) {
                    red[(q * CO + h * CQ + c) * 2 + 0] = s1[c];
                    red[(q * CO + h * CQ + c) * 2 + 1] = s2[c];
                }
            }
#pragma unroll
            for (int c = 0; c < CQ; ++c) {
                s1[c] = 0.0f;
                s2[c] = 0.0f;
            }
            epi_sync();
            if (et < CO) {
                float S1 = 0.0f, S2 = 0.0f;
                for (int qq = 0; qq < 4; ++qq) {  // fixed quadrant order
                    S1 += red[(qq * CO + et) * 2 + 0];
                    S2 += red[(qq * CO + et) * 2 + 1];
                }
                const float kc = apply_act(a.act, a.b ? __ldg(a.b + et) : 0.0f);
                const Moments<double> m =
                    moments_from_sums((double)nzv * a.Ho * a.Wo, (double)kc, (double)S1, (double)S2);
                double *pp = a.partial + (((size_t)n * a.nchunks + g) * a.Co + et) * 3;
                pp[0] = m.n;
                pp[1] = m.mean;
                pp[2] = m.m2;
            }
            __threadfence();
            epi_sync();
            if (et == 0) s_last = (atomicAdd(a.tickets + n, 1) == a.nchunks - 1);
            epi_sync();
            if (s_last) {
                __threadfence();
                for (int c = et; c < a.Co; c += kEpiThreads) {
                    const Moments<double> m = mean_chunks_merged(a, n, c);
                    sch[c * 3 + 0] = m.n;
                    sch[c * 3 + 1] = m.mean;
                    sch[c * 3 + 2] = m.m2;
                }
                epi_sync();
                for (int c = et; c < a.Co; c += kEpiThreads) mean_write_output(a, n, c, sch);
                if (et == 0) a.tickets[n] = 0;
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
    if (tid == 0 && atomicAdd(a.tickets + a.N + 1, 1) == (int)gridDim.x - 1) {
        a.tickets[a.N] = 0;
        a.tickets[a.N + 1] = 0;
    }
}

struct T3Inst {
    int K, CO, ZG, WBYTES, HALO;
    Mean3dKernel fn;
    const char *name;
};
#define CN_T3_INST(K, CO)                                                                     \
    {K, CO, T3<K, CO>::ZG, T3<K, CO>::WBYTES, T3<K, CO>::HALO, k_conv3d_tc_mean<K, CO>, \
     "k_conv3d_tc_mean<" #K "," #CO ">"}
const T3Inst kT3Inst[] = {CN_T3_INST(3, 16), CN_T3_INST(4, 16), CN_T3_INST(3, 32), CN_T3_INST(4, 32)};
#undef CN_T3_INST

}  // namespace

int tc3_mean_plan(const conv_norm_desc &d, Mean3dArgs &a, Mean3dConfig &cfg) {
    if (d.conv != CN_CONV3D || d.groups != 1 || d.C_in < 1 || d.C_in > 4) return CN_ERR_UNSUPPORTED;
    const T3Inst *inst = nullptr;
    for (const T3Inst &in : kT3Inst)
        if (in.K == d.k && in.CO == d.C_out) inst = &in;
    if (!inst) return CN_ERR_UNSUPPORTED;
    // whole-row tiles of up to 128 positions; the TMA box is a whole row wide
    if (d.W % 4 != 0 || d.W > 128 || !tma_available()) return CN_ERR_UNSUPPORTED;
    const char *e = getenv("CN_NO_TC");
    if (e && atoi(e)) return CN_ERR_UNSUPPORTED;
    const int K = d.k, CO = d.C_out, ZG = inst->ZG, NU = ZG + K - 1;
    const int Do = d.D - K + 1, Ho = d.H - K + 1, Wo = d.W - K + 1;
    if (Do < 1 || Ho < 1 || Wo < 1) return CN_ERR_UNSUPPORTED;
    const int rb = 128 / d.W;
    const int rows_in = rb + K - 1;
    // farthest operand row an MMA reads: tile row 127 + the largest ky offset
    // (+1 row for the zero-padded pair of an odd k)
    const int far = 127 + (K - 1 + (K & 1)) * d.W;
    const int pp = (std::max(rows_in * d.W, far + 1) + 7) & ~7;
    const int stage_bytes = 2 * NU * pp * 16;
    const int land = d.C_in * NU * rows_in * d.W * 4;
    const int halo = (32 % d.W) != 0;
    const int smem = 2 * stage_bytes + ((land + 127) & ~127) + inst->WBYTES +
                     (halo ? inst->HALO * 4 : 0) + 4 * CO * 2 * 4 + CO * 3 * 8;
    if (smem > kT3SmemLimit) return CN_ERR_UNSUPPORTED;
    // one item = one group of ZG output planes of one sample: a function of
    // the sample's shape only, so a sample's result (its items' merge order)
    // does not depend on the batch it is part of
    const int nchunks = (Do + ZG - 1) / ZG;
    const long long items = (long long)d.N * nchunks;
    if (items > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;

    a.tc = 1;
    a.tc_xmap_base = nullptr;
    a.tc_rb = rb;
    a.tc_nband = (Ho + rb - 1) / rb;
    a.tc_pp = pp;
    a.tc_stage = stage_bytes;
    a.tc_land = land;
    a.tc_halo = halo;
    a.tc_wmagic = (uint32_t)(((1ull << 32) + (uint64_t)d.W - 1) / (uint64_t)d.W);
    a.use_tma = 0;
    a.tmap_base = nullptr;
    a.N = d.N;
    a.Ci = d.C_in;
    a.Co = d.C_out;
    a.D = d.D;
    a.H = d.H;
    a.W = d.W;
    a.Do = Do;
    a.Ho = Ho;
    a.Wo = Wo;
    a.nseg = 1;
    a.rows = 0;
    a.rows_per_cta = 0;
    a.nchunks = nchunks;
    a.ncob = 1;
    a.wco = 0;
    a.wrows = 0;
    a.planes_max = NU;
    a.pitch = d.W;
    a.nbuf = 2;
    a.buf_stride = 0;
    a.items = (int)items;
    a.vec16 = 1;
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
    cfg.COT = CO;
    cfg.threads = kT3Threads;
    cfg.smem = smem;
    cfg.grid = (int)std::min<long long>(items, 148);  // refined from the device in mean3d_prepare
    return CN_OK;
}

// Encodes the input tensor map for this x (cached while x stays the same):
// x as (W, H, D, N * C_in), box (W, rb + k - 1 rows, ZG + k - 1 planes, C_in).
int tc3_bind_x(Mean3dArgs &a) {
    if (a.tc_xmap_base == a.x) return CN_OK;
    const int K = a.D - a.Do + 1;
    const uint64_t dims[4] = {(uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.D, (uint64_t)a.N * a.Ci};
    const uint64_t strides[3] = {(uint64_t)a.W * 4, (uint64_t)a.H * a.W * 4,
                                 (uint64_t)a.D * a.H * a.W * 4};
    const uint32_t box[4] = {(uint32_t)a.W, (uint32_t)(a.tc_rb + K - 1), (uint32_t)a.planes_max,
                             (uint32_t)a.Ci};
    const int st = encode_tmap_f32_4d(&a.tc_xmap, a.x, dims, strides, box);
    if (st != CN_OK) return st;
    a.tc_xmap_base = a.x;
    return CN_OK;
}

}  // namespace cn
