// Variant 2, tensor-core transposed conv: grouped ConvTranspose2d (stride 1,
// padding 0, 8 input and 8 output channels per group, k = 3) as an implicit
// GEMM on the 5th-generation tensor cores, for the l2_p19 problem shape
// (ConvTranspose2d 64 -> 64, groups 8, k = 3, then GELU and GroupNorm(8)).
//
// The transposed conv as a correlation.  With xp = x padded by k - 1 zeros
// on every side and the filter flipped, wf[ci][co][ky][kx] =
// w[ci][co][k-1-ky][k-1-kx] (the adjoint derivation of the page),
//   y[n][co][i][j] = b[co] + sum_{ci in group} sum_{ky,kx} xp[ci][i+ky][j+kx] wf[ci][co][ky][kx],
// an ordinary stride-1 correlation with Ho = H + k - 1, Wo = W + k - 1.
//
// GEMM.  A unit is ZG = 6 output rows (a band) x 30 output columns (a
// segment) of one (sample, group).  Its input is ZG + k - 1 = 8 padded rows
// of 32 positions; a tile packs four units (of one group, so of one filter)
// as the four 32-lane quadrants of M = 128.  Per input row u of the tile,
//   Dacc[m][(zg, co, kx)] += sum_ci X[u][m][ci] * wf[ci][co][u - zg][kx]
// (wf = 0 where u - zg is not a tap) with N = (zg, co, kx) = 6 * 8 * 3 = 144
// columns and K = the group's 8 input channels, and the output is the
// kx-shifted sum of accumulator rows, done by the epilogue with warp
// shuffles inside a quadrant:
//   y[r0 + zg][c0 + m] = sum_kx Dacc[m + kx][(zg, co, kx)],  m < 30.
// The filter operand of input row u holds taps ky = u - zg: blocks of one
// sequence stored with ky descending and zero blocks at both ends, so B for
// every u is a window of it (the same scheme as the tensor-core Conv3d).
//
// Precision: split TF32 (v = hi + lo, hi = the tf32 part the tensor core
// reads, lo = the exact remainder): W X ~= Wh Xh + Wl Xh + Wh Xl, three MMAs
// of K = 8 per input row: Xh(c0..7) x Wh, [Xh | Xl](c0..3) x [Wl | Wh], and
// the same for channels 4..7.  The conv then matches an fp32 conv to ~1e-6
// relative.
//
// Operands (K-major, no swizzle, a core matrix is 8 rows x 16 bytes): an
// operand stage is [input row u][Xh c0-3 | Xh c4-7 | Xl c0-3 | Xl c4-7][128
// positions][4 channels]; the filter is [Wl c0-3 | Wl c4-7 | Wh c0-3 | Wh
// c4-7][block][(co, kx) rows][4 channels].  The leading-byte offset of a
// descriptor picks the second K half anywhere, so the three MMAs differ in
// their start addresses and offsets only.
//
// Warp roles (one persistent CTA per SM; the CTAs are split evenly over the
// conv groups, each claims tiles of its group from a counter and builds its
// group's filter operand once):
//   warp 0      producer: four TMA tensor copies per tile (36 columns x 8
//               rows x 8 channels each, zero fill outside x: the padding)
//               into one of two landing buffers; tiles are claimed two
//               ahead, so the claim's round trip is off the critical path;
//   warps 2-5   converters, warp 2 + q for unit q: landing [c][row][col]
//               -> the unit's quadrant of the operand stage;
//   warp 1      MMA issuer (one thread): 24 MMAs per tile into one of two
//               TMEM accumulators;
//   warps 6-21  epilogue, thread = position: warp (q, h) reads quadrant q
//               (unit q) and output channels 2h, 2h + 1 of all its rows
//               (every column it needs with one TMEM wait, after which the
//               accumulator is released; the channel pair in packed fp32x2
//               arithmetic): the kx sum, bias, activation, the pre-norm
//               store, and per-channel sums about the unit's first value,
//               written as the unit's partial (count, K, S1, S2) for the
//               statistics pass.
// The statistics and normalize passes that follow are the ones of the other
// 2-D paths (k_group_stats, k_norm_apply).
#include "cn_common.cuh"
#include "cn_internal.h"
#include "cn_tcgen05.cuh"

#include <algorithm>
#include <cstdlib>

namespace cn {
namespace {

constexpr int kK = 3;                       // filter extent
constexpr int kCig = 8, kCog = 8;           // channels per group
constexpr int kZG = 6;                      // output rows per unit
constexpr int kRowsIn = kZG + kK - 1;       // staged input rows per unit
constexpr int kSegV = 32 - (kK - 1);        // valid output columns per unit
constexpr int kBoxW = 36;                   // TMA box columns (16-byte aligned start, +3)
constexpr int kN = kZG * kCog * kK;         // MMA N: (zg, co, kx)
constexpr int kAccCols = 256;               // TMEM columns per accumulator (two)
constexpr int kArr = 128 * 16;              // one [128 positions][4 ch] operand array
constexpr int kRowBytes = 4 * kArr;         // Xh c0-3 | Xh c4-7 | Xl c0-3 | Xl c4-7
constexpr int kStageBytes = kRowsIn * kRowBytes;
constexpr int kUnitLand = kCig * kRowsIn * kBoxW * 4;  // one unit's TMA box
constexpr int kLandBytes = 4 * kUnitLand;
constexpr int kBlk = kCog * kK * 16;        // one ky block: (co, kx) rows x 4 channels
constexpr int kNB = 2 * kZG + kK - 2;       // blocks of one ky sequence
constexpr int kC = kZG + kK - 2;            // block i holds ky = kC - i
constexpr int kSeq = kNB * kBlk;            // one sequence
constexpr int kFiltBytes = 4 * kSeq;
constexpr int kNLand = 2;                   // landing buffers
constexpr int kSmemBytes = 2 * kStageBytes + kNLand * kLandBytes + kFiltBytes;
constexpr int kConvWarps = 4;               // warps 2-5, one unit of a tile each
constexpr int kEpiWarp0 = 2 + kConvWarps;   // epilogue: warps 6-21
constexpr int kEpiRows = kZG;               // output rows per epilogue warp
constexpr int kEpiCo = 2;                   // output channels per epilogue warp
constexpr int kRowParts = kZG / kEpiRows;   // a unit's rows split over this many warps
constexpr int kEpiWarps = 4 * kRowParts * (kCog / kEpiCo);  // six per TMEM lane quadrant
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
static_assert(kZG % kEpiRows == 0 && kCog % kEpiCo == 0 && kEpiCo % 2 == 0, "epilogue split");
static_assert(kEpiCo * kK == 6 || kEpiCo * kK == 12, "TMEM loads of a warp's row columns");
static_assert(kN % 16 == 0 && kN <= kAccCols, "MMA N");
static_assert((kZG - 1) * kCog * kK + (kCog - kEpiCo) * kK + 8 <= kAccCols,
              "an epilogue row's 8-column load stays inside the accumulator");
static_assert(kBlk % 128 == 0, "a block is whole 8-row core-matrix groups");
static_assert(kUnitLand % 128 == 0, "landing units stay 128-byte aligned");
static_assert(kSmemBytes <= 227 * 1024 - 1024, "shared memory");

template <int ACT>
CN_DEV float2 act_v2(float2 t) {
    if (ACT == ACT_HARDSWISH) return make_float2(hardswish(t.x), hardswish(t.y));
    if (ACT == ACT_GELU) return gelu_erf2(t);
    return t;
}

// Unit u of a group (over samples, bands, segments) -> its sample, band, segment.
struct Unit {
    int n, band, seg;
};
CN_DEV Unit unit_of(const Full2dArgs &a, int u) {
    Unit r;
    r.n = u / a.tct_U;
    const int rem = u - r.n * a.tct_U;
    r.band = rem / a.tct_nseg;
    r.seg = rem - r.band * a.tct_nseg;
    return r;
}
// First x column of a unit's TMA box: 16-byte aligned, at or left of the
// unit's first padded column (x column 30 seg - (k - 1)); off = the unit's
// first column inside the box (0..3).
CN_DEV int box_col(int seg, int &off) {
    const int c = seg * kSegV - (kK - 1);
    const int c4 = c >= 0 ? (c & ~3) : -((-c + 3) & ~3);
    off = c - c4;
    return c4;
}

template <int ACT>
__global__ void __launch_bounds__(kThreads, 1) k_convt2d_tc(const __grid_constant__ Full2dArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t land_full[kNLand], land_empty[kNLand];
    // st_full[b]: the converters wrote stage b; st_empty[b]: its MMAs are done
    __shared__ __align__(8) uint64_t st_full[2], st_empty[2];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], fin_bar;
    __shared__ int s_land_tile[kNLand], s_st_tile[2], s_acc_tile[2];  // tile or -1 to stop
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned char *stage0 = smem_raw;
    auto stage = [&](int b) { return stage0 + (size_t)b * kStageBytes; };
    unsigned char *land0 = stage0 + 2 * (size_t)kStageBytes;
    auto land = [&](int b) { return land0 + (size_t)b * kLandBytes; };
    unsigned char *filt = land0 + kNLand * (size_t)kLandBytes;

    // this CTA's group and its place among the group's CTAs
    const int g = (int)blockIdx.x / a.tct_ctas_g;
    const int cta_in_g = (int)blockIdx.x - g * a.tct_ctas_g;
    const int units_g = a.N * a.tct_U;

    // ---- setup: the group's filter operand, barriers, TMEM ----
    {
        // [lo | hi][channel half][block i: ky = kC - i][(co, kx) rows][4 channels]
        float *wf = reinterpret_cast<float *>(filt);
        for (int e = tid; e < kFiltBytes / 4; e += blockDim.x) {
            const int j = e & 3;
            int r = e >> 2;
            const int row = r % (kCog * kK);
            r /= kCog * kK;
            const int i = r % kNB;
            const int seq = r / kNB;  // part * 2 + half
            const int ky = kC - i;
            float v = 0.0f;
            if (ky >= 0 && ky < kK) {
                const int ci = (seq & 1) * 4 + j, co = row / kK, kx = row - co * kK;
                // PyTorch's transposed-conv weight (C_in, C_out / groups, k, k), flipped
                const float x = __ldg(a.w + (((size_t)(g * kCig + ci) * kCog + co) * kK + (kK - 1 - ky)) * kK +
                                      (kK - 1 - kx));
                v = (seq >> 1) ? x : tf32_rest(x);
            }
            wf[e] = v;
        }
    }
    if (tid == 0) {
        for (int i = 0; i < kNLand; ++i) {
            mbar_init(&land_full[i], 1);
            mbar_init(&land_empty[i], kConvWarps);
        }
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
                     "r"(2 * kAccCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    fence_proxy_async();  // the filter operand is read by the MMAs
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    int *abort_p = const_cast<int *>(&s_abort);
    auto wait = [&](uint64_t *bar, uint32_t par) {
        return tc_wait_sleep(bar, par, abort_p, a.err, a.wait_ns);
    };
    int *work = a.tickets + a.N;  // [G] per-group work counters, then the exit counter

    if (warp == 0) {
        // ---------------- producer ----------------
        // Lane 0 claims tiles two ahead of the one it arms (the claim's round
        // trip overlaps a whole tile) and issues the four copies of each.
        if (lane == 0) {
            int k = 0;
            int cur = cta_in_g;  // the tile armed next; later ones from the group's counter
            int nxt = a.tct_ctas_g + atomicAdd(work + g, 1);  // past the last tile: a stop
            for (;; ++k) {
                const int lb = k % kNLand;
                if (k >= kNLand && !wait(&land_empty[lb], ((k / kNLand) - 1) & 1)) break;
                const int tile = cur < a.tct_tiles_g ? cur : -1;
                s_land_tile[lb] = tile;
                if (tile < 0) {
                    mbar_arrive(&land_full[lb]);
                    ++k;
                    break;
                }
                cur = nxt;
                if (cur < a.tct_tiles_g) nxt = a.tct_ctas_g + atomicAdd(work + g, 1);
                // failure-path test hook: the first landing stage of CTA 0
                // stays unarmed, a phase nothing completes
                if (a.stall && blockIdx.x == 0 && k == 0) continue;
                const int nv = min(4, units_g - 4 * tile);
                mbar_arrive_expect_tx(&land_full[lb], (uint32_t)(nv * kUnitLand));
                for (int q = 0; q < nv; ++q) {
                    const Unit U = unit_of(a, 4 * tile + q);
                    int off;
                    const int c4 = box_col(U.seg, off);
                    tma_load_4d(land(lb) + (size_t)q * kUnitLand, &a.tct_xmap, c4, U.band * kZG - (kK - 1),
                                g * kCig, U.n, &land_full[lb]);
                }
            }
            // copies still in flight (only after an abort) land before the CTA
            // exits; in a normal run these phases are long complete
            for (int j = max(0, k - kNLand); j < k; ++j)
                if (!(a.stall && blockIdx.x == 0 && j == 0))
                    mbar_wait_bounded(&land_full[j % kNLand], (j / kNLand) & 1, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_tf32(128, kN);
            const uint32_t wb = smem_u32(filt);
            // B windows: input row u reads blocks kC - u .. kC - u + ZG - 1
            const uint64_t b_hh = umma_desc(wb + 2 * kSeq + kC * kBlk, kSeq, 128);      // [Wh c0-3 | Wh c4-7]
            const uint64_t b_c1 = umma_desc(wb + kC * kBlk, 2 * kSeq, 128);             // [Wl c0-3 | Wh c0-3]
            const uint64_t b_c2 = umma_desc(wb + kSeq + kC * kBlk, 2 * kSeq, 128);      // [Wl c4-7 | Wh c4-7]
            for (int k = 0;; ++k) {
                const int b = k & 1;
                if (!wait(&st_full[b], (k >> 1) & 1)) break;
                const int tile = s_st_tile[b];
                if (k >= 2 && !wait(&acc_empty[b], ((k >> 1) - 1) & 1)) break;
                tc_fence_after();  // the epilogue's reads of this accumulator are done
                s_acc_tile[b] = tile;
                mbar_arrive(&acc_full[b]);  // publishes the tile (1 of 2 arrivals)
                if (tile < 0) {
                    mbar_arrive(&acc_full[b]);
                    break;
                }
                const uint32_t d = tmem + (uint32_t)(b * kAccCols);
                const uint32_t sa = smem_u32(stage(b));
                const uint64_t a_hh = umma_desc(sa, kArr, 128);               // [Xh c0-3 | Xh c4-7]
                const uint64_t a_c1 = umma_desc(sa, 2 * kArr, 128);           // [Xh c0-3 | Xl c0-3]
                const uint64_t a_c2 = umma_desc(sa + kArr, 2 * kArr, 128);    // [Xh c4-7 | Xl c4-7]
#pragma unroll
                for (int u = 0; u < kRowsIn; ++u) {
                    // descriptors are linear in the start address (16-byte units)
                    const uint64_t au = (uint64_t)((u * kRowBytes) >> 4);
                    const uint64_t bu = (uint64_t)((u * kBlk) >> 4);  // window start kC - u
                    umma_tf32(d, a_hh + au, b_hh - bu, idesc, u > 0 ? 1u : 0u);
                    umma_tf32(d, a_c1 + au, b_c1 - bu, idesc, 1u);
                    umma_tf32(d, a_c2 + au, b_c2 - bu, idesc, 1u);
                }
                umma_commit(&st_empty[b]);
                umma_commit(&acc_full[b]);  // the tile's MMAs are done (2 of 2)
            }
            // every MMA issued by this thread completes before TMEM is freed
            umma_commit(&fin_bar);
            mbar_wait_bounded(&fin_bar, 0, kWaitLimitNs);
        }
    } else if (warp < kEpiWarp0) {
        // ---------------- converters ----------------
        // Warp 2 + q converts unit q of each tile: lane i takes position i
        // of the unit's 8 staged rows (loads of a warp: 32 consecutive words;
        // stores: 32 consecutive 16-byte rows).  The landing buffer and the
        // operand stage are both released after the stores (releasing the
        // landing buffer right after the loads measured slower).
        static_assert(kConvWarps == 4, "one unit of a tile per converter warp");
        const int q = warp - 2;
        for (int k = 0;; ++k) {
            const int lb = k % kNLand, b = k & 1;
            if (!wait(&land_full[lb], (k / kNLand) & 1)) break;
            const int tile = s_land_tile[lb];
            if (k >= 2 && !wait(&st_empty[b], ((k >> 1) - 1) & 1)) break;
            bool wrote = false;
            if (tile >= 0 && 4 * tile + q < units_g) {
                int off;
                box_col(unit_of(a, 4 * tile + q).seg, off);
                const float *s = reinterpret_cast<const float *>(land(lb)) + (size_t)q * (kUnitLand / 4) + off + lane;
                float4 *dst = reinterpret_cast<float4 *>(stage(b)) + q * 32 + lane;
                if (CN_CHECK(q * (kUnitLand / 4) + (kCig - 1) * kRowsIn * kBoxW + (kRowsIn - 1) * kBoxW + off + lane <
                                 kLandBytes / 4,
                             a.err)) {
                    // all 64 loads in flight before the first store
                    float v[kRowsIn][8];
#pragma unroll
                    for (int u = 0; u < kRowsIn; ++u)
#pragma unroll
                        for (int c = 0; c < 8; ++c) v[u][c] = s[c * kRowsIn * kBoxW + u * kBoxW];
#pragma unroll
                    for (int u = 0; u < kRowsIn; ++u) {
                        float4 *row = dst + u * (kRowBytes / 16);
                        row[0] = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
                        row[128] = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
                        row[256] = make_float4(tf32_rest(v[u][0]), tf32_rest(v[u][1]), tf32_rest(v[u][2]),
                                               tf32_rest(v[u][3]));
                        row[384] = make_float4(tf32_rest(v[u][4]), tf32_rest(v[u][5]), tf32_rest(v[u][6]),
                                               tf32_rest(v[u][7]));
                    }
                    wrote = true;
                }
            }
            if (wrote) fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                if (warp == 2) s_st_tile[b] = tile;
                mbar_arrive(&land_empty[lb]);
                mbar_arrive(&st_full[b]);
            }
            if (tile < 0) break;
        }
    } else {
        // ---------------- epilogue ----------------
        const int e = warp - kEpiWarp0;
        const int q = warp & 3;                  // TMEM lane quadrant = unit of the tile
        const int rp = (e >> 2) % kRowParts;     // output rows kEpiRows rp ..
        const int h = (e >> 2) / kRowParts;      // output channels kEpiCo h ..
        const int co0 = g * kCog + kEpiCo * h;
        constexpr int NV = kEpiCo * kK;          // a warp's columns of one output row
        constexpr int NP = kEpiCo / 2;           // channel pairs
        float2 bias2[NP];
#pragma unroll
        for (int c = 0; c < NP; ++c)
            bias2[c] = a.b ? make_float2(__ldg(a.b + co0 + 2 * c), __ldg(a.b + co0 + 2 * c + 1))
                           : make_float2(0.0f, 0.0f);
        for (int k = 0;; ++k) {
            const int b = k & 1;
            if (!wait(&acc_full[b], (k >> 1) & 1)) break;
            const int tile = s_acc_tile[b];
            if (tile < 0) break;
            tc_fence_after();
            const int unit = 4 * tile + q;
            if (unit < units_g) {  // uniform per warp
                const Unit U = unit_of(a, unit);
                const int r0 = U.band * kZG + kEpiRows * rp, c0 = U.seg * kSegV;
                const int rows_ok = max(0, min(kEpiRows, a.Ho - r0));
                const int col = c0 + lane;
                const bool col_ok = lane < kSegV && col < a.Wo;
                const uint32_t tq = tmem + (uint32_t)(b * kAccCols) + ((uint32_t)(q * 32) << 16);
                // every column this warp needs, then one wait (a row's six
                // columns by one 8-column load: the two past them are unused
                // and stay inside the accumulator's allocation)
                uint32_t v[kEpiRows][NV == 6 ? 8 : NV];
#pragma unroll
                for (int zi = 0; zi < kEpiRows; ++zi) {
                    const uint32_t ta = tq + (uint32_t)((kEpiRows * rp + zi) * kCog * kK + kEpiCo * h * kK);
                    if (NV == 12) {
                        tmem_ld8(ta, v[zi]);
                        tmem_ld4(ta + 8, v[zi] + 8);
                    } else {
                        tmem_ld8(ta, v[zi]);
                    }
                }
                tmem_wait_ld();
                // the accumulator is in registers: release it for the tile
                // after next, whose MMAs then overlap this tile's arithmetic
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[b]);
                // kx sums by lane shifts (the next two positions' columns),
                // then the channel pairs in packed arithmetic
                float2 y[kEpiRows][NP];
#pragma unroll
                for (int zi = 0; zi < kEpiRows; ++zi)
#pragma unroll
                    for (int c = 0; c < NP; ++c) {
                        const uint32_t *w0 = v[zi] + 2 * c * kK, *w1 = w0 + kK;
                        float2 acc = make_float2(__uint_as_float(w0[0]), __uint_as_float(w1[0]));
#pragma unroll
                        for (int kx = 1; kx < kK; ++kx)
                            acc = add2(acc, make_float2(__shfl_down_sync(0xffffffffu, __uint_as_float(w0[kx]), kx),
                                                        __shfl_down_sync(0xffffffffu, __uint_as_float(w1[kx]), kx)));
                        y[zi][c] = act_v2<ACT>(add2(acc, bias2[c]));
                    }
                // shift of the warp's sums: its first value (row r0, column
                // c0: inside the output whenever the warp has rows)
                float2 ksh[NP], s1[NP], s2[NP];
                float *obase = a.out + ((size_t)U.n * a.Co + co0) * (size_t)a.S + (size_t)r0 * a.Wo + col;
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    ksh[c] = make_float2(__shfl_sync(0xffffffffu, y[0][c].x, 0),
                                         __shfl_sync(0xffffffffu, y[0][c].y, 0));
                    s1[c] = make_float2(0.0f, 0.0f);
                    s2[c] = s1[c];
                }
#pragma unroll
                for (int zi = 0; zi < kEpiRows; ++zi) {
                    const bool ok = col_ok && zi < rows_ok;
#pragma unroll
                    for (int c = 0; c < NP; ++c) {
                        float2 dl = add2(y[zi][c], make_float2(-ksh[c].x, -ksh[c].y));
                        if (!ok) dl = make_float2(0.0f, 0.0f);
                        s1[c] = add2(s1[c], dl);
                        s2[c] = fma2(dl, dl, s2[c]);
                        float *o = obase + (size_t)(2 * c) * a.S + (size_t)zi * a.Wo;
                        if (ok && CN_CHECK((size_t)(o - a.out) + (size_t)a.S < (size_t)a.N * a.Co * a.S, a.err)) {
                            o[0] = y[zi][c].x;
                            o[a.S] = y[zi][c].y;
                        }
                    }
                }
                // Warp sums of the four values (S1, S2 of the two channels) by
                // reduce-scatter: halve the values each lane carries (xor 16,
                // then xor 8), then a butterfly over the last three lane bits.
                // Lane 0 ends with S1 of channel co0, lane 8 S1 of co0 + 1,
                // lane 16 and 24 the S2 values.
                static_assert(NP == 1, "reduce-scatter of one channel pair");
                const bool hi16 = lane & 16, hi8 = lane & 8;
                float2 keep = hi16 ? s2[0] : s1[0];
                const float2 send = hi16 ? s1[0] : s2[0];
                keep.x += __shfl_xor_sync(0xffffffffu, send.x, 16);
                keep.y += __shfl_xor_sync(0xffffffffu, send.y, 16);
                float r = hi8 ? keep.y : keep.x;
                r += __shfl_xor_sync(0xffffffffu, hi8 ? keep.x : keep.y, 8);
#pragma unroll
                for (int o = 4; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
                const float r2 = __shfl_down_sync(0xffffffffu, r, 16);  // the S2 of lanes 0 and 8
                if ((lane & ~8) == 0) {
                    const float cnt = (float)(rows_ok * min(kSegV, a.Wo - c0));
                    const int ui = U.band * a.tct_nseg + U.seg;
                    // partials [n][channel][unit][row part]
                    const size_t pi = (((size_t)U.n * a.Co + co0 + (hi8 ? 1 : 0)) * a.tct_U + ui) * kRowParts + rp;
                    if (CN_CHECK(pi < (size_t)a.N * a.Co * a.tct_U * kRowParts, a.err))
                        a.partial[pi] = make_float4(cnt, hi8 ? ksh[0].y : ksh[0].x, r, r2);
                }
            } else {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[b]);
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
                     "r"(2 * kAccCols)
                     : "memory");
    // the last CTA to leave resets the work counters for the next launch
    if (tid == 0 && atomicAdd(work + a.tct_G, 1) == (int)gridDim.x - 1) {
        for (int i = 0; i <= a.tct_G; ++i) work[i] = 0;
    }
}

}  // namespace

// Plans the tensor-core transposed conv; CN_ERR_UNSUPPORTED when the problem
// does not fit it (the CUDA-core kernel then takes it).
int tct_plan(const conv_norm_desc &d, Full2dArgs &a, Full2dConfig &cfg) {
    if (d.conv != CN_CONVT2D) return CN_ERR_UNSUPPORTED;
    if (d.C_in / d.groups != kCig || d.C_out / d.groups != kCog || d.k != kK) return CN_ERR_UNSUPPORTED;
    // x rows must be 16-byte multiples for the tensor map
    if (d.W % 4 != 0 || !tma_available()) return CN_ERR_UNSUPPORTED;
    const char *e = getenv("CN_NO_TC");
    if (e && atoi(e)) return CN_ERR_UNSUPPORTED;
    const int Ho = d.H + kK - 1, Wo = d.W + kK - 1;
    const int nseg = (Wo + kSegV - 1) / kSegV, nband = (Ho + kZG - 1) / kZG;
    const long long U = (long long)nseg * nband;
    const long long units_g = (long long)d.N * U;
    const long long tiles_g = (units_g + 3) / 4;
    if (units_g > 0x3fffffffLL || (long long)d.groups * tiles_g > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;

    a.tc = 0;
    a.tct = 1;
    a.tct_xmap_base = nullptr;
    a.wait_ns = kWaitLimitNs;
    a.tct_G = d.groups;
    a.tct_nseg = nseg;
    a.tct_nband = nband;
    a.tct_U = (int)U;
    a.tct_tiles_g = (int)tiles_g;
    a.tct_ctas_g = 1;  // set from the device by full2d_prepare
    a.use_bulk = 1;
    a.use_tma = 0;
    a.N = d.N;
    a.Ci = d.C_in;
    a.Co = d.C_out;
    a.H = d.H;
    a.W = d.W;
    a.Ho = Ho;
    a.Wo = Wo;
    a.Cig = kCig;
    a.Cog = kCog;
    a.KD = 1;
    a.Din = 1;
    a.Dv = 1;
    a.row_tiles = nband;
    a.col_tiles = nseg;
    a.ncob = 0;
    a.nchunk = 0;
    a.wstage = 0;
    a.ntiles = (int)U;  // partials per channel: one per unit and row part
    a.wsp = kRowParts;
    a.items = (int)(d.groups * tiles_g);
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

    switch (d.act) {
        case CN_ACT_NONE:
            cfg.kern = k_convt2d_tc<ACT_NONE>;
            cfg.names = "k_convt2d_tc<0>,k_group_stats,k_norm_apply";
            break;
        case CN_ACT_HARDSWISH:
            cfg.kern = k_convt2d_tc<ACT_HARDSWISH>;
            cfg.names = "k_convt2d_tc<1>,k_group_stats,k_norm_apply";
            break;
        case CN_ACT_GELU_ERF:
            cfg.kern = k_convt2d_tc<ACT_GELU>;
            cfg.names = "k_convt2d_tc<2>,k_group_stats,k_norm_apply";
            break;
        default:
            return CN_ERR_UNSUPPORTED;
    }
    cfg.K = kK;
    cfg.RW = 0;
    cfg.COT = kCog;
    cfg.VECW = 0;
    cfg.transposed = 1;
    cfg.threads = kThreads;
    cfg.smem = kSmemBytes;
    cfg.grid = d.groups;  // refined from the device in full2d_prepare
    cfg.prep_grid = 0;
    return apply_config(d, a, cfg);
}

// Persistent grid: the same number of CTAs for every group (each builds its
// group's filter once), as many as the SMs allow, capped by the group's tiles.
int tct_prepare(Full2dConfig &cfg, Full2dArgs &a, int sms) {
    a.tct_ctas_g = std::max(1, std::min(sms / std::max(1, a.tct_G), a.tct_tiles_g));
    const long long grid = (long long)a.tct_G * a.tct_ctas_g;
    if (grid > 0x7fffffffLL) return CN_ERR_UNSUPPORTED;
    cfg.grid = a.tct_tiles_g > 0 ? (int)grid : 0;
    return CN_OK;
}

// Encodes the input tensor map for this x (cached while x stays the same):
// x as (W, H, C_in, N), box (36 columns, 8 rows, 8 channels, 1).
int tct_bind_x(Full2dArgs &a) {
    if (a.tct_xmap_base == a.x) return CN_OK;
    const uint64_t dims[4] = {(uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.Ci, (uint64_t)a.N};
    const uint64_t strides[3] = {(uint64_t)a.W * 4, (uint64_t)a.H * a.W * 4,
                                 (uint64_t)a.Ci * a.H * a.W * 4};
    const uint32_t box[4] = {(uint32_t)kBoxW, (uint32_t)kRowsIn, (uint32_t)kCig, 1u};
    const int st = encode_tmap_f32_4d(&a.tct_xmap, a.x, dims, strides, box);
    if (st != CN_OK) return st;
    a.tct_xmap_base = a.x;
    return CN_OK;
}

}  // namespace cn
