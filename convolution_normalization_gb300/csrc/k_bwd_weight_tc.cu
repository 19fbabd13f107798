// Backward of a dense Conv2d (groups 1), the filter gradient, on the
// 5th-generation tensor cores:
//   dw[co][ci][p][q] = sum_{n, i, j} dA[n][co][i][j] x[n][ci][i + p][j + q],
// a GEMM D[co][(ci, p, q)] over the positions (n, i, j) as the contraction.
// dA comes in rows padded with zeros to a multiple of 32 columns (its pitch
// Pq), so along a row segment the positions are consecutive and tap (p, q)
// of x is the segment moved by p rows and q columns.
//
// Tiles: M = 128 output channels, N = 16 input channels x k^2 taps, K = 32
// positions (one row segment of dA) a K-tile.  Split TF32 as in the forward
// kernels (v = hi + lo, hi the raw fp32 word the tensor core truncates):
//   dA * x ~= Ah*Xh + Al*Xh + Ah*Xl,
// per 8 positions three MMAs: [Ah(c) | Ah(c+1)].[Xh(c) | Xh(c+1)], and for
// each 4-position chunk c [Al(c) | Ah(c)].[Xh(c) | Xl(c)].  Operands are
// K-major without swizzle: core matrices of 8 rows x 4 positions; A holds
// its lo half before its hi half and B its hi half before its lo half, so
// every pairing is a positive offset; chunks are one 16-byte skew apart, so
// the converters' 16-byte stores of a quarter warp hit distinct banks.
//
// Roles (one CTA per SM): warp 0 producer (per K-tile a TMA box of dA,
// 32 positions x 128 channels, and one of x, (32 + k - 1 rounded up to 4)
// columns x k rows x 16 channels, zero fill past the edges); warps 2-9
// converters (landed tiles -> hi / lo operands); warp 1 lane 0 issues the
// MMAs into one TMEM accumulator for the CTA's whole run of K-tiles; at the
// end warps 2-5 read the accumulator (thread = output channel) and write the
// run's partial sums, which a fixed-order sum over the runs turns into dw.
// Every wait is bounded; a role that gives up stops the others.
#include "cn_common.cuh"
#include "cn_internal.h"
#include "cn_tcgen05.cuh"

#include <algorithm>
#include <cstdlib>
#include <new>

namespace cn {
namespace {

constexpr int kWtThreads = 320;  // warps 0 producer, 1 MMA, 2-9 converters (2-5 the epilogue)
constexpr int kWtConv0 = 2, kWtConvWarps = 8;
constexpr int kWtKT = 32;        // positions a K-tile
constexpr int kWtCi = 16;        // input channels an N tile
constexpr int kWtM = 128;        // output channels an M tile
constexpr int kWtStages = 2, kWtLand = 2;

template <int K>
struct WT {
    static constexpr int KK = K * K;
    static constexpr int NT = kWtCi * KK;                 // MMA N: (ci, p, q) of the tile
    static constexpr int NG = NT / 8;                     // 8-row groups of B
    static constexpr int ACH = (kWtM / 8) * 128 + 16;     // bytes between A's 4-position chunks (skewed)
    static constexpr int BCH = NG * 128 + 16;             // bytes between B's chunks
    static constexpr int AHALF = (kWtKT / 4) * ACH;       // one of A's lo / hi
    static constexpr int BHALF = (kWtKT / 4) * BCH;
    static constexpr int STAGE = (2 * AHALF + 2 * BHALF + 127) & ~127;
    static constexpr int BOXW = (kWtKT + K - 1 + 3) / 4 * 4;  // landed x columns (16-byte rows)
    static constexpr int LANDA = kWtM * kWtKT * 4;            // dA: [co][32]
    static constexpr int LANDB = kWtCi * K * BOXW * 4;        // x: [ci][k rows][BOXW]
    static constexpr int LAND = (LANDA + LANDB + 127) & ~127;
    static constexpr int SMEM = kWtStages * STAGE + kWtLand * LAND;
    static constexpr int TCOLS = NT <= 32 ? 32 : NT <= 64 ? 64 : NT <= 128 ? 128 : 256;
    static_assert(NT % 16 == 0 && NT <= 256, "MMA N");
};

struct WtArgs {
    CUtensorMap amap;  // dA rows of pitch Pq as (Pq, Ho, C_out, N), box (32, 1, 128, 1)
    CUtensorMap bmap;  // x as (W, H, C_in, N), box (BOXW, k, 16, 1)
    int *err;
    unsigned long long wait_ns;
    int N, Co, Ci, Ho, Pq, nseg;
    int mtiles, ntiles, nrun;  // tiles of M and N, runs of K-tiles per tile
    long long ktiles;          // K-tiles of one (M, N) tile: N * Ho * nseg
    long long kper;            // K-tiles a run
    float *part;               // [run][C_out][C_in * k * k]
};

template <int K>
__global__ void __launch_bounds__(kWtThreads, 1) k_bwd_weight_tc(const __grid_constant__ WtArgs a) {
    using P = WT<K>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t land_full[kWtLand], land_empty[kWtLand];
    __shared__ __align__(8) uint64_t st_full[kWtStages], st_empty[kWtStages], fin_bar;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned char *stages = smem_raw;
    unsigned char *lands = smem_raw + kWtStages * P::STAGE;
    int bx = blockIdx.x;
    const int run = bx % a.nrun;
    bx /= a.nrun;
    const int nt = bx % a.ntiles, mt = bx / a.ntiles;
    const long long kt0 = (long long)run * a.kper;
    const long long kt1 = kt0 + a.kper < a.ktiles ? kt0 + a.kper : a.ktiles;
    const int nk = (int)(kt1 > kt0 ? kt1 - kt0 : 0);

    if (tid == 0) {
        for (int i = 0; i < kWtLand; ++i) {
            mbar_init(&land_full[i], 1);
            mbar_init(&land_empty[i], kWtConvWarps);
        }
        for (int i = 0; i < kWtStages; ++i) {
            mbar_init(&st_full[i], kWtConvWarps);
            mbar_init(&st_empty[i], 1);
        }
        mbar_init(&fin_bar, 1);
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(P::TCOLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    int *abort_p = const_cast<int *>(&s_abort);
    auto wait = [&](uint64_t *bar, uint32_t par) { return tc_wait(bar, par, abort_p, a.err, a.wait_ns); };
    auto wait_warp = [&](uint64_t *bar, uint32_t par) { return __all_sync(0xffffffffu, wait(bar, par)); };
    bool mma_ok = true;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < nk; ++t) {
                const int lb = t % kWtLand;
                if (t >= kWtLand && !wait(&land_empty[lb], ((t / kWtLand) - 1) & 1)) break;
                long long kt = kt0 + t;
                const int n = (int)(kt / ((long long)a.Ho * a.nseg));
                const int rem = (int)(kt - (long long)n * a.Ho * a.nseg);
                const int i = rem / a.nseg, j0 = (rem - i * a.nseg) * kWtKT;
                unsigned char *L = lands + (size_t)lb * P::LAND;
                mbar_arrive_expect_tx(&land_full[lb], (uint32_t)(P::LANDA + P::LANDB));
                tma_load_4d(L, &a.amap, j0, i, mt * kWtM, n, &land_full[lb]);
                tma_load_4d(L + P::LANDA, &a.bmap, j0, i, nt * kWtCi, n, &land_full[lb]);
                issued = t + 1;
            }
            // copies in flight land before the CTA exits
            for (int t = issued - kWtLand > 0 ? issued - kWtLand : 0; t < issued; ++t)
                mbar_wait_bounded(&land_full[t % kWtLand], (t / kWtLand) & 1, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t id = idesc_tf32(128, P::NT);
            for (int t = 0; t < nk; ++t) {
                const int b = t % kWtStages;
                if (!wait(&st_full[b], (t / kWtStages) & 1)) {
                    mma_ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sb = smem_u32(stages + (size_t)b * P::STAGE);
                const uint32_t alo = sb, ahi = sb + P::AHALF, bhi = sb + 2 * P::AHALF, blo = bhi + P::BHALF;
#pragma unroll
                for (int s = 0; s < kWtKT / 8; ++s) {
                    const int c0 = 2 * s, c1 = 2 * s + 1;
                    // hi*hi over the 8 positions
                    umma_tf32(tmem, umma_desc(ahi + c0 * P::ACH, P::ACH, 128), umma_desc(bhi + c0 * P::BCH, P::BCH, 128),
                              id, (t > 0 || s > 0) ? 1u : 0u);
                    // the cross terms of each 4-position chunk
                    umma_tf32(tmem, umma_desc(alo + c0 * P::ACH, P::AHALF, 128),
                              umma_desc(bhi + c0 * P::BCH, P::BHALF, 128), id, 1u);
                    umma_tf32(tmem, umma_desc(alo + c1 * P::ACH, P::AHALF, 128),
                              umma_desc(bhi + c1 * P::BCH, P::BHALF, 128), id, 1u);
                }
                umma_commit(&st_empty[b]);
            }
            // every MMA completes before the accumulator is read or freed
            umma_commit(&fin_bar);
            mbar_wait_bounded(&fin_bar, 0, kWaitLimitNs);
        }
    } else {
        // ---------------- converters ----------------
        const int ct = tid - 32 * kWtConv0;  // 0 .. 255
        for (int t = 0; t < nk; ++t) {
            const int lb = t % kWtLand, b = t % kWtStages;
            if (!wait_warp(&land_full[lb], (t / kWtLand) & 1)) break;
            if (t >= kWtStages && !wait_warp(&st_empty[b], ((t / kWtStages) - 1) & 1)) break;
            const float *LA = reinterpret_cast<const float *>(lands + (size_t)lb * P::LAND);
            const float *LB = LA + kWtM * kWtKT;
            unsigned char *S = stages + (size_t)b * P::STAGE;
            // A: dA [co][32] -> (lo | hi) cores (chunk c, co group, row co % 8);
            // a quarter warp reads one row's 128 bytes and stores to 8
            // chunks, one bank group apart thanks to the skew
            for (int e = ct; e < kWtM * (kWtKT / 4); e += 32 * kWtConvWarps) {
                const int c = e & (kWtKT / 4 - 1), co = e >> 3;
                const float4 v = *reinterpret_cast<const float4 *>(LA + co * kWtKT + 4 * c);
                const int off = c * P::ACH + (co >> 3) * 128 + (co & 7) * 16;
                if (!CN_CHECK(off + 16 <= P::AHALF, a.err)) continue;
                *reinterpret_cast<float4 *>(S + P::AHALF + off) = v;
                *reinterpret_cast<float4 *>(S + off) =
                    make_float4(tf32_rest(v.x), tf32_rest(v.y), tf32_rest(v.z), tf32_rest(v.w));
            }
            // B: x [ci][p][col] -> (hi | lo) cores of rows (ci, p, q), the
            // chunk's 4 positions read at column 4c + q
            for (int e = ct; e < P::NT * (kWtKT / 4); e += 32 * kWtConvWarps) {
                const int nn = e % P::NT, c = e / P::NT;
                const int ci = nn / P::KK, pq = nn - ci * P::KK, p = pq / K, q = pq - p * K;
                const float *src = LB + (ci * K + p) * P::BOXW + 4 * c + q;
                const float4 v = make_float4(src[0], src[1], src[2], src[3]);
                const int off = 2 * P::AHALF + c * P::BCH + (nn >> 3) * 128 + (nn & 7) * 16;
                if (!CN_CHECK(off + 16 <= 2 * P::AHALF + P::BHALF, a.err)) continue;
                *reinterpret_cast<float4 *>(S + off) = v;
                *reinterpret_cast<float4 *>(S + P::BHALF + off) =
                    make_float4(tf32_rest(v.x), tf32_rest(v.y), tf32_rest(v.z), tf32_rest(v.w));
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&land_empty[lb]);
                mbar_arrive(&st_full[b]);
            }
        }
    }

    // ---- epilogue: the run's sums, thread = output channel ----
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp >= kWtConv0 && warp < kWtConv0 + 4 && nk > 0 && !*abort_p) {
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        const int co = mt * kWtM + 32 * q + lane;
        const int NN = a.Ci * P::KK;
        float *dst = a.part + ((size_t)run * a.Co + co) * NN + (size_t)nt * P::NT;
#pragma unroll 1
        for (int c0 = 0; c0 < P::NT; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
            tmem_wait_ld();
            if (co < a.Co && CN_CHECK(nt * P::NT + c0 + 16 <= NN && run < a.nrun, a.err))
#pragma unroll
                for (int u = 0; u < 16; ++u) dst[c0 + u] = __uint_as_float(v[u]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(P::TCOLS)
                     : "memory");
    (void)mma_ok;
}

typedef void (*WtKernel)(WtArgs);
struct WtInst {
    int K, smem;
    WtKernel fn;
};
const WtInst kWtInst[] = {{1, WT<1>::SMEM, k_bwd_weight_tc<1>},
                          {2, WT<2>::SMEM, k_bwd_weight_tc<2>},
                          {3, WT<3>::SMEM, k_bwd_weight_tc<3>}};
const WtInst *wt_inst(int K) {
    for (const WtInst &w : kWtInst)
        if (w.K == K) return &w;
    return nullptr;
}

}  // namespace

struct BwdWtState {
    WtArgs a;
    const WtInst *inst = nullptr;
    int grid = 0, W = 0, H = 0, K = 0;
    const float *amap_base = nullptr, *bmap_base = nullptr;
};

// Plans the tensor-core dw of a dense Conv2d: C_out a multiple of 128,
// C_in of 16, k <= 3, x rows a multiple of 4 columns; dA supplied with rows
// of pitch Pq = Wo rounded up to 32 (zeros past Wo).
int bwd_wt_plan(int N, int C_out, int C_in, int H, int W, int k, int sms, int *err, BwdWtState **out, int *nrun,
                int *pitch) {
    *out = nullptr;
    if (C_out % kWtM != 0 || C_in % kWtCi != 0 || k < 1 || k > 3 || W % 4 != 0 || !tma_available())
        return CN_ERR_UNSUPPORTED;
    const char *e = getenv("CN_NO_TC");
    if (e && atoi(e)) return CN_ERR_UNSUPPORTED;
    const WtInst *inst = wt_inst(k);
    if (!inst || inst->smem > 227 * 1024) return CN_ERR_UNSUPPORTED;
    const int Ho = H - k + 1, Wo = W - k + 1;
    if (Ho < 1 || Wo < 1) return CN_ERR_UNSUPPORTED;
    BwdWtState *st = new (std::nothrow) BwdWtState();
    if (!st) return CN_ERR_ALLOC;
    WtArgs &a = st->a;
    a.err = err;
    a.wait_ns = kWaitLimitNs;
    a.N = N;
    a.Co = C_out;
    a.Ci = C_in;
    a.Ho = Ho;
    a.nseg = (Wo + kWtKT - 1) / kWtKT;
    a.Pq = a.nseg * kWtKT;
    a.mtiles = C_out / kWtM;
    a.ntiles = C_in / kWtCi;
    a.ktiles = (long long)N * Ho * a.nseg;
    const long long tiles = (long long)a.mtiles * a.ntiles;
    a.nrun = (int)std::max(1LL, std::min(a.ktiles, (long long)std::max(1, sms) / std::max(1LL, tiles)));
    a.kper = (a.ktiles + a.nrun - 1) / a.nrun;
    a.nrun = (int)((a.ktiles + a.kper - 1) / a.kper);
    st->grid = (int)(tiles * a.nrun);
    st->inst = inst;
    st->W = W;
    st->H = H;
    st->K = k;
    if (raise_dyn_smem(reinterpret_cast<const void *>(inst->fn), inst->smem) != cudaSuccess) {
        cudaGetLastError();
        delete st;
        return CN_ERR_UNSUPPORTED;
    }
    *out = st;
    *nrun = a.nrun;
    *pitch = a.Pq;
    return CN_OK;
}

void bwd_wt_destroy(BwdWtState *st) { delete st; }
void bwd_wt_set_err(BwdWtState *st, int *err) { st->a.err = err; }

// dA with rows of pitch Pq ([N][C_out][Ho][Pq]), x ([N][C_in][H][W]); writes
// part[run][C_out][C_in k k].
int bwd_wt_launch(BwdWtState *st, const float *dAq, const float *x, float *part, cudaStream_t s) {
    WtArgs &a = st->a;
    const int K = st->K;
    if (st->amap_base != dAq) {
        const uint64_t dims[4] = {(uint64_t)a.Pq, (uint64_t)a.Ho, (uint64_t)a.Co, (uint64_t)a.N};
        const uint64_t strides[3] = {(uint64_t)a.Pq * 4, (uint64_t)a.Ho * a.Pq * 4, (uint64_t)a.Co * a.Ho * a.Pq * 4};
        const uint32_t box[4] = {(uint32_t)kWtKT, 1u, (uint32_t)kWtM, 1u};
        const int r = encode_tmap_f32_4d(&a.amap, dAq, dims, strides, box);
        if (r != CN_OK) return r;
        st->amap_base = dAq;
    }
    if (st->bmap_base != x) {
        const uint64_t dims[4] = {(uint64_t)st->W, (uint64_t)st->H, (uint64_t)a.Ci, (uint64_t)a.N};
        const uint64_t strides[3] = {(uint64_t)st->W * 4, (uint64_t)st->H * st->W * 4,
                                     (uint64_t)a.Ci * st->H * st->W * 4};
        const int boxw = (kWtKT + K - 1 + 3) / 4 * 4;
        const uint32_t box[4] = {(uint32_t)boxw, (uint32_t)K, (uint32_t)kWtCi, 1u};
        const int r = encode_tmap_f32_4d(&a.bmap, x, dims, strides, box);
        if (r != CN_OK) return r;
        st->bmap_base = x;
    }
    a.part = part;
    st->inst->fn<<<st->grid, kWtThreads, st->inst->smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? CN_OK : CN_ERR_CUDA;
}

}  // namespace cn
