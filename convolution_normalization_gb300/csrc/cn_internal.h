// Internal interfaces between the C-ABI layer (cn_api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda.h>

#include "../../include/conv_norm.h"

namespace cn {

// Per-launch timing events of a plan (conv_norm_plan_set_launch_events):
// record(i) marks the start of launch i, record(L) the end of the last one.
constexpr int kMaxLaunchEvents = 8;
struct LaunchEvents {
    cudaEvent_t ev[kMaxLaunchEvents];
    int n;  // 0: off
};
inline void record_launch(const LaunchEvents *e, int i, cudaStream_t s) {
    if (e && i < e->n) cudaEventRecord(e->ev[i], s);
}

// Tensor-map encoding (cn_tma_host.cu).
bool tma_available();
// Raises (never lowers) a kernel's dynamic shared-memory limit on the
// current device: plans of one kernel with different sizes live side by
// side, and each launch needs the limit at or above its own size.
cudaError_t raise_dyn_smem(const void *kern, int bytes);

// Backward dw of a dense Conv2d on the tensor cores (k_bwd_weight_tc.cu).
struct BwdWtState;
int bwd_wt_plan(int N, int C_out, int C_in, int H, int W, int k, int sms, int *err, BwdWtState **out, int *nrun,
                int *pitch);
void bwd_wt_destroy(BwdWtState *st);
void bwd_wt_set_err(BwdWtState *st, int *err);  // the device flag its bounded waits report to
int bwd_wt_launch(BwdWtState *st, const float *dAq, const float *x, float *part, cudaStream_t s);
int encode_tmap_f32_4d(CUtensorMap *map, const float *base, const uint64_t dims[4],
                       const uint64_t strides_bytes[3], const uint32_t box[4]);
int encode_tmap_f32_5d(CUtensorMap *map, const float *base, const uint64_t dims[5],
                       const uint64_t strides_bytes[4], const uint32_t box[5]);

// Upper bound on any device-side wait (ns of GPU wall time) before a kernel
// gives up, records CN_ERR_TIMEOUT in the plan's flag and carries on.  The
// tensor-core kernels take their progress-wait limit from their arguments
// (wait_ns, this value unless conv_norm_plan_set_wait_limit lowered it); the
// waits that drain copies and MMAs in flight before a CTA exits always use
// this one.
constexpr unsigned long long kWaitLimitNs = 200ull * 1000ull * 1000ull;

// ---------------------------------------------------------------------------
// Tensor-core Conv3d (k_conv3d_tc.cu), used by the spatial-mean and the
// softmax + pool variants: a stage is one band of rb output rows of a group
// of output depth planes; the fields describe its staged input and MMA tiles.
struct Tc3Args {
    CUtensorMap xmap;        // x as (W, H, D, N*C_in), box (W, rb + k - 1, planes, C_in)
    const float *xmap_base;  // x pointer the map was encoded for
    int *err;                // device error flag
    unsigned long long wait_ns;  // progress-wait limit (ns) before a timeout is recorded
    int stall;               // failure-path test hook: CTA 0 leaves its first copy unissued
    const float *x, *w, *b, *gamma, *beta;
    float *out;
    int N, Ci, Co, D, H, W, Do, Ho, Wo;
    int k, nu;        // filter extent; staged input planes per stage (plane group + k - 1)
    int rb;           // output rows per band: 128 / W
    int nband;        // bands per plane group
    int pp;           // operand positions per staged input plane
    int pad;          // 1: operand planes leave a 16-byte gap after every 8 positions (W % 8 == 0)
    int ppu;          // 16-byte units per staged operand plane: pp, or pp / 8 * 9 with pad
    int stage;        // bytes of one operand stage (hi and lo, all staged planes)
    int land;         // bytes of the raw input box of a stage
    int nland;        // landing buffers for it (1 or 2)
    int halo;         // 1: output rows cross 32-lane quadrants (W does not divide 32)
    uint32_t wmagic;  // ceil(2^32 / W): p / W = umulhi(p, wmagic) for p < 2^16
    int ngroups;      // plane groups per sample
    int nsplit;       // items per plane group, each ceil(nband / nsplit) bands
    int items;        // N * ngroups * nsplit
    int act, norm, G, affine;
    float eps, post_scale;
    int Pd, Ph, Pw;    // pool: pooled extents
    double inv_cnt, inv_cpg;  // mean: 1 / (Do Ho Wo), 1 / (channels per norm group)
    float4 *partial;   // mean: [N][ngroups * nsplit][Co] (count, K, S1, S2): an item's sums about
                       // K, its first value of the channel
    int *tickets;      // mean: [N] per-sample tickets, zero between launches
    int *work;         // [2] work / exit counters, zero between launches
};
typedef void (*Tc3Kernel)(Tc3Args);
struct Tc3Config {
    Tc3Kernel kern;
    const char *name;
    int threads, smem, grid;
};
// Plans the tensor-core kernel for a spatial-mean or a softmax + pool problem;
// CN_ERR_UNSUPPORTED when the problem does not fit it.
int tc3_plan(const conv_norm_desc &d, Tc3Args &a, Tc3Config &cfg);
int tc3_prepare(Tc3Config &cfg, const Tc3Args &a);  // smem attribute, persistent grid
int tc3_launch(const Tc3Config &cfg, Tc3Args &a, cudaStream_t s, const LaunchEvents *ev);
int tc3_launches(const Tc3Config &cfg);  // kernels one forward launches

// ---------------------------------------------------------------------------
// Variant 0: 3-D conv -> activation -> (GroupNorm | InstanceNorm | none)
// -> spatial mean.  One launch; the conv tensor is never written.
struct Mean3dArgs {
    int tc;           // 1: the tensor-core kernel (t) runs the problem
    int small;        // 1: the small-problem kernel (one CTA per (n, norm group)) runs it
    int sm_cpg;       // small: channels per normalization group (one CTA's channels)
    int sm_ngrp;      // small: normalization groups per sample
    int sm_nsplit;    // small: CTAs per (sample, normalization group), by output rows
    Tc3Args t;
    CUtensorMap tmap;           // x viewed as (W, H, D, N*C_in), box (pitch, H, planes_max, C_in)
    const float *tmap_base;     // x pointer the map was encoded for
    int use_tma;                // 1: stage with one TMA tensor copy per CTA
    int *err;                   // device error flag
    const float *x, *w, *b, *gamma, *beta;
    float *out;
    int N, Ci, Co, D, H, W, Do, Ho, Wo;
    int nseg;         // W-segments of RW outputs per output row
    int rows;         // Do * Ho * nseg thread-rows per sample
    int rows_per_cta; // 32 * wrows
    int nchunks;      // ceil(rows / rows_per_cta)
    int ncob;         // co blocks per sample
    int wco;          // warps (co-slices of 4 channels) per co block
    int wrows;        // row groups per CTA
    int planes_max;   // input depth planes staged per chunk
    int pitch;        // shared-memory row pitch in floats
    int nbuf;         // staging buffers (2: next chunk prefetched during compute)
    int buf_stride;   // floats per staging buffer (multiple of 32)
    int items;        // N * ncob * nchunks work items, ordered (cob, n, chunk)
    int vec16;        // 1: 16-byte cp.async staging is legal
    int act, norm, G, affine;
    float eps, post_scale;
    double *partial;  // [N][nchunks][Co][3]  (count, mean, M2); the tensor-core kernel's float4 sums
    int *tickets;     // [N] per-sample tickets (small kernel: [N * groups] per-group
                      // ones), then [2] work/exit counters; zero between launches
};
typedef void (*Mean3dKernel)(Mean3dArgs);
struct Mean3dConfig {
    Tc3Config tc3;    // the tensor-core kernel's launch, when args.tc
    Mean3dKernel kern;
    const char *name;
    int K, RW, COT;
    int threads, smem;
    int grid;         // persistent CTAs (set by mean3d_prepare from the device)
};
// Chooses tiling + instantiation; fills the geometry fields of args.
// Returns CN_OK or CN_ERR_UNSUPPORTED.
int mean3d_plan(const conv_norm_desc &d, Mean3dArgs &args, Mean3dConfig &cfg);
// The small-problem kernel (k_conv3d_mean_small.cu); CN_ERR_UNSUPPORTED when
// the problem is too large for it.
int small3d_plan(const conv_norm_desc &d, Mean3dArgs &args, Mean3dConfig &cfg);
size_t small3d_partial_bytes(const Mean3dArgs &a);
// Bytes of the partial-moment slots (the tensor-core kernel's float4 sums or
// the CUDA-core kernel's fp64 (count, mean, M2)).
size_t mean3d_partial_bytes(const Mean3dArgs &a);
size_t mean3d_tickets(const Mean3dArgs &a);  // ints after the partial slots
size_t mean3d_workspace(const Mean3dArgs &a);
int mean3d_prepare(Mean3dConfig &cfg, const Mean3dArgs &a);  // needs a device: smem attribute, grid
int mean3d_launch(const Mean3dConfig &cfg, Mean3dArgs &a, cudaStream_t s,
                  const LaunchEvents *ev = nullptr);
int mean3d_launches(const Mean3dConfig &cfg, const Mean3dArgs &a);  // kernels one forward launches

// ---------------------------------------------------------------------------
// Variant 1: 3-D conv -> channel softmax -> MaxPool3d(2,2) twice (= one
// 4x4x4 stride-4 max pool).  One launch, only the pooled output is written.
struct Pool3dArgs {
    CUtensorMap tmap;     // x viewed as (W, H, D, N*C_in), box (pxb, P, P, C_in)
    const float *tmap_base;
    int use_tma;
    int *err;
    const float *x, *w, *b;
    float *out;
    int N, Ci, D, H, W, Do, Ho, Wo;
    int Pd, Ph, Pw;      // pooled extents: floor(Do/4), floor(Ho/4), floor(Wo/4)
    long long nvox;      // N * Pd * Ph * Pw
    float post_scale;    // > 0: multiplies the pooled value
    int tc;              // 1: the tensor-core kernel (t) runs the problem
    Tc3Args t;
    int vox_per_cta;     // pooled voxels per CTA (16 threads each)
    int pw_pitch;        // shared-memory patch row pitch (floats), P rounded up to 4
    int vox_stride;      // floats per staged voxel patch
};
typedef void (*Pool3dKernel)(Pool3dArgs);
struct Pool3dConfig {
    Tc3Config tc3;       // the tensor-core kernel's launch, when args.tc
    Pool3dKernel kern;
    const char *name;
    int threads, smem, grid;
};
int pool3d_plan(const conv_norm_desc &d, Pool3dArgs &args, Pool3dConfig &cfg);
size_t pool3d_workspace(const Pool3dArgs &a);
int pool3d_prepare(Pool3dConfig &cfg, const Pool3dArgs &a);
int pool3d_launch(const Pool3dConfig &cfg, Pool3dArgs &a, cudaStream_t s,
                  const LaunchEvents *ev = nullptr);

// ---------------------------------------------------------------------------
// Variant 2: 2-D conv or transposed conv (groups) -> activation ->
// GroupNorm/InstanceNorm/none -> post scale, full output.
// Kernel A computes conv + activation for a tile, writes the pre-norm value
// to out and per-(n, c, tile) moments; the last CTA of each sample merges
// the moments into per-channel coefficients.  Kernel B rewrites out in place
// as (y - mu) * a + bb.
struct Full2dArgs {
    // Tensor-core conv (k_conv2d_tc, tc = 1): dense Conv2d as a split-TF32
    // implicit GEMM; the fields below tc_* describe its tiles and stages.
    CUtensorMap tc_xmap;        // x as (W, H, C_in, N), box (W, tc_R + K - 1, 4, 1)
    const float *tc_xmap_base;  // x pointer the map was encoded for
    int tc;
    int tc_K;                   // filter size
    int tc_R;                   // output rows per tile
    int tc_npos;                // MMA N: positions per tile (multiple of 32, <= 256)
    int tc_ngrp;                // 4-channel input groups = pipeline stages per tile
    int tc_xbuf_bytes;          // one interleaved input operand buffer (hi or lo)
    int tc_wblk_bytes;          // one (channel block, group) filter block, lo | hi
    int tc_stage_bytes;         // 2 * tc_xbuf_bytes + tc_wblk_bytes
    int tc_land_bytes;          // raw input box of a stage
    int tc_stages;              // operand stages in shared memory
    int tc_acc_cols;            // TMEM columns per accumulator (two are allocated)

    // Tensor-core grouped transposed conv (k_convt2d_tc, tct = 1): a unit is
    // 4 output rows x 30 output columns of one (n, group), a tile 4 units of
    // one group; the CTAs are split evenly over the groups.
    CUtensorMap tct_xmap;       // x as (W, H, C_in, N), box (36, 6, 8, 1)
    const float *tct_xmap_base; // x pointer the map was encoded for
    int tct;
    int tct_G;                  // conv groups
    int tct_nseg, tct_nband;    // column units per output row; row bands per plane
    int tct_U;                  // units per (n, group): nband * nseg
    int tct_tiles_g;            // tiles per group: ceil(N * U / 4)
    int tct_ctas_g;             // persistent CTAs per group (full2d_prepare)

    // CUDA-core kernel staging: use_tma = one tensor copy per stage (box
    // (pitch, rows_in, cib, 1) of x viewed as (W, H, C_in, N), zero fill
    // outside); else use_bulk = one bulk copy per row; else cp.async.
    CUtensorMap xmap;
    const float *xmap_base;     // x pointer xmap was encoded for
    int use_tma;
    int use_bulk;         // 1: rows staged with bulk async copies (W % 4 == 0)
    const float *x, *w, *b, *gamma, *beta;
    float *out;
    int N, Ci, Co, H, W, Ho, Wo;
    // Conv3d (full output) runs as 2-D samples (n, d) over depth-stacked
    // channels (ci, kd): Din input depth, KD depth taps (1 for 2-D), Dv
    // output depth planes per sample (1 for 2-D).  A stage's channels then
    // are cib/KD input channels x KD taps.
    int Din, KD, Dv;
    int Cig, Cog;         // conv channels per group (in, stacked with the depth taps / out)
    int TR, NT;           // CTA tile: TR output rows x NT row segments
    int row_tiles, col_tiles, ncob, ntiles;
    int wco, wsp;         // warps: channel slices x spatial groups
    int cib, nchunk;      // input channels per pipeline stage, stages per tile
    int nstage;           // stage buffers in shared memory (2..4)
    int rows_in, cols_in, pitch;
    int stage_floats;     // floats per pipeline stage (input + filter)
    int xstage;           // floats of the input part of a stage
    int wstage;           // floats of the filter part of a stage (cib * K*K * COB)
    int items;            // tiles: N * ncob * ntiles, claimed through the work counter
    float *wprep;         // filter regrouped per (channel block, chunk) stage layout
    int act, norm, NG, affine;
    float eps, post_scale;
    int apply_needed, vec4;
    long long S;          // Dv * Ho * Wo: one normalized (n, c) plane
    float4 *partial;      // [N][Co][ntiles * wsp]: per warp and tile (count, K, S1, S2),
                          // shifted sums S1 = sum(v - K), S2 = sum((v - K)^2) about
                          // one of the partial's own values K
    float4 *coef;         // [N][Co]: (mu, a, bb, 0)
    int *tickets;         // [N] (unused), then work counters (2, or one per group + 1
                          // for the tensor-core transposed conv), zero between launches
    int *err;
    unsigned long long wait_ns;  // tensor-core kernels: progress-wait limit (ns)
    int stall;                   // tensor-core kernels: failure-path test hook (see Tc3Args)
};
typedef void (*Full2dKernel)(Full2dArgs);
struct Full2dConfig {
    Full2dKernel kern;
    const char *names;
    int K, RW, COT, VECW, transposed;
    int threads, smem, grid;
    int apply_threads, apply_grid, apply_slices;  // normalize pass: 1-D grid, slices per plane
    int prep_grid;
    int fin_threads;
};
int full2d_plan(const conv_norm_desc &d, Full2dArgs &args, Full2dConfig &cfg);
// Launch shape of the normalize pass (k_conv2d_norm.cu), shared by every 2-D plan.
int apply_config(const conv_norm_desc &d, const Full2dArgs &a, Full2dConfig &cfg);
// Tensor-core path (k_conv2d_tc.cu): plan (CN_ERR_UNSUPPORTED when the problem
// does not fit it), filter-block bytes, x tensor map, filter pre-pass.
int tc2d_plan(const conv_norm_desc &d, Full2dArgs &args, Full2dConfig &cfg);
size_t tc2d_wprep_bytes(const Full2dArgs &a);
// Tensor-core grouped transposed conv (k_convt2d_tc.cu): plan
// (CN_ERR_UNSUPPORTED when the problem does not fit it), persistent grid for
// `sms` SMs, x tensor map.
int tct_plan(const conv_norm_desc &d, Full2dArgs &args, Full2dConfig &cfg);
int tct_prepare(Full2dConfig &cfg, Full2dArgs &a, int sms);
int tct_bind_x(Full2dArgs &a);
int tc2d_bind_x(Full2dArgs &a);
int tc2d_prep_launch(const Full2dConfig &cfg, const Full2dArgs &a, cudaStream_t s);
size_t full2d_workspace(const Full2dArgs &a);
size_t full2d_counter_bytes(const Full2dArgs &a);  // the tickets / work counters
void full2d_bind_workspace(Full2dArgs &a, char *base, int *err_flag);
int full2d_prepare(Full2dConfig &cfg, Full2dArgs &a);  // needs a device: smem attribute, grid
int full2d_launches(const Full2dConfig &cfg, const Full2dArgs &a);
int full2d_launch(const Full2dConfig &cfg, Full2dArgs &a, cudaStream_t s,
                  const LaunchEvents *ev = nullptr);  // may cache a tensor map in a

// Reads and clears the error flag of conv_norm_forward_noalloc on the current
// device after synchronizing the stream (cn_noalloc.cu).
int noalloc_check_device(cudaStream_t stream);

}  // namespace cn
