// C-ABI layer: descriptor validation, plans, dispatch to the kernel variants.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>

#include "cn_internal.h"

using namespace cn;

namespace {

enum Variant { V_MEAN3D = 0, V_POOL3D = 1, V_FULL2D = 2 };

constexpr int kMaxHostChunks = 16;

// Device staging for conv_norm_forward_host, created on its first call:
// buffers, per-chunk plans, and the upload / download streams and events
// that overlap chunk i+1's upload (and chunk i-1's download) with chunk i's
// kernels.  Odd chunks compute on a second stream: chunks share no device
// data (each sub-plan owns its workspace), so chunk i+1's CTAs can take the
// SMs that chunk i's last work items leave idle instead of waiting for the
// whole launch to drain.
struct HostStage {
    float *x = nullptr, *w = nullptr, *b = nullptr, *gamma = nullptr, *beta = nullptr,
          *out = nullptr;
    bool ready = false;
    int nchunk = 1, chunk_n = 0;
    conv_norm_plan_s *sub[kMaxHostChunks] = {};  // one plan per chunk (keeps its tensor map)
    cudaStream_t up = nullptr, down = nullptr, comp2 = nullptr;
    cudaEvent_t ev_up[kMaxHostChunks] = {}, ev_done[kMaxHostChunks] = {};
    cudaEvent_t ev_comp2 = nullptr;  // the caller's stream waits for comp2's chunks
};

}  // namespace

struct conv_norm_plan_s {
    conv_norm_desc d;
    int variant;
    int device;
    int64_t out_numel;
    int64_t x_numel, w_numel;
    void *ws = nullptr;  // [error flag | variant workspace]
    size_t ws_bytes = 0;
    int *err_flag = nullptr;
    int *counters = nullptr;  // tickets and work counters: zero between launches
    size_t counter_bytes = 0;
    int stall_pending = 0;    // conv_norm_plan_inject_stall: the next forward stalls
    Mean3dArgs mean_args;
    Mean3dConfig mean_cfg;
    Pool3dArgs pool_args;
    Pool3dConfig pool_cfg;
    Full2dArgs full_args;
    Full2dConfig full_cfg;
    HostStage stage;
    LaunchEvents events{};  // per-launch timing, off unless set
};

namespace {

bool is_finite(float v) { return std::isfinite(v); }

// Malformed problems -> CN_ERR_INVALID_ARG.
int check_wellformed(const conv_norm_desc &d) {
    if (d.conv < CN_CONV3D || d.conv > CN_CONVT2D) return CN_ERR_INVALID_ARG;
    if (d.N < 0 || d.C_in < 1 || d.C_out < 1 || d.H < 1 || d.W < 1 || d.D < 1 || d.k < 1 ||
        d.groups < 1)
        return CN_ERR_INVALID_ARG;
    if (d.C_in % d.groups || d.C_out % d.groups) return CN_ERR_INVALID_ARG;
    if (d.conv != CN_CONV3D && d.D != 1) return CN_ERR_INVALID_ARG;
    if (d.conv != CN_CONVT2D) {
        if (d.H < d.k || d.W < d.k) return CN_ERR_INVALID_ARG;
        if (d.conv == CN_CONV3D && d.D < d.k) return CN_ERR_INVALID_ARG;
    }
    if (d.has_bias != 0 && d.has_bias != 1) return CN_ERR_INVALID_ARG;
    if (d.act < CN_ACT_NONE || d.act > CN_ACT_SOFTMAX_C) return CN_ERR_INVALID_ARG;
    if (d.norm < CN_NORM_NONE || d.norm > CN_NORM_INSTANCE) return CN_ERR_INVALID_ARG;
    if (d.red < CN_RED_NONE || d.red > CN_RED_MAXPOOL2_X2) return CN_ERR_INVALID_ARG;
    if (d.affine != 0 && d.affine != 1) return CN_ERR_INVALID_ARG;
    if (d.norm == CN_NORM_GROUP && (d.num_groups < 1 || d.C_out % d.num_groups))
        return CN_ERR_INVALID_ARG;
    if (!is_finite(d.eps) || !is_finite(d.post_scale)) return CN_ERR_INVALID_ARG;
    if (d.norm != CN_NORM_NONE && !(d.eps > 0.0f)) return CN_ERR_INVALID_ARG;
    if (d.red == CN_RED_MAXPOOL2_X2 && d.conv != CN_CONV3D) return CN_ERR_INVALID_ARG;
    // element counts must stay far inside int64 (the kernels address memory
    // with 64-bit offsets; per-axis sizes and TMA coordinates are the
    // descriptor's 32-bit ints)
    const double big = (double)d.N * d.C_out * d.D * (double)(d.H + d.k) * (d.W + d.k);
    const double bigx = (double)d.N * d.C_in * d.D * (double)d.H * d.W;
    if (big > 4.0e18 || bigx > 4.0e18) return CN_ERR_INVALID_ARG;
    return CN_OK;
}

void conv_dims(const conv_norm_desc &d, int &Do, int &Ho, int &Wo) {
    if (d.conv == CN_CONVT2D) {
        Do = 1;
        Ho = d.H + d.k - 1;
        Wo = d.W + d.k - 1;
    } else {
        Do = d.conv == CN_CONV3D ? d.D - d.k + 1 : 1;
        Ho = d.H - d.k + 1;
        Wo = d.W - d.k + 1;
    }
}

int pick_variant(const conv_norm_desc &d, int &variant) {
    if (d.red == CN_RED_MEAN_SPATIAL) {
        if (d.conv != CN_CONV3D || d.act == CN_ACT_SOFTMAX_C) return CN_ERR_UNSUPPORTED;
        variant = V_MEAN3D;
        return CN_OK;
    }
    if (d.red == CN_RED_MAXPOOL2_X2) {
        // a positive post scale commutes with the max
        if (d.act != CN_ACT_SOFTMAX_C || d.norm != CN_NORM_NONE || !(d.post_scale > 0.0f))
            return CN_ERR_UNSUPPORTED;
        variant = V_POOL3D;
        return CN_OK;
    }
    // full output: Conv2d / ConvTranspose2d, and Conv3d as depth-stacked 2-D samples
    if (d.act == CN_ACT_SOFTMAX_C) return CN_ERR_UNSUPPORTED;
    variant = V_FULL2D;
    return CN_OK;
}

int plan_variant(conv_norm_plan_s &p) {
    switch (p.variant) {
        case V_MEAN3D:
            return mean3d_plan(p.d, p.mean_args, p.mean_cfg);
        case V_POOL3D:
            return pool3d_plan(p.d, p.pool_args, p.pool_cfg);
        default:
            return full2d_plan(p.d, p.full_args, p.full_cfg);
    }
}

int64_t numel_out(const conv_norm_desc &d) {
    int64_t dims[5];
    int nd = 0;
    conv_norm_output_shape(&d, dims, &nd);
    int64_t n = 1;
    for (int i = 0; i < nd; ++i) n *= dims[i];
    return n;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

const char *conv_norm_status_string(int s) {
    switch (s) {
        case CN_OK: return "ok";
        case CN_ERR_INVALID_ARG: return "invalid argument";
        case CN_ERR_UNSUPPORTED: return "unsupported problem";
        case CN_ERR_CUDA: return "CUDA error";
        case CN_ERR_TIMEOUT: return "device wait timed out";
        case CN_ERR_DEVICE_CHECK: return "device bounds check failed";
        case CN_ERR_ALLOC: return "allocation failed";
        default: return "unknown status";
    }
}

int conv_norm_output_shape(const conv_norm_desc *d, int64_t dims[5], int *ndim) {
    if (!d || !dims || !ndim) return CN_ERR_INVALID_ARG;
    int st = check_wellformed(*d);
    if (st != CN_OK) return st;
    int Do, Ho, Wo;
    conv_dims(*d, Do, Ho, Wo);
    dims[0] = d->N;
    dims[1] = d->C_out;
    if (d->red == CN_RED_MEAN_SPATIAL) {
        *ndim = 2;
    } else if (d->red == CN_RED_MAXPOOL2_X2) {
        dims[2] = Do / 4;
        dims[3] = Ho / 4;
        dims[4] = Wo / 4;
        *ndim = 5;
    } else if (d->conv == CN_CONV3D) {
        dims[2] = Do;
        dims[3] = Ho;
        dims[4] = Wo;
        *ndim = 5;
    } else {
        dims[2] = Ho;
        dims[3] = Wo;
        *ndim = 4;
    }
    return CN_OK;
}

int conv_norm_desc_validate(const conv_norm_desc *d) {
    if (!d) return CN_ERR_INVALID_ARG;
    int st = check_wellformed(*d);
    if (st != CN_OK) return st;
    conv_norm_plan_s *p = new (std::nothrow) conv_norm_plan_s();
    if (!p) return CN_ERR_ALLOC;
    p->d = *d;
    st = pick_variant(*d, p->variant);
    if (st == CN_OK) st = plan_variant(*p);
    delete p;
    return st;
}

int conv_norm_plan_create(const conv_norm_desc *d, conv_norm_plan *out) {
    if (!d || !out) return CN_ERR_INVALID_ARG;
    *out = nullptr;
    int st = check_wellformed(*d);
    if (st != CN_OK) return st;
    conv_norm_plan_s *p = new (std::nothrow) conv_norm_plan_s();
    if (!p) return CN_ERR_ALLOC;
    p->d = *d;
    st = pick_variant(*d, p->variant);
    if (st == CN_OK) st = plan_variant(*p);
    if (st != CN_OK) {
        delete p;
        return st;
    }
    if (cudaGetDevice(&p->device) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return CN_ERR_CUDA;
    }
    p->out_numel = numel_out(*d);
    p->x_numel = (int64_t)d->N * d->C_in * d->D * d->H * d->W;
    const int kd = d->conv == CN_CONV3D ? d->k : 1;
    p->w_numel = (int64_t)d->C_out * (d->C_in / d->groups) * kd * d->k * d->k;
    size_t vws = 0;
    switch (p->variant) {
        case V_MEAN3D:
            st = mean3d_prepare(p->mean_cfg, p->mean_args);
            vws = mean3d_workspace(p->mean_args);
            break;
        case V_POOL3D:
            st = pool3d_prepare(p->pool_cfg, p->pool_args);
            vws = pool3d_workspace(p->pool_args);
            break;
        default:
            st = full2d_prepare(p->full_cfg, p->full_args);
            vws = full2d_workspace(p->full_args);
            break;
    }
    if (st != CN_OK) {
        cudaGetLastError();
        delete p;
        return st;
    }
    p->ws_bytes = 256 + vws;
    if (cudaMalloc(&p->ws, p->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return CN_ERR_ALLOC;
    }
    if (cudaMemset(p->ws, 0, p->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p->ws);
        delete p;
        return CN_ERR_CUDA;
    }
    p->err_flag = static_cast<int *>(p->ws);
    char *vbase = static_cast<char *>(p->ws) + 256;
    switch (p->variant) {
        case V_MEAN3D: {
            Mean3dArgs &a = p->mean_args;
            const size_t part = mean3d_partial_bytes(a);
            a.partial = reinterpret_cast<double *>(vbase);
            a.tickets = reinterpret_cast<int *>(vbase + ((part + 255) & ~(size_t)255));
            a.err = p->err_flag;
            p->counters = a.tickets;
            p->counter_bytes = mean3d_tickets(a) * sizeof(int);
            break;
        }
        case V_POOL3D:
            p->pool_args.err = p->err_flag;
            p->pool_args.t.work = reinterpret_cast<int *>(vbase);  // zero between launches
            p->counters = p->pool_args.t.work;
            p->counter_bytes = pool3d_workspace(p->pool_args);
            break;
        default:
            full2d_bind_workspace(p->full_args, vbase, p->err_flag);
            p->counters = p->full_args.tickets;
            p->counter_bytes = full2d_counter_bytes(p->full_args);
            break;
    }
    *out = p;
    return CN_OK;
}

void conv_norm_plan_destroy(conv_norm_plan p) {
    if (!p) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    cudaFree(p->ws);
    cudaFree(p->stage.x);
    cudaFree(p->stage.w);
    cudaFree(p->stage.b);
    cudaFree(p->stage.gamma);
    cudaFree(p->stage.beta);
    cudaFree(p->stage.out);
    for (int i = 0; i < kMaxHostChunks; ++i) conv_norm_plan_destroy(p->stage.sub[i]);
    if (p->stage.up) cudaStreamDestroy(p->stage.up);
    if (p->stage.down) cudaStreamDestroy(p->stage.down);
    if (p->stage.comp2) cudaStreamDestroy(p->stage.comp2);
    if (p->stage.ev_comp2) cudaEventDestroy(p->stage.ev_comp2);
    for (int i = 0; i < kMaxHostChunks; ++i) {
        if (p->stage.ev_up[i]) cudaEventDestroy(p->stage.ev_up[i]);
        if (p->stage.ev_done[i]) cudaEventDestroy(p->stage.ev_done[i]);
    }
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    cudaGetLastError();
    delete p;
}

size_t conv_norm_workspace_bytes(conv_norm_plan p) { return p ? p->ws_bytes : 0; }

int conv_norm_plan_info(conv_norm_plan p, conv_norm_info *info) {
    if (!p || !info) return CN_ERR_INVALID_ARG;
    memset(info, 0, sizeof(*info));
    info->variant = p->variant;
    info->out_numel = p->out_numel;
    info->workspace_bytes = p->ws_bytes;
    switch (p->variant) {
        case V_MEAN3D:
            info->launches_per_forward = mean3d_launches(p->mean_cfg, p->mean_args);
            info->kernel_names = p->mean_cfg.name;
            info->grid_ctas = p->mean_cfg.grid;
            info->threads_per_cta = p->mean_cfg.threads;
            info->smem_bytes_per_cta = p->mean_cfg.smem;
            break;
        case V_POOL3D:
            info->launches_per_forward = p->pool_cfg.grid > 0 ? 1 : 0;
            info->kernel_names = p->pool_cfg.name;
            info->grid_ctas = p->pool_cfg.grid;
            info->threads_per_cta = p->pool_cfg.threads;
            info->smem_bytes_per_cta = p->pool_cfg.smem;
            break;
        default:
            info->launches_per_forward = full2d_launches(p->full_cfg, p->full_args);
            info->kernel_names = p->full_cfg.names;
            info->grid_ctas = p->full_cfg.grid;
            info->threads_per_cta = p->full_cfg.threads;
            info->smem_bytes_per_cta = p->full_cfg.smem;
            break;
    }
    return CN_OK;
}

static int forward_impl(conv_norm_plan p, const float *x, const float *w, const float *b,
                        const float *gamma, const float *beta, float *out, cudaStream_t s,
                        const LaunchEvents *ev = nullptr) {
    const conv_norm_desc &d = p->d;
    const bool need_aff = d.affine && d.norm != CN_NORM_NONE;
    // An empty problem launches nothing; its (zero-size) tensors may have null pointers.
    if (d.N == 0 || p->out_numel == 0) return CN_OK;
    if (!x || !w || !out) return CN_ERR_INVALID_ARG;
    if ((b != nullptr) != (d.has_bias == 1)) return CN_ERR_INVALID_ARG;
    if (need_aff && (!gamma || !beta)) return CN_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(w, 4)) return CN_ERR_INVALID_ARG;
    if (!need_aff) gamma = beta = nullptr;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    if (cur != p->device && cudaSetDevice(p->device) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    int st;
    const int stall = p->stall_pending;  // one forward only
    p->stall_pending = 0;
    switch (p->variant) {
        case V_MEAN3D: {
            Mean3dArgs &a = p->mean_args;  // keeps the encoded tensor map cached
            a.x = x; a.w = w; a.b = b; a.gamma = gamma; a.beta = beta; a.out = out;
            a.t.stall = stall;
            st = mean3d_launch(p->mean_cfg, a, s, ev);
            a.t.stall = 0;
            break;
        }
        case V_POOL3D: {
            Pool3dArgs &a = p->pool_args;  // keeps the encoded tensor map cached
            a.x = x; a.w = w; a.b = b; a.out = out;
            a.t.stall = stall;
            st = pool3d_launch(p->pool_cfg, a, s, ev);
            a.t.stall = 0;
            break;
        }
        default: {
            Full2dArgs &a = p->full_args;  // keeps the encoded tensor map cached
            a.x = x; a.w = w; a.b = b; a.gamma = gamma; a.beta = beta; a.out = out;
            a.stall = stall;
            st = full2d_launch(p->full_cfg, a, s, ev);
            a.stall = 0;
            break;
        }
    }
    if (st != CN_OK) cudaGetLastError();
    if (cur != p->device) cudaSetDevice(cur);
    return st;
}

int conv_norm_forward(conv_norm_plan p, const float *x, const float *w, const float *b,
                      const float *gamma, const float *beta, float *out, void *stream) {
    if (!p) return CN_ERR_INVALID_ARG;
    return forward_impl(p, x, w, b, gamma, beta, out, static_cast<cudaStream_t>(stream),
                        p->events.n ? &p->events : nullptr);
}

int conv_norm_plan_set_launch_events(conv_norm_plan p, void *const *events, int n) {
    if (!p) return CN_ERR_INVALID_ARG;
    if (n == 0) {
        p->events.n = 0;
        return CN_OK;
    }
    int L = 0;
    switch (p->variant) {
        case V_MEAN3D:
            L = mean3d_launches(p->mean_cfg, p->mean_args);
            break;
        case V_POOL3D:
            L = p->pool_cfg.grid > 0 ? 1 : 0;
            break;
        default:
            L = full2d_launches(p->full_cfg, p->full_args);
            break;
    }
    if (!events || n != L + 1 || n > kMaxLaunchEvents) return CN_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (!events[i]) return CN_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) p->events.ev[i] = static_cast<cudaEvent_t>(events[i]);
    p->events.n = n;
    return CN_OK;
}

static int stage_alloc(float **dst, int64_t n) {
    if (*dst || n <= 0) return CN_OK;
    if (cudaMalloc(reinterpret_cast<void **>(dst), (size_t)n * sizeof(float)) != cudaSuccess) {
        cudaGetLastError();
        *dst = nullptr;
        return CN_ERR_ALLOC;
    }
    return CN_OK;
}

// Sets up the staging of conv_norm_forward_host: the batch is cut into up
// to kMaxHostChunks chunks of whole samples (every step of the computation
// is per sample) so uploads, kernels and downloads of different chunks
// overlap.  One chunk when the batch is small or a sample's tensors are not
// 16-byte multiples.
static int host_stage_setup(conv_norm_plan p) {
    HostStage &hs = p->stage;
    const conv_norm_desc &d = p->d;
    const bool need_aff = d.affine && d.norm != CN_NORM_NONE;
    int st = CN_OK;
    if (st == CN_OK) st = stage_alloc(&hs.x, p->x_numel);
    if (st == CN_OK) st = stage_alloc(&hs.w, p->w_numel);
    if (st == CN_OK && d.has_bias) st = stage_alloc(&hs.b, d.C_out);
    if (st == CN_OK && need_aff) st = stage_alloc(&hs.gamma, d.C_out);
    if (st == CN_OK && need_aff) st = stage_alloc(&hs.beta, d.C_out);
    if (st == CN_OK) st = stage_alloc(&hs.out, p->out_numel);
    if (st != CN_OK) return st;
    const int64_t xs = p->x_numel / d.N, os = p->out_numel / d.N;
    // Measured on GB300 (host copies ~210 GB/s up, ~190 down, ~330 both
    // ways at once): about 6 MB of input per chunk, at most 16.  Only the
    // first chunk's upload and the last chunk's kernels and download stay
    // exposed, and with two compute streams a chunk's launch ramp overlaps
    // the previous chunk's tail; at 25 MB of input 4 chunks beat 2 and 8,
    // at 135 MB and 537 MB 16 chunks beat 8 by 1.4% and 1.9%, and at 101 MB
    // 8, 12 and 16 are within 1%.
    const double xbytes = (double)p->x_numel * 4;
    int nch = xbytes < 16.0 * 1024 * 1024 ? 1 : std::min(kMaxHostChunks, (int)(xbytes / 6.0e6));
    if (const char *e = getenv("CN_HOST_CHUNKS")) nch = std::max(1, std::min(kMaxHostChunks, atoi(e)));
    if (xs % 4 != 0 || os % 4 != 0) nch = 1;
    nch = std::min(nch, d.N);
    hs.chunk_n = (d.N + nch - 1) / nch;
    hs.nchunk = (d.N + hs.chunk_n - 1) / hs.chunk_n;
    // Each object is created only if missing, so a call after a failed setup
    // finishes it without leaking what the failed one made.
    auto stream = [](cudaStream_t &q) {
        return q || cudaStreamCreateWithFlags(&q, cudaStreamNonBlocking) == cudaSuccess;
    };
    auto event = [](cudaEvent_t &e) {
        return e || cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    };
    if (hs.nchunk > 1) {
        conv_norm_desc dc = d;
        for (int i = 0; i < hs.nchunk; ++i) {
            dc.N = std::min(hs.chunk_n, d.N - i * hs.chunk_n);
            if (!hs.sub[i] && (st = conv_norm_plan_create(&dc, &hs.sub[i])) != CN_OK) return st;
        }
        if (!stream(hs.up) || !stream(hs.down) || !stream(hs.comp2) || !event(hs.ev_comp2)) {
            cudaGetLastError();
            return CN_ERR_CUDA;
        }
        for (int i = 0; i < hs.nchunk; ++i)
            if (!event(hs.ev_up[i]) || !event(hs.ev_done[i])) {
                cudaGetLastError();
                return CN_ERR_CUDA;
            }
    }
    hs.ready = true;
    return CN_OK;
}

int conv_norm_forward_host(conv_norm_plan p, const float *x, const float *w, const float *b,
                           const float *gamma, const float *beta, float *out, void *stream) {
    if (!p) return CN_ERR_INVALID_ARG;
    const conv_norm_desc &d = p->d;
    const bool need_aff = d.affine && d.norm != CN_NORM_NONE;
    if (d.N == 0 || p->out_numel == 0) return CN_OK;
    if (!x || !w || !out) return CN_ERR_INVALID_ARG;
    if ((b != nullptr) != (d.has_bias == 1)) return CN_ERR_INVALID_ARG;
    if (need_aff && (!gamma || !beta)) return CN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    if (cur != p->device) cudaSetDevice(p->device);
    HostStage &hs = p->stage;
    int st = hs.ready ? CN_OK : host_stage_setup(p);
    bool ok = st == CN_OK;
    // The parameters go first on the stream that carries x: queued on a
    // compute stream instead, these small copies could wait on the copy
    // engine behind the large x uploads and hold every chunk's kernels back.
    cudaStream_t ps = hs.nchunk > 1 ? hs.up : s;
    ok = ok && cudaMemcpyAsync(hs.w, w, p->w_numel * 4, cudaMemcpyHostToDevice, ps) == cudaSuccess;
    if (b) ok = ok && cudaMemcpyAsync(hs.b, b, d.C_out * 4, cudaMemcpyHostToDevice, ps) == cudaSuccess;
    if (need_aff) {
        ok = ok && cudaMemcpyAsync(hs.gamma, gamma, d.C_out * 4, cudaMemcpyHostToDevice, ps) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(hs.beta, beta, d.C_out * 4, cudaMemcpyHostToDevice, ps) == cudaSuccess;
    }
    const float *db = b ? hs.b : nullptr;
    const float *dg = need_aff ? hs.gamma : nullptr, *dbe = need_aff ? hs.beta : nullptr;
    if (ok && hs.nchunk == 1) {
        ok = cudaMemcpyAsync(hs.x, x, p->x_numel * 4, cudaMemcpyHostToDevice, s) == cudaSuccess;
        if (ok) {
            st = forward_impl(p, hs.x, hs.w, db, dg, dbe, hs.out, s);
            ok = st == CN_OK;
        }
        ok = ok && cudaMemcpyAsync(out, hs.out, p->out_numel * 4, cudaMemcpyDeviceToHost, s) == cudaSuccess;
    } else if (ok) {
        const int64_t xs = p->x_numel / d.N, os = p->out_numel / d.N;
        // uploads run ahead on their own stream, after the parameters; a
        // chunk's kernels wait for its upload event, so for the parameters too
        for (int i = 0; ok && i < hs.nchunk; ++i) {
            const int64_t n0 = (int64_t)i * hs.chunk_n, nn = std::min<int64_t>(hs.chunk_n, d.N - n0);
            ok = cudaMemcpyAsync(hs.x + n0 * xs, x + n0 * xs, nn * xs * 4, cudaMemcpyHostToDevice,
                                 hs.up) == cudaSuccess &&
                 cudaEventRecord(hs.ev_up[i], hs.up) == cudaSuccess;
        }
        // even chunks compute on the caller's stream, odd ones on comp2;
        // downloads on their own stream
        for (int i = 0; ok && i < hs.nchunk; ++i) {
            const int64_t n0 = (int64_t)i * hs.chunk_n, nn = std::min<int64_t>(hs.chunk_n, d.N - n0);
            conv_norm_plan_s *sp = hs.sub[i];
            cudaStream_t cs = (i & 1) ? hs.comp2 : s;
            ok = cudaStreamWaitEvent(cs, hs.ev_up[i], 0) == cudaSuccess;
            if (ok) {
                st = forward_impl(sp, hs.x + n0 * xs, hs.w, db, dg, dbe, hs.out + n0 * os, cs);
                ok = st == CN_OK;
            }
            ok = ok && cudaEventRecord(hs.ev_done[i], cs) == cudaSuccess &&
                 cudaStreamWaitEvent(hs.down, hs.ev_done[i], 0) == cudaSuccess &&
                 cudaMemcpyAsync(out + n0 * os, hs.out + n0 * os, nn * os * 4, cudaMemcpyDeviceToHost,
                                 hs.down) == cudaSuccess;
        }
        ok = ok && cudaEventRecord(hs.ev_comp2, hs.comp2) == cudaSuccess &&
             cudaStreamWaitEvent(s, hs.ev_comp2, 0) == cudaSuccess;
    }
    // drain every stream this call used, after an error too, so that the
    // next call never overwrites staging buffers a queued copy or kernel uses
    for (cudaStream_t q : {hs.up, hs.comp2, hs.down})
        if (q && cudaStreamSynchronize(q) != cudaSuccess) ok = false;
    if (cudaStreamSynchronize(s) != cudaSuccess) ok = false;
    if (!ok) {
        if (st == CN_OK) st = CN_ERR_CUDA;
        cudaGetLastError();
    }
    if (cur != p->device) cudaSetDevice(cur);
    return st;
}

static bool has_tc_kernel(const conv_norm_plan_s *p);

int conv_norm_plan_set_wait_limit(conv_norm_plan p, uint64_t ns) {
    if (!p || ns == 0) return CN_ERR_INVALID_ARG;
    if (!has_tc_kernel(p)) return CN_ERR_UNSUPPORTED;
    switch (p->variant) {
        case V_MEAN3D: p->mean_args.t.wait_ns = ns; break;
        case V_POOL3D: p->pool_args.t.wait_ns = ns; break;
        default: p->full_args.wait_ns = ns; break;
    }
    return CN_OK;
}

static bool has_tc_kernel(const conv_norm_plan_s *p) {
    switch (p->variant) {
        case V_MEAN3D: return p->mean_args.tc != 0;
        case V_POOL3D: return p->pool_args.tc != 0;
        default: return p->full_args.tc || p->full_args.tct;
    }
}

int conv_norm_plan_inject_stall(conv_norm_plan p) {
    if (!p) return CN_ERR_INVALID_ARG;
    if (!has_tc_kernel(p)) return CN_ERR_UNSUPPORTED;
    p->stall_pending = 1;
    return CN_OK;
}

int conv_norm_plan_check_device(conv_norm_plan p, void *stream) {
    if (!p) return noalloc_check_device(static_cast<cudaStream_t>(stream));
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    int st = CN_OK;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        st = CN_ERR_CUDA;
    }
    // the plan's own flag, then those of the chunk plans conv_norm_forward_host runs
    for (int i = -1; st != CN_ERR_CUDA && i < kMaxHostChunks; ++i) {
        const conv_norm_plan_s *q = i < 0 ? p : p->stage.sub[i];
        if (!q) continue;
        int flag = 0;
        if (cudaMemcpy(&flag, q->err_flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            st = CN_ERR_CUDA;
        } else if (flag != 0) {
            const int zero = 0;
            cudaMemcpy(q->err_flag, &zero, sizeof(int), cudaMemcpyHostToDevice);
            // a kernel that gave up may have left tickets and work counters
            // part-way: zero them so the plan's next forward starts clean
            if (q->counters && q->counter_bytes) cudaMemset(q->counters, 0, q->counter_bytes);
            if (st != CN_ERR_TIMEOUT) st = flag == 1 ? CN_ERR_TIMEOUT : CN_ERR_DEVICE_CHECK;
        }
    }
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    return st;
}

}  // extern "C"
