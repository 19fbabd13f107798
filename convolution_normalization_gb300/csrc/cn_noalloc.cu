// conv_norm_forward_noalloc: the Conv3d -> activation -> norm -> spatial
// mean forward for callers that cannot allocate device memory.
//
// The regular path keeps the kernel's scratch (per-chunk partial moments and
// per-sample tickets) in a workspace that conv_norm_plan_create obtains with
// cudaMalloc.  Some callers cannot do that: an engine plugin or a real-time
// loop whose device memory was reserved up front by another allocator (a
// framework's caching allocator, a memory pool) gets a failed or
// device-synchronizing cudaMalloc, and code with a fixed device-memory
// budget must not grow it after start-up.  This entry point instead uses
// one fixed array in the library's own device globals, so it makes no
// allocation call of any kind.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "cn_internal.h"

// Largest scratch one call may use.  Every GPU that loads the library holds
// this much device memory in its globals until the process exits.
#define CN_NOALLOC_SCRATCH_BYTES (4u << 20)

// The kernel's scratch for conv_norm_forward_noalloc.  In host code this
// name is only a host-side stand-in: the device address must come from
// cudaGetSymbolAddress (scratch_device_address below).
static __device__ __align__(256) unsigned char g_cn_noalloc_scratch[CN_NOALLOC_SCRATCH_BYTES];
// Error flag of those calls (a bounded wait that gave up), read and cleared
// by conv_norm_plan_check_device(NULL, stream).  Same host-side caveat.
static __device__ int g_cn_noalloc_err;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};
void *g_err_ptr[kMaxDevices] = {};

// Device addresses of the scratch array and the error flag on the current
// device, looked up once per device (with that device current) and cached.
int scratch_device_address(int dev, void **out, int **err) {
    if (dev < 0 || dev >= kMaxDevices) return CN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr, *e = nullptr;
        if (cudaGetSymbolAddress(&p, g_cn_noalloc_scratch) != cudaSuccess || !p ||
            cudaGetSymbolAddress(&e, g_cn_noalloc_err) != cudaSuccess || !e) {
            cudaGetLastError();
            return CN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
        g_err_ptr[dev] = e;
    }
    *out = g_scratch_ptr[dev];
    *err = static_cast<int *>(g_err_ptr[dev]);
    return CN_OK;
}

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int conv_norm_forward_noalloc(const conv_norm_desc *d, const float *x, const float *w,
                                         const float *b, const float *gamma, const float *beta,
                                         float *out, void *stream) {
    if (!d) return CN_ERR_INVALID_ARG;
    int64_t dims[5];
    int nd = 0;
    int st = conv_norm_output_shape(d, dims, &nd);  // checks the descriptor is well formed
    if (st != CN_OK) return st;
    // Only the variant whose kernel needs scratch memory is offered here.
    if (d->conv != CN_CONV3D || d->red != CN_RED_MEAN_SPATIAL || d->act == CN_ACT_SOFTMAX_C)
        return CN_ERR_UNSUPPORTED;
    cn::Mean3dArgs a{};
    cn::Mean3dConfig cfg{};
    st = cn::mean3d_plan(*d, a, cfg);
    if (st != CN_OK) return st;
    if (d->N == 0) return CN_OK;
    // the scratch this problem needs: moments, then tickets (256-byte aligned)
    const size_t part = cn::mean3d_partial_bytes(a);
    const size_t part_al = (part + 255) & ~(size_t)255;
    const size_t tick_bytes = cn::mean3d_tickets(a) * sizeof(int);
    if (part_al + tick_bytes > CN_NOALLOC_SCRATCH_BYTES)
        return CN_ERR_UNSUPPORTED;
    const bool need_aff = d->affine && d->norm != CN_NORM_NONE;
    if (!x || !w || !out) return CN_ERR_INVALID_ARG;
    if ((b != nullptr) != (d->has_bias == 1)) return CN_ERR_INVALID_ARG;
    if (need_aff && (!gamma || !beta)) return CN_ERR_INVALID_ARG;
    if (!aligned_to(x, 16) || !aligned_to(out, 16) || !aligned_to(w, 4)) return CN_ERR_INVALID_ARG;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    void *base = nullptr;
    int *err = nullptr;
    st = scratch_device_address(dev, &base, &err);
    if (st != CN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    a.partial = static_cast<double *>(base);
    a.tickets = reinterpret_cast<int *>(static_cast<char *>(base) + part_al);
    a.err = err;
    // The array keeps the previous call's contents: the tickets and work
    // counters must start at zero (every partial-moment slot is overwritten
    // before it is read).
    if (cudaMemsetAsync(a.tickets, 0, tick_bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    st = cn::mean3d_prepare(cfg, a);
    if (st != CN_OK) {
        cudaGetLastError();
        return st;
    }
    a.x = x;
    a.w = w;
    a.b = b;
    a.gamma = need_aff ? gamma : nullptr;
    a.beta = need_aff ? beta : nullptr;
    a.out = out;
    st = cn::mean3d_launch(cfg, a, s);
    if (st != CN_OK) cudaGetLastError();
    return st;
}

// conv_norm_plan_check_device(NULL, stream): the flag of the no-allocation
// calls on the current device, after synchronizing the stream.
int cn::noalloc_check_device(cudaStream_t stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    void *base = nullptr;
    int *err = nullptr;
    int st = scratch_device_address(dev, &base, &err);
    if (st != CN_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    int flag = 0;
    if (cudaMemcpy(&flag, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return CN_ERR_CUDA;
    }
    if (flag == 0) return CN_OK;
    // clear it, and the scratch's tickets and counters (every call zeroes
    // the ones it uses before its kernel runs, so nothing else is needed)
    const int zero = 0;
    cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return flag == 1 ? CN_ERR_TIMEOUT : CN_ERR_DEVICE_CHECK;
}
