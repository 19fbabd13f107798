/*
 * conv_norm — fused convolution + normalization forward for GB300 (sm_103a).
 *
 * One call computes, on one GPU and on the caller's stream,
 *
 *   conv  ->  activation  ->  normalization  ->  post scale  ->  reduction
 *
 * for fp32 tensors in PyTorch's contiguous NCDHW / NCHW layout, stride 1,
 * padding 0.  The computation is the one four problem transcripts build
 * fused kernels for (their pages are named by problem id):
 *
 *   l2_p27  Conv3d(3->16, k) -> HardSwish -> GroupNorm(4) -> mean over D,H,W
 *   l2_p17  Conv2d(64->128, k=3) -> InstanceNorm2d -> divide by 2
 *   l2_p6   Conv3d(3->16, k=3) -> Softmax(dim=1) -> MaxPool3d(2) -> MaxPool3d(2)
 *   l2_p19  ConvTranspose2d(64->64, k=3, s=1, groups) -> GELU -> GroupNorm(8)
 *
 * Status codes: every function that returns int returns CN_OK (0) on
 * success and a negative CN_ERR_* value on failure; no function aborts the
 * process.  All tensors are caller-owned.  The library is not thread-safe
 * per plan: calls that use one plan must be ordered (one stream, or
 * explicit synchronization), because the plan's workspace is shared by its
 * launches.
 */
#ifndef CONV_NORM_H
#define CONV_NORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define CN_OK 0
#define CN_ERR_INVALID_ARG (-1)  /* bad descriptor, null/misaligned pointer  */
#define CN_ERR_UNSUPPORTED (-2)  /* valid problem, no kernel for this shape  */
#define CN_ERR_CUDA (-3)         /* a CUDA runtime call or launch failed     */
#define CN_ERR_TIMEOUT (-4)      /* a bounded device-side wait ran out       */
#define CN_ERR_DEVICE_CHECK (-5) /* a kernel's own bounds check tripped      */
#define CN_ERR_ALLOC (-6)        /* device or host allocation failed         */

/* ---- problem descriptor -------------------------------------------------- */
typedef enum { CN_CONV3D = 0, CN_CONV2D = 1, CN_CONVT2D = 2 } cn_conv_kind;
typedef enum {
    CN_ACT_NONE = 0,
    CN_ACT_HARDSWISH = 1, /* v * clamp(v + 3, 0, 6) / 6            (l2_p27) */
    CN_ACT_GELU_ERF = 2,  /* 0.5 v (1 + erf(v / sqrt 2)), exact     (l2_p19) */
    CN_ACT_SOFTMAX_C = 3  /* softmax over the channel axis          (l2_p6)  */
} cn_act;
typedef enum {
    CN_NORM_NONE = 0,
    CN_NORM_GROUP = 1,    /* per (n, group) over C/G channels x space (l2_p27, l2_p19) */
    CN_NORM_INSTANCE = 2  /* per (n, c) over space                    (l2_p17) */
} cn_norm;
typedef enum {
    CN_RED_NONE = 0,         /* full normalized tensor is the output            */
    CN_RED_MEAN_SPATIAL = 1, /* mean over all spatial axes -> (N, C_out) (l2_p27) */
    CN_RED_MAXPOOL2_X2 = 2   /* MaxPool3d(2,2) applied twice, floor mode (l2_p6) */
} cn_red;

/*
 * All fields are plain ints/floats so the struct has the same layout from C,
 * C++ and Python ctypes.
 *   conv        cn_conv_kind.  CN_CONV3D: x (N,C_in,D,H,W), weight
 *               (C_out, C_in/groups, k, k, k).  CN_CONV2D: x (N,C_in,H,W),
 *               weight (C_out, C_in/groups, k, k), D must be 1.
 *               CN_CONVT2D: transposed conv, stride 1, padding 0, x
 *               (N,C_in,H,W), weight (C_in, C_out/groups, k, k) (PyTorch's
 *               ConvTranspose2d layout), D must be 1.
 *   N           batch size; N = 0 is an empty problem (forward does nothing).
 *   k, groups   cubic/square kernel extent; channel groups of the conv.
 *   has_bias    0/1: whether a conv bias of length C_out is added.
 *   act         cn_act.   norm: cn_norm.  red: cn_red.
 *   num_groups  GroupNorm groups (C_out % num_groups == 0); ignored otherwise.
 *   affine      0/1: per-channel gamma/beta after normalization.
 *   eps         added to the variance inside the square root (> 0).
 *   post_scale  multiplies the normalized value (0.5 for "divide by 2").
 * Conv output extent per spatial axis: L - k + 1 (conv), L + k - 1 (convT).
 */
typedef struct {
    int conv;
    int N, C_in, C_out, D, H, W, k, groups;
    int has_bias;
    int act;
    int norm;
    int num_groups;
    int affine;
    float eps;
    float post_scale;
    int red;
} conv_norm_desc;

typedef struct conv_norm_plan_s *conv_norm_plan;

/* Facts about a created plan, for reporting (kernel names are static
 * strings owned by the library). */
typedef struct {
    int variant;               /* 0 mean-3d, 1 softmax-pool-3d, 2 full-2d */
    int launches_per_forward;  /* kernels one conv_norm_forward launches   */
    const char *kernel_names;  /* comma-separated, in launch order         */
    int64_t out_numel;         /* number of fp32 values written to out     */
    size_t workspace_bytes;    /* device workspace owned by the plan        */
    int grid_ctas;             /* CTAs of the main (conv) kernel            */
    int threads_per_cta;
    int smem_bytes_per_cta;
} conv_norm_info;

/* ---- host-only queries (need no GPU) ------------------------------------- */

/* Checks a descriptor.  Returns CN_OK, CN_ERR_INVALID_ARG for a malformed
 * problem (e.g. C_in % groups != 0, kernel larger than the input) or
 * CN_ERR_UNSUPPORTED for a valid problem this library has no kernel for.
 * Supported: spatial mean after Conv3d (groups 1, k <= 4, C_out % 4 == 0);
 * the double max pool after Conv3d + channel softmax (C_out = 16, k <= 4, no
 * norm, post_scale > 0); the full output after Conv2d, ConvTranspose2d ((C_out/groups) % 4
 * == 0, k <= 4) or Conv3d (groups 1, C_out % 4 == 0, k <= 4), any activation
 * but softmax. */
int conv_norm_desc_validate(const conv_norm_desc *desc);

/* Writes the output shape implied by desc into dims[0..*ndim-1] (ndim <= 5):
 * (N, C_out) for CN_RED_MEAN_SPATIAL; (N, C_out, Do/4, Ho/4, Wo/4) with
 * floor division for CN_RED_MAXPOOL2_X2; the conv output shape otherwise. */
int conv_norm_output_shape(const conv_norm_desc *desc, int64_t dims[5], int *ndim);

/* Human-readable name of a status code (static string). */
const char *conv_norm_status_string(int status);

/* ---- plans ---------------------------------------------------------------- */

/* Cites: the module constructor of each problem page, whose arguments fix
 * the problem: in_channels, out_channels and kernel_size everywhere, the
 * group count on l2_p27, divide_by on l2_p17, the pool size on l2_p6, and
 * stride, groups and num_groups on l2_p19.  desc holds those arguments plus
 * the input extents each page's get_inputs fixes.
 * Validates desc, picks the kernel variant and its tiling for the CURRENT
 * CUDA device, and allocates the plan's device workspace there (partial
 * statistics, tickets, an error flag).  On success *out_plan owns that
 * memory until conv_norm_plan_destroy; on failure *out_plan is set to NULL.
 * Errors: CN_ERR_INVALID_ARG (NULL pointers, malformed desc),
 * CN_ERR_UNSUPPORTED, CN_ERR_CUDA (no device / attribute query failed),
 * CN_ERR_ALLOC (cudaMalloc or host allocation failed). */
int conv_norm_plan_create(const conv_norm_desc *desc, conv_norm_plan *out_plan);

/* Cites: no page passage (the pages' modules own their tensors through
 * PyTorch); this releases what conv_norm_plan_create acquired.
 * Frees the plan and its workspace.  NULL is ignored.  The caller must make
 * sure no forward that uses the plan is still running. */
void conv_norm_plan_destroy(conv_norm_plan plan);

/* Cites: the buffers of partial statistics that the pages' multi-pass
 * designs pass between kernels (l2_p19's three-kernel GroupNorm: partial
 * sums, group statistics, apply; l2_p27's per-block partial moments), kept
 * here in a plan-owned workspace.
 * Bytes of device workspace the plan owns (0 when none is needed; 0 for a
 * NULL plan). */
size_t conv_norm_workspace_bytes(conv_norm_plan plan);

/* Fills *info with the plan's variant, kernels and workspace size (a
 * reporting aid; no counterpart on the pages); returns CN_ERR_INVALID_ARG
 * for NULL arguments. */
int conv_norm_plan_info(conv_norm_plan plan, conv_norm_info *info);

/* ---- forward -------------------------------------------------------------- */

/*
 * Cites: ModelNew.forward(x) of each problem page (l2_p27: conv -> HardSwish
 * -> GroupNorm -> mean over D, H, W; l2_p17: conv -> InstanceNorm2d -> divide
 * by 2; l2_p6: conv -> Softmax(dim=1) -> MaxPool3d(2) twice; l2_p19:
 * ConvTranspose2d -> GELU -> GroupNorm), with the module's weights passed in.
 * Runs the fused forward asynchronously on cuda_stream (a cudaStream_t; NULL
 * is the legacy default stream).  All pointers are DEVICE pointers on the
 * plan's device, fp32, contiguous, 16-byte aligned:
 *   x      input, layout given by desc->conv                     (read)
 *   w      conv weight (layout in conv_norm_desc)                (read)
 *   b      bias (C_out), NULL iff has_bias == 0                  (read)
 *   gamma  (C_out), beta (C_out): NULL iff affine == 0 or norm == NONE
 *   out    output, shape from conv_norm_output_shape            (written)
 * out must not overlap the inputs.  No host synchronization happens and no
 * memory is allocated.  Errors: CN_ERR_INVALID_ARG (null/misaligned pointer,
 * NULL plan), CN_ERR_CUDA (launch failure; cudaGetLastError is cleared).
 * Device-side problems (a bounded wait that ran out) are reported later by
 * conv_norm_plan_check_device.
 */
int conv_norm_forward(conv_norm_plan plan, const float *x, const float *w,
                      const float *b, const float *gamma, const float *beta,
                      float *out, void *cuda_stream);

/*
 * Same computation with HOST buffers: copies x, w, b, gamma, beta to device
 * buffers owned by the plan, runs the forward on cuda_stream, copies the
 * result back into the host buffer out and synchronizes before returning.
 * Batches of more than about 16 MB of input are cut into chunks of whole
 * samples, about 6 MB of input each and at most 16 (every step is per
 * sample): chunk i+1 uploads on a
 * plan-owned stream while chunk i computes, even chunks on cuda_stream and
 * odd ones on a plan-owned compute stream (so one chunk's kernels can start
 * on the SMs the previous chunk's last work leaves idle), and each chunk's
 * result downloads on a third plan-owned stream as soon as it is done;
 * cuda_stream waits for the second compute stream before the call returns.
 * The first call allocates the staging buffers, the per-chunk plans, the
 * three streams and their events.  Pinned (page-locked) host memory gives
 * asynchronous full-bandwidth copies; pageable memory works too.  Errors as
 * conv_norm_forward, plus CN_ERR_ALLOC.
 */
int conv_norm_forward_host(conv_norm_plan plan, const float *x, const float *w,
                           const float *b, const float *gamma, const float *beta,
                           float *out, void *cuda_stream);

/*
 * Synchronizes cuda_stream, then reads and clears the plan's device error
 * flag and those of the chunk plans conv_norm_forward_host created.  Returns
 * CN_OK, CN_ERR_TIMEOUT (a bounded device wait gave up; the
 * output of that forward is undefined), CN_ERR_DEVICE_CHECK or CN_ERR_CUDA.
 * With plan == NULL it reads and clears the flag of the
 * conv_norm_forward_noalloc calls on the current device instead.
 * When a flag was set it also zeroes that plan's tickets and work counters,
 * which a kernel that gave up can leave part-way, so the plan's next
 * forward runs normally.
 */
int conv_norm_plan_check_device(conv_norm_plan plan, void *cuda_stream);

/*
 * Failure handling (no counterpart in the transcripts).  Every wait of a
 * kernel on another part of its work (a copy landing, an MMA finishing, a
 * pipeline slot freeing) is bounded: after the limit it records
 * CN_ERR_TIMEOUT in the plan's flag, the CTA stops its other roles, waits
 * (with the fixed 200 ms bound) for its own copies and MMAs in flight,
 * frees its tensor memory and exits.  This sets the limit of those progress
 * waits for the plan's tensor-core kernel, in ns of GPU wall time (default
 * 200 ms); a very short limit makes a forward give up on purpose, which is
 * how the timeout path is tested.  The CUDA-core kernels keep the fixed
 * limit.  The chunk plans of conv_norm_forward_host keep the default.
 * Errors: CN_ERR_INVALID_ARG (NULL plan, ns == 0), CN_ERR_UNSUPPORTED (the
 * plan runs no tensor-core kernel).
 */
int conv_norm_plan_set_wait_limit(conv_norm_plan plan, uint64_t ns);

/*
 * Failure-path test hook (no counterpart in the transcripts): the plan's
 * next forward runs its tensor-core kernel with the first input copy of
 * CTA 0 left unissued, a barrier phase that nothing completes.  That CTA's
 * waits run out after the plan's wait limit, it stops and exits as above,
 * the other CTAs finish their own work, and conv_norm_plan_check_device
 * then returns CN_ERR_TIMEOUT; the output of that forward is undefined.
 * Nothing faults and no wait is unbounded.  One forward only.
 * Errors: CN_ERR_INVALID_ARG (NULL plan), CN_ERR_UNSUPPORTED (the plan
 * runs no tensor-core kernel).
 */
int conv_norm_plan_inject_stall(conv_norm_plan plan);

/*
 * Optional per-launch timing (a measurement aid; no counterpart in the
 * transcripts).  After this call every conv_norm_forward on the plan records
 * events[i] on its stream just before the plan's i-th kernel launch and
 * events[L] after the last one, where L = conv_norm_info.launches_per_forward;
 * cudaEventElapsedTime(events[i], events[i+1]) is then the device time of
 * launch i (kernel names in order: conv_norm_info.kernel_names).
 *   events  array of n cudaEvent_t handles, created and owned by the caller,
 *           valid until the next call of this function (the handles are
 *           copied, the array may be freed after the call)
 *   n       L + 1, or 0 (events may be NULL) to stop recording
 * Errors: CN_ERR_INVALID_ARG for a NULL plan, n not in {0, L + 1}, or a NULL
 * handle.  conv_norm_forward_host does not record.
 */
int conv_norm_plan_set_launch_events(conv_norm_plan plan, void *const *events, int n);

/* ---- forward without any allocation ------------------------------------------ */

/*
 * No counterpart in the transcripts: this exists for callers that cannot
 * allocate device memory.  conv_norm_plan_create gets its workspace from
 * cudaMalloc; an engine plugin or a real-time loop whose device memory is
 * reserved up front by another allocator (a framework's caching allocator,
 * a memory pool) may see that call fail or synchronize the device, and some
 * programs must keep a fixed device-memory footprint after start-up.
 *
 * conv_norm_forward_noalloc runs the same computation as conv_norm_forward
 * for the spatial-mean problems (desc->conv == CN_CONV3D, desc->red ==
 * CN_RED_MEAN_SPATIAL; l2_p27's Conv3d -> HardSwish -> GroupNorm -> mean)
 * without a plan and without any allocation: the kernel's scratch (partial
 * moments and per-sample tickets) lives in one fixed array of 4 MiB in the
 * library's device globals, which every GPU that loads the library holds
 * until the process exits.  Arguments, layouts and alignment are those of
 * conv_norm_forward; x, w, b, gamma, beta and out are caller-owned device
 * pointers.  The call is asynchronous on cuda_stream.
 *
 * Limits and errors:
 *  - the scratch a problem needs is the workspace conv_norm_plan_create would
 *    allocate for it, less the plan's 256-byte flag (conv_norm_workspace_bytes
 *    of such a plan, minus 256); more than 4 MiB returns CN_ERR_UNSUPPORTED.
 *    It depends on the kernel the problem runs on: small batches (up to about
 *    16 M multiply-adds) 16 bytes per (sample, channel, row split) plus 4
 *    bytes per (sample, normalization group); the tensor-core kernel 16 bytes
 *    per (sample, item, channel) plus 4 bytes per sample (1 MB for N=512,
 *    16x32x32, k=4: 8 items a sample); the CUDA-core kernel 24 bytes per
 *    (sample, row chunk, channel) plus 4 bytes per sample;
 *  - other problem kinds return CN_ERR_UNSUPPORTED; malformed descriptors or
 *    null/misaligned pointers CN_ERR_INVALID_ARG; a failed launch CN_ERR_CUDA;
 *  - a bounded device wait that gives up is recorded in a flag of the
 *    library's device globals, which conv_norm_plan_check_device(NULL,
 *    stream) reads and clears.
 * All calls share the one array: calls whose work overlaps on the GPU (two
 * streams, or two host threads) race and give wrong results; order them.
 * Each call clears the tickets it needs before its kernel runs.
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress (device current at the time of the call); make that
 * first call before any stream capture on that device.
 */
int conv_norm_forward_noalloc(const conv_norm_desc *desc, const float *x, const float *w,
                              const float *b, const float *gamma, const float *beta,
                              float *out, void *cuda_stream);

/* ---- backward pass ----------------------------------------------------------- */

typedef struct conv_norm_bwd_plan_s *conv_norm_bwd_plan;

/* Cites: no page passage: the pages implement the forward only (l2_p27 notes
 * that its problem asks for no gradient).  The backward is the derivative of
 * the forward each page states (the chain rule through its layers).
 * A backward plan for the full-output 2-D block: desc with conv = CN_CONV2D
 * or CN_CONVT2D (any groups the forward takes), act none / HardSwish / GELU,
 * any norm, any post scale, red = CN_RED_NONE, N >= 1, and a forward that the
 * library supports for desc (the adjoint conv, C_in and C_out swapped, must
 * also be one: (C_in / groups) % 4 == 0).  Allocates, on the CURRENT device,
 * a workspace of N C_out H_out W_out floats (the conv output, then its
 * gradient) plus small per-plane and per-split buffers, and two forward plans
 * (the conv alone and its adjoint); for a dense Conv2d that fits the
 * tensor-core path also a third (the adjoint as a Conv2d of the gradient
 * padded by k - 1 zeros, with its output channels padded to a multiple of
 * 128) and that plan's input and output, about three more copies of the
 * gradient's size.
 * Errors: CN_ERR_INVALID_ARG, CN_ERR_UNSUPPORTED, CN_ERR_CUDA, CN_ERR_ALLOC. */
int conv_norm_bwd_plan_create(const conv_norm_desc *desc, conv_norm_bwd_plan *out_plan);

/* Cites: as conv_norm_bwd_plan_create.
 * Gradients of a loss L through the block, given dout = dL/d(out) (the
 * forward output's shape, NCHW fp32, 16-byte aligned) and the forward's
 * inputs x, w, b, gamma, beta (layouts as conv_norm_forward):
 *   dx (x's shape, 16-byte aligned), dw (w's shape), db (C_out; required
 *   iff has_bias), dgamma and dbeta (C_out; required iff the norm is affine,
 *   NULL otherwise).  All device pointers, written in full.
 * With A the conv output, y = act(A), mu and r = 1/sqrt(var + eps) per
 * (sample, norm group), xh = (y - mu) r and s the post scale:
 *   dy = r (s gamma dout - mean(s gamma dout) - xh mean(s gamma dout xh)),
 *   dA = dy act'(A) (HardSwish' = 0 / a/3 + 1/2 / 1 below -3 / on [-3, 3] /
 *   above 3), dgamma = s sum dout xh, dbeta = s sum dout, db = sum dA,
 *   dx = the adjoint conv of dA, dw = the correlation of dA with x.
 * Asynchronous on cuda_stream; allocates nothing; deterministic (fixed-order
 * sums).  Calls on one plan must not overlap.  Errors: CN_ERR_INVALID_ARG
 * (NULL plan or tensor, a gradient pointer given or missing against desc,
 * misalignment), CN_ERR_CUDA. */
int conv_norm_backward(conv_norm_bwd_plan plan, const float *x, const float *w, const float *b,
                       const float *gamma, const float *beta, const float *dout, float *dx,
                       float *dw, float *db, float *dgamma, float *dbeta, void *cuda_stream);

/* Cites: as conv_norm_bwd_plan_create.
 * Bytes of device memory the backward plan holds (its workspace and its
 * forward plans'); 0 for NULL. */
size_t conv_norm_bwd_workspace_bytes(conv_norm_bwd_plan plan);

/* Cites: as conv_norm_plan_check_device.
 * Synchronizes cuda_stream and reads and clears the error flags of the
 * backward plan's forward plans and of its own tensor-core kernels (CN_OK,
 * CN_ERR_TIMEOUT, CN_ERR_DEVICE_CHECK, CN_ERR_CUDA); CN_ERR_INVALID_ARG for
 * NULL. */
int conv_norm_bwd_check_device(conv_norm_bwd_plan plan, void *cuda_stream);

/* Cites: as conv_norm_plan_destroy.
 * Frees the backward plan and its forward plans; NULL is ignored; no call on
 * the plan may still be running. */
void conv_norm_bwd_plan_destroy(conv_norm_bwd_plan plan);

#ifdef __cplusplus
}
#endif
#endif /* CONV_NORM_H */
