/* fnospec.h -- C ABI of libfnospec, the FNO 2D spectral-convolution layer on one
 * GPU (sm_103a).
 *
 * The layer (TurboFNO: FFT-GEMM-iFFT fused operator page, sections 1 and 2.2;
 * orthonormal scaling per its section 3.1):
 *
 *   X = rfft2(x, norm="ortho")                    x : real [B][Cin][H][W]
 *   Z[b,o,k1,k2] = sum_i X[b,i,k1,k2] * W[i,o,r,k2]   on the retained modes
 *        k1 in R1 = {0..m1-1} U {H-m1..H-1},  k2 in R2 = {0..m2-1}
 *   y = irfft2(Z, s=(H, W), norm="ortho")         y : real [B][Cout][H][W]
 *
 * with every bin outside R1 x R2 zero.  The complex-to-real row step keeps only
 * the real part of the k2 = 0 bin (and of the k2 = W/2 bin when m2 = W/2 + 1),
 * as the half-spectrum (W/2 + 1 wide) convention of the FFT operator-optimisation
 * page (lpnh.cn/news/2688017, section 2.2) implies.
 *
 * Layouts (all dense, row-major, no padding, complex = interleaved re, im float):
 *   x  float     [B][Cin][H][W]
 *   w  complex64 [Cin][Cout][2*m1][m2]   retained row r: k1 = r for r < m1,
 *                                        k1 = H - 2*m1 + r for r >= m1
 *   y  float     [B][Cout][H][W]
 *   X  complex64 [B][Cin][2*m1][m2]      (stage entry points only)
 *   Z  complex64 [B][Cout][2*m1][m2]     (stage entry points only)
 *
 * Conventions shared by every entry point:
 *   - Tensor pointers are DEVICE pointers (cudaMalloc / caching allocators /
 *     managed memory) owned by the caller; the library never frees them.  Each
 *     must be 16-byte aligned.  Unregistered host memory is rejected.
 *   - Out-of-place only: outputs must not overlap inputs.
 *   - Work is enqueued on the given stream and returns without synchronising
 *     and without allocating (except the one-shot fno_spectral_conv2d, which
 *     caches a plan and a workspace on its first call per shape and stream).
 *   - Supported shapes: H and W in [2, 4096] (powers of two run on FFT kernels,
 *     other sizes on direct DFTs of the retained bins); 1 <= m1, 2*m1 <= H;
 *     1 <= m2 <= W/2 + 1; B, Cin, Cout >= 1; every tensor below 2^31 elements.
 *   - Errors detected on the host are returned immediately and nothing is
 *     enqueued.  Errors detected inside kernels set a word in device memory
 *     that fno_get_device_status reads and clears.
 *   - A runtime error already pending on the calling host thread (one that
 *     cudaPeekAtLastError would return, such as a launch the runtime rejected
 *     before the call) makes every entry point that enqueues work return
 *     FNO_ERR_CUDA before enqueuing anything.  The error is left pending: it
 *     belongs to the caller, who reads and clears it with cudaGetLastError.
 */
#ifndef FNOSPEC_H_
#define FNOSPEC_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FNO_OK = 0,
    FNO_ERR_INVALID_ARG = 1, /* null/misaligned/host pointer, bad size, aliasing */
    FNO_ERR_UNSUPPORTED = 2, /* shape or precision outside what is built      */
    FNO_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed     */
    FNO_ERR_WORKSPACE = 4,   /* workspace smaller than fno_plan_workspace_size  */
    FNO_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up              */
    FNO_ERR_DEVICE = 6       /* a kernel flagged an internal error              */
} fno_status_t;

typedef enum {
    /* fp32 storage and fp32 FMA for every stage. */
    FNO_PREC_FP32 = 0,
    /* Mode contraction on tcgen05 tensor cores with TF32 operands and fp32
     * accumulation when Cin >= 32 and Cout >= 32 (fp32 FMA otherwise);
     * transforms stay fp32.  Expected relative L2 error ~1e-3. */
    FNO_PREC_TF32 = 1,
    /* As FNO_PREC_TF32 but each operand is split into a TF32 high part and a
     * TF32 residual and three products are accumulated (hi*hi + hi*lo + lo*hi),
     * which recovers fp32-level accuracy on the tensor cores. */
    FNO_PREC_3XTF32 = 2
} fno_precision_t;

typedef struct fno_plan_s* fno_plan_t;

/* Human-readable name of a status code (static storage, never NULL).
 * The codes separate the failure classes the FFT operator-optimisation page
 * (lpnh.cn/news/2688017) tells apart when it debugs such an operator: section
 * 6.1 and the symptom table that closes section 6.2 (wrong arguments and
 * out-of-range layouts, unsupported sizes, runtime failures), plus the
 * device-side timeouts of this library's bounded waits. */
const char* fno_status_string(fno_status_t status);

/* Create a plan for one shape on the CURRENT device.  Host-side call: validates
 * the shape, chooses the kernels, builds the twiddle tables (computed in double
 * on the host, rounded once to float) and allocates them plus a device error
 * word.  *plan is set to NULL on failure.
 * Source for caching plans per shape: FFT operator-optimisation page, section
 * 5.3 (reuse plans and workspace across calls; query the workspace size once). */
fno_status_t fno_plan_create(fno_plan_t* plan, int B, int Cin, int Cout, int H, int W,
                             int m1, int m2, fno_precision_t prec);

/* Create a plan for the 1D layer over sequences of L points on the CURRENT
 * device: y = irfft(Z, n=L, norm="ortho") with X = rfft(x, norm="ortho") and
 * Z[b,o,k] = sum_i X[b,i,k] w[i,o,k] for the m retained modes k < m (the
 * others zero; C2R drops the imaginary part of the k = 0 and k = L/2 bins).
 * Sources: FFT operator-optimisation page, section 3.2 (the transform over a
 * sequence, a learned complex factor per frequency, the inverse back), with the
 * per-mode channel contraction of the TurboFNO page, section 2.2, in one
 * dimension.  Shapes: x float [B][Cin][L], w complex64 [Cin][Cout][m],
 * y float [B][Cout][L]; 2 <= L <= 4096, 1 <= m <= L/2 + 1 (pruned FFTs for
 * L = 512, 1024, 2048, 4096 with m <= 64, direct DFTs otherwise).  The returned plan serves every call taking a plan (execute, the
 * three stages, the backward, the block epilogue), with H = 1, W = L, and
 * 2*m1*m2 read as m wherever a size is stated.  Errors as fno_plan_create. */
fno_status_t fno_plan_create_1d(fno_plan_t* plan, int B, int Cin, int Cout, int L, int m,
                                fno_precision_t prec);

/* Bytes of device workspace fno_plan_execute needs (may be 0): the retained
 * spectra X and Z (and, on the shape-generic path, the row/column
 * intermediate).  Query once per plan and allocate once, as the FFT
 * operator-optimisation page, section 5.3, does with cuFFT's workspace size
 * query.  *bytes is written on FNO_OK; FNO_ERR_INVALID_ARG for NULL arguments. */
fno_status_t fno_plan_workspace_size(fno_plan_t plan, size_t* bytes);

/* Number of kernel launches one fno_plan_execute enqueues. */
fno_status_t fno_plan_launch_count(fno_plan_t plan, int* launches);

/* Copy a short description of the chosen kernels into buf (NUL-terminated). */
fno_status_t fno_plan_describe(fno_plan_t plan, char* buf, size_t len);

/* Describe kernel `index` (0-based, < fno_plan_launch_count) of one execute:
 * its name (NUL-terminated, truncated to name_len), the algorithmic bytes it
 * must move (compulsory reads + writes of its inputs and outputs, each once) and
 * its algorithmic floating-point operations.  Any output pointer may be NULL. */
fno_status_t fno_plan_kernel_info(fno_plan_t plan, int index, char* name, size_t name_len,
                                  size_t* bytes, size_t* flops);

/* Arm per-kernel timing for later executes: events[0] is recorded on the stream
 * before the first kernel and events[k + 1] after kernel k, so count must be
 * fno_plan_launch_count + 1.  The caller creates and owns the events.  Pass
 * events = NULL (count 0) to disarm.  Not thread-safe against a concurrent
 * execute of the same plan. */
fno_status_t fno_plan_record_events(fno_plan_t plan, cudaEvent_t* events, int count);

/* Run the whole layer y = irfft2(mix(rfft2(x), w)) on stream s: the fused
 * FFT -> per-mode contraction -> inverse FFT operator of the TurboFNO page,
 * sections 1 and 2.2 (low modes kept, every other bin zero, the complex
 * product per retained mode), with the orthonormal scale of its section 3.1,
 * as the stages a1-a5 in this header's preamble define it.
 * x: float [B][Cin][H][W]; w: complex64 [Cin][Cout][2*m1][m2];
 * y: float [B][Cout][H][W]; workspace: device buffer of at least
 * fno_plan_workspace_size bytes (NULL allowed when that size is 0), owned by the
 * caller and not used concurrently by another call. */
fno_status_t fno_plan_execute(fno_plan_t plan, const float* x, const void* w, float* y,
                              void* workspace, size_t workspace_bytes, cudaStream_t s);

/* Activation of the FNO block (fno_block_execute / fno_block_epilogue). */
typedef enum {
    FNO_ACT_NONE = 0, /* identity */
    FNO_ACT_GELU = 1  /* v/2 * (1 + erf(v / sqrt(2))), erf from the CUDA math library */
} fno_activation_t;

/* The FNO block around the spectral layer, in place over y:
 *   y[b][o][h][w] <- act(y[b][o][h][w] + bias[o] + sum_i w_pw[o][i] * x[b][i][h][w])
 * with y on entry the spectral layer's output for x (fno_plan_execute), w_pw the
 * 1x1 convolution weights float [Cout][Cin] (PyTorch's [Cout, Cin, 1, 1]), bias
 * float [Cout] or NULL (no bias).  This is the pointwise branch and activation
 * that the neural-operator block adds to the spectral path (the FFT operator-
 * optimisation page, section 5.2, fuses such a branch-add and GELU into the
 * last stage of its FFT convolution).  Needs Cin <= 256 and H*W a multiple of
 * 4 (FNO_ERR_UNSUPPORTED otherwise).  y must not overlap x, w_pw or bias.  Stream-ordered, no host
 * synchronisation, no allocation. */
fno_status_t fno_block_epilogue(fno_plan_t plan, const float* x, const float* w_pw,
                                const float* bias, fno_activation_t act, float* y,
                                cudaStream_t s);

/* fno_plan_execute followed by fno_block_epilogue: one FNO block
 *   y = act(layer(x, w) + w_pw x + bias)
 * with the plan's workspace (fno_plan_workspace_size bytes). */
fno_status_t fno_block_execute(fno_plan_t plan, const float* x, const void* w, const float* w_pw,
                               const float* bias, fno_activation_t act, float* y,
                               void* workspace, size_t workspace_bytes, cudaStream_t s);

/* Backward of the layer for a real loss L, given gy = dL/dy (float
 * [B][Cout][H][W]), on stream s:
 *   gx = dL/dx, float [B][Cin][H][W]: the layer applied to gy with w conjugated
 *        and transposed per mode (w^H[o][i] = conj(w[i][o]));
 *   gw = dL/dRe(w) + i dL/dIm(w), complex64 [Cin][Cout][2*m1][m2]:
 *        gw[i][o][r][k2] = c(k2) * sum_b conj(X[b][i][r][k2]) * G[b][o][r][k2],
 *        X and G the forward modes (fno_forward_modes) of x and of gy, c = 1 for
 *        k2 = 0 and k2 = W/2 and 2 for every other column (the Hermitian
 *        weights of the complex-to-real step).
 * Derived by differentiating the layer defined in the TurboFNO page, sections
 * 2.2 and 3.1 (truncated orthonormal rfft2, per-mode product, irfft2).
 * Either gx or gw may be NULL (that gradient is skipped, and x, respectively w,
 * may then be NULL too); at least one must be given.  Uses the plan's workspace
 * (fno_plan_workspace_size bytes, the same as the forward).  Outputs must not
 * overlap x, w, gy, each other or the workspace (FNO_ERR_INVALID_ARG).  The
 * backward computes in fp32 whatever the plan's precision. */
fno_status_t fno_plan_backward(fno_plan_t plan, const float* x, const void* w, const float* gy,
                               float* gx, void* gw, void* workspace, size_t workspace_bytes,
                               cudaStream_t s);

/* Release the plan's tables and error word (the counterpart of the plan cache
 * and reuse of the FFT operator-optimisation page, section 5.3: a plan lives as
 * long as its shape is in use).  Safe on NULL; always FNO_OK.  The caller must
 * make sure no work that uses the plan is still running. */
fno_status_t fno_plan_destroy(fno_plan_t plan);

/* One-shot form of fno_plan_execute with FNO_PREC_FP32: the layer of the
 * TurboFNO page (sections 1, 2.2 and 3.1) behind the plan and workspace cache
 * that the FFT operator-optimisation page, section 5.3, prescribes (plans and
 * workspaces keyed by shape, created on the first request and reused).  Keeps
 * an internal cache of plans keyed by (device, shape) and of workspaces keyed by
 * (device, shape, stream); the first call for a key allocates (cudaMalloc), so
 * make it before any stream capture.  Calls with the same key must not overlap
 * on the GPU (they share the workspace).  Errors: as fno_plan_create and
 * fno_plan_execute. */
fno_status_t fno_spectral_conv2d(const float* x, const void* w, float* y, int B, int Cin,
                                 int Cout, int H, int W, int m1, int m2, cudaStream_t s);

/* Free every cached plan and workspace of fno_spectral_conv2d (synchronises the
 * device first). */
fno_status_t fno_release_cache(void);

/* Stage a1+a2 (forward row and column transforms, pruned to the retained modes,
 * orthonormal scale applied): x float [B][Cin][H][W] -> X complex64
 * [B][Cin][2*m1][m2].  Needs the plan's workspace. */
fno_status_t fno_forward_modes(fno_plan_t plan, const float* x, void* X, void* workspace,
                               size_t workspace_bytes, cudaStream_t s);

/* Stage a3 (per-mode complex channel contraction): X complex64 [B][Cin][2*m1][m2],
 * w complex64 [Cin][Cout][2*m1][m2] -> Z complex64 [B][Cout][2*m1][m2].
 * Source: TurboFNO page, section 2.2 ((a+bi)(c+di) = (ac-bd) + (ad+bc)i per
 * retained mode). */
fno_status_t fno_mix_modes(fno_plan_t plan, const void* X, const void* w, void* Z,
                           cudaStream_t s);

/* Stage a4+a5 (zero-filled inverse column transform, complex-to-real row
 * transform, orthonormal scale applied): Z complex64 [B][Cout][2*m1][m2] ->
 * y float [B][Cout][H][W].  Needs the plan's workspace. */
fno_status_t fno_inverse_modes(fno_plan_t plan, const void* Z, float* y, void* workspace,
                               size_t workspace_bytes, cudaStream_t s);

/* The whole layer (same arguments, shapes and result as fno_spectral_conv2d,
 * fp32 path) for callers that cannot allocate device memory: this entry point
 * calls no cudaMalloc, cudaFree or other allocating routine.  The pages have no
 * counterpart; it exists for hosts that own every allocation themselves.  It
 * runs the shape-generic transform kernels (FFTs for powers of two, direct DFTs
 * otherwise) and the per-thread fp32 contraction, none of which waits on the
 * device, so there is no device status to query for it.
 * Its scratch (twiddle tables, error word, the spectra X and Z, the row/column
 * intermediate) lives in one static device array of 16 MiB that every GPU
 * loading the library holds until exit; shapes whose scratch does not fit
 * (2*m1*m2*8*B*(Cin+Cout) + 8*B*max(Cin,Cout)*H*m2 + 8*(H+W) bytes, plus
 * alignment) return FNO_ERR_UNSUPPORTED before anything is enqueued.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) while that device is current; make that first call
 * before any stream capture.  All calls share the array and each call
 * re-initialises what it reads, so calls that overlap on the GPU (different
 * streams, or several host threads) race and must be serialised by the
 * caller. */
fno_status_t fno_spectral_conv2d_noalloc(const float* x, const void* w, float* y, int B,
                                         int Cin, int Cout, int H, int W, int m1, int m2,
                                         cudaStream_t s);

/* Choose how fno_plan_execute runs the layer: enable != 0 runs the whole layer
 * as ONE cooperative launch (forward transforms, per-mode contraction and
 * inverse transforms as three phases of one persistent grid, separated by
 * grid-wide barriers; the retained spectra cross CTAs through the plan's
 * workspace inside the launch), enable = 0 as the regular three launches.  This
 * is the fused FFT -> GEMM -> iFFT operator of the TurboFNO page, sections 1
 * and 2.1-2.3 (no launch between the stages).  Served for square planes
 * H = W in {32, 64, 128, 256} with batch up to 16 (FNO_ERR_UNSUPPORTED
 * otherwise).  Plans start with it off: the three launches, which overlap
 * one another's start and end through programmatic dependent launch, are the
 * faster form at every shape it serves.  Host-only; changes
 * fno_plan_launch_count, so call it before fno_plan_record_events
 * (FNO_ERR_INVALID_ARG while events are armed, for a NULL plan or for a
 * backward's internal plan).  The grid barriers wait at most one second; a
 * wait that runs out is reported by fno_get_device_status as FNO_ERR_TIMEOUT.
 * Calls that use the same plan must not overlap on the GPU. */
fno_status_t fno_plan_set_single_launch(fno_plan_t plan, int enable);

/* Range-checked builds (libfnospec_debug.so, compiled with FNO_DEBUG): every
 * global store of the kernels on the execute, stage, backward and single-launch
 * paths is checked against the output ranges of its launch; a store outside
 * them is skipped (nothing is written, nothing traps) and bit 0 of the plan's
 * device error word is set, so fno_get_device_status returns FNO_ERR_DEVICE.
 * This test hook shortens the first output range of every launch of the plan
 * (and of its backward) by `bytes`, so that the last outputs count as out of
 * range without any access leaving its tensor.  bytes = 0 restores the true
 * ranges.  Returns FNO_ERR_UNSUPPORTED in release builds (no checks compiled),
 * FNO_ERR_INVALID_ARG for a NULL plan.  Host-only.  A stand-in for a memory
 * checker where none can run; the pages have no counterpart. */
fno_status_t fno_plan_debug_bounds_margin(fno_plan_t plan, size_t bytes);

/* Synchronise stream s, read and clear the plan's device error word.  Returns
 * FNO_OK, FNO_ERR_TIMEOUT or FNO_ERR_DEVICE (or FNO_ERR_CUDA if the copy fails).
 * This is the stage-by-stage fault check of the FFT operator-optimisation page,
 * sections 6.1 and 6.4 (find which step went wrong before looking at numbers),
 * for faults that only the kernels can see: a bounded wait that gave up.  The
 * plan's error word is shared with its backward; the caller owns s. */
fno_status_t fno_get_device_status(fno_plan_t plan, cudaStream_t s);

/* Test hook for the failure path: with enable != 0, every bounded wait inside
 * this plan's kernels (and its backward's) gives up at once, as if its time
 * limit had run out.  The kernel sets
 * FNO_DEVERR_TIMEOUT in the error word, lets its own asynchronous copies and
 * tensor-core work finish, frees what it holds and returns, so the context
 * stays usable; outputs of such calls are void and the next
 * fno_get_device_status returns FNO_ERR_TIMEOUT.  Kernels without waits
 * (the shape-generic transforms, the direct-DFT steps other than the inverse
 * rows, the short-row forward) are not affected.  enable = 0 restores normal
 * operation.  Host-synchronous: it synchronises the device before it writes
 * the flag, so call it between calls,
 * never during stream capture.  Returns FNO_ERR_INVALID_ARG for a NULL plan or
 * another current device, FNO_ERR_CUDA if the device copy fails.  A test hook
 * of this library: no page defines it. */
fno_status_t fno_plan_debug_force_timeout(fno_plan_t plan, int enable);

#ifdef __cplusplus
}
#endif

#endif /* FNOSPEC_H_ */
