// noalloc.cu -- fno_spectral_conv2d_noalloc: the whole layer without any
// device allocation, for callers that cannot call cudaMalloc (for example code
// that runs under a framework which owns every allocation, a real-time loop
// that must not enter the driver's allocator, or a plugin whose host
// application forbids allocation after start-up).
//
// Everything the regular path keeps in a plan or in a caller-provided workspace
// (the two twiddle tables, the device error word, and the intermediate
// spectra X, Z and T) lives in one file-scope __device__ array of
// kNoAllocScratchBytes.  Every GPU that loads this library holds that array
// until the process exits.  The caller still provides x, w and y.
#include <cmath>
#include <mutex>

#include "internal.h"

namespace {

// 16 MiB: enough for small layers (for example B=8, C=32, 64x64, m=16 needs
// about 4 MiB); larger shapes are rejected with FNO_ERR_UNSUPPORTED.
constexpr size_t kNoAllocScratchBytes = 16u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Host-side device addresses of g_noalloc_scratch, one per device, looked up
// once with cudaGetSymbolAddress while that device is current.  The symbol
// itself is only a host-side stand-in and must never be passed to a kernel.
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// x, w and y must be memory the GPU can reach (device, managed, or mapped
// host memory); unregistered host memory would fault, so it is refused.
bool reachable(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeUnregistered) return false;
    if (a.type == cudaMemoryTypeHost && a.devicePointer == nullptr) return false;
    return true;
}

// The error word in the scratch is cleared by every call but never read back:
// no status query covers this entry point.  Its stages must therefore stay on
// kernels that cannot fail on the device (the shape-generic and direct-DFT
// transforms and the per-thread contraction have no waits and no device-side
// checks); a kernel with bounded waits would report a timeout nowhere.  The
// direct-DFT pass kernels, which wait for their streamed twiddle tiles, run
// only with a plan's tables (g_irows, g_frows), which the plan below leaves
// null, and the column steps form their twiddles in the kernel without g_cols.
//
// Fills both twiddle tables e^{+2 pi i j / N} (double sincospi, rounded once
// to float) and clears the error word and the debug-flag word after it.  Nothing else in the scratch needs to
// start at zero: X, Z and T are fully written before they are read.
__global__ void noalloc_setup_kernel(float2* tw_h, int H, float2* tw_w, int W, unsigned* err) {
    const int n = H + W;
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x) {
        double s, c;
        if (j < H) {
            sincospi(2.0 * (double)j / (double)H, &s, &c);
            tw_h[j] = make_float2((float)c, (float)s);
        } else {
            const int k = j - H;
            sincospi(2.0 * (double)k / (double)W, &s, &c);
            tw_w[k] = make_float2((float)c, (float)s);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        err[0] = 0u;  // error bits
        err[1] = 0u;  // debug flags (none)
    }
}

}  // namespace

extern "C" fno_status_t fno_spectral_conv2d_noalloc(const float* x, const void* w, float* y,
                                                    int B, int Cin, int Cout, int H, int W,
                                                    int m1, int m2, cudaStream_t s) {
    // Shape rules of the regular path.
    if (B < 1 || Cin < 1 || Cout < 1 || H < 1 || W < 1 || m1 < 1 || m2 < 1)
        return FNO_ERR_INVALID_ARG;
    if (2LL * m1 > H || (long long)m2 > W / 2 + 1) return FNO_ERR_INVALID_ARG;
    // any size in [2, 4096]: powers of two take the shape-generic FFT stages,
    // other sizes the direct-DFT stages (the same [planes][H][m2] intermediate)
    if (H < 2 || W < 2 || H > 4096 || W > 4096) return FNO_ERR_UNSUPPORTED;
    if (!x || !w || !y) return FNO_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) |
         reinterpret_cast<uintptr_t>(y)) % 16)
        return FNO_ERR_INVALID_ARG;
    // an error left pending by the caller's earlier runtime calls is reported
    // before anything is enqueued, and left pending (as the plan entry points do)
    if (cudaPeekAtLastError() != cudaSuccess) return FNO_ERR_CUDA;
    if (!reachable(x) || !reachable(w) || !reachable(y)) return FNO_ERR_INVALID_ARG;

    // Scratch layout: tw_h | tw_w | err | X | Z | T, each 256-byte aligned.
    const size_t nm = 2ull * m1 * m2;
    const size_t planes = (size_t)B * (Cin > Cout ? Cin : Cout);
    size_t off = 0;
    const size_t off_th = off; off = align256(off + 8ull * H);
    const size_t off_tw = off; off = align256(off + 8ull * W);
    const size_t off_err = off; off = align256(off + 2 * sizeof(unsigned));
    const size_t off_X = off; off = align256(off + 8ull * B * Cin * nm);
    const size_t off_Z = off; off = align256(off + 8ull * B * Cout * nm);
    const size_t off_T = off; off = align256(off + 8ull * planes * H * m2);
    if (off > kNoAllocScratchBytes) return FNO_ERR_UNSUPPORTED;  // beyond the static scratch

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FNO_ERR_CUDA;
    unsigned char* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_ptr[dev]) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
                return FNO_ERR_CUDA;
            // shared-memory limits of the stage kernels (no allocation involved)
            if (stages_generic_init() != cudaSuccess) return FNO_ERR_CUDA;
            g_scratch_ptr[dev] = ptr;
        }
        base = static_cast<unsigned char*>(g_scratch_ptr[dev]);
    }

    // A plan on the stack that points into the scratch; the stage launchers
    // read only its shape fields and these pointers.
    fno_plan_s p{};
    p.B = B; p.Cin = Cin; p.Cout = Cout; p.H = H; p.W = W; p.m1 = m1; p.m2 = m2;
    p.nm = (int)nm;
    p.prec = FNO_PREC_FP32;
    p.device = dev;
    p.scale = (float)(1.0 / std::sqrt((double)H * (double)W));
    p.tw_h = reinterpret_cast<float2*>(base + off_th);
    p.tw_w = reinterpret_cast<float2*>(base + off_tw);
    p.err = reinterpret_cast<unsigned*>(base + off_err);
    float2* X = reinterpret_cast<float2*>(base + off_X);
    float2* Z = reinterpret_cast<float2*>(base + off_Z);
    float2* T = reinterpret_cast<float2*>(base + off_T);

    const int n = H + W;
    noalloc_setup_kernel<<<(n + 255) / 256, 256, 0, s>>>(p.tw_h, H, p.tw_w, W, p.err);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_forward_modes(p, x, X, T, s, nullptr);
    if (e == cudaSuccess) e = launch_mix_modes(p, X, static_cast<const float2*>(w), Z, s, nullptr);
    if (e == cudaSuccess) e = launch_inverse_modes(p, Z, y, T, s, nullptr);
    return e == cudaSuccess ? FNO_OK : FNO_ERR_CUDA;
}
