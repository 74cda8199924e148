// fnospec.cu -- host side of libfnospec: argument validation, plans, twiddle
// tables, workspace layout, the one-shot plan cache and the device error word.
// The declarations and their contracts are in include/fnospec.h.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "internal.h"

namespace {

constexpr int kMaxN = 4096;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

fno_status_t validate_shape(int B, int Cin, int Cout, int H, int W, int m1, int m2) {
    if (B < 1 || Cin < 1 || Cout < 1 || H < 1 || W < 1 || m1 < 1 || m2 < 1)
        return FNO_ERR_INVALID_ARG;
    if (2LL * m1 > H || (long long)m2 > W / 2 + 1) return FNO_ERR_INVALID_ARG;
    // powers of two run on the FFT kernels, other sizes on direct DFTs
    if (H < 2 || W < 2 || H > kMaxN || W > kMaxN) return FNO_ERR_UNSUPPORTED;
    const long long lim = (1LL << 31) - 1;
    if ((long long)B * Cin * H * W > lim || (long long)B * Cout * H * W > lim ||
        (long long)Cin * Cout * 2 * m1 * m2 > lim)
        return FNO_ERR_UNSUPPORTED;
    if ((long long)B * Cin > 65535 * 1024LL || (long long)B * Cout > 65535 * 1024LL)
        return FNO_ERR_UNSUPPORTED;
    return FNO_OK;
}

fno_status_t validate_shape_1d(int B, int Cin, int Cout, int L, int m) {
    if (B < 1 || Cin < 1 || Cout < 1 || L < 1 || m < 1) return FNO_ERR_INVALID_ARG;
    if ((long long)m > L / 2 + 1) return FNO_ERR_INVALID_ARG;
    if (L < 2 || L > kMaxN) return FNO_ERR_UNSUPPORTED;
    const long long lim = (1LL << 31) - 1;
    if ((long long)B * Cin * L > lim || (long long)B * Cout * L > lim ||
        (long long)Cin * Cout * m > lim)
        return FNO_ERR_UNSUPPORTED;
    return FNO_OK;
}

// A pointer the kernels can dereference: device or managed memory, or host
// memory that is registered/pinned and mapped (the GPU reaches it through UVA).
// Unregistered host memory would fault the GPU, so it is rejected here.
fno_status_t check_ptr(const void* p, bool required) {
    if (!p) return required ? FNO_ERR_INVALID_ARG : FNO_OK;
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return FNO_ERR_INVALID_ARG;
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error
        return FNO_ERR_INVALID_ARG;
    }
    if (attr.type == cudaMemoryTypeUnregistered) return FNO_ERR_INVALID_ARG;
    if (attr.type == cudaMemoryTypeHost && attr.devicePointer == nullptr) return FNO_ERR_INVALID_ARG;
    return FNO_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const char* pa = static_cast<const char*>(a);
    const char* pb = static_cast<const char*>(b);
    return pa < pb + nb && pb < pa + na;
}

fno_status_t check_device(const fno_plan_s* p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FNO_ERR_CUDA;
    return dev == p->device ? FNO_OK : FNO_ERR_INVALID_ARG;
}

// An error left pending by earlier runtime calls of this host thread (for
// example a kernel launch the runtime rejected, such as one with an invalid
// block size) belongs to the caller.  Entry points that enqueue work report it
// as FNO_ERR_CUDA before enqueuing anything and leave it pending, so the caller
// still reads it with cudaGetLastError (a sticky error of the context is
// reported the same way).
fno_status_t check_no_pending_error() {
    return cudaPeekAtLastError() == cudaSuccess ? FNO_OK : FNO_ERR_CUDA;
}

// e^{+2 pi i j / N} for j in [0, N), evaluated in double and rounded once.
std::vector<float2> twiddles(int N) {
    std::vector<float2> t(N);
    const double two_pi = 6.283185307179586476925286766559005768;
    for (int j = 0; j < N; ++j) {
        const double a = two_pi * (double)j / (double)N;
        t[j] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
    return t;
}

size_t x_bytes(const fno_plan_s* p) { return 4ull * p->B * p->Cin * p->H * p->W; }
size_t y_bytes(const fno_plan_s* p) { return 4ull * p->B * p->Cout * p->H * p->W; }
size_t w_bytes(const fno_plan_s* p) { return 8ull * p->Cin * p->Cout * p->nm; }
size_t X_bytes(const fno_plan_s* p) { return 8ull * p->B * p->Cin * p->nm; }
size_t Z_bytes(const fno_plan_s* p) { return 8ull * p->B * p->Cout * p->nm; }

fno_status_t check_ws(const fno_plan_s* p, const void* ws, size_t ws_bytes) {
    if (ws_bytes < p->ws_bytes) return FNO_ERR_WORKSPACE;
    if (p->ws_bytes == 0) return FNO_OK;
    return check_ptr(ws, true);
}

void set_kernel(fno_plan_s* p, int k, const char* name, size_t bytes, size_t flops) {
    std::snprintf(p->kernels[k].name, sizeof(p->kernels[k].name), "%s", name);
    p->kernels[k].bytes = bytes;
    p->kernels[k].flops = flops;
}

const char* mix_name(const fno_plan_s* p) {
    if (p->mix_path == 2) return p->tc_split == 3 ? "mix_tc_3xtf32" : "mix_tc_tf32";
    if (p->mix_path == 5) return p->tc_split == 3 ? "mix_tcm_3xtf32" : "mix_tcm_tf32";
    if (p->mix_path == 3) return p->adjoint ? "mix_wide_adj" : "mix_wide";
    if (p->mix_path == 4) return "mix_adj_fma";
    return p->mix_path == 1 ? "mix_tma" : "mix_fma";
}

double fft_flops(double L) { return 5.0 * L * std::log2(L); }

// Kernel list of the shape-generic path (stages_generic.cu + mix_fma.cu).
void describe_generic(fno_plan_s* p) {
    const size_t Pi = (size_t)p->B * p->Cin, Po = (size_t)p->B * p->Cout;
    const size_t Ti = 8ull * Pi * p->H * p->m2, To = 8ull * Po * p->H * p->m2;
    set_kernel(p, 0, "fwd_rows", x_bytes(p) + Ti, (size_t)(fft_flops(p->W) * Pi * p->H / 2));
    set_kernel(p, 1, "fwd_cols", Ti + X_bytes(p), (size_t)(fft_flops(p->H) * Pi * p->m2));
    set_kernel(p, 2, mix_name(p), X_bytes(p) + w_bytes(p) + Z_bytes(p),
               8ull * p->B * p->Cin * p->Cout * p->nm);
    set_kernel(p, 3, "inv_cols", Z_bytes(p) + To, (size_t)(fft_flops(p->H) * Po * p->m2));
    set_kernel(p, 4, "inv_rows", To + y_bytes(p), (size_t)(fft_flops(p->W) * Po * p->H / 2));
    p->launches = 5;
}

// Kernel list of the fused path (stages_fused.cu + mix_fma.cu).
void describe_fused(fno_plan_s* p) {
    const size_t Pi = (size_t)p->B * p->Cin, Po = (size_t)p->B * p->Cout;
    int k = 0;
    if (p->P > 1) set_kernel(p, k++, "zero_X", X_bytes(p), 0);
    const double fl_f = Pi * (fft_flops(p->W) * p->H / 2 + fft_flops(p->R) * p->m2 * p->P);
    const double fl_i = Po * (fft_flops(p->W) * p->H / 2 + fft_flops(p->Ri) * p->m2 * p->Pi);
    set_kernel(p, k++, "fwd_fused", x_bytes(p) + X_bytes(p), (size_t)fl_f);
    set_kernel(p, k++, mix_name(p), X_bytes(p) + w_bytes(p) + Z_bytes(p),
               8ull * p->B * p->Cin * p->Cout * p->nm);
    set_kernel(p, k++, "inv_fused", Z_bytes(p) + y_bytes(p), (size_t)fl_i);
    p->launches = k;
}

// Kernel list of the 1D layer (stages_dft.cu row transforms + a contraction).
void describe_1d(fno_plan_s* p) {
    const size_t Pi = (size_t)p->B * p->Cin, Po = (size_t)p->B * p->Cout;
    set_kernel(p, 0, "dft1_fwd", x_bytes(p) + X_bytes(p), 8ull * Pi * p->W * p->m2);
    set_kernel(p, 1, mix_name(p), X_bytes(p) + w_bytes(p) + Z_bytes(p),
               8ull * p->B * p->Cin * p->Cout * p->nm);
    set_kernel(p, 2, "dft1_inv", Z_bytes(p) + y_bytes(p), 4ull * Po * p->W * p->m2);
    p->launches = 3;
}

// Kernel list of the single-launch layer (layer_persistent.cu), or of the
// regular path when single_launch is off.
void describe_launches(fno_plan_s* p) {
    if (p->single_launch) {
        set_kernel(p, 0, "layer_persistent", x_bytes(p) + w_bytes(p) + y_bytes(p),
                   8ull * p->B * p->Cin * p->Cout * p->nm);
        p->launches = 1;
    } else {
        describe_fused(p);
    }
}

cudaError_t run_forward(const fno_plan_s& p, const float* x, float2* X, float2* T, cudaStream_t s,
                        fno_launch_ctx* ctx) {
    if (p.dims == 1)
        return p.path == 2 ? launch_forward_rows1d(p, x, X, s, ctx) : launch_forward_1d(p, x, X, s, ctx);
    return p.path == 1 ? launch_forward_fused(p, x, X, s, ctx) : launch_forward_modes(p, x, X, T, s, ctx);
}

cudaError_t run_inverse(const fno_plan_s& p, const float2* Z, float* y, float2* T, cudaStream_t s,
                        fno_launch_ctx* ctx) {
    if (p.dims == 1)
        return p.path == 2 ? launch_inverse_rows1d(p, Z, y, s, ctx) : launch_inverse_1d(p, Z, y, s, ctx);
    return p.path == 1 ? launch_inverse_fused(p, Z, y, s, ctx) : launch_inverse_modes(p, Z, y, T, s, ctx);
}

// after_own_forward: the previous kernel on s is this library's forward stage.
cudaError_t run_mix(const fno_plan_s& p, const float2* X, const float2* w, float2* Z, cudaStream_t s,
                    fno_launch_ctx* ctx, bool after_own_forward) {
    if (p.mix_path == 2) return launch_mix_tc(p, X, w, Z, p.tc_split, s, ctx);
    if (p.mix_path == 5) return launch_mix_tcm(p, X, w, Z, p.tc_split, after_own_forward, s, ctx);
    if (p.mix_path == 3) return launch_mix_wide(p, X, w, Z, after_own_forward, s, ctx);
    if (p.mix_path == 4) return launch_mix_adjoint_fma(p, X, w, Z, s, ctx);
    return p.mix_path == 1 ? launch_mix_tma(p, X, w, Z, s, ctx) : launch_mix_modes(p, X, w, Z, s, ctx);
}


fno_status_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return FNO_OK;
    return FNO_ERR_CUDA;
}

// Kernel attributes (dynamic shared-memory limits) are held per device, so
// the set-up runs once for every device a plan is created on, with that
// device current.  g_init_done[d] is written under g_init_mu only.
constexpr int kMaxDevices = 64;
std::mutex g_init_mu;
bool g_init_done[kMaxDevices] = {};

fno_plan_s* plan_new(int dims, int B, int Cin, int Cout, int H, int W, int m1, int m2,
                     fno_precision_t prec, fno_plan_s* parent);

cudaError_t init_device() {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_init_mu);
    if (g_init_done[dev]) return cudaSuccess;
    e = stages_generic_init();
    if (e == cudaSuccess) e = stages_dft_init();
    if (e == cudaSuccess) e = stages_fused_init();
    if (e == cudaSuccess) e = stages_big_init();
    if (e == cudaSuccess) e = mix_init();
    if (e == cudaSuccess) e = mix_tma_init();
    if (e == cudaSuccess) e = mix_wide_init();
    if (e == cudaSuccess) e = block_init();
    if (e == cudaSuccess) e = block_tc_init();
    if (e == cudaSuccess) e = mix_tc_init();
    if (e == cudaSuccess) e = mix_tcm_init();
    if (e == cudaSuccess) e = layer_persistent_init();
    if (e == cudaSuccess) g_init_done[dev] = true;
    return e;
}

// A plan and its adjoint (the backward's plan: channels swapped, contraction
// with w conjugated and transposed, tables and error word shared).
fno_status_t plan_pair(fno_plan_t* out, int dims, int B, int Cin, int Cout, int H, int W, int m1,
                       int m2, fno_precision_t prec) {
    if (prec != FNO_PREC_FP32 && prec != FNO_PREC_TF32 && prec != FNO_PREC_3XTF32)
        return FNO_ERR_INVALID_ARG;
    if (init_device() != cudaSuccess) return FNO_ERR_CUDA;
    fno_plan_s* p = plan_new(dims, B, Cin, Cout, H, W, m1, m2, prec, nullptr);
    if (!p) return FNO_ERR_CUDA;
    p->adj = plan_new(dims, B, Cout, Cin, H, W, m1, m2, FNO_PREC_FP32, p);
    if (!p->adj) {
        fno_plan_destroy(p);
        return FNO_ERR_CUDA;
    }
    *out = p;
    return FNO_OK;
}

}  // namespace

extern "C" {

const char* fno_status_string(fno_status_t s) {
    switch (s) {
        case FNO_OK: return "FNO_OK";
        case FNO_ERR_INVALID_ARG: return "FNO_ERR_INVALID_ARG: invalid argument";
        case FNO_ERR_UNSUPPORTED: return "FNO_ERR_UNSUPPORTED: shape or precision not supported";
        case FNO_ERR_CUDA: return "FNO_ERR_CUDA: CUDA runtime error";
        case FNO_ERR_WORKSPACE: return "FNO_ERR_WORKSPACE: workspace too small";
        case FNO_ERR_TIMEOUT: return "FNO_ERR_TIMEOUT: device-side wait timed out";
        case FNO_ERR_DEVICE: return "FNO_ERR_DEVICE: kernel reported an internal error";
    }
    return "unknown fno_status_t";
}

fno_status_t fno_plan_create(fno_plan_t* out, int B, int Cin, int Cout, int H, int W, int m1,
                             int m2, fno_precision_t prec) {
    if (!out) return FNO_ERR_INVALID_ARG;
    *out = nullptr;
    fno_status_t st = validate_shape(B, Cin, Cout, H, W, m1, m2);
    if (st != FNO_OK) return st;
    return plan_pair(out, 2, B, Cin, Cout, H, W, m1, m2, prec);
}

fno_status_t fno_plan_create_1d(fno_plan_t* out, int B, int Cin, int Cout, int L, int m,
                                fno_precision_t prec) {
    if (!out) return FNO_ERR_INVALID_ARG;
    *out = nullptr;
    fno_status_t st = validate_shape_1d(B, Cin, Cout, L, m);
    if (st != FNO_OK) return st;
    return plan_pair(out, 1, B, Cin, Cout, 1, L, 0, m, prec);
}

}  // extern "C"

namespace {

// A plan for (B, Cin, Cout, ...).  With a parent, it is that plan's adjoint:
// the parent's tables and error word are shared and the contraction is the
// conjugate-transpose one (fp32).  dims = 1 is the 1D layer over W = L points
// with m2 = m modes (H = 1, m1 = 0).  Returns nullptr on a CUDA error.
fno_plan_s* plan_new(int dims, int B, int Cin, int Cout, int H, int W, int m1, int m2,
                     fno_precision_t prec, fno_plan_s* parent) {
    fno_plan_s* p = new fno_plan_s();
    std::memset(p, 0, sizeof(*p));
    p->dims = dims;
    p->B = B; p->Cin = Cin; p->Cout = Cout; p->H = H; p->W = W; p->m1 = m1; p->m2 = m2;
    p->adjoint = parent != nullptr;
    p->nm = dims == 1 ? m2 : 2 * m1 * m2;
    p->prec = prec;
    p->scale = (float)(1.0 / std::sqrt((double)H * (double)W));
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
        delete p;
        return nullptr;
    }

    int Rf = 0, Ri = 0;
    // path: 0 shape-generic (FFT or direct-DFT stages), 1 fused transforms,
    // 2 the 1D layer on the long-row FFT kernels
    if (dims == 1) p->path = rows1d_supported(W, m2) ? 2 : 0;
    else p->path = fused_supported(W, H, m1, m2, &Rf, &Ri) ? 1 : 0;
    p->R = p->path == 1 ? Rf : H;
    p->P = H / p->R;
    p->Ri = p->path == 1 ? Ri : H;
    p->Pi = H / p->Ri;
    p->mix_path = mix_tma_supported(B, Cin, Cout, p->nm) ? 1 : 0;
    // 32-mode blocks move w and X as 256-byte rows (measured faster than the
    // 4-mode mix_tma at every workload: 128x128 44.7 -> 38.2 us, 256x256 222 ->
    // 207 us, 2048x2048 25.2 -> 19.8 us)
    if (mix_wide_supported(B, Cin, Cout, p->nm)) p->mix_path = 3;
    p->tc_split = prec == FNO_PREC_3XTF32 ? 3 : 1;
    // tensor cores for the contraction only where it is a real dense product
    // (Cin, Cout >= 32): the weight-in-TMEM kernel for batches up to 16, the
    // shared-memory-operand kernel for larger batches
    if (prec != FNO_PREC_FP32 && Cin >= 32 && Cout >= 32) {
        if (mix_tcm_supported(B, Cin, Cout, p->nm))
            p->mix_path = 5;
        else if (mix_tc_supported(B, Cin, Cout, p->nm, p->tc_split))
            p->mix_path = 2;
    }
    if (p->adjoint) p->mix_path = mix_wide_supported(B, Cin, Cout, p->nm) ? 3 : 4;

    // workspace: X | Z | T (T only on the shape-generic path)
    size_t off = 0;
    p->off_X = off; off = align_up(off + X_bytes(p), 256);
    p->off_Z = off; off = align_up(off + Z_bytes(p), 256);
    p->off_T = off;
    if (p->path == 0 && dims == 2) {
        const size_t planes = (size_t)B * (Cin > Cout ? Cin : Cout);
        off = align_up(off + 8ull * planes * H * m2, 256);
    }
    p->ws_bytes = off;
    if (dims == 1) {
        describe_1d(p);
        if (p->path == 2) {
            std::snprintf(p->kernels[0].name, sizeof(p->kernels[0].name), "rows1d_fwd");
            std::snprintf(p->kernels[2].name, sizeof(p->kernels[2].name), "rows1d_inv");
            p->kernels[0].flops = (size_t)(fft_flops(W) * p->B * Cin / 2);
            p->kernels[2].flops = (size_t)(fft_flops(W) * p->B * Cout / 2);
        }
        std::snprintf(p->desc, sizeof(p->desc), "1d-%s: rows(L=%d,m=%d)|%s|irows",
                      p->path == 2 ? "fft" : "dft", W, m2, mix_name(p));
    } else if (p->path == 1) {
        describe_fused(p);
        std::snprintf(p->desc, sizeof(p->desc),
                      "fused: fwd-rows+cols(W=%d,R=%d,P=%d)|%s|inv-cols+rows(R=%d,P=%d)", W,
                      p->R, p->P, mix_name(p), p->Ri, p->Pi);
        // the single-launch layer (fno_plan_set_single_launch) is opt-in: measured
        // slower than the three launches with programmatic dependent launch at
        // every shape it serves (64x64 B8 C32: 38.7 against 18.6 us; 128x128
        // B16 C64: 187 against 83 us)
    } else if (dft_path(H, W)) {
        describe_generic(p);
        std::snprintf(p->kernels[0].name, sizeof(p->kernels[0].name), "dft_rows");
        std::snprintf(p->kernels[1].name, sizeof(p->kernels[1].name), "dft_cols");
        std::snprintf(p->kernels[3].name, sizeof(p->kernels[3].name), "dft_icols");
        std::snprintf(p->kernels[4].name, sizeof(p->kernels[4].name), "dft_irows");
        std::snprintf(p->desc, sizeof(p->desc),
                      "direct-dft: rows(W=%d)|cols(H=%d)|%s|icols|irows", W, H, mix_name(p));
    } else {
        describe_generic(p);
        std::snprintf(p->desc, sizeof(p->desc),
                      "generic: rows-fft(W=%d)|cols-fft(H=%d)|%s|icols-fft|irows-fft", W, H,
                      mix_name(p));
    }

    if (parent) {
        p->shares_tables = true;
        p->tw_h = parent->tw_h;
        p->tw_w = parent->tw_w;
        p->g_irows = parent->g_irows;
        p->g_frows = parent->g_frows;
        p->g_cols = parent->g_cols;
        p->err = parent->err;
        return p;
    }
    std::vector<float2> th = twiddles(H), tw = twiddles(W);
    cudaError_t e = cudaMalloc(&p->tw_h, sizeof(float2) * H);
    if (e == cudaSuccess) e = cudaMalloc(&p->tw_w, sizeof(float2) * W);
    // err[0]: error bits, err[1]: debug flags (see fno_plan_debug_force_timeout)
    if (e == cudaSuccess) e = cudaMalloc(&p->err, 2 * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMalloc(&p->gbar, sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemset(p->gbar, 0, sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemcpy(p->tw_h, th.data(), sizeof(float2) * H, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(p->tw_w, tw.data(), sizeof(float2) * W, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(p->err, 0, 2 * sizeof(unsigned));
    // the direct-DFT inverse rows stream their twiddle tiles from the plan
    if (e == cudaSuccess && p->path == 0 && (dims == 1 || dft_path(H, W))) {
        const std::vector<float> g = dft_irows_table(W, m2, (double)p->scale);
        if (!g.empty()) {
            e = cudaMalloc(&p->g_irows, sizeof(float) * g.size());
            if (e == cudaSuccess)
                e = cudaMemcpy(p->g_irows, g.data(), sizeof(float) * g.size(),
                               cudaMemcpyHostToDevice);
        }
        // the forward rows carry the 1D layer's 1/sqrt(L); in 2D the columns
        // apply the scale
        const std::vector<float> f = dft_frows_table(W, m2, dims == 1 ? (double)p->scale : 1.0);
        if (e == cudaSuccess && !f.empty()) {
            e = cudaMalloc(&p->g_frows, sizeof(float) * f.size());
            if (e == cudaSuccess)
                e = cudaMemcpy(p->g_frows, f.data(), sizeof(float) * f.size(),
                               cudaMemcpyHostToDevice);
        }
        // the column steps of the 2D direct-DFT path
        if (e == cudaSuccess && dims == 2) {
            const std::vector<float2> c = dft_cols_table(H, m1);
            e = cudaMalloc(&p->g_cols, sizeof(float2) * c.size());
            if (e == cudaSuccess)
                e = cudaMemcpy(p->g_cols, c.data(), sizeof(float2) * c.size(),
                               cudaMemcpyHostToDevice);
        }
    }
    if (e != cudaSuccess) {
        fno_plan_destroy(p);
        return nullptr;
    }
    return p;
}

}  // namespace

extern "C" {

fno_status_t fno_plan_workspace_size(fno_plan_t p, size_t* bytes) {
    if (!p || !bytes) return FNO_ERR_INVALID_ARG;
    *bytes = p->ws_bytes;
    return FNO_OK;
}

fno_status_t fno_plan_launch_count(fno_plan_t p, int* n) {
    if (!p || !n) return FNO_ERR_INVALID_ARG;
    *n = p->launches;
    return FNO_OK;
}

fno_status_t fno_plan_kernel_info(fno_plan_t p, int index, char* name, size_t name_len,
                                  size_t* bytes, size_t* flops) {
    if (!p || index < 0 || index >= p->launches) return FNO_ERR_INVALID_ARG;
    if (name && name_len) std::snprintf(name, name_len, "%s", p->kernels[index].name);
    if (bytes) *bytes = p->kernels[index].bytes;
    if (flops) *flops = p->kernels[index].flops;
    return FNO_OK;
}

fno_status_t fno_plan_record_events(fno_plan_t p, cudaEvent_t* events, int count) {
    if (!p) return FNO_ERR_INVALID_ARG;
    if (!events) {
        p->events = nullptr;
        p->nevents = 0;
        return FNO_OK;
    }
    if (count != p->launches + 1) return FNO_ERR_INVALID_ARG;
    p->events = events;
    p->nevents = count;
    return FNO_OK;
}

fno_status_t fno_plan_describe(fno_plan_t p, char* buf, size_t len) {
    if (!p || !buf || len == 0) return FNO_ERR_INVALID_ARG;
    std::snprintf(buf, len, "%s", p->desc);
    return FNO_OK;
}

fno_status_t fno_plan_destroy(fno_plan_t p) {
    if (!p) return FNO_OK;
    if (p->adj) fno_plan_destroy(p->adj);
    if (!p->shares_tables) {
        if (p->tw_h) cudaFree(p->tw_h);
        if (p->tw_w) cudaFree(p->tw_w);
        if (p->g_irows) cudaFree(p->g_irows);
        if (p->g_frows) cudaFree(p->g_frows);
        if (p->g_cols) cudaFree(p->g_cols);
        if (p->err) cudaFree(p->err);
        if (p->gbar) cudaFree(p->gbar);
    }
    delete p;
    return FNO_OK;
}

fno_status_t fno_plan_backward(fno_plan_t p, const float* x, const void* w, const float* gy,
                               float* gx, void* gw, void* ws, size_t ws_bytes, cudaStream_t s) {
    if (!p || !p->adj) return FNO_ERR_INVALID_ARG;
    if (check_no_pending_error() != FNO_OK) return FNO_ERR_CUDA;
    if (!gx && !gw) return FNO_ERR_INVALID_ARG;
    fno_status_t st;
    if ((st = check_device(p)) != FNO_OK) return st;
    if ((st = check_ptr(gy, true)) != FNO_OK) return st;
    if ((st = check_ptr(w, gx != nullptr)) != FNO_OK) return st;
    if ((st = check_ptr(x, gw != nullptr)) != FNO_OK) return st;
    if ((st = check_ptr(gx, false)) != FNO_OK) return st;
    if ((st = check_ptr(gw, false)) != FNO_OK) return st;
    if ((st = check_ws(p, ws, ws_bytes)) != FNO_OK) return st;
    // outputs overlap no input, no other output and not the workspace
    const void* ins[3] = {x, w, gy};
    const size_t in_bytes[3] = {x_bytes(p), w_bytes(p), y_bytes(p)};
    const void* outs[2] = {gx, gw};
    const size_t out_bytes[2] = {x_bytes(p), w_bytes(p)};
    for (int o = 0; o < 2; ++o) {
        if (!outs[o]) continue;
        for (int i = 0; i < 3; ++i)
            if (ins[i] && overlaps(outs[o], out_bytes[o], ins[i], in_bytes[i]))
                return FNO_ERR_INVALID_ARG;
        if (p->ws_bytes && overlaps(outs[o], out_bytes[o], ws, p->ws_bytes))
            return FNO_ERR_INVALID_ARG;
    }
    if (gx && gw && overlaps(gx, out_bytes[0], gw, out_bytes[1])) return FNO_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
        if (ins[i] && p->ws_bytes && overlaps(ws, p->ws_bytes, ins[i], in_bytes[i]))
            return FNO_ERR_INVALID_ARG;

    const fno_plan_s& q = *p->adj;  // B, Cout -> Cin, w conjugated and transposed
    char* base = static_cast<char*>(ws);
    float2* A = reinterpret_cast<float2*>(base + p->off_X);  // B*Cin*nm: dL/dX, then X
    float2* G = reinterpret_cast<float2*>(base + p->off_Z);  // B*Cout*nm: forward modes of gy
    float2* T = reinterpret_cast<float2*>(base + p->off_T);
    cudaError_t e = run_forward(q, gy, G, T, s, nullptr);
    if (e == cudaSuccess && gx)
        e = run_mix(q, G, static_cast<const float2*>(w), A, s, nullptr, true);
    if (e == cudaSuccess && gx) e = run_inverse(q, A, gx, T, s, nullptr);
    if (e == cudaSuccess && gw) e = run_forward(*p, x, A, T, s, nullptr);
    if (e == cudaSuccess && gw)
        e = wgrad_wide_supported(p->nm) ? launch_wgrad_wide(*p, A, G, static_cast<float2*>(gw), s)
                        : launch_wgrad(A, G, static_cast<float2*>(gw), p->B, p->Cin, p->Cout,
                                       p->nm, p->m2, p->W, s);
    return cuda_status(e);
}

fno_status_t fno_plan_execute(fno_plan_t p, const float* x, const void* w, float* y, void* ws,
                              size_t ws_bytes, cudaStream_t s) {
    if (!p) return FNO_ERR_INVALID_ARG;
    if (check_no_pending_error() != FNO_OK) return FNO_ERR_CUDA;
    fno_status_t st;
    if ((st = check_device(p)) != FNO_OK) return st;
    if ((st = check_ptr(x, true)) != FNO_OK) return st;
    if ((st = check_ptr(w, true)) != FNO_OK) return st;
    if ((st = check_ptr(y, true)) != FNO_OK) return st;
    if ((st = check_ws(p, ws, ws_bytes)) != FNO_OK) return st;
    if (overlaps(y, y_bytes(p), x, x_bytes(p)) || overlaps(y, y_bytes(p), w, w_bytes(p)))
        return FNO_ERR_INVALID_ARG;
    if (p->ws_bytes && (overlaps(ws, p->ws_bytes, x, x_bytes(p)) ||
                        overlaps(ws, p->ws_bytes, y, y_bytes(p)) ||
                        overlaps(ws, p->ws_bytes, w, w_bytes(p))))
        return FNO_ERR_INVALID_ARG;
    char* base = static_cast<char*>(ws);
    float2* X = reinterpret_cast<float2*>(base + p->off_X);
    float2* Z = reinterpret_cast<float2*>(base + p->off_Z);
    float2* T = reinterpret_cast<float2*>(base + p->off_T);
    fno_launch_ctx ctx;
    ctx.events = p->events;
    ctx.count = p->nevents;
    cudaError_t e = ctx.mark(s);
    if (p->single_launch) {
        if (e == cudaSuccess)
            e = launch_layer_persistent(*p, x, static_cast<const float2*>(w), y, X, Z, s, &ctx);
        return cuda_status(e);
    }
    if (e == cudaSuccess) e = run_forward(*p, x, X, T, s, &ctx);
    if (e == cudaSuccess) e = run_mix(*p, X, static_cast<const float2*>(w), Z, s, &ctx, true);
    if (e == cudaSuccess) e = run_inverse(*p, Z, y, T, s, &ctx);
    return cuda_status(e);
}

namespace {

fno_status_t check_block_args(const fno_plan_s* p, const float* x, const float* w_pw,
                              const float* bias, fno_activation_t act, const float* y) {
    fno_status_t st;
    if ((st = check_device(p)) != FNO_OK) return st;
    if (act != FNO_ACT_NONE && act != FNO_ACT_GELU) return FNO_ERR_INVALID_ARG;
    if (!block_supported(p->Cin) || (p->H * p->W) % 4 != 0) return FNO_ERR_UNSUPPORTED;
    if ((st = check_ptr(x, true)) != FNO_OK) return st;
    if ((st = check_ptr(w_pw, true)) != FNO_OK) return st;
    if ((st = check_ptr(bias, false)) != FNO_OK) return st;
    if ((st = check_ptr(y, true)) != FNO_OK) return st;
    const size_t wpw_bytes = 4ull * p->Cin * p->Cout, bias_bytes = 4ull * p->Cout;
    if (overlaps(y, y_bytes(p), x, x_bytes(p)) || overlaps(y, y_bytes(p), w_pw, wpw_bytes) ||
        (bias && overlaps(y, y_bytes(p), bias, bias_bytes)))
        return FNO_ERR_INVALID_ARG;
    return FNO_OK;
}

}  // namespace

fno_status_t fno_block_epilogue(fno_plan_t p, const float* x, const float* w_pw, const float* bias,
                                fno_activation_t act, float* y, cudaStream_t s) {
    if (!p) return FNO_ERR_INVALID_ARG;
    if (check_no_pending_error() != FNO_OK) return FNO_ERR_CUDA;
    fno_status_t st = check_block_args(p, x, w_pw, bias, act, y);
    if (st != FNO_OK) return st;
    return cuda_status(launch_block_epilogue(*p, x, w_pw, bias, (int)act, y, false, s));
}

fno_status_t fno_block_execute(fno_plan_t p, const float* x, const void* w, const float* w_pw,
                               const float* bias, fno_activation_t act, float* y, void* ws,
                               size_t ws_bytes, cudaStream_t s) {
    if (!p) return FNO_ERR_INVALID_ARG;
    if (check_no_pending_error() != FNO_OK) return FNO_ERR_CUDA;
    fno_status_t st = check_block_args(p, x, w_pw, bias, act, y);
    if (st != FNO_OK) return st;
    st = fno_plan_execute(p, x, w, y, ws, ws_bytes, s);
    if (st != FNO_OK) return st;
    // the kernel just before is the plan's own inverse stage (launched either with
    // programmatic serialisation, after its own wait, or normally), so w_pw and
    // bias may be read before the epilogue's launch wait
    return cuda_status(launch_block_epilogue(*p, x, w_pw, bias, (int)act, y, true, s));
}

fno_status_t fno_forward_modes(fno_plan_t p, const float* x, void* X, void* ws, size_t ws_bytes,
                               cudaStream_t s) {
    if (!p) return FNO_ERR_INVALID_ARG;
    if (check_no_pending_error() != FNO_OK) return FNO_ERR_CUDA;
    fno_status_t st;
    if ((st = check_device(p)) != FNO_OK) return st;
    if ((st = check_ptr(x, true)) != FNO_OK) return st;
    if ((st = check_ptr(X, true)) != FNO_OK) return st;
    if ((st = check_ws(p, ws, ws_bytes)) != FNO_OK) return st;
    if (overlaps(X, X_bytes(p), x, x_bytes(p))) return FNO_ERR_INVALID_ARG;
    if (overlaps(ws, p->ws_bytes, x, x_bytes(p)) || overlaps(ws, p->ws_bytes, X, X_bytes(p)))
        return FNO_ERR_INVALID_ARG;
    float2* T = reinterpret_cast<float2*>(static_cast<char*>(ws) + p->off_T);
    return cuda_status(run_forward(*p, x, static_cast<float2*>(X), T, s, nullptr));
}

fno_status_t fno_mix_modes(fno_plan_t p, const void* X, const void* w, void* Z, cudaStream_t s) {
    if (!p) return FNO_ERR_INVALID_ARG;
    if (check_no_pending_error() != FNO_OK) return FNO_ERR_CUDA;
    fno_status_t st;
    if ((st = check_device(p)) != FNO_OK) return st;
    if ((st = check_ptr(X, true)) != FNO_OK) return st;
    if ((st = check_ptr(w, true)) != FNO_OK) return st;
    if ((st = check_ptr(Z, true)) != FNO_OK) return st;
    if (overlaps(Z, Z_bytes(p), X, X_bytes(p)) || overlaps(Z, Z_bytes(p), w, w_bytes(p)))
        return FNO_ERR_INVALID_ARG;
    return cuda_status(run_mix(*p, static_cast<const float2*>(X), static_cast<const float2*>(w),
                               static_cast<float2*>(Z), s, nullptr, false));
}

fno_status_t fno_inverse_modes(fno_plan_t p, const void* Z, float* y, void* ws, size_t ws_bytes,
                               cudaStream_t s) {
    if (!p) return FNO_ERR_INVALID_ARG;
    if (check_no_pending_error() != FNO_OK) return FNO_ERR_CUDA;
    fno_status_t st;
    if ((st = check_device(p)) != FNO_OK) return st;
    if ((st = check_ptr(Z, true)) != FNO_OK) return st;
    if ((st = check_ptr(y, true)) != FNO_OK) return st;
    if ((st = check_ws(p, ws, ws_bytes)) != FNO_OK) return st;
    if (overlaps(y, y_bytes(p), Z, Z_bytes(p))) return FNO_ERR_INVALID_ARG;
    if (overlaps(ws, p->ws_bytes, y, y_bytes(p)) || overlaps(ws, p->ws_bytes, Z, Z_bytes(p)))
        return FNO_ERR_INVALID_ARG;
    float2* T = reinterpret_cast<float2*>(static_cast<char*>(ws) + p->off_T);
    return cuda_status(run_inverse(*p, static_cast<const float2*>(Z), y, T, s, nullptr));
}

fno_status_t fno_plan_debug_force_timeout(fno_plan_t p, int enable) {
    if (!p) return FNO_ERR_INVALID_ARG;
    fno_status_t st = check_device(p);
    if (st != FNO_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return FNO_ERR_CUDA;
    const unsigned flags = enable ? 1u : 0u;
    if (cudaMemcpy(p->err + 1, &flags, sizeof(flags), cudaMemcpyHostToDevice) != cudaSuccess)
        return FNO_ERR_CUDA;
    return FNO_OK;
}

fno_status_t fno_plan_debug_bounds_margin(fno_plan_t p, size_t bytes) {
    if (!p || p->adjoint) return FNO_ERR_INVALID_ARG;
#ifdef FNO_DEBUG
    p->dbg_margin = bytes;
    if (p->adj) p->adj->dbg_margin = bytes;
    return FNO_OK;
#else
    (void)bytes;
    return FNO_ERR_UNSUPPORTED;  // only the range-checked build checks stores
#endif
}

fno_status_t fno_plan_set_single_launch(fno_plan_t p, int enable) {
    if (!p || p->adjoint) return FNO_ERR_INVALID_ARG;
    if (enable && !layer_persistent_supported(*p)) return FNO_ERR_UNSUPPORTED;
    if (p->events) return FNO_ERR_INVALID_ARG;  // armed events are sized for the launch count
    p->single_launch = enable ? 1 : 0;
    describe_launches(p);
    if (p->single_launch)
        std::snprintf(p->desc, sizeof(p->desc), "single-launch: fwd-fused(W=%d)|mix|inv-fused",
                      p->W);
    else
        std::snprintf(p->desc, sizeof(p->desc),
                      "fused: fwd-rows+cols(W=%d,R=%d,P=%d)|%s|inv-cols+rows(R=%d,P=%d)", p->W,
                      p->R, p->P, mix_name(p), p->Ri, p->Pi);
    return FNO_OK;
}

fno_status_t fno_get_device_status(fno_plan_t p, cudaStream_t s) {
    if (!p) return FNO_ERR_INVALID_ARG;
    unsigned word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, p->err, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->err, 0, sizeof(unsigned), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return FNO_ERR_CUDA;
    if (word & FNO_DEVERR_TIMEOUT) return FNO_ERR_TIMEOUT;
    if (word) return FNO_ERR_DEVICE;
    return FNO_OK;
}

}  // extern "C"

// ---- one-shot API with a plan/workspace cache ------------------------------
namespace {

using PlanKey = std::tuple<int, int, int, int, int, int, int, int>;           // dev + shape
using WsKey = std::tuple<int, int, int, int, int, int, int, int, uintptr_t>;  // + stream

struct Cache {
    std::mutex mu;
    std::map<PlanKey, fno_plan_t> plans;
    std::map<WsKey, std::pair<void*, size_t>> ws;
};

Cache& cache() {
    static Cache* c = new Cache();  // intentionally leaked: no teardown-order issues at exit
    return *c;
}

}  // namespace

extern "C" fno_status_t fno_spectral_conv2d(const float* x, const void* w, float* y, int B,
                                            int Cin, int Cout, int H, int W, int m1, int m2,
                                            cudaStream_t s) {
    fno_status_t st = validate_shape(B, Cin, Cout, H, W, m1, m2);
    if (st != FNO_OK) return st;
    if (check_no_pending_error() != FNO_OK) return FNO_ERR_CUDA;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FNO_ERR_CUDA;
    Cache& c = cache();
    fno_plan_t plan = nullptr;
    void* ws = nullptr;
    size_t wsb = 0;
    {
        std::lock_guard<std::mutex> lock(c.mu);
        PlanKey pk{dev, B, Cin, Cout, H, W, m1, m2};
        auto it = c.plans.find(pk);
        if (it == c.plans.end()) {
            st = fno_plan_create(&plan, B, Cin, Cout, H, W, m1, m2, FNO_PREC_FP32);
            if (st != FNO_OK) return st;
            c.plans[pk] = plan;
        } else {
            plan = it->second;
        }
        WsKey wk{dev, B, Cin, Cout, H, W, m1, m2, reinterpret_cast<uintptr_t>(s)};
        auto jt = c.ws.find(wk);
        if (jt == c.ws.end()) {
            wsb = plan->ws_bytes;
            if (wsb && cudaMalloc(&ws, wsb) != cudaSuccess) return FNO_ERR_CUDA;
            c.ws[wk] = {ws, wsb};
        } else {
            ws = jt->second.first;
            wsb = jt->second.second;
        }
    }
    return fno_plan_execute(plan, x, w, y, ws, wsb, s);
}

extern "C" fno_status_t fno_release_cache(void) {
    Cache& c = cache();
    std::lock_guard<std::mutex> lock(c.mu);
    if (cudaDeviceSynchronize() != cudaSuccess) return FNO_ERR_CUDA;
    for (auto& kv : c.ws)
        if (kv.second.first) cudaFree(kv.second.first);
    for (auto& kv : c.plans) fno_plan_destroy(kv.second);
    c.ws.clear();
    c.plans.clear();
    return FNO_OK;
}
