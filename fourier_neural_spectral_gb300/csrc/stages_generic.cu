// stages_generic.cu -- shape-generic kernels for every supported shape.
//
// Stage a1 (forward row transform): pairs of real rows are packed into one
//   complex row z = x_a + i x_b, transformed with a full W-point FFT, and the two
//   real-input spectra are separated, X_a[k] = (Z[k] + conj Z[-k]) / 2,
//   X_b[k] = (Z[k] - conj Z[-k]) / (2i); only k2 < m2 is kept.
// Stage a2 (forward column transform): H-point FFT of each kept column, keeping
//   the 2*m1 retained rows, times 1/sqrt(HW).
// Stage a4 (inverse column transform): the retained rows are placed in a zeroed
//   H-point column and inverse transformed.
// Stage a5 (complex-to-real row transform): pairs of rows are packed as
//   U = S_a + i S_b with S the Hermitian extension of the kept bins (imaginary
//   parts of k2 = 0 and k2 = W/2 dropped), inverse transformed, and the real and
//   imaginary parts are the two output rows, times 1/sqrt(HW).
// Stage a3 (per-mode contraction) is in mix_fma.cu.
//
// Intermediate T (row transform output / inverse column output) is complex64
// [planes][H][m2] in the plan's workspace.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fno {
namespace {

constexpr int kThreads = 256;
constexpr int kSeqElems = 2048;  // complex elements per buffer per CTA

__device__ __forceinline__ int kept_row(int r, int H, int m1) { return r < m1 ? r : H - 2 * m1 + r; }

// ---- a1: forward row transform of row pairs -------------------------------
__global__ void __launch_bounds__(kThreads)
fwd_rows_kernel(const float* __restrict__ x, float2* __restrict__ T, long long npairs, int W,
                int m2, int S, const float2* __restrict__ tw FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    extern __shared__ float2 smem[];
    float2* a = smem;
    float2* b = smem + (size_t)S * W;
    const long long pair0 = (long long)blockIdx.x * S;
    const int lw = ilog2(W);
    for (int e = threadIdx.x; e < S * W; e += blockDim.x) {
        const int s = e >> lw, n = e & (W - 1);
        const long long pr = pair0 + s;
        float2 v = make_float2(0.f, 0.f);
        if (pr < npairs) {
            v.x = x[(2 * pr) * W + n];
            v.y = x[(2 * pr + 1) * W + n];
        }
        a[e] = v;
    }
    __syncthreads();
    const float2* res = stockham_radix2<false>(a, b, W, S, tw);
    for (int e = threadIdx.x; e < S * m2; e += blockDim.x) {
        const int s = e / m2, k = e - s * m2;
        const long long pr = pair0 + s;
        if (pr >= npairs) continue;
        const float2 zk = res[s * W + k];
        const float2 zm = res[s * W + ((W - k) & (W - 1))];
        const float2 sum = make_float2(0.5f * (zk.x + zm.x), 0.5f * (zk.y - zm.y));
        // (Z[k] - conj Z[-k]) / (2i)
        const float2 dif = make_float2(0.5f * (zk.y + zm.y), -0.5f * (zk.x - zm.x));
        if (FNO_DBG_OK(&T[(2 * pr) * m2 + k], sizeof(float2))) T[(2 * pr) * m2 + k] = sum;
        if (FNO_DBG_OK(&T[(2 * pr + 1) * m2 + k], sizeof(float2))) T[(2 * pr + 1) * m2 + k] = dif;
    }
}

// ---- a2: forward column transform, keep retained rows, scale ---------------
__global__ void __launch_bounds__(kThreads)
fwd_cols_kernel(const float2* __restrict__ T, float2* __restrict__ X, int H, int m1, int m2,
                int S, float scale, const float2* __restrict__ tw FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    extern __shared__ float2 smem[];
    float2* a = smem;
    float2* b = smem + (size_t)S * H;
    const long long plane = blockIdx.x;
    const int c0 = blockIdx.y * S;
    const int ns = min(S, m2 - c0);
    const float2* Tp = T + plane * H * m2;
    for (int e = threadIdx.x; e < S * H; e += blockDim.x) {
        const int h = e / S, s = e - h * S;
        a[s * H + h] = s < ns ? Tp[(long long)h * m2 + c0 + s] : make_float2(0.f, 0.f);
    }
    __syncthreads();
    const float2* res = stockham_radix2<false>(a, b, H, S, tw);
    const int R = 2 * m1;
    float2* Xp = X + plane * R * m2;
    for (int e = threadIdx.x; e < R * S; e += blockDim.x) {
        const int r = e / S, s = e - r * S;
        if (s < ns && FNO_DBG_OK(&Xp[(long long)r * m2 + c0 + s], sizeof(float2)))
            Xp[(long long)r * m2 + c0 + s] = cscale(res[s * H + kept_row(r, H, m1)], scale);
    }
}

// ---- a4: inverse column transform of the zero-filled retained rows ---------
__global__ void __launch_bounds__(kThreads)
inv_cols_kernel(const float2* __restrict__ Z, float2* __restrict__ T, int H, int m1, int m2,
                int S, const float2* __restrict__ tw FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    extern __shared__ float2 smem[];
    float2* a = smem;
    float2* b = smem + (size_t)S * H;
    const long long plane = blockIdx.x;
    const int c0 = blockIdx.y * S;
    const int ns = min(S, m2 - c0);
    const int R = 2 * m1;
    const float2* Zp = Z + plane * R * m2;
    for (int e = threadIdx.x; e < S * H; e += blockDim.x) {
        const int h = e / S, s = e - h * S;
        int r = -1;
        if (h < m1) r = h;
        else if (h >= H - m1) r = h - H + R;
        a[s * H + h] = (s < ns && r >= 0) ? Zp[(long long)r * m2 + c0 + s] : make_float2(0.f, 0.f);
    }
    __syncthreads();
    const float2* res = stockham_radix2<true>(a, b, H, S, tw);
    float2* Tp = T + plane * H * m2;
    for (int e = threadIdx.x; e < S * H; e += blockDim.x) {
        const int h = e / S, s = e - h * S;
        if (s < ns && FNO_DBG_OK(&Tp[(long long)h * m2 + c0 + s], sizeof(float2)))
            Tp[(long long)h * m2 + c0 + s] = res[s * H + h];
    }
}

// ---- a5: complex-to-real row transform of row pairs -------------------------
__global__ void __launch_bounds__(kThreads)
inv_rows_kernel(const float2* __restrict__ T, float* __restrict__ y, long long npairs, int W,
                int m2, int S, float scale, const float2* __restrict__ tw FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    extern __shared__ float2 smem[];
    float2* a = smem;
    float2* b = smem + (size_t)S * W;
    const long long pair0 = (long long)blockIdx.x * S;
    const int lw = ilog2(W);
    const int half = W >> 1;
    for (int e = threadIdx.x; e < S * W; e += blockDim.x) {
        const int s = e >> lw, k = e & (W - 1);
        const long long pr = pair0 + s;
        float2 u = make_float2(0.f, 0.f);
        if (pr < npairs) {
            const float2* Ta = T + (2 * pr) * m2;
            const float2* Tb = Ta + m2;
            if (k == 0 || k == half) {
                if (k < m2) u = make_float2(Ta[k].x, Tb[k].x);
            } else if (k < half) {
                if (k < m2) {
                    const float2 va = Ta[k], vb = Tb[k];
                    u = make_float2(va.x - vb.y, va.y + vb.x);      // Va + i Vb
                }
            } else {
                const int kk = W - k;
                if (kk < m2) {
                    const float2 va = Ta[kk], vb = Tb[kk];
                    u = make_float2(va.x + vb.y, vb.x - va.y);      // conj Va + i conj Vb
                }
            }
        }
        a[e] = u;
    }
    __syncthreads();
    const float2* res = stockham_radix2<true>(a, b, W, S, tw);
    for (int e = threadIdx.x; e < S * W; e += blockDim.x) {
        const int s = e >> lw, n = e & (W - 1);
        const long long pr = pair0 + s;
        if (pr >= npairs) continue;
        const float2 v = res[e];
        if (FNO_DBG_OK(&y[(2 * pr) * W + n], sizeof(float))) y[(2 * pr) * W + n] = v.x * scale;
        if (FNO_DBG_OK(&y[(2 * pr + 1) * W + n], sizeof(float)))
            y[(2 * pr + 1) * W + n] = v.y * scale;
    }
}

int seqs_for(int L) { return L >= kSeqElems ? 1 : kSeqElems / L; }

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t stages_generic_init() {
    // Largest dynamic shared memory any launch below asks for: two buffers of
    // max(kSeqElems, 4096) complex elements.
    const int bytes = 2 * (int)sizeof(float2) * 4096;
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fwd_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(inv_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(inv_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e;
}

cudaError_t launch_forward_modes(const fno_plan_s& p, const float* x, float2* X, float2* T,
                                 cudaStream_t s, fno_launch_ctx* ctx) {
    if (dft_path(p.H, p.W)) return launch_forward_dft(p, x, X, T, s, ctx);
    const long long npairs = (long long)p.B * p.Cin * p.H / 2;
    {
        const int S = seqs_for(p.W);
        const size_t smem = 2 * sizeof(float2) * (size_t)S * p.W;
        const long long grid = (npairs + S - 1) / S;
        fwd_rows_kernel<<<(unsigned)grid, kThreads, smem, s>>>(
            x, T, npairs, p.W, p.m2, S, p.tw_w FNO_DBG_ARG1(T, 16ull * npairs * p.m2, p));
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess && ctx) e = ctx->mark(s);
        if (e != cudaSuccess) return e;
    }
    {
        const int S = std::min(seqs_for(p.H), p.m2);
        const size_t smem = 2 * sizeof(float2) * (size_t)S * p.H;
        dim3 grid((unsigned)(p.B * p.Cin), (p.m2 + S - 1) / S);
        fwd_cols_kernel<<<grid, kThreads, smem, s>>>(
            T, X, p.H, p.m1, p.m2, S, p.scale, p.tw_h FNO_DBG_ARG1(X, 8ull * p.B * p.Cin * p.nm, p));
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess && ctx) e = ctx->mark(s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_inverse_modes(const fno_plan_s& p, const float2* Z, float* y, float2* T,
                                 cudaStream_t s, fno_launch_ctx* ctx) {
    if (dft_path(p.H, p.W)) return launch_inverse_dft(p, Z, y, T, s, ctx);
    {
        const int S = std::min(seqs_for(p.H), p.m2);
        const size_t smem = 2 * sizeof(float2) * (size_t)S * p.H;
        dim3 grid((unsigned)(p.B * p.Cout), (p.m2 + S - 1) / S);
        inv_cols_kernel<<<grid, kThreads, smem, s>>>(
            Z, T, p.H, p.m1, p.m2, S, p.tw_h FNO_DBG_ARG1(T, 8ull * p.B * p.Cout * p.H * p.m2, p));
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess && ctx) e = ctx->mark(s);
        if (e != cudaSuccess) return e;
    }
    {
        const long long npairs = (long long)p.B * p.Cout * p.H / 2;
        const int S = seqs_for(p.W);
        const size_t smem = 2 * sizeof(float2) * (size_t)S * p.W;
        const long long grid = (npairs + S - 1) / S;
        inv_rows_kernel<<<(unsigned)grid, kThreads, smem, s>>>(
            T, y, npairs, p.W, p.m2, S, p.scale, p.tw_w FNO_DBG_ARG1(y, 8ull * npairs * p.W, p));
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess && ctx) e = ctx->mark(s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
