// stages_dft.cu -- the transforms for grids whose H or W is not a power of two,
// as pruned direct DFTs (the FFT kernels need power-of-two lengths).  With few
// retained modes (the layer keeps m2 columns and 2*m1 rows) a direct sum per
// retained bin costs W (or H) multiply-adds, which is the right order for
// these sizes.  All four steps are the layer's definition written out:
//   rows, forward:   T[q][h][k2]  = sum_w x[q][h][w] e^{-2 pi i k2 w / W},   k2 < m2
//   cols, forward:   X[q][r][k2]  = s * sum_h T[q][h][k2] e^{-2 pi i k1(r) h / H}
//   cols, inverse:   V[q][h][k2]  = sum_r Z[q][r][k2] e^{+2 pi i k1(r) h / H}
//   rows, inverse:   y[q][h][w]   = s * sum_k2 c(k2) Re(V[q][h][k2] e^{+2 pi i k2 w / W})
// with q a (batch, channel) plane, s = 1/sqrt(HW), k1(r) = r for r < m1 and
// H - 2*m1 + r otherwise, c = 1 for k2 = 0 and k2 = W/2 and 2 otherwise (TurboFNO
// page, sections 2.2 and 3.1; the half-spectrum width W/2 + 1 of the FFT
// operator-optimisation page, section 2.2).  Twiddles come from the plan's
// tables e^{+2 pi i j / N}, indexed by the exact integer (k * n) mod N.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fno {
namespace {

constexpr int kDftThreads = 256;
constexpr int kWarps = kDftThreads / 32;
constexpr int kRowsPerWarp = 4;  // column steps: output rows (or h) per warp

__device__ __forceinline__ int kr(int r, int H, int m1) { return r < m1 ? r : H - 2 * m1 + r; }

// One CTA per RB consecutive rows (of all planes, flattened); rows and the
// twiddle table in shared memory; warp j computes the (row, k2) outputs j,
// j + 8, ..., lanes striding over w, then a shuffle reduction.
__global__ void __launch_bounds__(kDftThreads)
dft_rows_fwd_kernel(const float* __restrict__ x, float2* __restrict__ T, long long nrows, int W,
                    int m2, int RB, float out_scale, const float2* __restrict__ tw_w) {
    extern __shared__ float2 dsm[];
    float2* tw = dsm;                                  // [W]
    float* xs = reinterpret_cast<float*>(dsm + W);     // [RB][W]
    const long long row0 = (long long)blockIdx.x * RB;
    const int nr = (int)std::min<long long>(RB, nrows - row0);
    for (int i = threadIdx.x; i < W; i += kDftThreads) tw[i] = tw_w[i];
    for (int i = threadIdx.x; i < nr * W; i += kDftThreads) xs[i] = __ldg(&x[row0 * W + i]);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int job = warp; job < nr * m2; job += kWarps) {
        const int r = job / m2, k2 = job - r * m2;
        const float* xr = xs + r * W;
        float re = 0.f, im = 0.f;
        int idx = (int)(((long long)k2 * lane) % W);
        const int step = (int)(((long long)k2 * 32) % W);
        for (int w = lane; w < W; w += 32) {
            const float v = xr[w];
            const float2 t = tw[idx];           // e^{+2 pi i k2 w / W}
            re = fmaf(v, t.x, re);
            im = fmaf(-v, t.y, im);             // conjugate: forward sign
            idx += step;
            if (idx >= W) idx -= W;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            re += __shfl_xor_sync(0xffffffffu, re, o);
            im += __shfl_xor_sync(0xffffffffu, im, o);
        }
        if (lane == 0) T[(row0 + r) * m2 + k2] = make_float2(re * out_scale, im * out_scale);
    }
}

// Forward columns: warp = (plane, 4 consecutive retained rows r), lanes over
// k2 (in blocks of 32); per h one coalesced read of T[q][h][k2] serves the 4
// rows, whose twiddles are warp-uniform.
__global__ void __launch_bounds__(kDftThreads)
dft_cols_fwd_kernel(const float2* __restrict__ T, float2* __restrict__ X, long long planes, int H,
                    int m1, int m2, float scale, const float2* __restrict__ tw_h) {
    const int lane = threadIdx.x & 31;
    const int R = 2 * m1, rg = (R + kRowsPerWarp - 1) / kRowsPerWarp;
    const long long job = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (job >= planes * rg) return;
    const long long q = job / rg;
    const int r0 = (int)(job - q * rg) * kRowsPerWarp;
    const float2* Tq = T + q * H * m2;
    for (int kb = 0; kb < m2; kb += 32) {
        const int k2 = kb + lane;
        float2 acc[kRowsPerWarp];
        int k1[kRowsPerWarp], idx[kRowsPerWarp];  // idx = (k1 * h) mod H, stepped with h
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            acc[j] = make_float2(0.f, 0.f);
            k1[j] = r0 + j < R ? kr(r0 + j, H, m1) : 0;
            idx[j] = 0;
        }
        for (int h = 0; h < H; ++h) {
            const float2 v = k2 < m2 ? __ldg(&Tq[(size_t)h * m2 + k2]) : make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) {
                float2 t = __ldg(&tw_h[idx[j]]);
                t.y = -t.y;  // e^{-2 pi i k1 h / H}
                cmac(acc[j], v, t);
                idx[j] += k1[j];
                if (idx[j] >= H) idx[j] -= H;
            }
        }
        if (k2 < m2) {
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j)
                if (r0 + j < R) X[(q * R + r0 + j) * m2 + k2] = cscale(acc[j], scale);
        }
    }
}

// Inverse columns: warp = (plane, 4 consecutive h), lanes over k2; per retained
// row r one coalesced read of Z[q][r][k2] serves the 4 h.
__global__ void __launch_bounds__(kDftThreads)
dft_cols_inv_kernel(const float2* __restrict__ Z, float2* __restrict__ T, long long planes, int H,
                    int m1, int m2, const float2* __restrict__ tw_h) {
    const int lane = threadIdx.x & 31;
    const int R = 2 * m1, hg = (H + kRowsPerWarp - 1) / kRowsPerWarp;
    const long long job = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (job >= planes * hg) return;
    const long long q = job / hg;
    const int h0 = (int)(job - q * hg) * kRowsPerWarp;
    const float2* Zq = Z + q * R * m2;
    for (int kb = 0; kb < m2; kb += 32) {
        const int k2 = kb + lane;
        float2 acc[kRowsPerWarp];
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) acc[j] = make_float2(0.f, 0.f);
        for (int r = 0; r < R; ++r) {
            const float2 v = k2 < m2 ? __ldg(&Zq[(size_t)r * m2 + k2]) : make_float2(0.f, 0.f);
            const int k1 = kr(r, H, m1);
            int idx = (int)(((long long)k1 * h0) % H);  // (k1 * h) mod H for h = h0 + j
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) {
                cmac(acc[j], v, __ldg(&tw_h[idx]));  // e^{+2 pi i k1 h / H}
                idx += k1;
                if (idx >= H) idx -= H;
            }
        }
        if (k2 < m2) {
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j)
                if (h0 + j < H) T[(q * H + h0 + j) * m2 + k2] = acc[j];
        }
    }
}

// Inverse rows: CTA = RB consecutive rows of V (all planes flattened), the row
// values c(k2) V[k2] and the twiddle table in shared memory; thread per output
// w (strided), sum over k2 of Re(c V e^{+2 pi i k2 w / W}).
__global__ void __launch_bounds__(kDftThreads)
dft_rows_inv_kernel(const float2* __restrict__ T, float* __restrict__ y, long long nrows, int W,
                    int m2, int RB, float scale, const float2* __restrict__ tw_w) {
    extern __shared__ float2 dsm[];
    float2* tw = dsm;            // [W]
    float2* vs = dsm + W;        // [RB][m2], times c(k2)
    const long long row0 = (long long)blockIdx.x * RB;
    const int nr = (int)std::min<long long>(RB, nrows - row0);
    for (int i = threadIdx.x; i < W; i += kDftThreads) tw[i] = tw_w[i];
    for (int i = threadIdx.x; i < nr * m2; i += kDftThreads) {
        const int k2 = i % m2;
        const float c = (k2 == 0 || 2 * k2 == W) ? 1.f : 2.f;
        vs[i] = cscale(__ldg(&T[row0 * m2 + i]), c);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nr * W; i += kDftThreads) {
        const int r = i / W, w = i - r * W;
        const float2* v = vs + r * m2;
        float acc = 0.f;
        int idx = 0;
        for (int k2 = 0; k2 < m2; ++k2) {
            const float2 t = tw[idx];  // e^{+2 pi i k2 w / W}
            acc = fmaf(v[k2].x, t.x, acc);
            acc = fmaf(-v[k2].y, t.y, acc);
            idx += w;
            if (idx >= W) idx -= W;
        }
        y[(row0 + r) * W + w] = acc * scale;
    }
}

int rows_per_cta(int W) { return std::max(1, std::min(16, 16384 / W)); }

}  // namespace
}  // namespace fno

using namespace fno;

bool dft_path(int H, int W) {
    const auto pow2 = [](int v) { return v >= 1 && (v & (v - 1)) == 0; };
    return !pow2(H) || !pow2(W);
}

cudaError_t stages_dft_init() {
    // largest requests: W = 4096 (4 rows per CTA): 32 KB of twiddles + 64 KB of x
    // rows, or 4 rows of m2 <= 2049 values
    const int fwd = (int)(sizeof(float2) * 4096 + sizeof(float) * 4 * 4096);
    const int inv = (int)(sizeof(float2) * 4096 + sizeof(float2) * 4 * 2049);
    cudaError_t e = cudaFuncSetAttribute(dft_rows_fwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, fwd);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dft_rows_inv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 inv);
    return e;
}

cudaError_t launch_forward_dft(const fno_plan_s& p, const float* x, float2* X, float2* T,
                               cudaStream_t s, fno_launch_ctx* ctx) {
    const long long planes = (long long)p.B * p.Cin, nrows = planes * p.H;
    const int RB = rows_per_cta(p.W);
    const size_t smem = sizeof(float2) * p.W + sizeof(float) * (size_t)RB * p.W;
    dft_rows_fwd_kernel<<<(unsigned)((nrows + RB - 1) / RB), kDftThreads, smem, s>>>(
        x, T, nrows, p.W, p.m2, RB, 1.f, p.tw_w);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    if (e != cudaSuccess) return e;
    const long long jobs = planes * ((2 * p.m1 + kRowsPerWarp - 1) / kRowsPerWarp);
    dft_cols_fwd_kernel<<<(unsigned)((jobs + kWarps - 1) / kWarps), kDftThreads, 0, s>>>(
        T, X, planes, p.H, p.m1, p.m2, p.scale, p.tw_h);
    e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_dft(const fno_plan_s& p, const float2* Z, float* y, float2* T,
                               cudaStream_t s, fno_launch_ctx* ctx) {
    const long long planes = (long long)p.B * p.Cout, nrows = planes * p.H;
    const long long jobs = planes * ((p.H + kRowsPerWarp - 1) / kRowsPerWarp);
    dft_cols_inv_kernel<<<(unsigned)((jobs + kWarps - 1) / kWarps), kDftThreads, 0, s>>>(
        Z, T, planes, p.H, p.m1, p.m2, p.tw_h);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    if (e != cudaSuccess) return e;
    const int RB = rows_per_cta(p.W);
    const size_t smem = sizeof(float2) * p.W + sizeof(float2) * (size_t)RB * p.m2;
    dft_rows_inv_kernel<<<(unsigned)((nrows + RB - 1) / RB), kDftThreads, smem, s>>>(
        T, y, nrows, p.W, p.m2, RB, p.scale, p.tw_w);
    e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

// The 1D layer (plan with dims = 1, W = L, m2 = m retained modes): the row
// transforms alone, orthonormal scale 1/sqrt(L) applied on each side.
cudaError_t launch_forward_1d(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s,
                              fno_launch_ctx* ctx) {
    const long long nrows = (long long)p.B * p.Cin;
    const int RB = rows_per_cta(p.W);
    const size_t smem = sizeof(float2) * p.W + sizeof(float) * (size_t)RB * p.W;
    dft_rows_fwd_kernel<<<(unsigned)((nrows + RB - 1) / RB), kDftThreads, smem, s>>>(
        x, X, nrows, p.W, p.m2, RB, p.scale, p.tw_w);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_1d(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s,
                              fno_launch_ctx* ctx) {
    const long long nrows = (long long)p.B * p.Cout;
    const int RB = rows_per_cta(p.W);
    const size_t smem = sizeof(float2) * p.W + sizeof(float2) * (size_t)RB * p.m2;
    dft_rows_inv_kernel<<<(unsigned)((nrows + RB - 1) / RB), kDftThreads, smem, s>>>(
        Z, y, nrows, p.W, p.m2, RB, p.scale, p.tw_w);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
