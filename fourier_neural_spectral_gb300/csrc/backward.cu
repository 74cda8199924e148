// backward.cu -- the kernels only the backward of the layer needs.
//
// For a real loss L with g = dL/dy (gradient convention dL/dRe + i dL/dIm for
// complex values), differentiating the layer's sums gives
//   dL/dZ[b,o,k1,k2] = c(k2) * G[b,o,k1,k2],  G = the layer's forward modes of g,
//   dL/dx = the layer applied to g with w conjugated and transposed per mode
//           (the weights c(k2) cancel through the per-mode channel mixing),
//   dL/dw[i,o,r,k2] = c(k2) * sum_b conj(X[b,i,r,k2]) * G[b,o,r,k2],
// with c = 1 for k2 = 0 and k2 = W/2 and 2 otherwise (the weights of the
// complex-to-real step).  The transforms are the forward stages' kernels; this
// file holds the weight gradient and the shape-generic adjoint contraction.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fno {
namespace {

constexpr int kWgModes = 32;  // modes per CTA (one per lane)
constexpr int kWgO = 8;       // output channels per thread
constexpr int kWgI = 4;       // input channels per CTA (one per warp)

// gw[i][o][m] = c(k2) * sum_b conj(X[b][i][m]) * G[b][o][m], m = r*m2 + k2.
// CTA: 32 consecutive modes (lanes) x 4 input channels (warps) x 8 output
// channels (per thread).  The 4 warps read the same G rows (L1 hits); every
// load and store is a lane-contiguous 256-byte row.
__global__ void __launch_bounds__(32 * kWgI)
wgrad_kernel(const float2* __restrict__ X, const float2* __restrict__ G, float2* __restrict__ gw,
             int B, int Cin, int Cout, int nm, int m2, int W) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m = blockIdx.x * kWgModes + lane;
    const int o0 = blockIdx.y * kWgO;
    const int i = blockIdx.z * kWgI + warp;
    if (m >= nm || i >= Cin) return;
    float2 acc[kWgO];
#pragma unroll
    for (int j = 0; j < kWgO; ++j) acc[j] = make_float2(0.f, 0.f);
    for (int b = 0; b < B; ++b) {
        float2 xv = __ldg(&X[((size_t)b * Cin + i) * nm + m]);
        xv.y = -xv.y;  // conj
#pragma unroll
        for (int j = 0; j < kWgO; ++j) {
            if (o0 + j < Cout) cmac(acc[j], xv, __ldg(&G[((size_t)b * Cout + o0 + j) * nm + m]));
        }
    }
    const int k2 = m % m2;
    const float c = (k2 == 0 || 2 * k2 == W) ? 1.f : 2.f;
#pragma unroll
    for (int j = 0; j < kWgO; ++j)
        if (o0 + j < Cout) gw[((size_t)i * Cout + o0 + j) * nm + m] = cscale(acc[j], c);
}

// GX[b][i][m] = sum_o G[b][o][m] * conj(w[i][o][m]); one thread per output,
// modes fastest.  w is [Cin_w][Cout_w][nm].
__global__ void __launch_bounds__(256)
mix_adjoint_fma_kernel(const float2* __restrict__ G, const float2* __restrict__ w,
                       float2* __restrict__ GX, int B, int Cin_w, int Cout_w, int nm) {
    const size_t n = (size_t)B * Cin_w * nm;
    for (size_t t = blockIdx.x * (size_t)blockDim.x + threadIdx.x; t < n;
         t += (size_t)gridDim.x * blockDim.x) {
        const int m = (int)(t % nm);
        const size_t bi = t / nm;
        const int i = (int)(bi % Cin_w);
        const int b = (int)(bi / Cin_w);
        float2 acc = make_float2(0.f, 0.f);
        for (int o = 0; o < Cout_w; ++o) {
            float2 wv = __ldg(&w[((size_t)i * Cout_w + o) * nm + m]);
            wv.y = -wv.y;
            cmac(acc, __ldg(&G[((size_t)b * Cout_w + o) * nm + m]), wv);
        }
        GX[t] = acc;
    }
}

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t launch_wgrad(const float2* X, const float2* G, float2* gw, int B, int Cin, int Cout,
                         int nm, int m2, int W, cudaStream_t s) {
    const dim3 grid((nm + kWgModes - 1) / kWgModes, (Cout + kWgO - 1) / kWgO,
                    (Cin + kWgI - 1) / kWgI);
    wgrad_kernel<<<grid, 32 * kWgI, 0, s>>>(X, G, gw, B, Cin, Cout, nm, m2, W);
    return cudaGetLastError();
}

// p is an adjoint plan: p.Cin = w's Cout (reduction), p.Cout = w's Cin (outputs).
cudaError_t launch_mix_adjoint_fma(const fno_plan_s& p, const float2* G, const float2* w,
                                   float2* GX, cudaStream_t s, fno_launch_ctx* ctx) {
    const size_t n = (size_t)p.B * p.Cout * p.nm;
    const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, 152 * 16);
    mix_adjoint_fma_kernel<<<blocks, 256, 0, s>>>(G, w, GX, p.B, p.Cout, p.Cin, p.nm);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
