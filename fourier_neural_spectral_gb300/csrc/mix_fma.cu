// mix_fma.cu -- stage a3 on fp32 FMA: the per-mode complex channel contraction
//   Z[b,o,m] = sum_i X[b,i,m] * w[i,o,m],   (a+bi)(c+di) = (ac-bd) + (ad+bc)i
// (TurboFNO: FFT-GEMM-iFFT fused operator page, section 2.2).
//
// Layouts: X [B][Cin][NM], w [Cin][Cout][NM], Z [B][Cout][NM], complex64, with
// NM = 2*m1*m2 retained modes innermost, so 32 consecutive modes are one 256-byte
// segment of every operand.
//
// CTA tile: 32 modes (one per lane) x 16 output channels (2 per warp, 8 warps)
// x BT batch rows (all accumulators in registers).  Input channels stream
// through shared memory IC at a time.  Each w element is read from HBM by
// exactly one CTA when B <= BT.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fno {
namespace {

constexpr int kModes = 32;
constexpr int kOT = 16;
constexpr int kIC = 4;
constexpr int kThreads = 256;

template <int BT>
__global__ void __launch_bounds__(kThreads)
mix_fma_kernel(const float2* __restrict__ X, const float2* __restrict__ w, float2* __restrict__ Z,
               int B, int Cin, int Cout, int NM) {
    __shared__ float2 sX[kIC][BT][kModes];
    __shared__ float2 sW[kIC][kOT][kModes];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int m0 = blockIdx.x * kModes;
    const int o0 = blockIdx.y * kOT;
    const int b0 = blockIdx.z * BT;
    float2 acc[BT][2];
#pragma unroll
    for (int bb = 0; bb < BT; ++bb) acc[bb][0] = acc[bb][1] = make_float2(0.f, 0.f);

    for (int i0 = 0; i0 < Cin; i0 += kIC) {
        for (int e = threadIdx.x; e < kIC * BT * kModes; e += kThreads) {
            const int mm = e % kModes, bb = (e / kModes) % BT, ii = e / (kModes * BT);
            const int m = m0 + mm, b = b0 + bb, i = i0 + ii;
            sX[ii][bb][mm] = (m < NM && b < B && i < Cin) ? X[((long long)b * Cin + i) * NM + m]
                                                          : make_float2(0.f, 0.f);
        }
        for (int e = threadIdx.x; e < kIC * kOT * kModes; e += kThreads) {
            const int mm = e % kModes, oo = (e / kModes) % kOT, ii = e / (kModes * kOT);
            const int m = m0 + mm, o = o0 + oo, i = i0 + ii;
            sW[ii][oo][mm] = (m < NM && o < Cout && i < Cin) ? w[((long long)i * Cout + o) * NM + m]
                                                             : make_float2(0.f, 0.f);
        }
        __syncthreads();
#pragma unroll
        for (int ii = 0; ii < kIC; ++ii) {
            const float2 w0 = sW[ii][2 * warp][lane];
            const float2 w1 = sW[ii][2 * warp + 1][lane];
#pragma unroll
            for (int bb = 0; bb < BT; ++bb) {
                const float2 xv = sX[ii][bb][lane];
                cmac(acc[bb][0], xv, w0);
                cmac(acc[bb][1], xv, w1);
            }
        }
        __syncthreads();
    }
    const int m = m0 + lane;
    if (m >= NM) return;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int o = o0 + 2 * warp + j;
        if (o >= Cout) continue;
#pragma unroll
        for (int bb = 0; bb < BT; ++bb) {
            const int b = b0 + bb;
            if (b < B) Z[((long long)b * Cout + o) * NM + m] = acc[bb][j];
        }
    }
}

template <int BT>
cudaError_t launch_bt(const float2* X, const float2* w, float2* Z, int B, int Cin, int Cout,
                      int NM, cudaStream_t s, fno_launch_ctx* ctx) {
    dim3 grid((NM + kModes - 1) / kModes, (Cout + kOT - 1) / kOT, (B + BT - 1) / BT);
    mix_fma_kernel<BT><<<grid, kThreads, 0, s>>>(X, w, Z, B, Cin, Cout, NM);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

}  // namespace
}  // namespace fno

cudaError_t mix_init() { return cudaSuccess; }

cudaError_t launch_mix_modes(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                             cudaStream_t s, fno_launch_ctx* ctx) {
    using namespace fno;
    if (p.B <= 1) return launch_bt<1>(X, w, Z, p.B, p.Cin, p.Cout, p.nm, s, ctx);
    if (p.B <= 2) return launch_bt<2>(X, w, Z, p.B, p.Cin, p.Cout, p.nm, s, ctx);
    if (p.B <= 4) return launch_bt<4>(X, w, Z, p.B, p.Cin, p.Cout, p.nm, s, ctx);
    if (p.B <= 8) return launch_bt<8>(X, w, Z, p.B, p.Cin, p.Cout, p.nm, s, ctx);
    return launch_bt<16>(X, w, Z, p.B, p.Cin, p.Cout, p.nm, s, ctx);
}
