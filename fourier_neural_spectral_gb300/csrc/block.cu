// block.cu -- the FNO block's epilogue around the spectral layer:
//   out[b,o,p] = act(y[b,o,p] + bias[o] + sum_i w_pw[o,i] * x[b,i,p]),  p = h*W + w,
// written in place over y (the spectral layer's output), act = identity or GELU
// (v/2 * (1 + erf(v / sqrt(2)))).  The pointwise branch is the 1x1 convolution
// that the neural-operator block adds to the spectral path before its
// activation.  It cannot be folded into the inverse transform kernel (each
// output plane needs every input plane), so it is one kernel over pixel tiles:
//   * one resident wave of CTAs, each with an equal share of the (batch row,
//     128-pixel tile) units for 32 or 64 output channels; lane l owns pixels
//     4l .. 4l + 3 of a tile, warp w output channels 8w .. 8w + 7;
//   * the CTA's block of w_pw is loaded once into shared memory as [Cin][OB]
//     (a warp reads its 8 weights of an input channel as one broadcast);
//   * x streams through a 3-stage ring of 32-channel tiles ([32][128] floats)
//     filled by TMA from a producer warp (3D tensor map over [B][Cin][P], so
//     channels past Cin and pixels past P arrive as zeros) that runs on across
//     tile boundaries, released through per-stage "empty" mbarriers;
//   * each tile's y rows are prefetched into L2 when the tile starts; the
//     epilogue reads them, adds the accumulators and the bias, applies the
//     activation and stores, 16 bytes per lane.
// Launched with programmatic stream serialisation (see common.cuh): y is read
// only after griddep_wait(); w_pw and bias, inputs no kernel of the library
// writes, are read before it when the kernel just before this one is the
// library's inverse stage (early = 1).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace fno {
namespace {

constexpr int kPx = 128;    // pixels per tile
constexpr int kJ = 8;       // output channels per warp
constexpr int kICh = 32;    // input channels per stage
constexpr int kStages = 3;
constexpr uint32_t kStageBytes = kICh * kPx * sizeof(float);  // 16 KB
constexpr int kMaxCin = 256;

// OB = 8 * CW output channels per CTA (CW consumer warps) and one producer warp.
template <int CW>
constexpr int block_threads() { return 32 * (CW + 1); }

// w_pw's block is held for Cin rounded up to whole 32-channel chunks (zero rows
// past Cin, matching the zero-filled x channels), so every chunk runs 32 steps.
inline int padded_cin(int Cin) { return (Cin + kICh - 1) / kICh * kICh; }

template <int CW>
size_t block_smem_bytes(int Cin) {
    return 128 + (size_t)kStages * kStageBytes + (size_t)padded_cin(Cin) * (8 * CW) * sizeof(float);
}

__device__ __forceinline__ float act_apply(float v, int act) {
    return act == FNO_ACT_GELU ? 0.5f * v * (1.f + erff(v * 0.70710678118654752440f)) : v;
}

// The grid is one resident wave: gridDim.x CTAs per block of 8*CW output
// channels, CTA j taking the units [j*U/n, (j+1)*U/n) of the U = B * ntiles
// (batch row, 128-pixel tile) pairs, tile-major within a batch row; the
// producer's ring runs on across unit boundaries.
template <int CW>
__global__ void __launch_bounds__(block_threads<CW>(), CW == 8 ? 2 : 3)
block_epilogue_kernel(const __grid_constant__ CUtensorMap tmX, const float* __restrict__ w_pw,
                      const float* __restrict__ bias, float* __restrict__ y, int B, int Cin,
                      int Cout, int P, int act, int early, unsigned* __restrict__ err) {
    constexpr int OB = 8 * CW;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStages;
    float* stages = reinterpret_cast<float*>(smem + 128);
    float* ws = stages + kStages * kICh * kPx;  // [Cin][OB]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ntiles = (P + kPx - 1) / kPx;
    const long long U = (long long)B * ntiles;
    const int u0 = (int)(U * blockIdx.x / gridDim.x);
    const int u1 = (int)(U * (blockIdx.x + 1) / gridDim.x);
    const int o0 = blockIdx.y * OB;
    const int nch = (Cin + kICh - 1) / kICh;
    const int nwork = (u1 - u0) * nch;  // (unit, chunk) pairs, unit-major

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        fence_barrier_init();
    }
    if (!early) griddep_wait();
    // the CTA's block of w_pw, transposed: ws[i][o] = w_pw[o0 + o][i], zero for
    // i >= Cin up to the padded channel count
    const int cinp = nch * kICh;
    for (int idx = tid; idx < cinp * OB; idx += block_threads<CW>()) {
        const int i = idx / OB, o = idx - i * OB;
        ws[idx] = (o0 + o < Cout && i < Cin) ? __ldg(&w_pw[(size_t)(o0 + o) * Cin + i]) : 0.f;
    }
    __syncthreads();

    if (warp == CW) {
        // ---- producer: x tiles [32 channels][128 pixels] ------------------
        if (lane == 0) {
            prefetch_tensormap(&tmX);
            griddep_wait();
            griddep_launch_dependents();
            int issued = 0;
            for (int k = 0; k < nwork; ++k) {
                const int s = k % kStages;
                if (k >= kStages &&
                    !wait_parity_bounded(&empty[s], (uint32_t)((k / kStages - 1) & 1), err))
                    break;
                const int u = u0 + k / nch, c = k - (k / nch) * nch;
                const int bu = u / ntiles, t = u - bu * ntiles;
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                tma_load_3d(stages + (size_t)s * kICh * kPx, &tmX, t * kPx, c * kICh, bu, &full[s]);
                issued = k + 1;
            }
            // no copy may be in flight when the CTA leaves (bounded waits)
            for (int k = issued > kStages ? issued - kStages : 0; k < issued; ++k)
                wait_parity_bounded(&full[k % kStages], (uint32_t)((k / kStages) & 1), nullptr);
        } else {
            griddep_wait();
            griddep_launch_dependents();
        }
        return;
    }

    // ---- consumers --------------------------------------------------------
    griddep_wait();  // y is the previous kernel's output
    griddep_launch_dependents();
    float bo[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
        const int o = o0 + warp * kJ + j;
        bo[j] = bias && o < Cout ? __ldg(&bias[o]) : 0.f;
    }
    int k = 0;
    for (int u = u0; u < u1; ++u) {
        const int b = u / ntiles, t = u - b * ntiles;
        const int p = t * kPx + 4 * lane;
        const bool pin = p < P;  // P is a multiple of 4: all 4 pixels in, or none
        // pull this tile's y rows into L2 now; they are read after the accumulation
        if (pin) {
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                const int o = o0 + warp * kJ + j;
                if (o < Cout)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(y + ((size_t)b * Cout + o) * P + p));
            }
        }
        float acc[kJ][4];
#pragma unroll
        for (int j = 0; j < kJ; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;
        for (int c = 0; c < nch; ++c, ++k) {
            const int s = k % kStages;
            if (!wait_parity_bounded(&full[s], (uint32_t)((k / kStages) & 1), err))
                return;  // err is set; the rest of y is left as it was
            const float4* xs = reinterpret_cast<const float4*>(stages + (size_t)s * kICh * kPx) + lane;
            const float* wb = ws + (size_t)(c * kICh) * OB + warp * kJ;
#pragma unroll 2
            for (int ii = 0; ii < kICh; ++ii) {
                const float4 xv = xs[ii * (kPx / 4)];
                const float4 w0 = *reinterpret_cast<const float4*>(wb + ii * OB);
                const float4 w1 = *reinterpret_cast<const float4*>(wb + ii * OB + 4);
                const float wv[kJ] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int j = 0; j < kJ; ++j) {
                    acc[j][0] = fmaf(wv[j], xv.x, acc[j][0]);
                    acc[j][1] = fmaf(wv[j], xv.y, acc[j][1]);
                    acc[j][2] = fmaf(wv[j], xv.z, acc[j][2]);
                    acc[j][3] = fmaf(wv[j], xv.w, acc[j][3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (!pin) continue;
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const int o = o0 + warp * kJ + j;
            if (o >= Cout) break;
            float4* yp = reinterpret_cast<float4*>(y + ((size_t)b * Cout + o) * P + p);
            const float4 yv = *yp;
            *yp = make_float4(act_apply(yv.x + acc[j][0] + bo[j], act),
                              act_apply(yv.y + acc[j][1] + bo[j], act),
                              act_apply(yv.z + acc[j][2] + bo[j], act),
                              act_apply(yv.w + acc[j][3] + bo[j], act));
        }
    }
}

// 3D tensor map over x [B][Cin][P] floats: dims (P, Cin, B), box (128, 32, 1).
bool encode_x_map(CUtensorMap* map, const float* x, int B, int Cin, int P) {
    fno_encode_tiled_fn enc = fno_get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)P, (cuuint64_t)Cin, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)P * 4, (cuuint64_t)Cin * P * 4};
    cuuint32_t box[3] = {kPx, kICh, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(x), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t block_init() {
    cudaError_t e = cudaFuncSetAttribute(block_epilogue_kernel<4>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)block_smem_bytes<4>(kMaxCin));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(block_epilogue_kernel<8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)block_smem_bytes<8>(kMaxCin));
    return e;
}

bool block_supported(int Cin) { return Cin >= 1 && Cin <= kMaxCin; }

cudaError_t launch_block_epilogue(const fno_plan_s& p, const float* x, const float* w_pw,
                                  const float* bias, int act, float* y, bool after_own_inverse,
                                  cudaStream_t s) {
    // up to 64 output channels the pointwise branch runs on the tensor cores
    // (block_tc.cu); wider blocks keep this fp32 kernel
    if (block_tc_supported(p.Cin, p.Cout))
        return launch_block_tc(p, x, w_pw, bias, act, y, after_own_inverse, s);
    const int P = p.H * p.W;
    CUtensorMap mx;
    if (!encode_x_map(&mx, x, p.B, p.Cin, P)) return cudaErrorInvalidValue;
    const int cw = p.Cout <= 32 ? 4 : 8;
    const int ob = 8 * cw;
    const int ntiles = (P + kPx - 1) / kPx;
    const int oblocks = (p.Cout + ob - 1) / ob;
    // one resident wave: CTAs per SM (occupancy at this shared-memory size)
    // times the SMs, split over the output-channel blocks
    int sms = 0, per_sm = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p.device);
    if (e == cudaSuccess)
        e = cw == 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                          &per_sm, block_epilogue_kernel<4>, block_threads<4>(),
                          block_smem_bytes<4>(p.Cin))
                    : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                          &per_sm, block_epilogue_kernel<8>, block_threads<8>(),
                          block_smem_bytes<8>(p.Cin));
    if (e != cudaSuccess) return e;
    const long long units = (long long)p.B * ntiles;
    const long long per_oblock = std::max(1LL, (long long)std::max(1, per_sm) * sms / oblocks);
    const dim3 grid((unsigned)std::min(units, per_oblock), oblocks, 1);
    const int early = after_own_inverse ? 1 : 0;
    if (cw == 4)
        return launch_pdl(block_epilogue_kernel<4>, grid, dim3(block_threads<4>()),
                          block_smem_bytes<4>(p.Cin), s, mx, w_pw, bias, y, p.B, p.Cin, p.Cout, P,
                          act, early, p.err);
    return launch_pdl(block_epilogue_kernel<8>, grid, dim3(block_threads<8>()),
                      block_smem_bytes<8>(p.Cin), s, mx, w_pw, bias, y, p.B, p.Cin, p.Cout, P, act,
                      early, p.err);
}
