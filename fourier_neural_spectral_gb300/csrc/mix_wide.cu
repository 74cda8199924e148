// mix_wide.cu -- stage a3 on fp32 FMA over blocks of 32 consecutive modes:
//   Z[b,o,m] = sum_i X[b,i,m] * w[i,o,m]     (complex, per retained mode m)
// (TurboFNO: FFT-GEMM-iFFT fused operator page, section 2.2.)
//
// A CTA owns the modes m0..m0+31 (one per lane), 8 output channels and BT
// batch rows (the power of two >= B, at most 16).  Per input channel, w and X
// of 32 consecutive modes are 256-byte rows, which TMA moves at full width:
//   * w is viewed as a 3D tensor [Cin][Cout][2*NM floats] and X as
//     [B][Cin][2*NM floats]; both stream through a ring of shared-memory stages,
//     one TMA box of each per stage (w: 32 modes x 8 outputs x IC inputs, X:
//     32 modes x IC inputs x BT), completion tracked by one mbarrier per stage;
//   * warp (oh, bh) accumulates 4 output channels x JB batch rows for its lane's
//     mode in registers; every shared-memory read is a lane-contiguous 8-byte
//     load (conflict-free), and each thread does 4*JB complex MACs per 4 + JB
//     loads.
// Every wait is bounded (see tma.cuh); on a timeout the CTA drains its copies
// and returns with the error word set.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace fno {
namespace {

constexpr int kModes = 32;  // modes per CTA (one per lane)
constexpr int kOCB = 8;     // output channels per CTA
constexpr int kJO = 4;      // output channels per thread (two warp halves)
constexpr int kNST = 2;     // ring depth
// Stage size and ring depth, measured (128x128 / 256x256 / 2048x2048 contraction, us):
// 4 x 12 KB 37.6 / 206 / 19.9, 3 x 18 KB 36.1 / 208 / 18.6, 2 x 24 KB 35.3 / 197 / 18.8,
// 6 x 8 KB 45.8 / 201 / 20.7: fewer, larger stages (fewer CTA barriers) win.
constexpr size_t kStageTarget = 24 * 1024;

struct MixWideCfg {
    int BT, JB, NBW, IC;
    size_t stage_bytes, smem;
};

MixWideCfg mix_wide_cfg(int B, int Cin) {
    MixWideCfg c;
    int bt = 1;
    while (bt < B && bt < 16) bt <<= 1;
    c.BT = bt;
    c.JB = std::max(1, bt / 2);
    c.NBW = bt / c.JB;
    const size_t row = (size_t)kModes * sizeof(float2);  // 256 bytes
    c.IC = (int)std::max<size_t>(1, std::min<size_t>(Cin, kStageTarget / (row * (kOCB + bt))));
    c.stage_bytes = row * c.IC * (kOCB + bt);
    c.smem = 128 + (size_t)kNST * c.stage_bytes;
    return c;
}

// Threads: 64 * NBW.  Warp w: oh = w & 1 (output channels o0 + 4*oh .. + 3),
// bh = w >> 1 (batch rows b0 + JB*bh .. + JB - 1); lane = mode m0 + lane.
template <int JB>
__global__ void __launch_bounds__(128)
mix_wide_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                float2* __restrict__ Z, int B, int Cin, int Cout, int NM, int IC, int BT,
                unsigned* __restrict__ err) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    unsigned char* stages = smem + 128;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int oh = warp & 1, bh = warp >> 1;
    const int m0 = blockIdx.x * kModes, o0 = blockIdx.y * kOCB, b0 = blockIdx.z * BT;
    const int nch = (Cin + IC - 1) / IC;
    const uint32_t w_bytes = (uint32_t)(kModes * sizeof(float2)) * kOCB * IC;
    const uint32_t stage_bytes = w_bytes + (uint32_t)(kModes * sizeof(float2)) * IC * BT;

    if (tid == 0) {
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
        for (int s = 0; s < kNST; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    int issued = 0;  // stages handed to the TMA unit (thread 0 only)
    if (tid == 0) {
        for (; issued < kNST && issued < nch; ++issued) {
            unsigned char* st = stages + (size_t)issued * stage_bytes;
            mbar_arrive_expect_tx(&bars[issued], stage_bytes);
            tma_load_3d(st, &tmW, 2 * m0, o0, issued * IC, &bars[issued]);
            tma_load_3d(st + w_bytes, &tmX, 2 * m0, issued * IC, b0, &bars[issued]);
        }
    }

    float2 acc[kJO][JB];
#pragma unroll
    for (int j = 0; j < kJO; ++j)
#pragma unroll
        for (int bb = 0; bb < JB; ++bb) acc[j][bb] = make_float2(0.f, 0.f);

    int consumed = 0;
    bool timed_out = false;
    for (int c = 0; c < nch; ++c) {
        const int s = c % kNST;
        const bool ok = wait_parity_bounded(&bars[s], (uint32_t)((c / kNST) & 1), err);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        consumed = c + 1;
        const unsigned char* st = stages + (size_t)s * stage_bytes;
        // w stage [IC][kOCB][32 modes], X stage [BT][IC][32 modes]
        const float2* Ws = reinterpret_cast<const float2*>(st) + (oh * kJO) * kModes + lane;
        const float2* Xs = reinterpret_cast<const float2*>(st + w_bytes) + (bh * JB) * IC * kModes + lane;
        const int ni = min(IC, Cin - c * IC);
        for (int ii = 0; ii < ni; ++ii) {
            float2 wv[kJO], xv[JB];
#pragma unroll
            for (int j = 0; j < kJO; ++j) wv[j] = Ws[(ii * kOCB + j) * kModes];
#pragma unroll
            for (int bb = 0; bb < JB; ++bb) xv[bb] = Xs[(bb * IC + ii) * kModes];
#pragma unroll
            for (int j = 0; j < kJO; ++j)
#pragma unroll
                for (int bb = 0; bb < JB; ++bb) cmac(acc[j][bb], xv[bb], wv[j]);
        }
        __syncthreads();  // every thread is done with stage s
        if (tid == 0 && issued < nch) {
            unsigned char* st2 = stages + (size_t)s * stage_bytes;
            mbar_arrive_expect_tx(&bars[s], stage_bytes);
            tma_load_3d(st2, &tmW, 2 * m0, o0, issued * IC, &bars[s]);
            tma_load_3d(st2 + w_bytes, &tmX, 2 * m0, issued * IC, b0, &bars[s]);
            ++issued;
        }
    }
    if (timed_out) {
        // drain: wait (bounded) for every copy still in flight, then leave
        if (tid == 0)
            for (int c = consumed; c < issued; ++c)
                wait_parity_bounded(&bars[c % kNST], (uint32_t)((c / kNST) & 1), err);
        __syncthreads();
        return;
    }

    const int m = m0 + lane;
    if (m >= NM) return;
#pragma unroll
    for (int j = 0; j < kJO; ++j) {
        const int o = o0 + oh * kJO + j;
        if (o >= Cout) break;
#pragma unroll
        for (int bb = 0; bb < JB; ++bb) {
            const int b = b0 + bh * JB + bb;
            if (b >= B) break;
            Z[((size_t)b * Cout + o) * NM + m] = acc[j][bb];
        }
    }
}

template <int JB>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(mix_wide_kernel<JB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                227 * 1024);
}

// 3D tensor map over a complex64 array [d2][d1][NM] viewed as floats: dims
// (2*NM, d1, d2), box (64 floats = 32 modes, b1, b2), out-of-range elements
// filled with zeros.
bool encode_wide_map(CUtensorMap* map, const float2* base, int NM, int d1, int d2, int b1,
                     int b2) {
    fno_encode_tiled_fn enc = fno_get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)NM * 2, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)NM * 8, (cuuint64_t)d1 * NM * 8};
    cuuint32_t box[3] = {2 * kModes, (cuuint32_t)b1, (cuuint32_t)b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float2*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t mix_wide_init() {
    cudaError_t e = set_attr<1>();
    if (e == cudaSuccess) e = set_attr<2>();
    if (e == cudaSuccess) e = set_attr<4>();
    if (e == cudaSuccess) e = set_attr<8>();
    return e;
}

bool mix_wide_supported(int B, int Cin, int Cout, int nm) {
    (void)Cout;
    if (nm < kModes || (nm & 1) || B < 1 || Cin < 1) return false;
    return mix_wide_cfg(B, Cin).smem <= 227 * 1024;
}

cudaError_t launch_mix_wide(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                            cudaStream_t s, fno_launch_ctx* ctx) {
    const MixWideCfg c = mix_wide_cfg(p.B, p.Cin);
    CUtensorMap mw, mx;
    if (!encode_wide_map(&mw, w, p.nm, p.Cout, p.Cin, kOCB, c.IC) ||
        !encode_wide_map(&mx, X, p.nm, p.Cin, p.B, c.IC, c.BT))
        return cudaErrorInvalidValue;
    const dim3 grid((p.nm + kModes - 1) / kModes, (p.Cout + kOCB - 1) / kOCB,
                    (p.B + c.BT - 1) / c.BT);
    const int threads = 64 * c.NBW;
    switch (c.JB) {
        case 1:
            mix_wide_kernel<1><<<grid, threads, c.smem, s>>>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm,
                                                             c.IC, c.BT, p.err);
            break;
        case 2:
            mix_wide_kernel<2><<<grid, threads, c.smem, s>>>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm,
                                                             c.IC, c.BT, p.err);
            break;
        case 4:
            mix_wide_kernel<4><<<grid, threads, c.smem, s>>>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm,
                                                             c.IC, c.BT, p.err);
            break;
        default:
            mix_wide_kernel<8><<<grid, threads, c.smem, s>>>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm,
                                                             c.IC, c.BT, p.err);
            break;
    }
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
