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
//     loads;
//   * a producer warp refills each stage once all consumer warps have released
//     it (one "full" and one "empty" mbarrier per stage, no CTA-wide barrier).
// Every wait is bounded (see tma.cuh); after a timeout the error word is set,
// the producer waits (bounded) for its copies in flight and the CTA returns.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace fno {
namespace {

constexpr int kModes = 32;  // modes per CTA (one per lane)
constexpr size_t kRowBytes = kModes * sizeof(float2);  // 256

// Per batch tile BT (a power of two <= 16): output channels per CTA (OCB) and
// per thread (JO), batch rows per thread (JB), consumer warps (OCB/JO along the
// outputs x BT/JB along the batch), ring depth and input channels per stage.
// Stage size and ring depth, measured (128x128 / 256x256 / 2048x2048
// contraction, us): 4 x 12 KB 37.6 / 206 / 19.9, 3 x 18 KB 36.1 / 208 / 18.6,
// 2 x 24 KB 35.3 / 197 / 18.8, 6 x 8 KB 45.8 / 201 / 20.7.  An 8 x 8 thread tile
// over 16 outputs per CTA (two CTAs per SM, half the X re-reads) measured the
// same at 128x128 (35.4 against 35.0 us), as did 8 x 4 tiles and the
// three-multiplication complex product: the FMA stream of this loop is the
// bound, not its loads.
template <int BT>
struct WideTile {
    static constexpr int OCB = 8;
    static constexpr int JO = 4;
    static constexpr int JB = BT >= 2 ? BT / 2 : 1;
    static constexpr int NOW = OCB / JO;  // consumer warps along the outputs
    static constexpr int NBW = BT / JB;   // consumer warps along the batch
    static constexpr int NST = 2;
    static constexpr int MinBlocks = 4;
    static constexpr size_t StageTarget = 24 * 1024;
    static constexpr int IC = (int)(StageTarget / (kRowBytes * (OCB + BT)));
    static constexpr int Consumers = NOW * NBW;  // warps
    static constexpr int Threads = 32 * (Consumers + 1);  // + one producer warp
    static constexpr uint32_t WBytes = (uint32_t)(kRowBytes * OCB * IC);
    static constexpr uint32_t StageBytes = (uint32_t)(kRowBytes * IC * (OCB + BT));
    static constexpr size_t Smem = 128 + (size_t)NST * StageBytes;
};

int wide_bt(int B) {
    int bt = 1;
    while (bt < B && bt < 16) bt <<= 1;
    return bt;
}

size_t wide_smem(int bt) {
    switch (bt) {
        case 1: return WideTile<1>::Smem;
        case 2: return WideTile<2>::Smem;
        case 4: return WideTile<4>::Smem;
        case 8: return WideTile<8>::Smem;
        default: return WideTile<16>::Smem;
    }
}

// Warps 0 .. Consumers-1 compute: warp w takes output channels o0 + 4*(w & 1)
// .. + 3 and batch rows b0 + JB*(w >> 1) .. + JB - 1 of its lane's mode
// m0 + lane.  The last warp is the producer: its lane 0 refills a stage with
// TMA once every consumer warp has released it (per-stage "empty" mbarrier),
// so consumer warps never wait for one another.  Input channels past Cin in
// the last stage arrive as zeros (TMA fill) and add nothing.
//
// The same pipeline serves three products (MODE); rows / red / Cout below are
// the launch's row count, reduction length and output channel count:
//   kMix   Z[b,o,m] = sum_i X[b,i,m] w[i,o,m]          rows b, reduction i;
//   kAdj   GX[b,i,m] = sum_o G[b,o,m] conj(w[i,o,m])   (the backward's adjoint
//          contraction) rows b, reduction over w's output channels, outputs
//          w's input channels: same tensor map over w, box order (32 modes x
//          IC reductions x 8 outputs) landing as [8][IC][32 modes];
//   kWgrad gw[i,o,m] = c(k2) sum_b conj(X[b,i,m]) G[b,o,m]  (the weight
//          gradient) rows i, reduction b: the "w" operand is G [B][Cout][NM]
//          (box 32 modes x 8 outputs x IC batch rows, as kMix) and the "X"
//          operand is X [B][Cin][NM] with box 32 modes x BT rows x IC batch
//          rows, landing as [IC][BT][32 modes]; c = 1 at k2 = 0 and k2 = W/2,
//          else 2.
enum { kMix = 0, kAdj = 1, kWgrad = 2 };

template <int BT, int MODE>
__global__ void __launch_bounds__(WideTile<BT>::Threads, WideTile<BT>::MinBlocks)
mix_wide_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                float2* __restrict__ Z, int rows, int red, int Cout, int NM, int m2, int W,
                int early_w, unsigned* __restrict__ err FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    using T = WideTile<BT>;
    constexpr int JB = T::JB, IC = T::IC, kOCB = T::OCB, kJO = T::JO, kNST = T::NST;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kNST;
    unsigned char* stages = smem + 128;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // blockIdx.x enumerates (mode block, output block) with the output blocks
    // of one mode block consecutive, so CTAs that share an X tile run together
    const int nob = (Cout + kOCB - 1) / kOCB;
    const int m0 = (blockIdx.x / nob) * kModes, o0 = (blockIdx.x % nob) * kOCB;
    const int b0 = blockIdx.z * BT;
    const int nch = (red + IC - 1) / IC;

    if (tid == 0) {
        for (int s = 0; s < kNST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], T::Consumers);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == T::Consumers) {
        // ---- producer --------------------------------------------------
        if (lane == 0) {
            prefetch_tensormap(&tmW);
            prefetch_tensormap(&tmX);
            const auto load_w = [&](int c) {
                unsigned char* st = stages + (size_t)(c % kNST) * T::StageBytes;
                mbar_arrive_expect_tx(&full[c % kNST], T::StageBytes);
                if (MODE == kAdj)
                    tma_load_3d(st, &tmW, 2 * m0, c * IC, o0, &full[c % kNST]);
                else
                    tma_load_3d(st, &tmW, 2 * m0, o0, c * IC, &full[c % kNST]);
            };
            const auto load_x = [&](int c) {
                unsigned char* st = stages + (size_t)(c % kNST) * T::StageBytes;
                if (MODE == kWgrad)
                    tma_load_3d(st + T::WBytes, &tmX, 2 * m0, b0, c * IC, &full[c % kNST]);
                else
                    tma_load_3d(st + T::WBytes, &tmX, 2 * m0, c * IC, b0, &full[c % kNST]);
            };
            // early_w: the kernel just before this one is the library's own
            // forward stage, which never writes the "w" operand (w is an input, G
            // comes from an earlier kernel), so the first stages' w boxes may be
            // fetched before griddep_wait().  Callers of the standalone stage
            // entry point get no such guarantee and pass early_w = 0.
            const int pre = nch < kNST ? nch : kNST;
            if (early_w)
                for (int c = 0; c < pre; ++c) load_w(c);
            griddep_wait();
            griddep_launch_dependents();
            for (int c = 0; c < pre; ++c) {
                if (!early_w) load_w(c);
                load_x(c);
            }
            int issued = pre;
            for (int c = pre; c < nch; ++c) {
                const int s = c % kNST;
                // stage s last held chunk c - kNST: wait until every consumer let it go
                if (!wait_parity_bounded(&empty[s], (uint32_t)((c / kNST - 1) & 1), err)) break;
                load_w(c);
                load_x(c);
                issued = c + 1;
            }
            // no copy may be in flight when the CTA leaves: the last kNST issued
            // chunks are the only ones not known to have landed (bounded waits)
            for (int c = issued > kNST ? issued - kNST : 0; c < issued; ++c)
                wait_parity_bounded(&full[c % kNST], (uint32_t)((c / kNST) & 1), nullptr);
        } else {
            griddep_wait();
            griddep_launch_dependents();
        }
        return;
    }

    // ---- consumers ------------------------------------------------------
    griddep_wait();  // Z may still be read by an earlier kernel until then
    griddep_launch_dependents();
    const int oh = warp % T::NOW, bh = warp / T::NOW;
    float2 acc[kJO][JB];
#pragma unroll
    for (int j = 0; j < kJO; ++j)
#pragma unroll
        for (int bb = 0; bb < JB; ++bb) acc[j][bb] = make_float2(0.f, 0.f);

    for (int c = 0; c < nch; ++c) {
        const int s = c % kNST;
        if (!wait_parity_bounded(&full[s], (uint32_t)((c / kNST) & 1), err)) return;
        const unsigned char* st = stages + (size_t)s * T::StageBytes;
        // w stage [IC][kOCB][32 modes] ([kOCB][IC][32 modes] for kAdj),
        // X stage [BT][IC][32 modes] ([IC][BT][32 modes] for kWgrad)
        const float2* Ws = reinterpret_cast<const float2*>(st) +
                           (MODE == kAdj ? oh * kJO * IC : oh * kJO) * kModes + lane;
        const float2* Xs = reinterpret_cast<const float2*>(st + T::WBytes) +
                           (MODE == kWgrad ? bh * JB : bh * JB * IC) * kModes + lane;
#pragma unroll
        for (int ii = 0; ii < IC; ++ii) {
            float2 wv[kJO], xv[JB];
#pragma unroll
            for (int j = 0; j < kJO; ++j) {
                wv[j] = Ws[(MODE == kAdj ? j * IC + ii : ii * kOCB + j) * kModes];
                if (MODE == kAdj) wv[j].y = -wv[j].y;
            }
#pragma unroll
            for (int bb = 0; bb < JB; ++bb) {
                xv[bb] = Xs[(MODE == kWgrad ? ii * BT + bb : bb * IC + ii) * kModes];
                if (MODE == kWgrad) xv[bb].y = -xv[bb].y;
            }
#pragma unroll
            for (int j = 0; j < kJO; ++j)
#pragma unroll
                for (int bb = 0; bb < JB; ++bb) cmac(acc[j][bb], xv[bb], wv[j]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with stage s
    }

    const int m = m0 + lane;
    if (m >= NM) return;
    float c = 1.f;
    if (MODE == kWgrad) {
        const int k2 = m % m2;
        c = (k2 == 0 || 2 * k2 == W) ? 1.f : 2.f;
    }
#pragma unroll
    for (int j = 0; j < kJO; ++j) {
        const int o = o0 + oh * kJO + j;
        if (o >= Cout) break;
#pragma unroll
        for (int bb = 0; bb < JB; ++bb) {
            const int r = b0 + bh * JB + bb;
            if (r >= rows) break;
            if (FNO_DBG_OK(&Z[((size_t)r * Cout + o) * NM + m], sizeof(float2)))
                Z[((size_t)r * Cout + o) * NM + m] =
                    MODE == kWgrad ? cscale(acc[j][bb], c) : acc[j][bb];
        }
    }
}

template <int BT>
cudaError_t set_attr() {
    cudaError_t e = cudaFuncSetAttribute(mix_wide_kernel<BT, kMix>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)WideTile<BT>::Smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mix_wide_kernel<BT, kAdj>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)WideTile<BT>::Smem);
    if (e == cudaSuccess && BT == 16)
        e = cudaFuncSetAttribute(mix_wide_kernel<16, kWgrad>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)WideTile<16>::Smem);
    return e;
}

// Cin / Cout of the plan are the launch's reduction and output channel counts
// (an adjoint plan has them swapped relative to w).
template <int BT>
cudaError_t launch_bt(const CUtensorMap& mw, const CUtensorMap& mx, float2* Z, const fno_plan_s& p,
                      int early_w, cudaStream_t s) {
    constexpr int kOCB = WideTile<BT>::OCB;
    const dim3 grid(((p.nm + kModes - 1) / kModes) * ((p.Cout + kOCB - 1) / kOCB), 1,
                    (p.B + BT - 1) / BT);
    if (p.adjoint)
        return launch_pdl(mix_wide_kernel<BT, kAdj>, grid, WideTile<BT>::Threads,
                          WideTile<BT>::Smem, s, mw, mx, Z, p.B, p.Cin, p.Cout, p.nm, p.m2, p.W,
                          early_w, p.err FNO_DBG_ARG1(Z, 8ull * p.B * p.Cout * p.nm, p));
    return launch_pdl(mix_wide_kernel<BT, kMix>, grid, WideTile<BT>::Threads, WideTile<BT>::Smem,
                      s, mw, mx, Z, p.B, p.Cin, p.Cout, p.nm, p.m2, p.W, early_w, p.err
                      FNO_DBG_ARG1(Z, 8ull * p.B * p.Cout * p.nm, p));
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
    if (e == cudaSuccess) e = set_attr<16>();
    return e;
}

bool mix_wide_supported(int B, int Cin, int Cout, int nm) {
    (void)Cout;
    if (nm < kModes || (nm & 1) || B < 1 || Cin < 1) return false;
    return wide_smem(wide_bt(B)) <= kMaxDynSmem;
}

cudaError_t launch_mix_wide(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                            bool after_own_forward, cudaStream_t s, fno_launch_ctx* ctx) {
    const int early_w = after_own_forward ? 1 : 0;
    // batch tile: the power of two >= B (at most 16), halved while the grid
    // would have fewer than two CTAs per SM (few modes and outputs); smaller
    // tiles re-read w, which such shapes hold in L2
    int bt = wide_bt(p.B);
    const auto ctas = [&](int b) {
        return (long long)((p.nm + kModes - 1) / kModes) * ((p.Cout + 7) / 8) * ((p.B + b - 1) / b);
    };
    while (bt > 2 && ctas(bt) < 2 * 152) bt >>= 1;
    int ic = 0, kOCB = 0;
    switch (bt) {
        case 1: ic = WideTile<1>::IC; kOCB = WideTile<1>::OCB; break;
        case 2: ic = WideTile<2>::IC; kOCB = WideTile<2>::OCB; break;
        case 4: ic = WideTile<4>::IC; kOCB = WideTile<4>::OCB; break;
        case 8: ic = WideTile<8>::IC; kOCB = WideTile<8>::OCB; break;
        default: ic = WideTile<16>::IC; kOCB = WideTile<16>::OCB; break;
    }
    // w is [Cin_w][Cout_w][NM]: for an adjoint plan Cin_w = p.Cout (its outputs)
    // and Cout_w = p.Cin (its reduction), boxes (32 modes, IC, OCB)
    CUtensorMap mw, mx;
    const bool ok_w = p.adjoint ? encode_wide_map(&mw, w, p.nm, p.Cin, p.Cout, ic, kOCB)
                                : encode_wide_map(&mw, w, p.nm, p.Cout, p.Cin, kOCB, ic);
    if (!ok_w || !encode_wide_map(&mx, X, p.nm, p.Cin, p.B, ic, bt))
        return cudaErrorInvalidValue;
    cudaError_t e;
    switch (bt) {
        case 1: e = launch_bt<1>(mw, mx, Z, p, early_w, s); break;
        case 2: e = launch_bt<2>(mw, mx, Z, p, early_w, s); break;
        case 4: e = launch_bt<4>(mw, mx, Z, p, early_w, s); break;
        case 8: e = launch_bt<8>(mw, mx, Z, p, early_w, s); break;
        default: e = launch_bt<16>(mw, mx, Z, p, early_w, s); break;
    }
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

// The weight gradient's tile is fixed (16 rows); the 256-byte TMA rows need an
// even mode count (a 16-byte row pitch).
bool wgrad_wide_supported(int nm) { return nm >= kModes && (nm & 1) == 0; }

// Weight gradient gw[i][o][m] = c(k2) * sum_b conj(X[b][i][m]) * G[b][o][m] for
// the plan p (X [B][Cin][nm], G [B][Cout][nm], gw [Cin][Cout][nm]).
cudaError_t launch_wgrad_wide(const fno_plan_s& p, const float2* X, const float2* G, float2* gw,
                              cudaStream_t s) {
    using T = WideTile<16>;
    constexpr int kOCB = T::OCB;
    CUtensorMap mg, mx;
    if (!encode_wide_map(&mg, G, p.nm, p.Cout, p.B, kOCB, T::IC) ||
        !encode_wide_map(&mx, X, p.nm, p.Cin, p.B, 16, T::IC))
        return cudaErrorInvalidValue;
    const dim3 grid(((p.nm + kModes - 1) / kModes) * ((p.Cout + kOCB - 1) / kOCB), 1,
                    (p.Cin + 15) / 16);
    // G comes from an earlier kernel than the forward stage just before this one
    return launch_pdl(mix_wide_kernel<16, kWgrad>, grid, T::Threads, T::Smem, s, mg, mx, gw,
                      p.Cin, p.B, p.Cout, p.nm, p.m2, p.W, 1, p.err
                      FNO_DBG_ARG1(gw, 8ull * p.Cin * p.Cout * p.nm, p));
}
