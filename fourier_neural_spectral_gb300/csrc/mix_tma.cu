// mix_tma.cu -- stage a3 on fp32 FMA with the weights streamed by TMA:
//   Z[b,o,m] = sum_i X[b,i,m] * w[i,o,m]     (complex, per retained mode m)
// (TurboFNO: FFT-GEMM-iFFT fused operator page, section 2.2.)
//
// w dominates the traffic (it is read exactly once); X and Z are small.
// A CTA owns 4 consecutive modes m0..m0+3, OC output channels (one thread
// each) and BT batch rows:
//   * w is viewed as a 3D tensor [Cin][Cout][2*NM floats] and X as
//     [B][Cin][2*NM floats]; both stream through a 4- or 6-deep ring of shared-memory
//     stages, one TMA box of each per stage (w: 4 modes x OC x IC, X: 4 modes x
//     IC x BT), completion tracked by one mbarrier per stage;
//   * X values are read with broadcast loads (all lanes of a warp want the same
//     element); each thread keeps BTT x 4 complex accumulators in registers.
// Every wait is bounded (see tma.cuh); on a timeout the CTA drains its copies
// and returns with the error word set.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace fno {
namespace {

constexpr int kMaxStages = 6;

struct MixTmaCfg {
    int OC, IC, BT, BTT, NBH, OT, NST;
    size_t w_off, x_off, stage_bytes, smem;
};

__host__ __device__ inline size_t round128(size_t v) { return (v + 127) / 128 * 128; }

MixTmaCfg mix_tma_cfg(int B, int Cin, int Cout) {
    MixTmaCfg c;
    c.OC = std::min(256, (Cout + 31) / 32 * 32);
    int bt = 1;
    while (bt < B && bt < 16) bt <<= 1;
    c.BT = bt;
    c.BTT = std::min(bt, 8);
    c.NBH = bt / c.BTT;
    c.OT = c.OC >= 64 ? 2 : 1;  // output channels per thread
    if (c.OC / c.OT * c.NBH > 256) c.OC = 256 * c.OT / c.NBH;
    c.IC = std::max(1, std::min(Cin, 8192 / (32 * c.OC)));
    // one stage: w box (8 floats, OC, IC) then X box (8 floats, IC, BT)
    c.w_off = 0;
    c.x_off = (size_t)32 * c.OC * c.IC;
    c.stage_bytes = c.x_off + (size_t)32 * c.IC * c.BT;
    // ring depth: 4 stages when the batch tile is large (more CTAs per SM for
    // the FMA-heavy case), 6 when the weights stream nearly unused (HBM-bound)
    c.NST = c.BT >= 8 ? 4 : kMaxStages;
    c.smem = 128 + (size_t)c.NST * round128(c.stage_bytes);
    return c;
}

// Threads: (OC / OT) x NBH.  Thread t handles the OT output channels
// o0 + (t % (OC/OT)) + j * (OC/OT) and batch rows b0 + (t / (OC/OT)) * BTT .. + BTT.
template <int BTT, int OT>
__global__ void __launch_bounds__(256)
mix_tma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               float2* __restrict__ Z, int B, int Cin, int Cout, int NM, int OC, int IC, int BT,
               int kStages, unsigned* __restrict__ err) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    unsigned char* stages = smem + 128;
    const int tid = threadIdx.x;
    const int OS = OC / OT;  // stride between a thread's output channels
    const int ol = tid % OS, bh = tid / OS;
    const int m0 = blockIdx.x * 4, o0 = blockIdx.y * OC, b0 = blockIdx.z * BT;
    const int nch = (Cin + IC - 1) / IC;
    const uint32_t w_bytes = 32u * OC * IC;
    const uint32_t stage_bytes = w_bytes + 32u * IC * BT;
    const uint32_t stage_stride = (stage_bytes + 127u) / 128u * 128u;

    if (tid == 0) {
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    int issued = 0;  // stages handed to the TMA unit (thread 0 only)
    if (tid == 0) {
        for (; issued < kStages && issued < nch; ++issued) {
            unsigned char* st = stages + (size_t)issued * stage_stride;
            mbar_arrive_expect_tx(&bars[issued], stage_bytes);
            tma_load_3d(st, &tmW, 2 * m0, o0, issued * IC, &bars[issued]);
            tma_load_3d(st + w_bytes, &tmX, 2 * m0, issued * IC, b0, &bars[issued]);
        }
    }

    float2 acc[OT][BTT][4];
#pragma unroll
    for (int j = 0; j < OT; ++j)
#pragma unroll
        for (int bb = 0; bb < BTT; ++bb)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[j][bb][q] = make_float2(0.f, 0.f);

    // the two 16-byte halves of a thread's 32-byte w row are read in an order
    // that makes each quarter-warp touch 8 distinct 16-byte bank groups
    const int h = (tid >> 2) & 1;
    int consumed = 0;
    bool timed_out = false;
    for (int c = 0; c < nch; ++c) {
        const int s = c % kStages;
        const bool ok = wait_parity_bounded(&bars[s], (uint32_t)((c / kStages) & 1), err);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        consumed = c + 1;
        const unsigned char* st = stages + (size_t)s * stage_stride;
        const float4* Wst = reinterpret_cast<const float4*>(st);
        const float4* Xst = reinterpret_cast<const float4*>(st + w_bytes);  // [BT][IC][4 modes]
        const int ni = min(IC, Cin - c * IC);
        for (int ii = 0; ii < ni; ++ii) {
            float2 w[OT][4];
#pragma unroll
            for (int j = 0; j < OT; ++j) {
                const float4* wrow = Wst + (ii * OC + ol + j * OS) * 2;
                const float4 p0 = wrow[h], p1 = wrow[1 - h];
                const float4 lo = h ? p1 : p0, hi = h ? p0 : p1;
                w[j][0] = make_float2(lo.x, lo.y);
                w[j][1] = make_float2(lo.z, lo.w);
                w[j][2] = make_float2(hi.x, hi.y);
                w[j][3] = make_float2(hi.z, hi.w);
            }
#pragma unroll
            for (int bb = 0; bb < BTT; ++bb) {
                const float4* xr = Xst + ((bh * BTT + bb) * IC + ii) * 2;
                const float4 xa = xr[0], xb = xr[1];
                const float2 x0 = make_float2(xa.x, xa.y), x1 = make_float2(xa.z, xa.w);
                const float2 x2 = make_float2(xb.x, xb.y), x3 = make_float2(xb.z, xb.w);
#pragma unroll
                for (int j = 0; j < OT; ++j) {
                    cmac(acc[j][bb][0], x0, w[j][0]);
                    cmac(acc[j][bb][1], x1, w[j][1]);
                    cmac(acc[j][bb][2], x2, w[j][2]);
                    cmac(acc[j][bb][3], x3, w[j][3]);
                }
            }
        }
        __syncthreads();  // every thread is done with stage s
        if (tid == 0 && issued < nch) {
            unsigned char* st2 = stages + (size_t)s * stage_stride;
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
                wait_parity_bounded(&bars[c % kStages], (uint32_t)((c / kStages) & 1), nullptr);
        __syncthreads();
        return;
    }

    const bool vec = (NM & 3) == 0 && m0 + 3 < NM;
#pragma unroll
    for (int j = 0; j < OT; ++j) {
        const int o = o0 + ol + j * OS;
        if (o >= Cout) break;
#pragma unroll
        for (int bb = 0; bb < BTT; ++bb) {
            const int b = b0 + bh * BTT + bb;
            if (b >= B) break;
            float2* zp = Z + ((size_t)b * Cout + o) * NM + m0;
            if (vec) {
                reinterpret_cast<float4*>(zp)[0] =
                    make_float4(acc[j][bb][0].x, acc[j][bb][0].y, acc[j][bb][1].x, acc[j][bb][1].y);
                reinterpret_cast<float4*>(zp)[1] =
                    make_float4(acc[j][bb][2].x, acc[j][bb][2].y, acc[j][bb][3].x, acc[j][bb][3].y);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (m0 + q < NM) zp[q] = acc[j][bb][q];
            }
        }
    }
}

template <int BTT>
cudaError_t launch_btt(const CUtensorMap& mw, const CUtensorMap& mx, float2* Z, int B, int Cin,
                       int Cout, int NM, const MixTmaCfg& c, unsigned* err, cudaStream_t s) {
    dim3 grid((NM + 3) / 4, (Cout + c.OC - 1) / c.OC, (B + c.BT - 1) / c.BT);
    const int threads = c.OC / c.OT * c.NBH;
    if (c.OT == 2)
        mix_tma_kernel<BTT, 2><<<grid, threads, c.smem, s>>>(mw, mx, Z, B, Cin, Cout, NM, c.OC,
                                                             c.IC, c.BT, c.NST, err);
    else
        mix_tma_kernel<BTT, 1><<<grid, threads, c.smem, s>>>(mw, mx, Z, B, Cin, Cout, NM, c.OC,
                                                             c.IC, c.BT, c.NST, err);
    return cudaGetLastError();
}

template <int BTT>
cudaError_t set_attr() {
    cudaError_t e = cudaFuncSetAttribute(mix_tma_kernel<BTT, 1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mix_tma_kernel<BTT, 2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    return e;
}

}  // namespace
}  // namespace fno

using namespace fno;

fno_encode_tiled_fn fno_get_encode_tiled() {
    static fno_encode_tiled_fn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (fno_encode_tiled_fn) nullptr;
        return reinterpret_cast<fno_encode_tiled_fn>(p);
    }();
    return fn;
}

cudaError_t mix_tma_init() {
    cudaError_t e = set_attr<1>();
    if (e == cudaSuccess) e = set_attr<2>();
    if (e == cudaSuccess) e = set_attr<4>();
    if (e == cudaSuccess) e = set_attr<8>();
    if (e == cudaSuccess && !fno_get_encode_tiled()) e = cudaErrorNotSupported;
    return e;
}

bool mix_tma_supported(int B, int Cin, int Cout, int nm) {
    if (Cout < 32 || (nm & 1)) return false;
    return mix_tma_cfg(B, Cin, Cout).smem <= 227 * 1024;
}

// Encode a 3D tensor map over a complex64 array [d2][d1][NM] viewed as floats:
// dims (2*NM, d1, d2), box (8 floats = 4 modes, b1, b2).  Out-of-range box
// elements are filled with zeros.
static bool encode_modes_map(CUtensorMap* map, const float2* base, int NM, int d1, int d2,
                             int b1, int b2) {
    fno_encode_tiled_fn enc = fno_get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)NM * 2, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)NM * 8, (cuuint64_t)d1 * NM * 8};
    cuuint32_t box[3] = {8, (cuuint32_t)b1, (cuuint32_t)b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float2*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t launch_mix_tma(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                           cudaStream_t s, fno_launch_ctx* ctx) {
    const MixTmaCfg c = mix_tma_cfg(p.B, p.Cin, p.Cout);
    CUtensorMap mw, mx;
    if (!encode_modes_map(&mw, w, p.nm, p.Cout, p.Cin, c.OC, c.IC) ||
        !encode_modes_map(&mx, X, p.nm, p.Cin, p.B, c.IC, c.BT))
        return cudaErrorInvalidValue;
    cudaError_t e;
    switch (c.BTT) {
        case 1: e = launch_btt<1>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm, c, p.err, s); break;
        case 2: e = launch_btt<2>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm, c, p.err, s); break;
        case 4: e = launch_btt<4>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm, c, p.err, s); break;
        default: e = launch_btt<8>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm, c, p.err, s); break;
    }
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
