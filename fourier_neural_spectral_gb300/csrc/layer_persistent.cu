// layer_persistent.cu -- the whole layer (stages a1..a5) in one launch.
//
// The forward transform, the per-mode contraction and the inverse transform
// of the FFT -> GEMM -> iFFT operator (TurboFNO: FFT-GEMM-iFFT fused operator
// page, sections 1 and 2.1-2.3: one operator, no launches between its stages)
// run as three phases of one cooperative grid whose CTAs all stay resident:
//
//   phase F: CTA c transforms planes (b, i) = c, c + G, ... (G CTAs) with the
//            fused forward code (rows, then the kept columns) into X;
//   grid barrier;
//   phase M: CTA c computes contraction units c, c + G, ...: 32 consecutive
//            modes (one per lane) x 8 output channels (one per warp) x every
//            batch row, with X and w staged through shared memory 4 input
//            channels at a time; Z = sum_i X w per mode;
//   grid barrier;
//   phase I: CTA c transforms planes (b, o) = c, c + G, ... from Z with the
//            fused inverse code into y.
//
// The contraction is all-to-all over the channels of each mode, so a plane's
// inverse needs every input plane's forward: the spectra X and Z cross CTAs
// through the plan's workspace, written and read within the launch (at these
// sizes it stays in L2), and reads of what other CTAs wrote in the launch go
// through L2 (ld.global.cg), never through the read-only path.
//
// Grid barrier: each CTA adds one arrival to a 64-bit counter that only grows
// (over barriers and launches: every launch adds exactly two arrivals per CTA)
// and waits until it reaches the next multiple of the grid size.  Writes before
// the barrier are published by a device-scope fence before the arrival, and
// the waiting side fences after it sees the count.  The wait is bounded by
// kWaitLimitNs of %globaltimer; a wait that runs out (or the forced-timeout
// test hook) sets FNO_DEVERR_TIMEOUT and the CTA skips the remaining phases
// but still arrives at the remaining barrier, so the counter stays a multiple
// of the grid size for the next launch.  The launch is cooperative, so every
// CTA of the grid is resident and the barrier cannot wait for a CTA that has
// not started.
//
// Shapes: square planes H = W in {32, 64, 128, 256} (one column pass per
// plane), batch up to 16.  Run when a caller asks for it
// (fno_plan_set_single_launch); plans default to the three launches, which
// overlap through programmatic dependent launch and measure faster.
#include <algorithm>

#include "fused_rows.cuh"

namespace fno {
namespace {

constexpr int kPT = 256;       // threads per CTA (the fused transforms' block)
constexpr int kUM = 32;        // contraction unit: modes (one per lane)
constexpr int kUO = 8;         // output channels (one per warp)
constexpr int kUB = 16;        // batch rows (all of them, B <= 16)
constexpr int kUI = 4;         // input channels per shared-memory tile
constexpr size_t kMixSmem = sizeof(float2) * (size_t)kUI * (kUO + kUB) * kUM;

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// One grid-wide barrier (see the file comment).  Returns false, CTA-uniform,
// if the wait gave up.
__device__ bool grid_barrier(unsigned long long* ctr, unsigned* err) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned long long G = gridDim.x;
        const unsigned long long target = (atomicAdd(ctr, 1ull) + G) / G * G;
        int ok = 1;
        if (__ldg(err + 1) & 1u) {
            ok = 0;  // forced-timeout test hook
        } else if (ld_acquire_u64(ctr) < target) {
            const uint64_t t0 = global_ns();
            while (ld_acquire_u64(ctr) < target) {
                if (global_ns() - t0 > kWaitLimitNs) {
                    ok = 0;
                    break;
                }
                __nanosleep(256);
            }
        }
        if (!ok) atomicOr(err, 2u /* FNO_DEVERR_TIMEOUT */);
        __threadfence();
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

// Contraction unit u: modes m0 .. m0 + 31 (lane), output channels o0 .. o0 + 7
// (warp), batch rows 0 .. B - 1 (B <= 16).  X was written in this launch: read
// through L2.
__device__ __forceinline__ void mix_unit(unsigned char* smem, const float2* X,
                                         const float2* __restrict__ w, float2* Z, int B, int Cin,
                                         int Cout, int NM, int m0, int o0) {
    float2(*sX)[kUB][kUM] = reinterpret_cast<float2(*)[kUB][kUM]>(smem);
    float2(*sW)[kUO][kUM] =
        reinterpret_cast<float2(*)[kUO][kUM]>(smem + sizeof(float2) * kUI * kUB * kUM);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float2 acc[kUB];
#pragma unroll
    for (int b = 0; b < kUB; ++b) acc[b] = make_float2(0.f, 0.f);
    for (int i0 = 0; i0 < Cin; i0 += kUI) {
        for (int e = threadIdx.x; e < kUI * kUB * kUM; e += kPT) {
            const int mm = e % kUM, bb = (e / kUM) % kUB, ii = e / (kUM * kUB);
            const int m = m0 + mm, i = i0 + ii;
            sX[ii][bb][mm] = (m < NM && bb < B && i < Cin)
                                 ? __ldcg(&X[((size_t)bb * Cin + i) * NM + m])
                                 : make_float2(0.f, 0.f);
        }
        for (int e = threadIdx.x; e < kUI * kUO * kUM; e += kPT) {
            const int mm = e % kUM, oo = (e / kUM) % kUO, ii = e / (kUM * kUO);
            const int m = m0 + mm, o = o0 + oo, i = i0 + ii;
            sW[ii][oo][mm] = (m < NM && o < Cout && i < Cin)
                                 ? __ldg(&w[((size_t)i * Cout + o) * NM + m])
                                 : make_float2(0.f, 0.f);
        }
        __syncthreads();
#pragma unroll
        for (int ii = 0; ii < kUI; ++ii) {
            const float2 wv = sW[ii][warp][lane];
#pragma unroll
            for (int b = 0; b < kUB; ++b) cmac(acc[b], sX[ii][b][lane], wv);
        }
        __syncthreads();
    }
    const int m = m0 + lane, o = o0 + warp;
    if (m < NM && o < Cout) {
#pragma unroll
        for (int b = 0; b < kUB; ++b)
            if (b < B && FNO_DBG_OK(&Z[((size_t)b * Cout + o) * NM + m], sizeof(float2)))
                Z[((size_t)b * Cout + o) * NM + m] = acc[b];
    }
}

template <int W, int M1S, int M2S>
__global__ void __launch_bounds__(kPT, (W <= 128 ? 2 : 1))
layer_persistent_kernel(const float* __restrict__ x, const float2* __restrict__ w,
                        float* __restrict__ y, float2* X, float2* Z, int B, int Cin, int Cout,
                        int m1, int m2, float scale, const float2* __restrict__ tw_w,
                        const float2* __restrict__ tw_h, unsigned long long* gbar,
                        unsigned* __restrict__ err FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    constexpr int H = W, R = W;  // square planes, one column pass
    using C = FusedCfg<W, R>;
    extern __shared__ __align__(16) float2 sm[];
    float2* scr = sm;
    float2* Yv = sm + C::Scratch;  // Y (forward) / V (inverse): [R][ys]
    const int ys = kept_stride(M2S ? M2S : m2);
    const int G = gridDim.x;
    const int NM = 2 * m1 * m2;

    // ---- phase F: forward transforms of the input planes -----------------
    for (int plane = blockIdx.x; plane < B * Cin; plane += G)
        fwd_fused_plane<W, R, M1S, M2S>(scr, Yv, ys, x + (size_t)plane * H * W, X, H, m1, m2, 1,
                                        plane, 0, scale, tw_w, tw_h);
    bool ok = grid_barrier(gbar, err);

    // ---- phase M: the per-mode contraction ------------------------------
    if (ok) {
        const int nob = (Cout + kUO - 1) / kUO;
        const int units = ((NM + kUM - 1) / kUM) * nob;
        for (int u = blockIdx.x; u < units; u += G)
            mix_unit(reinterpret_cast<unsigned char*>(sm), X, w, Z, B, Cin, Cout, NM,
                     (u / nob) * kUM, (u % nob) * kUO);
    }
    ok = grid_barrier(gbar, err) && ok;

    // ---- phase I: inverse transforms of the output planes ---------------
    if (ok) {
        for (int plane = blockIdx.x; plane < B * Cout; plane += G) {
            columns_inverse<R, M1S, false, true>(scr, Yv, ys, Z + (size_t)plane * NM, H, m1, m2, 1,
                                                 0, tw_h);
            __syncthreads();
            inv_rows_plane<W, R, M2S>(scr, Yv, ys, y, H, m2, 1, plane, 0, scale, tw_w);
            __syncthreads();
        }
    }
}

template <int W>
size_t persistent_smem(int m2) {
    return std::max(fused_smem_bytes<W, W>(m2), kMixSmem);
}

// Dynamic shared memory a block may have besides the kernel's static shared
// memory (the barrier's flag): the device's opt-in limit minus that, rounded
// down to 1 KB.
constexpr size_t kSmemLimit = 227 * 1024 - 1024;

template <int W, int M1S, int M2S>
cudaError_t set_attr_one() {
    const int bytes = (int)std::min<size_t>(persistent_smem<W>(W / 2 + 1), kSmemLimit);
    return cudaFuncSetAttribute(layer_persistent_kernel<W, M1S, M2S>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int W, int M1S, int M2S>
cudaError_t launch_one(const fno_plan_s& p, const float* x, const float2* w, float* y, float2* X,
                       float2* Z, cudaStream_t s) {
    auto kern = layer_persistent_kernel<W, M1S, M2S>;
    const size_t smem = persistent_smem<W>(p.m2);
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int work = std::max(p.B * std::max(p.Cin, p.Cout), 1);
    const int grid = std::min(per_sm * p.sms, work);
    int B = p.B, Cin = p.Cin, Cout = p.Cout, m1 = p.m1, m2 = p.m2;
    float scale = p.scale;
    const float2* tw_w = p.tw_w;
    const float2* tw_h = p.tw_h;
    unsigned long long* gbar = p.gbar;
    unsigned* err = p.err;
#ifdef FNO_DEBUG
    // the spectra X and Z are adjacent in the workspace: one range covers both
    fno_dbg_ranges dbg = FNO_DBG_RANGES2(
        X, (size_t)((const char*)Z - (const char*)X) + 8ull * p.B * p.Cout * p.nm, y,
        4ull * p.B * p.Cout * p.H * p.W, p);
    void* args[] = {(void*)&x, (void*)&w, (void*)&y, (void*)&X, (void*)&Z, &B, &Cin, &Cout,
                    &m1, &m2, &scale, (void*)&tw_w, (void*)&tw_h, (void*)&gbar, (void*)&err,
                    (void*)&dbg};
#else
    void* args[] = {(void*)&x, (void*)&w, (void*)&y, (void*)&X, (void*)&Z, &B, &Cin, &Cout,
                    &m1, &m2, &scale, (void*)&tw_w, (void*)&tw_h, (void*)&gbar, (void*)&err};
#endif
    return cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kPT), args, smem, s);
}

template <int W>
cudaError_t launch_w(const fno_plan_s& p, const float* x, const float2* w, float* y, float2* X,
                     float2* Z, cudaStream_t s) {
    if (p.m1 == W / 4 && p.m2 == W / 4) return launch_one<W, W / 4, W / 4>(p, x, w, y, X, Z, s);
    return launch_one<W, 0, 0>(p, x, w, y, X, Z, s);
}

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t layer_persistent_init() {
    cudaError_t e = set_attr_one<32, 0, 0>();
    if (e == cudaSuccess) e = set_attr_one<32, 8, 8>();
    if (e == cudaSuccess) e = set_attr_one<64, 0, 0>();
    if (e == cudaSuccess) e = set_attr_one<64, 16, 16>();
    if (e == cudaSuccess) e = set_attr_one<128, 0, 0>();
    if (e == cudaSuccess) e = set_attr_one<128, 32, 32>();
    if (e == cudaSuccess) e = set_attr_one<256, 0, 0>();
    if (e == cudaSuccess) e = set_attr_one<256, 64, 64>();
    return e;
}

bool layer_persistent_supported(const fno_plan_s& p) {
    if (p.dims != 2 || p.path != 1 || p.H != p.W || p.P != 1 || p.Pi != 1) return false;
    if (p.W != 32 && p.W != 64 && p.W != 128 && p.W != 256) return false;
    if (p.B < 1 || p.B > kUB) return false;
    size_t smem = 0;
    switch (p.W) {
        case 32: smem = persistent_smem<32>(p.m2); break;
        case 64: smem = persistent_smem<64>(p.m2); break;
        case 128: smem = persistent_smem<128>(p.m2); break;
        default: smem = persistent_smem<256>(p.m2); break;
    }
    return smem <= kSmemLimit;
}

cudaError_t launch_layer_persistent(const fno_plan_s& p, const float* x, const float2* w,
                                    float* y, float2* X, float2* Z, cudaStream_t s,
                                    fno_launch_ctx* ctx) {
    cudaError_t e;
    switch (p.W) {
        case 32: e = launch_w<32>(p, x, w, y, X, Z, s); break;
        case 64: e = launch_w<64>(p, x, w, y, X, Z, s); break;
        case 128: e = launch_w<128>(p, x, w, y, X, Z, s); break;
        case 256: e = launch_w<256>(p, x, w, y, X, Z, s); break;
        default: return cudaErrorInvalidValue;
    }
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
