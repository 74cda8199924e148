// block_tc.cu -- the FNO block's epilogue with its pointwise branch on the
// tcgen05 tensor cores:
//   out[b,o,p] = act(y[b,o,p] + bias[o] + sum_i w_pw[o,i] * x[b,i,p]),  p = h*W + w,
// in place over y (the spectral layer's output), act = identity or GELU.  The
// 1x1 convolution is a dense product per batch row, D[p][o] = sum_i X^T[p][i]
// W^T[i][o] with M = 128 pixels per tile, N = Cout (<= 64) and K = Cin, which
// the tensor core takes in split TF32: each operand is split into its TF32
// part and the fp32 residual, and hi*hi + hi*lo + lo*hi are accumulated in
// fp32 (fp32 accuracy, as in the contraction kernels).
//
// Persistent: one CTA per SM takes every gridDim.x-th (batch row, 128-pixel
// tile) unit.  Warp roles:
//   warp 0    TMA producer: x in chunks of 16 channels ([16][128] floats, 3D
//             tensor map over [B][Cin][P], channels past Cin and pixels past P
//             read as zeros) into a ring of up to 12 stages;
//   warp 1    MMA issuer: per chunk 2 K steps x 3 products into the unit's
//             accumulator (128 lanes x N columns of tensor memory, two of them
//             so that a unit's read-out overlaps the next unit's products);
//   warps 2-5 converters: thread t owns pixel row t of the chunk and writes
//             the TF32 parts and residuals of its 16 channels as K-major
//             core-matrix tiles (16 bytes per 4 channels) in one of two operand
//             buffers;
//   warps 6-21 epilogue: warp w reads tensor-memory lanes 32 (w mod 4) .. + 31
//             (pixel rows), quarter (w - 6) / 4 of the accumulator columns, adds
//             them and the bias to the y tile in shared memory and applies the
//             activation;
//   warp 22   y tiles: lane 0 loads the units' y tiles ([Cout][128] floats)
//             into as many buffers (2 .. 4) as shared memory holds, writes each
//             finished tile back with a TMA store (pixels past P are not
//             written) and refills its buffer with the unit that many ahead as
//             soon as the store has read it.
// w_pw's split TF32 tiles ([Cin][N], K-major) are built once per CTA.
// Every wait is bounded (tma.cuh): after a timeout the error word is set, the
// producer and the store thread wait (bounded) for their copies in flight,
// every issued MMA completes before tensor memory is released, and the CTA
// returns; y is then partly written and void.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace fno {
namespace {

constexpr int kPx = 128;          // pixels per unit (MMA M)
constexpr int kCh = 16;           // input channels per chunk (2 MMA K steps)
constexpr int kMaxXS = 12;        // x ring depth at most
constexpr int kMaxY = 4;          // y tile buffers at most
constexpr int kConv = 128;        // converter threads (warps 2-5)
constexpr int kEpi = 512;         // epilogue threads (warps 6-21)
constexpr int kThreads = 64 + kConv + kEpi + 32;  // + the y tile warp (22)
constexpr uint32_t kXBytes = kCh * kPx * 4;      // 8 KB
constexpr uint32_t kATile = kPx * 8 * 4;         // one K step of A: 4 KB
constexpr uint32_t kASet = 2 * 2 * kATile;       // hi + lo, 2 K steps: 16 KB
constexpr size_t kSmemMax = kMaxDynSmem;  // less the range-checked build's static shared memory
constexpr int kMaxCinN = 4096;                   // padded Cin x N (w_pw tiles <= 32 KB)

__host__ __device__ inline int padded_cin(int Cin) { return (Cin + kCh - 1) / kCh * kCh; }
// MMA N: 16, 32 or 64 (a quarter of the columns per epilogue warp group)
inline int tc_n(int Cout) { return Cout <= 16 ? 16 : Cout <= 32 ? 32 : 64; }

// Shared memory: barriers | two operand sets | w_pw tiles (hi, lo) | bias |
// x ring (xs stages) | y tile buffers (ny).  The x loads and the y loads both
// cross DRAM latency (~5k cycles under load), so both rings are as deep as the
// budget allows: ny = 3 or 4 with at least 8 x stages where that fits, else
// 2 y buffers and the rest for x.
struct Layout {
    uint32_t off_a, off_b, off_bias, off_x, off_y, ybytes, ystride, bbytes;
    int xs, ny;
    size_t smem;
};

__host__ __device__ inline Layout layout(int Cinp, int N, int Cout) {
    Layout l;
    l.off_a = 1024;
    l.bbytes = (uint32_t)Cinp * (uint32_t)N * 4u;  // one of hi / lo
    l.off_b = l.off_a + 2 * kASet;
    l.off_bias = l.off_b + 2 * l.bbytes;
    l.off_x = l.off_bias + 1024;
    l.ybytes = (uint32_t)Cout * kPx * 4u;
    l.ystride = (l.ybytes + 1023u) & ~1023u;
    const size_t fixed = (size_t)l.off_x + 1024;  // + alignment slack
    const long long avail = (long long)kSmemMax - (long long)fixed;
    l.ny = 2;
    l.xs = 0;
    for (int ny = kMaxY; ny >= 2; --ny) {
        long long xs = (avail - (long long)ny * l.ystride) / kXBytes;
        if (xs > kMaxXS) xs = kMaxXS;
        if (xs >= 8 || ny == 2) {
            l.ny = ny;
            l.xs = xs > 0 ? (int)xs : 0;
            break;
        }
    }
    l.off_y = l.off_x + (uint32_t)l.xs * kXBytes;
    l.smem = fixed + (size_t)l.xs * kXBytes + (size_t)l.ny * l.ystride;
    return l;
}

// Byte offset of element (row, 4 k4 .. 4 k4 + 3) in a K-major no-swizzle tile
// of core matrices (8 rows x 16 bytes): LBO = 128 (along K), SBO = 256 (rows).
__device__ __forceinline__ uint32_t core_off(int row, int k4) {
    return (uint32_t)(((row >> 3) * 2 + k4) * 128 + (row & 7) * 16);
}

// TF32 part (round to nearest) and residual of four values.
__device__ __forceinline__ void split4(float4 v, float4& h, float4& l) {
    h = make_float4(to_tf32(v.x), to_tf32(v.y), to_tf32(v.z), to_tf32(v.w));
    l = make_float4(to_tf32(v.x - h.x), to_tf32(v.y - h.y), to_tf32(v.z - h.z),
                    to_tf32(v.w - h.w));
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1)
block_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                const float* __restrict__ w_pw, const float* __restrict__ bias, int B, int Cin,
                int Cout, int P, int act, int early, unsigned* __restrict__ err FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    const int Cinp = padded_cin(Cin);
    const Layout L = layout(Cinp, N, Cout);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [kMaxXS] x chunk landed
    uint64_t* empty = full + kMaxXS;                      // [kMaxXS] x chunk converted
    uint64_t* afull = empty + kMaxXS;                     // [2] operands written
    uint64_t* aempty = afull + 2;                         // [2] operands consumed
    uint64_t* dfull = aempty + 2;                         // [2] accumulator final
    uint64_t* dempty = dfull + 2;                         // [2] accumulator read out
    uint64_t* yfull = dempty + 2;                         // [kMaxY] y tile landed
    uint64_t* yready = yfull + kMaxY;                     // [kMaxY] y tile finished in smem
    uint64_t* done = yready + kMaxY;                      // every MMA completed
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    int* fail = reinterpret_cast<int*>(tslot + 1);
    unsigned char* xs = smem + L.off_x;
    unsigned char* as = smem + L.off_a;
    unsigned char* bs = smem + L.off_b;
    float* ys = reinterpret_cast<float*>(smem + L.off_y);
    const uint32_t ystride = L.ystride / 4u;  // floats between y buffers
    const int NY = L.ny, XS = L.xs;
    float* bsm = reinterpret_cast<float*>(smem + L.off_bias);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (P + kPx - 1) / kPx;
    const int units = B * ntiles;
    const int nu = (int)blockIdx.x < units ? (units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int nch = Cinp / kCh;
    const int G = nu * nch;
    const auto unit_b = [&](int j) { return ((int)blockIdx.x + j * (int)gridDim.x) / ntiles; };
    const auto unit_p0 = [&](int j) {
        return ((int)blockIdx.x + j * (int)gridDim.x) % ntiles * kPx;
    };

    if (tid == 0) {
        for (int s = 0; s < kMaxXS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConv);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&afull[t], kConv);
            mbar_init(&aempty[t], 1);
            mbar_init(&dfull[t], 1);
            mbar_init(&dempty[t], kEpi);
        }
        for (int t = 0; t < kMaxY; ++t) {
            mbar_init(&yfull[t], 1);
            mbar_init(&yready[t], kEpi);
        }
        mbar_init(done, 1);
        *fail = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tslot, 2 * N <= 32 ? 32 : (2 * N <= 64 ? 64 : 128));
    // w_pw^T as split TF32 K-major tiles: row o (N rows), K = input channel;
    // zero past Cin and Cout.  early: the kernel just before this one is the
    // library's inverse stage, which never writes w_pw or bias, so they may be
    // read before the programmatic-launch wait.
    if (!early) griddep_wait();
    for (int e = tid; e < (Cinp / 4) * N; e += kThreads) {
        const int o = e % N, i4 = e / N;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (o < Cout) {
            const float* wr = w_pw + (size_t)o * Cin + 4 * i4;
            if (4 * i4 < Cin) v.x = __ldg(wr);
            if (4 * i4 + 1 < Cin) v.y = __ldg(wr + 1);
            if (4 * i4 + 2 < Cin) v.z = __ldg(wr + 2);
            if (4 * i4 + 3 < Cin) v.w = __ldg(wr + 3);
        }
        float4 h, l;
        split4(v, h, l);
        // K step i4 / 2, half (i4 & 1) of its 8 channels
        const uint32_t off = (uint32_t)(i4 >> 1) * (uint32_t)N * 32u + core_off(o, i4 & 1);
        *reinterpret_cast<float4*>(bs + off) = h;
        *reinterpret_cast<float4*>(bs + L.bbytes + off) = l;
    }
    for (int o = tid; o < 64; o += kThreads) bsm[o] = (bias && o < Cout) ? __ldg(&bias[o]) : 0.f;
    fence_proxy_async_smem();  // w_pw tiles visible to the tensor core
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---- TMA producer ----
        if (lane == 0) {
            prefetch_tensormap(&tmX);
            prefetch_tensormap(&tmY);
            griddep_wait();  // y is the previous kernel's output
            griddep_launch_dependents();
            int issued = 0;
            for (int g = 0; g < G; ++g) {
                const int j = g / nch, c = g - j * nch, s = g % XS;
                if (g >= XS && !wait_parity_bounded(&empty[s], (uint32_t)((g / XS - 1) & 1), err)) {
                    atomicExch(fail, 1);
                    break;
                }
                if (*(volatile int*)fail) break;
                mbar_arrive_expect_tx(&full[s], kXBytes);
                tma_load_3d(xs + (size_t)s * kXBytes, &tmX, unit_p0(j), c * kCh, unit_b(j), &full[s]);
                issued = g + 1;
            }
            // no copy may be in flight when the CTA leaves
            for (int g = issued > XS ? issued - XS : 0; g < issued; ++g)
                wait_parity_bounded(&full[g % XS], (uint32_t)((g / XS) & 1), nullptr);
        } else {
            griddep_wait();
            griddep_launch_dependents();
        }
    } else if (warp == 1) {
        griddep_wait();
        griddep_launch_dependents();
        // ---- MMA issuer ----
        if (lane == 0) {
            const uint32_t idesc = idesc_tf32(kPx, N);
            const uint64_t a0 = smem_desc_noswz(as, 128, 256);
            const uint64_t b0 = smem_desc_noswz(bs, 128, 256);
            const uint64_t blo = (uint64_t)(L.bbytes >> 4);
            for (int g = 0; g < G; ++g) {
                const int j = g / nch, c = g - j * nch, a = g & 1, d = j & 1;
                if (!wait_parity_bounded(&afull[a], (uint32_t)((g >> 1) & 1), err)) {
                    atomicExch(fail, 1);
                    break;
                }
                // a unit's first chunk overwrites its accumulator: the read-out
                // of the unit two back must be done
                if (c == 0 && j >= 2 &&
                    !wait_parity_bounded(&dempty[d], (uint32_t)((j / 2 - 1) & 1), err)) {
                    atomicExch(fail, 1);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t dt = tmem + (uint32_t)(d * N);
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const uint64_t ah = a0 + (uint64_t)((a * kASet + ks * kATile) >> 4);
                    const uint64_t al = ah + (uint64_t)((2 * kATile) >> 4);
                    const uint64_t bh = b0 + (uint64_t)(((uint32_t)(2 * c + ks) * N * 32u) >> 4);
                    mma_tf32(dt, ah, bh, idesc, c > 0 || ks > 0);
                    mma_tf32(dt, ah, bh + blo, idesc, true);
                    mma_tf32(dt, al, bh, idesc, true);
                }
                mma_commit(&aempty[a]);
                if (c == nch - 1) mma_commit(&dfull[d]);
            }
            if (*(volatile int*)fail) {
                // the epilogue may be waiting for an accumulator that will not be
                // finished: release it (the output is void after a timeout)
                mma_commit(&dfull[0]);
                mma_commit(&dfull[1]);
            }
            mma_commit(done);
            if (!wait_parity_bounded(done, 0, nullptr)) {
                atomicExch(fail, 1);
                atomicOr(err, 2u /* FNO_DEVERR_TIMEOUT */);
            }
        }
    } else if (warp < 6) {
        griddep_wait();
        griddep_launch_dependents();
        // ---- converters: pixel row ct of each chunk ----
        const int ct = tid - 64;
        for (int g = 0; g < G; ++g) {
            const int s = g % XS, a = g & 1;
            bool ok = wait_parity_bounded(&full[s], (uint32_t)((g / XS) & 1), err);
            if (ok && g >= 2) ok = wait_parity_bounded(&aempty[a], (uint32_t)(((g - 2) >> 1) & 1), err);
            if (!ok) atomicExch(fail, 1);
            if (!ok || *(volatile int*)fail) break;
            const float* xc = reinterpret_cast<const float*>(xs + (size_t)s * kXBytes) + ct;
            unsigned char* ah = as + (size_t)a * kASet;
#pragma unroll
            for (int k4 = 0; k4 < kCh / 4; ++k4) {
                const float4 v = make_float4(xc[(4 * k4) * kPx], xc[(4 * k4 + 1) * kPx],
                                             xc[(4 * k4 + 2) * kPx], xc[(4 * k4 + 3) * kPx]);
                float4 h, l;
                split4(v, h, l);
                const uint32_t off = (uint32_t)(k4 >> 1) * kATile + core_off(ct, k4 & 1);
                *reinterpret_cast<float4*>(ah + off) = h;
                *reinterpret_cast<float4*>(ah + 2 * kATile + off) = l;
            }
            fence_proxy_async_smem();  // the tiles visible to the tensor core
            mbar_arrive(&afull[a]);
            mbar_arrive(&empty[s]);
        }
    } else if (warp < 22) {
        griddep_wait();
        griddep_launch_dependents();
        // ---- epilogue: pixel row 32 (warp mod 4) + lane, columns eh * N / 4 .. ----
        constexpr int NH = N / 4;
        const int q = warp & 3;
        const int pr = 32 * q + lane;
        const int et = tid - 64 - kConv;  // 0 .. 511
        const int eh = et >> 7;
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        for (int j = 0; j < nu; ++j) {
            const int d = j & 1, yb = j % NY;
            const uint32_t yph = (uint32_t)((j / NY) & 1);
            // every MMA of the unit completes before its accumulator is read
            // (bounded, not cut short by a forced timeout)
            const bool dok = wait_parity_bounded(&dfull[d], (uint32_t)((j >> 1) & 1), nullptr);
            if (!__all_sync(0xffffffffu, dok)) {
                atomicExch(fail, 1);
                atomicOr(err, 2u /* FNO_DEVERR_TIMEOUT */);
                break;
            }
            tc_fence_after_sync();
            float acc[NH];
            if constexpr (NH == 16) {
                tmem_ld16(trow + (uint32_t)(d * N + eh * NH), acc);
            } else if constexpr (NH == 8) {
                tmem_ld8(trow + (uint32_t)(d * N + eh * NH), acc);
            } else {
                tmem_ld4(trow + (uint32_t)(d * N + eh * NH), acc);
            }
            tmem_ld_wait();
            tc_fence_before_sync();
            mbar_arrive(&dempty[d]);  // the accumulator may be overwritten
            if (!wait_parity_bounded(&yfull[yb], yph, err)) {
                atomicExch(fail, 1);
                break;
            }
            // the thread's NH values: all loads, then the arithmetic (NH
            // independent chains, so the activation's latency overlaps), then
            // all stores
            float* yt = ys + (size_t)yb * ystride + (size_t)(eh * NH) * kPx + pr;
            const float* bt = bsm + eh * NH;
            const int nv = Cout - eh * NH;  // rows of this quarter inside the tile
            float yv[NH];
#pragma unroll
            for (int u = 0; u < NH; ++u) yv[u] = u < nv ? yt[u * kPx] : 0.f;
            if (act == FNO_ACT_GELU) {
#pragma unroll
                for (int u = 0; u < NH; ++u) {
                    const float v = yv[u] + acc[u] + bt[u];
                    yv[u] = 0.5f * v * (1.f + erff(v * 0.70710678118654752440f));
                }
            } else {
#pragma unroll
                for (int u = 0; u < NH; ++u) yv[u] += acc[u] + bt[u];
            }
#pragma unroll
            for (int u = 0; u < NH; ++u)
                if (u < nv) yt[u * kPx] = yv[u];
            fence_proxy_async_smem();  // the finished tile visible to the TMA store
            mbar_arrive(&yready[yb]);
        }
    } else {
        griddep_wait();  // y is the previous kernel's output
        griddep_launch_dependents();
        // ---- y tiles: loads ahead, stores behind ----
        if (lane == 0) {
            prefetch_tensormap(&tmY);
            int yissued = 0;
            const auto load_y = [&](int jj) {
                const int yb = jj % NY;
                mbar_arrive_expect_tx(&yfull[yb], L.ybytes);
                tma_load_3d(ys + (size_t)yb * ystride, &tmY, unit_p0(jj), 0, unit_b(jj), &yfull[yb]);
                yissued = jj + 1;
            };
            for (int jj = 0; jj < NY && jj < nu; ++jj) load_y(jj);
            int j = 0;
            for (; j < nu; ++j) {
                const int yb = j % NY;
                if (!wait_parity_bounded(&yready[yb], (uint32_t)((j / NY) & 1), err)) {
                    atomicExch(fail, 1);
                    break;
                }
                tma_store_3d(&tmY, ys + (size_t)yb * ystride, unit_p0(j), 0, unit_b(j));
                bulk_commit();
                bulk_wait_read0();  // the store has read the buffer
                if (j + NY < nu) load_y(j + NY);
            }
            bulk_wait_read0();  // every store has read its buffer
            // after a timeout: the y loads still in flight land before the CTA leaves
            for (int jj = j; jj < yissued; ++jj)
                wait_parity_bounded(&yfull[jj % NY], (uint32_t)((jj / NY) & 1), nullptr);
        }
    }

    tc_fence_before_sync();
    __syncthreads();  // the issuer has seen every MMA complete; no copy in flight
    if (warp == 1) tmem_dealloc(tmem, 2 * N <= 32 ? 32 : (2 * N <= 64 ? 64 : 128));
}

// 3D tensor map over a float array [B][C][P]: dims (P, C, B), box (128, bc, 1).
bool encode_map(CUtensorMap* map, const float* base, int B, int C, int P, int bc) {
    fno_encode_tiled_fn enc = fno_get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)P, (cuuint64_t)C, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)P * 4, (cuuint64_t)C * P * 4};
    cuuint32_t box[3] = {kPx, (cuuint32_t)bc, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(block_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemMax);
}

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t block_tc_init() {
    cudaError_t e = set_attr<16>();
    if (e == cudaSuccess) e = set_attr<32>();
    if (e == cudaSuccess) e = set_attr<64>();
    return e;
}

// Output channels up to 64 (one accumulator of N <= 64 columns per unit) and
// w_pw's split tiles within 32 KB.
bool block_tc_supported(int Cin, int Cout) {
    return Cin >= 1 && Cout >= 1 && Cout <= 64 &&
           (long long)padded_cin(Cin) * tc_n(Cout) <= kMaxCinN &&
           layout(padded_cin(Cin), tc_n(Cout), Cout).xs >= 4;
}

cudaError_t launch_block_tc(const fno_plan_s& p, const float* x, const float* w_pw,
                            const float* bias, int act, float* y, bool after_own_inverse,
                            cudaStream_t s) {
    const int P = p.H * p.W;
    CUtensorMap mx, my;
    if (!encode_map(&mx, x, p.B, p.Cin, P, kCh) || !encode_map(&my, y, p.B, p.Cout, P, p.Cout))
        return cudaErrorInvalidValue;
    const int N = tc_n(p.Cout);
    const int units = p.B * ((P + kPx - 1) / kPx);
    const int grid = units < p.sms ? units : p.sms;
    const size_t smem = layout(padded_cin(p.Cin), N, p.Cout).smem;
#define FNO_BLOCK_TC(NV)                                                                     \
    launch_pdl(block_tc_kernel<NV>, dim3(grid), dim3(kThreads), smem, s, mx, my, w_pw, bias, \
               p.B, p.Cin, p.Cout, P, act, after_own_inverse ? 1 : 0, p.err                 \
               FNO_DBG_ARG1(y, 4ull * p.B * p.Cout * P, p))
    if (N == 16) return FNO_BLOCK_TC(16);
    if (N == 32) return FNO_BLOCK_TC(32);
    return FNO_BLOCK_TC(64);
#undef FNO_BLOCK_TC
}
