// mix_tc.cu -- stage a3 on the tcgen05 tensor cores (TF32 operands, fp32
// accumulation in tensor memory):
//   Z[b,o,m] = sum_i X[b,i,m] * w[i,o,m]     (complex, per retained mode m)
// (TurboFNO: FFT-GEMM-iFFT fused operator page, sections 2.2-2.3: the per-mode
// complex product run on tensor cores.)
//
// Real form used per mode, for a block of 64 output channels:
//   D[(c,o), (c',b)] = sum_i A[(c,o), i] * Bop[i, (c',b)]
//   A[(c,o), i] = Re w[i,o] (c = 0) or Im w[i,o] (c = 1)      M = 128 rows
//   Bop[i, (c',b)] = Re X[b,i] (c' = 0) or Im X[b,i] (c' = 1) N = 2*Bp columns
//   Re Z[b,o] = D[(0,o),(0,b)] - D[(1,o),(1,b)],
//   Im Z[b,o] = D[(0,o),(1,b)] + D[(1,o),(0,b)]
// so each w and X element enters the products exactly once.  Bp is the batch
// rounded up to a multiple of 8; missing batch rows and channels are zeros.
//
// A CTA owns 4 consecutive modes and one block of 64 output channels and runs
// a warp-specialised pipeline over chunks of 8 input channels (one MMA K step):
//   warp 0: TMA producer -- the w box (4 modes x 64 channels x 8) and the X box
//           (4 modes x 8 x Bp) into a 3-stage ring (32-byte rows: one L2 sector
//           per row, so no sector is fetched twice);
//   warps 2-5: converters -- re-lay every stage into the canonical K-major
//           core-matrix tiles of each mode (rounding to TF32; for the split
//           variant also the TF32 residual), 2-deep tile ring;
//   warp 1: MMA issuer -- tcgen05.mma into 4 TMEM accumulators of N columns,
//           committing each tile's MMAs to the barrier that frees it.
// Stages and tiles hand over through mbarriers only (no CTA-wide barrier in
// the loop).  The epilogue reads TMEM with tcgen05.ld, combines the four real
// products into Z and stores it.
// With SPLIT = 3 each operand is split as hi + lo (both TF32) and
// hi*hi + hi*lo + lo*hi are accumulated, which recovers fp32-level accuracy.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace fno {
namespace {

constexpr int kQ = 4;        // modes per CTA (one 32-byte TMA row = one L2 sector)
constexpr int kIC = 8;       // input channels per chunk = MMA K (tf32)
constexpr int kNST = 3;      // TMA ring depth (two CTAs fit per SM)
constexpr int kNT = 2;       // operand tile ring depth
constexpr int kOB = 64;      // output channels per CTA (M = 2 * kOB = 128)
constexpr int kConv = 128;   // converter threads (warps 2..5)
constexpr int kT = 64 + kConv;

struct TcCfg {
    int Bp, N, ncols, split;
    uint32_t w_bytes, x_bytes, stage, tileA, tileB, tileset, off_stages, off_tiles;
    size_t smem;
};

__host__ __device__ inline uint32_t r1024(uint32_t v) { return (v + 1023u) & ~1023u; }

TcCfg tc_cfg(int B, int split) {
    TcCfg c;
    c.split = split;
    c.Bp = (B + 7) / 8 * 8;
    c.N = 2 * c.Bp;
    int cols = 32;
    while (cols < kQ * c.N) cols <<= 1;
    c.ncols = cols;
    c.w_bytes = 8u * kQ * kOB * kIC;          // 16 KB
    c.x_bytes = 8u * kQ * kIC * c.Bp;
    c.stage = r1024(c.w_bytes) + r1024(c.x_bytes);
    c.tileA = 128u * kIC * 4u;                // 4 KB
    c.tileB = (uint32_t)c.N * kIC * 4u;
    // one tile set: per mode A then B, for hi (and lo when split)
    c.tileset = r1024((c.tileA + c.tileB) * kQ * (split == 3 ? 2 : 1));
    c.off_stages = 1024;
    c.off_tiles = c.off_stages + kNST * c.stage;
    c.smem = (size_t)c.off_tiles + kNT * c.tileset + 1024;  // +1 KB alignment slack
    return c;
}

// Byte offset of element (row, k) (k < 8) inside a K-major no-swizzle tile of
// core matrices: core (row / 8, k / 4) at ((row / 8) * 2 + k / 4) * 128, row
// (row % 8) at 16-byte stride inside it.  LBO = 128, SBO = 256.
__device__ __forceinline__ uint32_t core_off(int row, int k4) {
    return (uint32_t)(((row >> 3) * 2 + k4) * 128 + (row & 7) * 16);
}

__device__ __forceinline__ float4 tf32x4(float4 v) {
    return make_float4(to_tf32(v.x), to_tf32(v.y), to_tf32(v.z), to_tf32(v.w));
}
__device__ __forceinline__ float4 sub4(float4 a, float4 b) {
    return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w);
}

// Write the TF32 operand rows (and for SPLIT = 3 the residual rows, kQ*(tileA +
// tileB) further on) of 4 consecutive K values.
template <int SPLIT>
__device__ __forceinline__ void put_row(unsigned char* tile, uint32_t lo_off, int row, int kh,
                                        float4 v) {
    const float4 h = tf32x4(v);
    *reinterpret_cast<float4*>(tile + core_off(row, kh)) = h;
    if (SPLIT == 3) *reinterpret_cast<float4*>(tile + lo_off + core_off(row, kh)) = tf32x4(sub4(v, h));
}

// Warp roles: warp 0 lane 0 issues the TMA loads, warp 1 lane 0 issues the
// MMAs, warps 2..5 convert TMA stages into operand tiles and run the
// epilogue.  Barriers: full[s] (TMA landed), empty[s] (converters done with
// stage s), tfull[t] (tile t written), tempty[t] (MMAs reading tile t done),
// done (all MMAs done).
template <int SPLIT>
__global__ void __launch_bounds__(kT)
mix_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              float2* __restrict__ Z, int B, int Cin, int Cout, int NM, int Bp, int N,
              int ncols, uint32_t stage_bytes, uint32_t x_off, uint32_t tileA, uint32_t tileB,
              uint32_t tileset, uint32_t off_stages, uint32_t off_tiles,
              unsigned* __restrict__ err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [kNST]
    uint64_t* empty = full + kNST;                        // [kNST]
    uint64_t* tfull = empty + kNST;                       // [kNT]
    uint64_t* tempty = tfull + kNT;                       // [kNT]
    uint64_t* done = tempty + kNT;                        // [1]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    int* fail = reinterpret_cast<int*>(tslot + 1);
    unsigned char* stages = smem + off_stages;
    unsigned char* tiles = smem + off_tiles;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * kQ, o0 = blockIdx.y * kOB;
    const int nch = (Cin + kIC - 1) / kIC;
    const uint32_t tx = 8u * kQ * kOB * kIC + 8u * kQ * kIC * Bp;
    const uint32_t lo_off = kQ * (tileA + tileB);

    if (tid == 0) {
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
        for (int s = 0; s < kNST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConv);
        }
        for (int t = 0; t < kNT; ++t) {
            mbar_init(&tfull[t], kConv);
            mbar_init(&tempty[t], 1);
        }
        mbar_init(done, 1);
        *fail = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tslot, (uint32_t)ncols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---- TMA producer ----
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c % kNST;
                if (c >= kNST &&
                    !wait_parity_bounded(&empty[s], (uint32_t)(((c - kNST) / kNST) & 1), err)) {
                    atomicExch(fail, 1);
                    break;
                }
                if (*(volatile int*)fail) break;
                unsigned char* st = stages + (size_t)s * stage_bytes;
                mbar_arrive_expect_tx(&full[s], tx);
                tma_load_3d(st, &tmW, 2 * m0, o0, c * kIC, &full[s]);
                tma_load_3d(st + x_off, &tmX, 2 * m0, c * kIC, 0, &full[s]);
                issued = c + 1;
            }
            // No copy may be in flight when the ring is reused or the CTA leaves.
            // Chunk c was refilled only after the converters had waited for
            // chunk c - kNST, so only the last kNST issued chunks may still be
            // landing (bounded waits that no error flag cuts short).
            for (int c = issued > kNST ? issued - kNST : 0; c < issued; ++c)
                wait_parity_bounded(&full[c % kNST], (uint32_t)((c / kNST) & 1), nullptr);
        }
    } else if (warp == 1) {
        // ---- MMA issuer ----
        if (lane == 0) {
            const uint32_t idesc = idesc_tf32(128, N);
            for (int c = 0; c < nch; ++c) {
                const int t = c % kNT;
                if (!wait_parity_bounded(&tfull[t], (uint32_t)((c / kNT) & 1), err)) {
                    atomicExch(fail, 1);
                    break;
                }
                tc_fence_after_sync();
                const unsigned char* ts = tiles + (size_t)t * tileset;
#pragma unroll
                for (int q = 0; q < kQ; ++q) {
                    const unsigned char* A = ts + q * (tileA + tileB);
                    const unsigned char* Bt = A + tileA;
                    const uint32_t d = tmem + (uint32_t)(q * N);
                    const uint64_t ah = smem_desc_noswz(A, 128, 256);
                    const uint64_t bh = smem_desc_noswz(Bt, 128, 256);
                    mma_tf32(d, ah, bh, idesc, c > 0);
                    if (SPLIT == 3) {
                        const uint64_t al = smem_desc_noswz(A + lo_off, 128, 256);
                        const uint64_t bl = smem_desc_noswz(Bt + lo_off, 128, 256);
                        mma_tf32(d, ah, bl, idesc, true);
                        mma_tf32(d, al, bh, idesc, true);
                    }
                }
                mma_commit(&tempty[t]);
            }
            mma_commit(done);  // arrives when every MMA above has completed
        }
    } else {
        // ---- converters: warps 2..5 ----
        const int ct = tid - 64;
        for (int c = 0; c < nch; ++c) {
            const int s = c % kNST, t = c % kNT;
            bool ok = wait_parity_bounded(&full[s], (uint32_t)((c / kNST) & 1), err);
            if (ok && c >= kNT)
                ok = wait_parity_bounded(&tempty[t], (uint32_t)(((c - kNT) / kNT) & 1), err);
            if (!ok) atomicExch(fail, 1);
            if (*(volatile int*)fail) break;
            tc_fence_after_sync();
            const unsigned char* st = stages + (size_t)s * stage_bytes;
            unsigned char* ts = tiles + (size_t)t * tileset;
            {   // w: thread (o = ct % 64, kh = ct / 64) -> channels 4*kh .. 4*kh + 3
                const int o = ct & 63, kh = ct >> 6;
                const int h = (o >> 2) & 1;  // order of the two 16-byte halves (bank spread)
                float4 wv[4][2];  // [channel][half]: (re, im) of modes 2*half, 2*half + 1
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    const float4* row =
                        reinterpret_cast<const float4*>(st + ((4 * kh + ii) * kOB + o) * (8 * kQ));
                    const float4 p0 = row[h], p1 = row[1 - h];
                    wv[ii][0] = h ? p1 : p0;
                    wv[ii][1] = h ? p0 : p1;
                }
#pragma unroll
                for (int q = 0; q < kQ; ++q) {
                    unsigned char* A = ts + q * (tileA + tileB);
                    const int hh = q >> 1;
                    const float4 re = (q & 1) == 0
                        ? make_float4(wv[0][hh].x, wv[1][hh].x, wv[2][hh].x, wv[3][hh].x)
                        : make_float4(wv[0][hh].z, wv[1][hh].z, wv[2][hh].z, wv[3][hh].z);
                    const float4 im = (q & 1) == 0
                        ? make_float4(wv[0][hh].y, wv[1][hh].y, wv[2][hh].y, wv[3][hh].y)
                        : make_float4(wv[0][hh].w, wv[1][hh].w, wv[2][hh].w, wv[3][hh].w);
                    put_row<SPLIT>(A, lo_off, o, kh, re);
                    put_row<SPLIT>(A, lo_off, 64 + o, kh, im);
                }
            }
            if (ct < 2 * Bp) {  // X: thread (b = ct % Bp, kh = ct / Bp)
                const int b = ct % Bp, kh = ct / Bp;
                float4 xv[4][2];
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    const float4* row = reinterpret_cast<const float4*>(
                        st + x_off + (b * kIC + 4 * kh + ii) * (8 * kQ));
                    xv[ii][0] = row[0];
                    xv[ii][1] = row[1];
                }
#pragma unroll
                for (int q = 0; q < kQ; ++q) {
                    unsigned char* Bt = ts + q * (tileA + tileB) + tileA;
                    const int hh = q >> 1;
                    const float4 re = (q & 1) == 0
                        ? make_float4(xv[0][hh].x, xv[1][hh].x, xv[2][hh].x, xv[3][hh].x)
                        : make_float4(xv[0][hh].z, xv[1][hh].z, xv[2][hh].z, xv[3][hh].z);
                    const float4 im = (q & 1) == 0
                        ? make_float4(xv[0][hh].y, xv[1][hh].y, xv[2][hh].y, xv[3][hh].y)
                        : make_float4(xv[0][hh].w, xv[1][hh].w, xv[2][hh].w, xv[3][hh].w);
                    put_row<SPLIT>(Bt, lo_off, b, kh, re);
                    put_row<SPLIT>(Bt, lo_off, Bp + b, kh, im);
                }
            }
            fence_proxy_async_smem();  // tiles visible to the tensor core
            mbar_arrive(&empty[s]);
            mbar_arrive(&tfull[t]);
        }
    }

    // ---- epilogue: wait for the last MMA, then TMEM -> Z ----
    // every issued MMA must complete before TMEM is read or released: this wait
    // is not cut short by a forced timeout (the issuer always commits `done`)
    bool ok = true;
    if (warp >= 2) ok = wait_parity_bounded(done, 0, nullptr);
    if (!ok) {
        atomicExch(fail, 1);
        atomicOr(err, 2u /* FNO_DEVERR_TIMEOUT */);
    }
    __syncthreads();
    const bool good = *(volatile int*)fail == 0;
    tc_fence_after_sync();
    if (good && warp >= 2) {
        const int quarter = warp & 3;                  // TMEM lanes 32*quarter ..
        const uint32_t trow = tmem + ((uint32_t)(32 * quarter) << 16);
        float* Ds = reinterpret_cast<float*>(stages);  // [64][N + 1]; the ring is idle
        const int ld = N + 1;
        for (int q = 0; q < kQ; ++q) {
            if (quarter >= 2) {  // rows (1, o): imaginary parts of w
                const int o = 32 * (quarter - 2) + lane;
                for (int n0 = 0; n0 < N; n0 += 16) {
                    float r[16];
                    tmem_ld16(trow + (uint32_t)(q * N + n0), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) Ds[o * ld + n0 + j] = r[j];
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
            if (quarter < 2) {   // rows (0, o)
                const int o = 32 * quarter + lane;
                const int og = o0 + o;
                for (int n0 = 0; n0 < Bp; n0 += 8) {
                    float r0[8], r1[8];
                    tmem_ld8(trow + (uint32_t)(q * N + n0), r0);       // columns (0, b)
                    tmem_ld8(trow + (uint32_t)(q * N + Bp + n0), r1);  // columns (1, b)
                    tmem_ld_wait();
                    if (og < Cout) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int b = n0 + j;
                            if (b < B) {
                                const float zr = r0[j] - Ds[o * ld + Bp + b];
                                const float zi = r1[j] + Ds[o * ld + b];
                                Z[((size_t)b * Cout + og) * NM + m0 + q] = make_float2(zr, zi);
                            }
                        }
                    }
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, (uint32_t)ncols);
}

template <int SPLIT>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(mix_tc_kernel<SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                227 * 1024);
}

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t mix_tc_init() {
    cudaError_t e = set_attr<1>();
    if (e == cudaSuccess) e = set_attr<3>();
    return e;
}

bool mix_tc_supported(int B, int Cin, int Cout, int nm, int split) {
    (void)Cin;
    (void)Cout;
    if (B > 32 || (nm % kQ)) return false;
    const TcCfg c = tc_cfg(B, split);
    return c.smem <= 227 * 1024 && c.ncols <= 512;
}

static bool encode_map(CUtensorMap* map, const float2* base, int NM, int d1, int d2, int b1,
                       int b2) {
    fno_encode_tiled_fn enc = fno_get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)NM * 2, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)NM * 8, (cuuint64_t)d1 * NM * 8};
    cuuint32_t box[3] = {2 * kQ, (cuuint32_t)b1, (cuuint32_t)b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float2*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_mix_tc(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                          int split, cudaStream_t s, fno_launch_ctx* ctx) {
    const TcCfg c = tc_cfg(p.B, split);
    CUtensorMap mw, mx;
    if (!encode_map(&mw, w, p.nm, p.Cout, p.Cin, kOB, kIC) ||
        !encode_map(&mx, X, p.nm, p.Cin, p.B, kIC, c.Bp))
        return cudaErrorInvalidValue;
    dim3 grid(p.nm / kQ, (p.Cout + kOB - 1) / kOB, 1);  // nm % kQ == 0 checked at plan time
    const uint32_t x_off = r1024(c.w_bytes);
    if (split == 3)
        mix_tc_kernel<3><<<grid, kT, c.smem, s>>>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm, c.Bp, c.N,
                                                  c.ncols, c.stage, x_off, c.tileA, c.tileB,
                                                  c.tileset, c.off_stages, c.off_tiles, p.err);
    else
        mix_tc_kernel<1><<<grid, kT, c.smem, s>>>(mw, mx, Z, p.B, p.Cin, p.Cout, p.nm, c.Bp, c.N,
                                                  c.ncols, c.stage, x_off, c.tileA, c.tileB,
                                                  c.tileset, c.off_stages, c.off_tiles, p.err);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
