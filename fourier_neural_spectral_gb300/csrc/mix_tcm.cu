// mix_tcm.cu -- stage a3 on the tcgen05 tensor cores with the weight operand
// held in tensor memory:
//   Z[b,o,m] = sum_i X[b,i,m] * w[i,o,m]     (complex, per retained mode m)
// (TurboFNO: FFT-GEMM-iFFT fused operator page, sections 2.2-2.3: the per-mode
// complex product on tensor cores; the real 2 x 2 block form below.)
//
// Real form per mode m, for a block of 64 output channels and Bp batch rows
// (Bp = 8 or 16; missing rows, channels and modes are TMA zero fill):
//   D[(o,c), (c',b)] = sum_i A[(o,c), i] * Bop[i, (c',b)]
//   A[(o,c), i]     = Re w[i,o] (c = 0) or Im w[i,o] (c = 1)   M = 128 rows 2o + c
//   Bop[i, (c',b)]  = Re X[b,i] (c' = 0) or Im X[b,i] (c' = 1) N = 2*Bp columns c'*Bp + b
//   Re Z[b,o] = D[(o,0),(0,b)] - D[(o,1),(1,b)],  Im Z[b,o] = D[(o,0),(1,b)] + D[(o,1),(0,b)]
// Rows 2o and 2o + 1 are neighbouring lanes of one warp, so the combination is
// one shuffle.  With SPLIT = 3 each operand is split into a TF32 high part and
// a TF32 residual and hi*hi + hi*lo + lo*hi are accumulated in fp32, which
// keeps the product at fp32 accuracy; SPLIT = 1 uses the high parts alone.
//
// A CTA owns 8 consecutive modes (one 64-byte row per (channel, channel) pair)
// and 64 output channels, and runs over the input channels in chunks of 8
// (one MMA K step):
//   warp 0: TMA producer -- the w box (8 modes x 64 outputs x 8 inputs, 32 KB)
//           and the X box (8 modes x 8 inputs x Bp) into a 3-stage ring, both
//           with the 64-byte swizzle (16-byte chunk index XOR row bits 1-2), so
//           that the converters' 16-byte reads of consecutive rows fall on
//           distinct banks;
//   warps 2-9: converters -- warp w may address TMEM lanes 32q .. 32q + 31
//           (q = w mod 4), i.e. rows (o, c) with o = 16q + lane/2, c = lane mod 2;
//           warps w and w + 4 split the 8 modes in halves.  Each thread reads its
//           w rows for the 8 inputs of the chunk (the two lanes of a row pair
//           read the same addresses, one shared-memory wavefront) and writes the
//           TF32 parts of its row for its 4 modes into tensor memory
//           (tcgen05.st), so the tensor core reads the weight operand from
//           tensor memory and never from shared memory; X is re-laid into
//           canonical K-major core-matrix tiles in shared memory (the B
//           operand);
//   warp 1: MMA issuer -- per chunk and mode, 1 or 3 tcgen05.mma (A from
//           tensor memory, B from shared memory) into the mode's accumulator
//           (N columns of TMEM), committing each chunk to the barrier that
//           frees its operand buffers.
// Tensor memory: 8 accumulators of N columns, then two operand buffers of
// 8 modes x 16 columns (8 high, 8 residual); 512 columns, one CTA per SM
// (its shared memory, about 218 KB, admits no second one).
// The split: high = v rounded to TF32 (add half a TF32 unit to the magnitude
// bits, clear the 13 low mantissa bits: two integer operations), residual =
// v - high exactly in fp32, which the tensor core reads as TF32 (dropping at
// most 2^-10 of a residual that is itself below 2^-11 |v|).
// The grid is persistent: one CTA per SM takes every gridDim.x-th (mode block,
// output block) unit, and the producer streams the chunks of its units back to
// back, so a unit's first data and its read-out overlap the neighbouring
// units' copies.  After a unit's last chunk the converter warps wait for its
// MMAs, read the accumulators (tcgen05.ld), combine them, stage the unit's Z
// in shared memory, release the accumulators to the next unit and copy the
// staged rows out with coalesced 16-byte stores (whole 64-byte runs of Z).
// Every wait is bounded (tma.cuh); after a timeout the error word is set, the
// producer waits for its copies in flight, every issued MMA completes before
// tensor memory is read or released, and the CTA returns.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace fno {
namespace {

constexpr int kQM = 8;      // modes per CTA (64-byte rows)
constexpr int kIC = 8;      // input channels per chunk = MMA K (tf32)
constexpr int kOB = 64;     // output channels per CTA (M = 128 = 64 x Re/Im)
constexpr int kNST = 3;     // TMA ring depth
constexpr int kNT = 2;      // operand buffers (A in TMEM, B in shared memory)
constexpr int kConv = 256;  // converter threads (warps 2..9: two per TMEM lane quarter)
constexpr int kThreads = 64 + kConv;
constexpr uint32_t kRow = kQM * 8;                 // 64 bytes
constexpr uint32_t kWBytes = kIC * kOB * kRow;     // 32 KB
constexpr uint32_t kTmemCols = 512;

template <int BP>
struct TcmCfg {
    static constexpr int N = 2 * BP;
    static constexpr uint32_t XBytes = BP * kIC * kRow;
    static constexpr uint32_t Stage = kWBytes + XBytes;           // a multiple of 1 KB
    static constexpr uint32_t BTile = N * kIC * 4;                // one mode, hi or lo
    static constexpr uint32_t BSet = 2 * kQM * BTile;             // hi + lo, 8 modes
    static constexpr uint32_t OffStages = 1024;
    static constexpr uint32_t OffB = OffStages + kNST * Stage;
    static constexpr uint32_t OffZ = OffB + kNT * BSet;           // Z staging
    static constexpr uint32_t ZBytes = BP * kOB * kRow;           // [Bp][64 o][8 modes]
    static constexpr size_t Smem = OffZ + ZBytes + 1024;          // + alignment slack
    static constexpr uint32_t DCols = kQM * N;                    // accumulators
    static constexpr uint32_t ACols = kQM * 2 * kIC;              // one operand buffer
    static_assert(Stage % 1024 == 0 && BSet % 1024 == 0, "1 KB aligned buffers");
    static_assert(DCols + kNT * ACols <= kTmemCols, "tensor memory budget");
};

// Byte offset of element (n, k) (k < 8) in a K-major no-swizzle tile of core
// matrices (8 rows x 16 bytes): core (n / 8, k / 4) at ((n / 8) * 2 + k / 4) *
// 128, row n % 8 at 16-byte stride inside it: LBO = 128, SBO = 256.
__device__ __forceinline__ uint32_t core_off(int n, int k) {
    return (uint32_t)(((n >> 3) * 2 + (k >> 2)) * 128 + (n & 7) * 16 + (k & 3) * 4);
}

// Physical byte offset of 16-byte chunk j of 64-byte row r under the 64-byte
// TMA swizzle (chunk bits 4-5 XOR address bits 7-8; buffers 1 KB aligned).
__device__ __forceinline__ uint32_t swz64(uint32_t r, uint32_t j) {
    return r * kRow + ((j ^ ((r >> 1) & 3u)) << 4);
}

// TF32 high part of v: round to nearest on the magnitude (ties away from
// zero), 10 explicit mantissa bits kept.
__device__ __forceinline__ float tf32_hi(float v) {
    return __uint_as_float((__float_as_uint(v) + 0x1000u) & 0xffffe000u);
}

template <int BP, int SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
mix_tcm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               float2* __restrict__ Z, int B, int Cin, int Cout, int NM, int early_w,
               unsigned* __restrict__ err FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    using C = TcmCfg<BP>;
    constexpr int N = C::N;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [kNST] stage landed
    uint64_t* empty = full + kNST;                        // [kNST] stage converted
    uint64_t* afull = empty + kNST;                       // [kNT] operands written
    uint64_t* aempty = afull + kNT;                       // [kNT] operands consumed
    uint64_t* dfull = aempty + kNT;                       // unit's accumulators final
    uint64_t* dempty = dfull + 1;                         // unit's accumulators read out
    uint64_t* done = dempty + 1;                          // every MMA completed
    uint64_t* zready = done + 1;                          // unit's Z staged
    uint64_t* zfree = zready + 1;                         // staged Z copied out
    uint32_t* tslot = reinterpret_cast<uint32_t*>(zfree + 1);
    int* fail = reinterpret_cast<int*>(tslot + 1);
    unsigned char* stages = smem + C::OffStages;
    unsigned char* bsets = smem + C::OffB;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = (Cin + kIC - 1) / kIC;
    const int nob = (Cout + kOB - 1) / kOB;
    const int units = ((NM + kQM - 1) / kQM) * nob;
    // this CTA's units: blockIdx.x, blockIdx.x + gridDim.x, ...; unit u is mode
    // block u / nob and output block u % nob (the output blocks of one mode
    // block are consecutive, so their shared X boxes stay in L2)
    const int nu = blockIdx.x < units ? (units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int G = nu * nch;  // chunks of this CTA, unit-major
    const auto unit_m0 = [&](int k) { return ((int)blockIdx.x + k * (int)gridDim.x) / nob * kQM; };
    const auto unit_o0 = [&](int k) { return ((int)blockIdx.x + k * (int)gridDim.x) % nob * kOB; };

    if (tid == 0) {
        for (int s = 0; s < kNST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConv);
        }
        for (int t = 0; t < kNT; ++t) {
            mbar_init(&afull[t], kConv);
            mbar_init(&aempty[t], 1);
        }
        mbar_init(dfull, 1);
        mbar_init(dempty, kConv);
        mbar_init(done, 1);
        mbar_init(zready, kConv);
        mbar_init(zfree, kConv);
        *fail = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tslot, kTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // ---- TMA producer: the CTA's chunks, unit after unit ----
        if (lane == 0) {
            prefetch_tensormap(&tmW);
            prefetch_tensormap(&tmX);
            const int pre = G < kNST ? G : kNST;
            const auto load_w = [&](int g) {
                const int k = g / nch, c = g - k * nch;
                unsigned char* st = stages + (size_t)(g % kNST) * C::Stage;
                mbar_arrive_expect_tx(&full[g % kNST], C::Stage);
                tma_load_3d(st, &tmW, 2 * unit_m0(k), unit_o0(k), c * kIC, &full[g % kNST]);
            };
            const auto load_x = [&](int g) {
                const int k = g / nch, c = g - k * nch;
                unsigned char* st = stages + (size_t)(g % kNST) * C::Stage;
                tma_load_3d(st + kWBytes, &tmX, 2 * unit_m0(k), c * kIC, 0, &full[g % kNST]);
            };
            // early_w: the kernel just before is the library's own forward stage,
            // which never writes w, so the first w boxes may be fetched before
            // the programmatic-launch wait
            if (early_w)
                for (int g = 0; g < pre; ++g) load_w(g);
            griddep_wait();
            griddep_launch_dependents();
            for (int g = 0; g < pre; ++g) {
                if (!early_w) load_w(g);
                load_x(g);
            }
            int issued = pre;
            for (int g = pre; g < G; ++g) {
                const int s = g % kNST;
                if (!wait_parity_bounded(&empty[s], (uint32_t)((g / kNST - 1) & 1), err)) {
                    atomicExch(fail, 1);
                    break;
                }
                if (*(volatile int*)fail) break;
                load_w(g);
                load_x(g);
                issued = g + 1;
            }
            // no copy may be in flight when the CTA leaves: only the last kNST
            // issued chunks are not known to have landed
            for (int g = issued > kNST ? issued - kNST : 0; g < issued; ++g)
                wait_parity_bounded(&full[g % kNST], (uint32_t)((g / kNST) & 1), nullptr);
        } else {
            griddep_wait();
            griddep_launch_dependents();
        }
    } else if (warp == 1) {
        griddep_wait();
        griddep_launch_dependents();
        // ---- MMA issuer ----
        // One thread issues every MMA, so the loop body is kept to immediate
        // offsets: a shared-memory descriptor's address field is the byte
        // address / 16, so a tile b bytes further is the base descriptor + b/16
        // (every offset here is a multiple of 16 and stays below 256 KB).
        if (lane == 0) {
            const uint32_t idesc = idesc_tf32(128, N);
            const uint64_t bdesc0 = smem_desc_noswz(bsets, 128, 256);
            for (int g = 0; g < G; ++g) {
                const int k = g / nch, c = g - k * nch;
                const int t = g % kNT;
                if (!wait_parity_bounded(&afull[t], (uint32_t)((g / kNT) & 1), err)) {
                    atomicExch(fail, 1);
                    break;
                }
                // a unit's first chunk overwrites the accumulators: the previous
                // unit's must have been read out
                if (c == 0 && k > 0 &&
                    !wait_parity_bounded(dempty, (uint32_t)((k - 1) & 1), err)) {
                    atomicExch(fail, 1);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t abuf = tmem + C::DCols + (uint32_t)t * C::ACols;
                const uint64_t bbuf = bdesc0 + (uint64_t)((t * C::BSet) >> 4);
                const bool acc0 = c > 0;
                // the products of a mode go to the same accumulator: issue them
                // term by term over the modes
#pragma unroll
                for (int term = 0; term < (SPLIT == 3 ? 3 : 1); ++term) {
#pragma unroll
                    for (int m = 0; m < kQM; ++m) {
                        const uint32_t bofs = (uint32_t)((term == 1 ? kQM + m : m) * C::BTile) >> 4;
                        mma_tf32_ts(tmem + (uint32_t)(m * N),
                                    abuf + (uint32_t)(m * 2 * kIC + (term == 2 ? kIC : 0)),
                                    bbuf + bofs, idesc, term > 0 || acc0);
                    }
                }
                mma_commit(&aempty[t]);
                if (c == nch - 1) mma_commit(dfull);
            }
            mma_commit(done);  // arrives once every MMA above has completed
            // the issuer waits for it before the CTA may release tensor memory
            // (not cut short by a forced timeout)
            if (!wait_parity_bounded(done, 0, nullptr)) {
                atomicExch(fail, 1);
                atomicOr(err, 2u /* FNO_DEVERR_TIMEOUT */);
            }
        }
    } else {
        griddep_wait();  // X is the previous kernel's output; Z may still be read
        griddep_launch_dependents();
        // ---- converters and epilogue: warps 2..9 ----
        const int ct = tid - 64;
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int hm = (warp - 2) >> 2;         // modes 4*hm .. 4*hm + 3
        const int o = 16 * q + (lane >> 1);     // output channel within the block
        const int cw = lane & 1;                // 0: Re w, 1: Im w
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        // w row (i, o) starts at byte (i*64 + o)*64; its 16-byte chunk j sits at
        // chunk j ^ ((o >> 1) & 3) (64-byte swizzle; i*64 leaves bits 7-8 alone)
        const uint32_t wsw = (uint32_t)((o >> 1) & 3);
        const uint32_t wofs0 = (uint32_t)o * kRow + (((2 * hm) ^ wsw) << 4);
        const uint32_t wofs1 = (uint32_t)o * kRow + (((2 * hm + 1) ^ wsw) << 4);
        // X: input xi of the chunk, batch row xb, mode pairs 2*xh and 2*xh + 1
        const int xi = ct & 7, xb = (ct >> 3) & 15, xh = ct >> 7;
        const uint32_t xr = (uint32_t)(xb * kIC + xi);
        const uint32_t xsw = (xr >> 1) & 3u;
        unsigned char* zst = smem + C::OffZ;
        for (int g = 0; g < G; ++g) {
            const int k = g / nch, c = g - k * nch;
            const int s = g % kNST, t = g % kNT;
            bool ok = wait_parity_bounded(&full[s], (uint32_t)((g / kNST) & 1), err);
            if (ok && g >= kNT)
                ok = wait_parity_bounded(&aempty[t], (uint32_t)(((g - kNT) / kNT) & 1), err);
            if (!ok) atomicExch(fail, 1);
            // the decision to stop is the warp's (tcgen05.st and wait::st below are
            // warp-collective: every lane executes them or none)
            if (__any_sync(0xffffffffu, !ok || *(volatile int*)fail != 0)) break;
            tc_fence_after_sync();
            const unsigned char* st = stages + (size_t)s * C::Stage;
            // w rows (i, o): this thread's component of modes 4*hm .. 4*hm + 3
            float v[kIC][4];
#pragma unroll
            for (int i = 0; i < kIC; ++i) {
                const unsigned char* row = st + (uint32_t)i * (kOB * kRow);
                const float4 p0 = *reinterpret_cast<const float4*>(row + wofs0);
                const float4 p1 = *reinterpret_cast<const float4*>(row + wofs1);
                v[i][0] = cw ? p0.y : p0.x;
                v[i][1] = cw ? p0.w : p0.z;
                v[i][2] = cw ? p1.y : p1.x;
                v[i][3] = cw ? p1.w : p1.z;
            }
            const uint32_t abuf = trow + C::DCols + (uint32_t)t * C::ACols;
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                float a[16];
#pragma unroll
                for (int i = 0; i < kIC; ++i) {
                    const float h = SPLIT == 3 ? tf32_hi(v[i][mm]) : to_tf32(v[i][mm]);
                    a[i] = h;
                    a[kIC + i] = SPLIT == 3 ? v[i][mm] - h : 0.f;
                }
                tmem_st16(abuf + (uint32_t)((4 * hm + mm) * 2 * kIC), a);
            }
            // X rows (b, i) -> B tiles: row n = b (Re) and Bp + b (Im), column k = i
            if (xb < BP) {
                unsigned char* bset = bsets + (size_t)t * C::BSet;
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = 2 * xh + jj;
                    const float4 p = *reinterpret_cast<const float4*>(
                        st + kWBytes + xr * kRow + (((uint32_t)j ^ xsw) << 4));
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int m = 2 * j + h;
                        const float re = h ? p.z : p.x, im = h ? p.w : p.y;
                        const float rh = SPLIT == 3 ? tf32_hi(re) : to_tf32(re);
                        const float ih = SPLIT == 3 ? tf32_hi(im) : to_tf32(im);
                        unsigned char* hi = bset + m * C::BTile;
                        *reinterpret_cast<float*>(hi + core_off(xb, xi)) = rh;
                        *reinterpret_cast<float*>(hi + core_off(BP + xb, xi)) = ih;
                        if (SPLIT == 3) {
                            unsigned char* lo = bset + (kQM + m) * C::BTile;
                            *reinterpret_cast<float*>(lo + core_off(xb, xi)) = re - rh;
                            *reinterpret_cast<float*>(lo + core_off(BP + xb, xi)) = im - ih;
                        }
                    }
                }
            }
            fence_proxy_async_smem();  // B tiles visible to the tensor core
            tmem_st_wait();            // A rows written
            tc_fence_before_sync();
            mbar_arrive(&empty[s]);
            mbar_arrive(&afull[t]);
            if (c != nch - 1) continue;

            // ---- the unit's last chunk is in: read its accumulators out ----
            // every MMA of the unit must have completed before TMEM is read: this
            // wait is bounded but not cut short by a forced timeout
            const bool dok = wait_parity_bounded(dfull, (uint32_t)(k & 1), nullptr);
            if (!__all_sync(0xffffffffu, dok)) {
                atomicExch(fail, 1);
                atomicOr(err, 2u /* FNO_DEVERR_TIMEOUT */);
                break;
            }
            tc_fence_after_sync();
            // Z of the unit is staged in shared memory as [b][o][8 modes] (64-byte
            // rows, 16-byte chunks rotated by (row >> 1) & 3 against bank
            // conflicts) and then written out row by row, so that each warp store
            // covers whole 64-byte runs of Z instead of scattered 16-byte pieces
#pragma unroll 1
            for (int jp = 2 * hm; jp < 2 * hm + 2; ++jp) {
                float z[2][BP / 2][2];  // [mode of the pair][b = 2k + cw][re, im]
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = 2 * jp + h;
                    float d[N];
                    if constexpr (N == 32) {
                        tmem_ld32(trow + (uint32_t)(m * N), d);
                    } else {
                        tmem_ld16(trow + (uint32_t)(m * N), d);
                    }
                    tmem_ld_wait();
                    // even lane (Re w): Re Z = D[(o,0),(0,b)] - D[(o,1),(1,b)];
                    // odd lane (Im w):  Im Z = D[(o,1),(0,b)] + D[(o,0),(1,b)]
                    float val[BP];
#pragma unroll
                    for (int b = 0; b < BP; ++b) {
                        const float other = __shfl_xor_sync(0xffffffffu, d[BP + b], 1);
                        val[b] = cw ? d[b] + other : d[b] - other;
                    }
                    // lane cw keeps the complex values of the rows b = 2k + cw
#pragma unroll
                    for (int kk = 0; kk < BP / 2; ++kk) {
                        const float give = cw ? val[2 * kk] : val[2 * kk + 1];
                        const float got = __shfl_xor_sync(0xffffffffu, give, 1);
                        z[h][kk][0] = cw ? got : val[2 * kk];
                        z[h][kk][1] = cw ? val[2 * kk + 1] : got;
                    }
                }
                // the previous unit's rows must have been copied out of the staging
                // buffer by every converter thread (a bounded wait: a thread that
                // gave up earlier never arrives, and then this one gives up too)
                if (k > 0 && jp == 2 * hm &&
                    !wait_parity_bounded(zfree, (uint32_t)((k - 1) & 1), err))
                    atomicExch(fail, 1);
#pragma unroll
                for (int kk = 0; kk < BP / 2; ++kk) {
                    const uint32_t r = (uint32_t)((2 * kk + cw) * kOB + o);
                    *reinterpret_cast<float4*>(zst + swz64(r, (uint32_t)jp)) =
                        make_float4(z[0][kk][0], z[0][kk][1], z[1][kk][0], z[1][kk][1]);
                }
            }
            tc_fence_before_sync();
            mbar_arrive(dempty);  // the accumulators may be overwritten
            mbar_arrive(zready);
            if (!wait_parity_bounded(zready, (uint32_t)(k & 1), err)) atomicExch(fail, 1);
            {
                // row (b, o) of the tile is 64 contiguous bytes of Z: four lanes per
                // row, eight rows per warp store
                const int m0 = unit_m0(k), o0 = unit_o0(k);
#pragma unroll 4
                for (int e = ct; e < BP * kOB * 4; e += kConv) {
                    const int r = e >> 2, j = e & 3;
                    const int b = r / kOB, og = o0 + (r - b * kOB), mg = m0 + 2 * j;
                    const float4 v =
                        *reinterpret_cast<const float4*>(zst + swz64((uint32_t)r, (uint32_t)j));
                    if (b < B && og < Cout && mg < NM &&
                        FNO_DBG_OK(Z + ((size_t)b * Cout + og) * NM + mg, 2 * sizeof(float2)))
                        *reinterpret_cast<float4*>(Z + ((size_t)b * Cout + og) * NM + mg) = v;
                }
            }
            mbar_arrive(zfree);
        }
    }

    tc_fence_before_sync();
    __syncthreads();  // the issuer has seen every MMA complete; no copy in flight
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int BP, int SPLIT>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(mix_tcm_kernel<BP, SPLIT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)TcmCfg<BP>::Smem);
}

// 3D tensor map over a complex64 array [d2][d1][NM] viewed as floats: dims
// (2*NM, d1, d2), box (16 floats = 8 modes, b1, b2), 64-byte swizzle,
// out-of-range elements read as zeros (and not written by stores).
bool encode_map(CUtensorMap* map, const float2* base, int NM, int d1, int d2, int b1, int b2) {
    fno_encode_tiled_fn enc = fno_get_encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)NM * 2, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)NM * 8, (cuuint64_t)d1 * NM * 8};
    cuuint32_t box[3] = {2 * kQM, (cuuint32_t)b1, (cuuint32_t)b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float2*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BP, int SPLIT>
cudaError_t launch_bp(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                      int early_w, cudaStream_t s) {
    CUtensorMap mw, mx;
    if (!encode_map(&mw, w, p.nm, p.Cout, p.Cin, kOB, kIC) ||
        !encode_map(&mx, X, p.nm, p.Cin, p.B, kIC, BP))
        return cudaErrorInvalidValue;
    // persistent: one CTA per SM (tensor memory and shared memory admit one),
    // each taking every gridDim.x-th (mode block, output block) unit
    const int units = ((p.nm + kQM - 1) / kQM) * ((p.Cout + kOB - 1) / kOB);
    const int grid = units < p.sms ? units : p.sms;
    return launch_pdl(mix_tcm_kernel<BP, SPLIT>, dim3(grid), dim3(kThreads), TcmCfg<BP>::Smem, s,
                      mw, mx, Z, p.B, p.Cin, p.Cout, p.nm, early_w, p.err
                      FNO_DBG_ARG1(Z, 8ull * p.B * p.Cout * p.nm, p));
}

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t mix_tcm_init() {
    cudaError_t e = set_attr<8, 1>();
    if (e == cudaSuccess) e = set_attr<8, 3>();
    if (e == cudaSuccess) e = set_attr<16, 1>();
    if (e == cudaSuccess) e = set_attr<16, 3>();
    return e;
}

// Batch rows up to 16 (one N = 2 * Bp block); an even mode count keeps the
// tensor maps' row pitch (8 * nm bytes) a multiple of 16.
bool mix_tcm_supported(int B, int Cin, int Cout, int nm) {
    return B >= 1 && B <= 16 && Cin >= 1 && Cout >= 1 && nm >= 2 && (nm & 1) == 0;
}

cudaError_t launch_mix_tcm(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                           int split, bool after_own_forward, cudaStream_t s,
                           fno_launch_ctx* ctx) {
    const int early_w = after_own_forward ? 1 : 0;
    cudaError_t e;
    if (p.B <= 8)
        e = split == 3 ? launch_bp<8, 3>(p, X, w, Z, early_w, s)
                       : launch_bp<8, 1>(p, X, w, Z, early_w, s);
    else
        e = split == 3 ? launch_bp<16, 3>(p, X, w, Z, early_w, s)
                       : launch_bp<16, 1>(p, X, w, Z, early_w, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
