// stages_dft.cu -- the transforms for grids whose H or W is not a power of two
// (and the 1D layer's rows at lengths the FFT rows do not cover), as pruned
// direct DFTs (the FFT kernels need power-of-two lengths).  With few retained
// modes (the layer keeps m2 columns and 2*m1 rows) a direct sum per retained
// bin costs W (or H) multiply-adds, which is the right order for these sizes.
// All four steps are the layer's definition written out:
//   rows, forward:   T[q][h][k2]  = sum_w x[q][h][w] e^{-2 pi i k2 w / W},   k2 < m2
//   cols, forward:   X[q][r][k2]  = s * sum_h T[q][h][k2] e^{-2 pi i k1(r) h / H}
//   cols, inverse:   V[q][h][k2]  = sum_r Z[q][r][k2] e^{+2 pi i k1(r) h / H}
//   rows, inverse:   y[q][h][w]   = s * sum_k2 c(k2) Re(V[q][h][k2] e^{+2 pi i k2 w / W})
// with q a (batch, channel) plane, s = 1/sqrt(HW), k1(r) = r for r < m1 and
// H - 2*m1 + r otherwise, c = 1 for k2 = 0 and k2 = W/2 and 2 otherwise (TurboFNO
// page, sections 2.2 and 3.1; the half-spectrum width W/2 + 1 of the FFT
// operator-optimisation page, section 2.2).  Twiddles come from the plan's
// tables e^{+2 pi i j / N}, indexed by the exact integer (k * n) mod N.  Each
// step is a dense product with a twiddle matrix (the rows over all rows of all
// planes, the columns batched over planes), computed by register-tiled fp32
// kernels below.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fno {
namespace {

// The row steps as real matrix products over all rows of all planes (M rows):
//   forward  C[row][n] = sum_w x[row][w] F[w][n],  n = 2*k2 + c,  N = 2*m2:
//            F[w][2k2] = cos(2 pi k2 w / W), F[w][2k2 + 1] = -sin(2 pi k2 w / W),
//            so C is T (k2 < m2 interleaved as re, im) and K = W;
//   inverse  C[row][w] = scale * sum_j V'[row][j] G[j][w],  j = 2*k2 + c, K = 2*m2:
//            V'[row][j] = c(k2) * (re or im of V[row][k2]),
//            G[2k2][w] = cos(2 pi k2 w / W), G[2k2 + 1][w] = -sin(2 pi k2 w / W),
//            the real part of sum_k2 c(k2) V[k2] e^{+2 pi i k2 w / W}, N = W.
// The twiddle operand is filled per K chunk from the table e^{+2 pi i j / W} at
// the exact index (k2 * w) mod W, kept incrementally (one division per thread
// per launch).  CTA: 256 threads, BM x BN outputs, each thread TM rows x 8
// columns in registers: grouped (columns tx*4 .. +3 and BN/2 + tx*4 .. +3,
// stored as float4 when rows start on 16 bytes) or interleaved (columns
// tx + NX*j, so that eight lanes store 32 contiguous bytes); per K step one
// shared-memory float4 of A (TM = 4) and two float4 of twiddles (grouped) feed
// TM * 8 fused multiply-adds.  The chunks are double buffered: the next chunk
// of A is loaded into registers and its twiddles are formed while the current
// one is multiplied.  With few output tiles the K
// range is split over CTAs (ksplit > 1) that add their partial sums into C,
// which the launcher has zeroed.
constexpr int kGT = 256;  // threads per CTA
constexpr int kGBK = 16;  // K chunk
constexpr int kGTN = 8;   // columns per thread

template <int BN, int TM>
struct RowGemm {
    static constexpr int NX = BN / kGTN;  // threads along N
    static constexpr int NY = kGT / NX;   // threads along M
    static constexpr int BM = NY * TM;
    static constexpr int AS = BM + 4;     // As row stride (floats)
    static constexpr int AE = BM * kGBK / kGT;  // A elements per thread per chunk
    static constexpr int BE = BN * kGBK / kGT;  // twiddle elements per thread per chunk
    static constexpr int KS = kGT / BN;         // twiddle row step between a thread's elements
    // CTAs per SM the registers are sized for (<64, 2>: 64 registers; TM = 4:
    // at most 128)
    static constexpr int MinBlocks = TM == 2 ? 4 : 2;
};

template <int BN, int TM, bool FWD, bool GROUPED>
__global__ void __launch_bounds__(kGT, (RowGemm<BN, TM>::MinBlocks))
dft_rows_gemm_kernel(const float* __restrict__ A, float* __restrict__ C, long long M, int K,
                     int N, int W, float scale, const float2* __restrict__ tw, int ksplit,
                     int kper FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    using G = RowGemm<BN, TM>;
    __shared__ __align__(16) float As[2][kGBK][G::AS];
    __shared__ __align__(16) float Bs[2][kGBK][BN];
    const int ntiles = (N + BN - 1) / BN;
    const int ks = blockIdx.x % ksplit;
    const int tile = blockIdx.x / ksplit;
    const long long row0 = (long long)(tile / ntiles) * G::BM;
    const int n0 = (tile % ntiles) * BN;
    const int kbeg = ks * kper, kend = min(K, kbeg + kper);
    const int tid = threadIdx.x, tx = tid % G::NX, ty = tid / G::NX;

    // this thread's A elements: rows tid / 16 + 16 i, column tid % 16 of a chunk
    const int akk = tid % kGBK, ar = tid / kGBK;
    // this thread's twiddle elements: column nn, rows kr + KS * i of a chunk
    const int nn = tid % BN, kr = tid / BN;
    const int n = n0 + nn;
    // twiddle index (freq * pos) mod W at the chunk start, its step between the
    // thread's elements and its advance per chunk
    int tbase, tstep, tadv;
    bool imag;
    if (FWD) {  // freq = n / 2 fixed, pos = k
        const int freq = n >> 1;
        imag = n & 1;
        tbase = (int)(((long long)freq * (kbeg + kr)) % W);
        tstep = (int)(((long long)freq * G::KS) % W);
        tadv = (int)(((long long)freq * kGBK) % W);
    } else {    // pos = n fixed, freq = k / 2 (the parity of k is the thread's)
        imag = kr & 1;
        const int pos = n < N ? n : 0;
        tbase = (int)(((long long)((kbeg + kr) >> 1) * pos) % W);
        tstep = (int)(((long long)(G::KS / 2) * pos) % W);
        tadv = (int)(((long long)(kGBK / 2) * pos) % W);
    }
    const auto add_mod = [W](int a, int b) { a += b; return a >= W ? a - W : a; };

    float ra[G::AE];
    const auto load_a = [&](int k0) {
#pragma unroll
        for (int i = 0; i < G::AE; ++i) {
            const long long row = row0 + ar + (kGT / kGBK) * i;
            const int k = k0 + akk;
            float v = 0.f;
            if (row < M && k < kend) {
                v = __ldg(&A[row * K + k]);
                if (!FWD) {
                    const int k2 = k >> 1;
                    if (k2 != 0 && 2 * k2 != W) v += v;  // c(k2) = 2
                }
            }
            ra[i] = v;
        }
    };
    const auto store_chunk = [&](int buf, int k0) {
#pragma unroll
        for (int i = 0; i < G::AE; ++i) As[buf][akk][ar + (kGT / kGBK) * i] = ra[i];
        int idx = tbase;
#pragma unroll
        for (int i = 0; i < G::BE; ++i) {
            const int k = k0 + kr + G::KS * i;
            float v = 0.f;
            if (k < kend && n < N) {
                const float2 t = __ldg(&tw[idx]);
                v = imag ? -t.y : t.x;
            }
            Bs[buf][kr + G::KS * i][nn] = v;
            idx = add_mod(idx, tstep);
        }
        tbase = add_mod(tbase, tadv);
    };

    float acc[TM][kGTN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < kGTN; ++j) acc[i][j] = 0.f;

    load_a(kbeg);
    store_chunk(0, kbeg);
    __syncthreads();
    int buf = 0;
    for (int k0 = kbeg; k0 < kend; k0 += kGBK) {
        const bool more = k0 + kGBK < kend;
        if (more) load_a(k0 + kGBK);
#pragma unroll
        for (int kk = 0; kk < kGBK; ++kk) {
            float av[TM];
            if constexpr (TM == 4) {
                const float4 a = *reinterpret_cast<const float4*>(&As[buf][kk][ty * TM]);
                av[0] = a.x; av[1] = a.y; av[2] = a.z; av[3] = a.w;
            } else {
#pragma unroll
                for (int i = 0; i < TM; ++i) av[i] = As[buf][kk][ty * TM + i];
            }
            float bv[kGTN];
            if constexpr (GROUPED) {  // columns tx*4 .. +3 and BN/2 + tx*4 .. +3
                const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
                const float4 b1 =
                    *reinterpret_cast<const float4*>(&Bs[buf][kk][BN / 2 + tx * 4]);
                bv[0] = b0.x; bv[1] = b0.y; bv[2] = b0.z; bv[3] = b0.w;
                bv[4] = b1.x; bv[5] = b1.y; bv[6] = b1.z; bv[7] = b1.w;
            } else {                  // columns tx + NX*j
#pragma unroll
                for (int j = 0; j < kGTN; ++j) bv[j] = Bs[buf][kk][tx + G::NX * j];
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < kGTN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (more) store_chunk(buf ^ 1, k0 + kGBK);
        __syncthreads();
        buf ^= 1;
    }
    // rows of C start on 16 bytes when N % 4 == 0 (C itself is 256-byte aligned)
    const bool vec = GROUPED && ksplit == 1 && (N & 3) == 0;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const long long row = row0 + ty * TM + i;
        if (row >= M) break;
        float* Cr = C + row * N;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int nb = n0 + (GROUPED ? g * (BN / 2) + tx * 4 : 0);
            if (vec && nb + 3 < N) {
                if (FNO_DBG_OK(&Cr[nb], 4 * sizeof(float)))
                    *reinterpret_cast<float4*>(&Cr[nb]) =
                    make_float4(acc[i][4 * g] * scale, acc[i][4 * g + 1] * scale,
                                acc[i][4 * g + 2] * scale, acc[i][4 * g + 3] * scale);
                continue;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = 4 * g + q;
                const int nj = GROUPED ? nb + q : n0 + tx + G::NX * j;
                if (nj < N && FNO_DBG_OK(&Cr[nj], sizeof(float))) {
                    if (ksplit == 1) Cr[nj] = acc[i][j] * scale;
                    else atomicAdd(&Cr[nj], acc[i][j] * scale);
                }
            }
        }
    }
}

// The column steps as complex matrix products batched over the planes q, with
// the columns c = (q, k2) of all planes side by side:
//   forward  X_q[r][k2] = s * sum_h F[r][h] T_q[h][k2],  F[r][h] = e^{-2 pi i k1(r) h / H},
//   inverse  T_q[h][k2] = sum_r G[h][r] Z_q[r][k2],      G[h][r] = e^{+2 pi i k1(r) h / H},
// i.e. C[m][c] = alpha * sum_k A[m][k] B[k][c], with B[k][(q, k2)] at
// (q*KB + k)*m2 + k2 and C[m][(q, k2)] at (q*MC + m)*m2 + k2.  A is formed per K
// chunk from the table e^{+2 pi i j / H} (forward: index kept incrementally).
// CTA: 128 threads, 32 rows x 32 complex columns; each thread 4 rows x 2
// columns (columns tx and tx + 16, so that 16 lanes store 128 contiguous
// bytes); per K step two float4 of A and two float2 of B feed 32 fused
// multiply-adds.  Chunks of 16 are double buffered.
constexpr int kCT = 128;   // threads
constexpr int kCBK = 16;   // K chunk
constexpr int kCBM = 32;   // rows per CTA
constexpr int kCBN = 32;   // complex columns per CTA

template <bool FWD>
__global__ void __launch_bounds__(kCT)
dft_cols_gemm_kernel(const float2* __restrict__ Bsrc, float2* __restrict__ Cdst, int M, int K,
                     long long ncols, int m2, int KB, int MC, int H, int m1, float alpha,
                     const float2* __restrict__ tw_h FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    __shared__ __align__(16) float2 As[2][kCBK][kCBM];
    __shared__ __align__(16) float2 Bs[2][kCBK][kCBN];
    const int mtiles = (M + kCBM - 1) / kCBM;
    const int m0 = (int)(blockIdx.x % mtiles) * kCBM;
    const long long c0 = (long long)(blockIdx.x / mtiles) * kCBN;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;  // ty < 8: rows ty*4 .. +3

    // loader roles: B column cc = tid % 32, K rows tid / 32 + 4 i; A row mm = tid % 32,
    // K rows tid / 32 + 4 i
    const int lc = tid % 32, lk = tid / 32;
    const long long bc = c0 + lc;
    const bool bvalid = bc < ncols;
    const long long bq = bvalid ? bc / m2 : 0;
    const int bk2 = bvalid ? (int)(bc - bq * m2) : 0;
    const float2* Bcol = Bsrc + (size_t)bq * KB * m2 + bk2;
    const int am = m0 + lc;
    const bool avalid = am < M;
    const auto k1_of = [H, m1](int r) { return r < m1 ? r : H - 2 * m1 + r; };
    // forward: A[m][k] = conj(tab[(k1(m) * k) mod H]), k1 fixed per thread
    const int ak1 = FWD && avalid ? k1_of(am) : 0;
    int abase = FWD ? (int)(((long long)ak1 * lk) % H) : 0;
    const int astep = FWD ? (int)(((long long)ak1 * 4) % H) : 0;
    const int aadv = FWD ? (int)(((long long)ak1 * kCBK) % H) : 0;

    float2 rb[4];
    const auto load_b = [&](int k0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = k0 + lk + 4 * i;
            rb[i] = bvalid && k < K ? __ldg(&Bcol[(size_t)k * m2]) : make_float2(0.f, 0.f);
        }
    };
    const auto store_chunk = [&](int buf, int k0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) Bs[buf][lk + 4 * i][lc] = rb[i];
        int idx = abase;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = k0 + lk + 4 * i;
            float2 a = make_float2(0.f, 0.f);
            if (avalid && k < K) {
                if (FWD) {
                    a = __ldg(&tw_h[idx]);
                    a.y = -a.y;
                } else {
                    a = __ldg(&tw_h[(int)(((long long)k1_of(k) * am) % H)]);
                }
            }
            As[buf][lk + 4 * i][lc] = a;
            if (FWD) {
                idx += astep;
                if (idx >= H) idx -= H;
            }
        }
        if (FWD) {
            abase += aadv;
            if (abase >= H) abase -= H;
        }
    };

    float2 acc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);

    load_b(0);
    store_chunk(0, 0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < K; k0 += kCBK) {
        const bool more = k0 + kCBK < K;
        if (more) load_b(k0 + kCBK);
#pragma unroll
        for (int kk = 0; kk < kCBK; ++kk) {
            const float4 a01 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a23 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4 + 2]);
            const float2 av[4] = {make_float2(a01.x, a01.y), make_float2(a01.z, a01.w),
                                  make_float2(a23.x, a23.y), make_float2(a23.z, a23.w)};
            const float2 bv[2] = {Bs[buf][kk][tx], Bs[buf][kk][tx + 16]};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) cmac(acc[i][j], av[i], bv[j]);
        }
        if (more) store_chunk(buf ^ 1, k0 + kCBK);
        __syncthreads();
        buf ^= 1;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const long long c = c0 + tx + 16 * j;
        if (c >= ncols) continue;
        const long long q = c / m2;
        const int k2 = (int)(c - q * m2);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = m0 + ty * 4 + i;
            if (m < M && FNO_DBG_OK(&Cdst[((size_t)q * MC + m) * m2 + k2], sizeof(float2)))
                Cdst[((size_t)q * MC + m) * m2 + k2] = cscale(acc[i][j], alpha);
        }
    }
}

// One row step as the matrix product above: M rows, contraction length K, N
// outputs per row.  Narrow forward outputs (2*m2 <= 32) take 32-column tiles of
// 256 rows; otherwise 64 columns by 128 rows, or by 64 rows when that would
// leave fewer than two CTAs per SM.  An inverse whose rows do not start on 16
// bytes (W % 4 != 0) takes 64 by 64 tiles with interleaved columns.  If the tiles still number fewer
// than two per SM, the K range is split over CTAs (chunks of at least 64) whose
// partial sums are added into C after it is zeroed; their order of addition
// varies from run to run.
template <bool FWD>
cudaError_t launch_rows_gemm(const float* A, float* C, long long M, int K, int N, int W,
                             float scale, const float2* tw, const fno_plan_s& p, cudaStream_t s) {
    constexpr long long kWant = 2 * 152;
    const auto tiles = [&](int bn, int bm) {
        return ((M + bm - 1) / bm) * (long long)((N + bn - 1) / bn);
    };
    int cfg;  // 0: <32, 4>, 1: <64, 4>, 2: <64, 2>, 3: <64, 2> with interleaved columns
    long long t;
    if (!FWD && (N & 3) != 0) {
        // rows of y that do not start on 16 bytes: interleaved columns (8 lanes
        // store 32 contiguous bytes) at four CTAs per SM.  Measured at 421x421:
        // 578 us, against 722 us with grouped columns
        cfg = 3;
        t = tiles(64, RowGemm<64, 2>::BM);
    } else if (FWD && N <= 32) {
        cfg = 0;
        t = tiles(32, RowGemm<32, 4>::BM);
    } else if (tiles(64, RowGemm<64, 4>::BM) >= kWant) {
        cfg = 1;
        t = tiles(64, RowGemm<64, 4>::BM);
    } else {
        cfg = 2;
        t = tiles(64, RowGemm<64, 2>::BM);
    }
    int ksplit = 1;
    if (t < kWant && K >= 2 * 64) {
        ksplit = (int)std::min<long long>((kWant + t - 1) / t, K / 64);
    }
    int kper = (K + ksplit - 1) / ksplit;
    kper = (kper + kGBK - 1) / kGBK * kGBK;
    ksplit = (K + kper - 1) / kper;
    if (ksplit > 1) {
        cudaError_t e = cudaMemsetAsync(C, 0, sizeof(float) * (size_t)M * N, s);
        if (e != cudaSuccess) return e;
    }
    const unsigned grid = (unsigned)(t * ksplit);
    if (cfg == 0)
        dft_rows_gemm_kernel<32, 4, FWD, true><<<grid, kGT, 0, s>>>(A, C, M, K, N, W, scale, tw,
                                                                    ksplit, kper FNO_DBG_ARG1(C, 4ull * M * N, p));
    else if (cfg == 1)
        dft_rows_gemm_kernel<64, 4, FWD, true><<<grid, kGT, 0, s>>>(A, C, M, K, N, W, scale, tw,
                                                                    ksplit, kper FNO_DBG_ARG1(C, 4ull * M * N, p));
    else if (cfg == 2)
        dft_rows_gemm_kernel<64, 2, FWD, true><<<grid, kGT, 0, s>>>(A, C, M, K, N, W, scale, tw,
                                                                    ksplit, kper FNO_DBG_ARG1(C, 4ull * M * N, p));
    else
        dft_rows_gemm_kernel<64, 2, FWD, false><<<grid, kGT, 0, s>>>(A, C, M, K, N, W, scale, tw,
                                                                     ksplit, kper FNO_DBG_ARG1(C, 4ull * M * N, p));
    return cudaGetLastError();
}

template <bool FWD>
cudaError_t launch_cols_gemm(const float2* B, float2* C, int M, int K, long long planes, int m2,
                             int KB, int MC, int H, int m1, float alpha, const float2* tw_h,
                             const fno_plan_s& p, cudaStream_t s) {
    const long long ncols = planes * m2;
    const long long grid = (long long)((M + kCBM - 1) / kCBM) * ((ncols + kCBN - 1) / kCBN);
    dft_cols_gemm_kernel<FWD><<<(unsigned)grid, kCT, 0, s>>>(
        B, C, M, K, ncols, m2, KB, MC, H, m1, alpha, tw_h
        FNO_DBG_ARG1(C, 8ull * planes * MC * m2, p));
    return cudaGetLastError();
}

}  // namespace
}  // namespace fno

using namespace fno;

bool dft_path(int H, int W) {
    const auto pow2 = [](int v) { return v >= 1 && (v & (v - 1)) == 0; };
    return !pow2(H) || !pow2(W);
}

cudaError_t stages_dft_init() { return cudaSuccess; }  // static shared memory only

cudaError_t launch_forward_dft(const fno_plan_s& p, const float* x, float2* X, float2* T,
                               cudaStream_t s, fno_launch_ctx* ctx) {
    const long long planes = (long long)p.B * p.Cin, nrows = planes * p.H;
    cudaError_t e = launch_rows_gemm<true>(x, reinterpret_cast<float*>(T), nrows, p.W, 2 * p.m2,
                                           p.W, 1.f, p.tw_w, p, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    if (e != cudaSuccess) return e;
    e = launch_cols_gemm<true>(T, X, 2 * p.m1, p.H, planes, p.m2, p.H, 2 * p.m1, p.H, p.m1,
                               p.scale, p.tw_h, p, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_dft(const fno_plan_s& p, const float2* Z, float* y, float2* T,
                               cudaStream_t s, fno_launch_ctx* ctx) {
    const long long planes = (long long)p.B * p.Cout, nrows = planes * p.H;
    cudaError_t e = launch_cols_gemm<false>(Z, T, p.H, 2 * p.m1, planes, p.m2, 2 * p.m1, p.H,
                                            p.H, p.m1, 1.f, p.tw_h, p, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    if (e != cudaSuccess) return e;
    e = launch_rows_gemm<false>(reinterpret_cast<const float*>(T), y, nrows, 2 * p.m2, p.W, p.W,
                                p.scale, p.tw_w, p, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

// The 1D layer (plan with dims = 1, W = L, m2 = m retained modes): the row
// transforms alone, orthonormal scale 1/sqrt(L) applied on each side.
cudaError_t launch_forward_1d(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s,
                              fno_launch_ctx* ctx) {
    const long long nrows = (long long)p.B * p.Cin;
    cudaError_t e = launch_rows_gemm<true>(x, reinterpret_cast<float*>(X), nrows, p.W, 2 * p.m2,
                                           p.W, p.scale, p.tw_w, p, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_1d(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s,
                              fno_launch_ctx* ctx) {
    const long long nrows = (long long)p.B * p.Cout;
    cudaError_t e = launch_rows_gemm<false>(reinterpret_cast<const float*>(Z), y, nrows,
                                            2 * p.m2, p.W, p.W, p.scale, p.tw_w, p, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
