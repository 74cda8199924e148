// stages_dft.cu -- the transforms for grids whose H or W is not a power of two,
// as pruned direct DFTs (the FFT kernels need power-of-two lengths).  With few
// retained modes (the layer keeps m2 columns and 2*m1 rows) a direct sum per
// retained bin costs W (or H) multiply-adds, which is the right order for
// these sizes.  All four steps are the layer's definition written out:
//   rows, forward:   T[q][h][k2]  = sum_w x[q][h][w] e^{-2 pi i k2 w / W},   k2 < m2
//   cols, forward:   X[q][r][k2]  = s * sum_h T[q][h][k2] e^{-2 pi i k1(r) h / H}
//   cols, inverse:   V[q][h][k2]  = sum_r Z[q][r][k2] e^{+2 pi i k1(r) h / H}
//   rows, inverse:   y[q][h][w]   = s * sum_k2 c(k2) Re(V[q][h][k2] e^{+2 pi i k2 w / W})
// with q a (batch, channel) plane, s = 1/sqrt(HW), k1(r) = r for r < m1 and
// H - 2*m1 + r otherwise, c = 1 for k2 = 0 and k2 = W/2 and 2 otherwise (TurboFNO
// page, sections 2.2 and 3.1; the half-spectrum width W/2 + 1 of the FFT
// operator-optimisation page, section 2.2).  Twiddles come from the plan's
// tables e^{+2 pi i j / N}, indexed by the exact integer (k * n) mod N.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fno {
namespace {

constexpr int kDftThreads = 256;
constexpr int kWarps = kDftThreads / 32;
constexpr int kRowsPerWarp = 4;  // column steps: output rows (or h) per warp

__device__ __forceinline__ int kr(int r, int H, int m1) { return r < m1 ? r : H - 2 * m1 + r; }

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
// columns in registers; per K step one shared-memory float4 of A (TM = 4) and
// two of twiddles feed TM * 8 fused multiply-adds.  The chunks are double
// buffered: the next chunk of A is loaded into registers and its twiddles are
// formed while the current one is multiplied.  With few output tiles the K
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

template <int BN, int TM, bool FWD>
__global__ void __launch_bounds__(kGT, (RowGemm<BN, TM>::MinBlocks))
dft_rows_gemm_kernel(const float* __restrict__ A, float* __restrict__ C, long long M, int K,
                     int N, int W, float scale, const float2* __restrict__ tw, int ksplit,
                     int kper) {
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
            if constexpr (FWD) {  // columns tx*8 .. tx*8 + 7
                const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * kGTN]);
                const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * kGTN + 4]);
                bv[0] = b0.x; bv[1] = b0.y; bv[2] = b0.z; bv[3] = b0.w;
                bv[4] = b1.x; bv[5] = b1.y; bv[6] = b1.z; bv[7] = b1.w;
            } else {              // columns tx + NX*j: stores of 8 lanes are contiguous
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
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const long long row = row0 + ty * TM + i;
        if (row >= M) break;
        float* Cr = C + row * N;
#pragma unroll
        for (int j = 0; j < kGTN; ++j) {
            const int nj = n0 + (FWD ? tx * kGTN + j : tx + G::NX * j);
            if (nj < N) {
                if (ksplit == 1) Cr[nj] = acc[i][j] * scale;
                else atomicAdd(&Cr[nj], acc[i][j] * scale);
            }
        }
    }
}

// Forward columns: warp = (plane, 4 consecutive retained rows r), lanes over
// k2 (in blocks of 32); per h one coalesced read of T[q][h][k2] serves the 4
// rows, whose twiddles are warp-uniform.
__global__ void __launch_bounds__(kDftThreads)
dft_cols_fwd_kernel(const float2* __restrict__ T, float2* __restrict__ X, long long planes, int H,
                    int m1, int m2, float scale, const float2* __restrict__ tw_h) {
    const int lane = threadIdx.x & 31;
    const int R = 2 * m1, rg = (R + kRowsPerWarp - 1) / kRowsPerWarp;
    const long long job = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (job >= planes * rg) return;
    const long long q = job / rg;
    const int r0 = (int)(job - q * rg) * kRowsPerWarp;
    const float2* Tq = T + q * H * m2;
    for (int kb = 0; kb < m2; kb += 32) {
        const int k2 = kb + lane;
        float2 acc[kRowsPerWarp];
        int k1[kRowsPerWarp], idx[kRowsPerWarp];  // idx = (k1 * h) mod H, stepped with h
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            acc[j] = make_float2(0.f, 0.f);
            k1[j] = r0 + j < R ? kr(r0 + j, H, m1) : 0;
            idx[j] = 0;
        }
        for (int h = 0; h < H; ++h) {
            const float2 v = k2 < m2 ? __ldg(&Tq[(size_t)h * m2 + k2]) : make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) {
                float2 t = __ldg(&tw_h[idx[j]]);
                t.y = -t.y;  // e^{-2 pi i k1 h / H}
                cmac(acc[j], v, t);
                idx[j] += k1[j];
                if (idx[j] >= H) idx[j] -= H;
            }
        }
        if (k2 < m2) {
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j)
                if (r0 + j < R) X[(q * R + r0 + j) * m2 + k2] = cscale(acc[j], scale);
        }
    }
}

// Inverse columns: warp = (plane, 4 consecutive h), lanes over k2; per retained
// row r one coalesced read of Z[q][r][k2] serves the 4 h.
__global__ void __launch_bounds__(kDftThreads)
dft_cols_inv_kernel(const float2* __restrict__ Z, float2* __restrict__ T, long long planes, int H,
                    int m1, int m2, const float2* __restrict__ tw_h) {
    const int lane = threadIdx.x & 31;
    const int R = 2 * m1, hg = (H + kRowsPerWarp - 1) / kRowsPerWarp;
    const long long job = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (job >= planes * hg) return;
    const long long q = job / hg;
    const int h0 = (int)(job - q * hg) * kRowsPerWarp;
    const float2* Zq = Z + q * R * m2;
    for (int kb = 0; kb < m2; kb += 32) {
        const int k2 = kb + lane;
        float2 acc[kRowsPerWarp];
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) acc[j] = make_float2(0.f, 0.f);
        for (int r = 0; r < R; ++r) {
            const float2 v = k2 < m2 ? __ldg(&Zq[(size_t)r * m2 + k2]) : make_float2(0.f, 0.f);
            const int k1 = kr(r, H, m1);
            int idx = (int)(((long long)k1 * h0) % H);  // (k1 * h) mod H for h = h0 + j
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) {
                cmac(acc[j], v, __ldg(&tw_h[idx]));  // e^{+2 pi i k1 h / H}
                idx += k1;
                if (idx >= H) idx -= H;
            }
        }
        if (k2 < m2) {
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j)
                if (h0 + j < H) T[(q * H + h0 + j) * m2 + k2] = acc[j];
        }
    }
}

// One row step as the matrix product above: M rows, contraction length K, N
// outputs per row.  The forward takes 32-column tiles of 256 rows for narrow
// outputs (2*m2 <= 32), else 64 columns by 128 rows, or by 64 rows when that
// would leave fewer than two CTAs per SM; the inverse always 64 by 64.  If the tiles still number fewer
// than two per SM, the K range is split over CTAs (chunks of at least 64) whose
// partial sums are added into C after it is zeroed; their order of addition
// varies from run to run.
template <bool FWD>
cudaError_t launch_rows_gemm(const float* A, float* C, long long M, int K, int N, int W,
                             float scale, const float2* tw, cudaStream_t s) {
    constexpr long long kWant = 2 * 152;
    const auto tiles = [&](int bn, int bm) {
        return ((M + bm - 1) / bm) * (long long)((N + bn - 1) / bn);
    };
    int cfg;  // 0: <32, 4>, 1: <64, 4>, 2: <64, 2>
    long long t;
    if (!FWD) {
        // the inverse's K (2*m2) is short and its output (y) large: the
        // 64-register tile at four CTAs per SM
        cfg = 2;
        t = tiles(64, RowGemm<64, 2>::BM);
    } else if (N <= 32) {
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
        dft_rows_gemm_kernel<32, 4, FWD><<<grid, kGT, 0, s>>>(A, C, M, K, N, W, scale, tw,
                                                              ksplit, kper);
    else if (cfg == 1)
        dft_rows_gemm_kernel<64, 4, FWD><<<grid, kGT, 0, s>>>(A, C, M, K, N, W, scale, tw,
                                                              ksplit, kper);
    else
        dft_rows_gemm_kernel<64, 2, FWD><<<grid, kGT, 0, s>>>(A, C, M, K, N, W, scale, tw,
                                                              ksplit, kper);
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
                                           p.W, 1.f, p.tw_w, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    if (e != cudaSuccess) return e;
    const long long jobs = planes * ((2 * p.m1 + kRowsPerWarp - 1) / kRowsPerWarp);
    dft_cols_fwd_kernel<<<(unsigned)((jobs + kWarps - 1) / kWarps), kDftThreads, 0, s>>>(
        T, X, planes, p.H, p.m1, p.m2, p.scale, p.tw_h);
    e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_dft(const fno_plan_s& p, const float2* Z, float* y, float2* T,
                               cudaStream_t s, fno_launch_ctx* ctx) {
    const long long planes = (long long)p.B * p.Cout, nrows = planes * p.H;
    const long long jobs = planes * ((p.H + kRowsPerWarp - 1) / kRowsPerWarp);
    dft_cols_inv_kernel<<<(unsigned)((jobs + kWarps - 1) / kWarps), kDftThreads, 0, s>>>(
        Z, T, planes, p.H, p.m1, p.m2, p.tw_h);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    if (e != cudaSuccess) return e;
    e = launch_rows_gemm<false>(reinterpret_cast<const float*>(T), y, nrows, 2 * p.m2, p.W, p.W,
                                p.scale, p.tw_w, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

// The 1D layer (plan with dims = 1, W = L, m2 = m retained modes): the row
// transforms alone, orthonormal scale 1/sqrt(L) applied on each side.
cudaError_t launch_forward_1d(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s,
                              fno_launch_ctx* ctx) {
    const long long nrows = (long long)p.B * p.Cin;
    cudaError_t e = launch_rows_gemm<true>(x, reinterpret_cast<float*>(X), nrows, p.W, 2 * p.m2,
                                           p.W, p.scale, p.tw_w, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_1d(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s,
                              fno_launch_ctx* ctx) {
    const long long nrows = (long long)p.B * p.Cout;
    cudaError_t e = launch_rows_gemm<false>(reinterpret_cast<const float*>(Z), y, nrows,
                                            2 * p.m2, p.W, p.W, p.scale, p.tw_w, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
