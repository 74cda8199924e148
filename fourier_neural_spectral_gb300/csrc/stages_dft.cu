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
#include <cmath>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "tma.cuh"

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

// Packed fp32 pairs for the row kernels below: fma.rn.f32x2 does two fused
// multiply-adds (each rounded as fmaf) in one instruction, halving the issue
// slots of their multiply-add streams.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 dup2(float a) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(a));
    return r;
}
__device__ __forceinline__ f32x2 ffma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float2 unpack2(f32x2 v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

// The inverse row step for K = 2*m2 <= 64 with whole rows per CTA
// (dft_irows_kernel): y[row][w] = sum_k V[row][k] G[k][w] with
//   G[2k2][w] = s c(k2) cos(2 pi k2 w / W),  G[2k2 + 1][w] = -s c(k2) sin(2 pi k2 w / W)
// (s = the output scale, c(k2) the Hermitian weight), the same product as the
// inverse of dft_rows_gemm_kernel with the weights moved into G.  The output
// rows (W floats each, consecutive in memory) start on 16 bytes only when
// row * W = 0 (mod 4), so each thread takes 8 rows of one residue class
// (row = 0, 1, 2 or 3 mod 4, hence one shift sh = row * W mod 4) and the
// columns w = 4 m - sh: every float4 it stores is aligned, and a warp's 16
// lanes along the row write 256 contiguous bytes.  Quads cut by the row ends
// are stored element by element.  The CTA owns 128 rows; their V (128 x K,
// contiguous) stays in shared memory, and the columns go by in passes of 64
// (every gridDim.y-th pass: with few rows the passes are shared out).  G is a
// plan constant: the plan builds, per pass, the tile Bs[sh][k][q] =
// G[k][64 pass + q - sh] (zero outside [0, W)) for the four shifts
// (dft_irows_table), and the kernel streams each pass's tile into one of two
// shared-memory buffers with a bulk copy while the other is in use.  Per K
// step a thread does two float4 loads of V, one float4 of G and 32 fused
// multiply-adds (16 packed pair instructions).
constexpr int kIRM = 128;     // rows per CTA
constexpr int kIRKMax = 64;   // largest K this kernel takes
constexpr int kIRP = 64;      // columns per pass

__host__ __device__ inline int irows_passes(int W) { return (W + 3 + kIRP - 1) / kIRP; }
// V, two tile buffers, two mbarriers
size_t irows_smem(int K) {
    return sizeof(float) * ((size_t)K * kIRM + 2ull * 4 * K * kIRP) + 2 * sizeof(uint64_t);
}

__global__ void __launch_bounds__(256, 3)
dft_irows_kernel(const float* __restrict__ A, float* __restrict__ y, long long M, int K, int W,
                 const float* __restrict__ G, unsigned* __restrict__ err FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    extern __shared__ __align__(16) float sm_ir[];
    const int tile = 4 * K * kIRP;   // floats per pass tile
    float* As = sm_ir;               // [K][16 ty][8 j]: row 32 (ty / 4) + ty % 4 + 4 j
    float* Bs = sm_ir + K * kIRM;    // [2][4 sh][K][64 q]
    uint64_t* bar = reinterpret_cast<uint64_t*>(Bs + 2 * tile);
    const uint32_t tbytes = (uint32_t)tile * 4u;
    const int tid = threadIdx.x;
    const long long R0 = (long long)blockIdx.x * kIRM;
    const int npass = irows_passes(W);
    const int first = blockIdx.y, step = gridDim.y;
    const int nmine = (npass - first + step - 1) / step;  // >= 1 (gridDim.y <= npass)

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
        for (int i = 0; i < 2 && i < nmine; ++i) {
            mbar_arrive_expect_tx(&bar[i], tbytes);
            bulk_load(Bs + i * tile, G + (size_t)(first + i * step) * tile, tbytes, &bar[i]);
        }
    }
    // V of the CTA's rows: 128 * K consecutive floats (zeros past M)
    {
        const long long base = R0 * K;
        const long long total = M * (long long)K;
        for (int e = tid; e < kIRM * K; e += 256) {
            const int rl = e / K, k = e - rl * K;
            const float v = base + e < total ? __ldg(A + base + e) : 0.f;
            const int ty = ((rl >> 5) << 2) | (rl & 3), j = (rl & 31) >> 2;
            As[k * kIRM + ty * 8 + j] = v;
        }
    }
    __syncthreads();
    const int tx = tid & 15, ty = tid >> 4;
    const long long rbase = R0 + ((ty >> 2) << 5) + (ty & 3);  // rows rbase + 4 j
    const int sh = (int)(((rbase & 3) * (W & 3)) & 3);          // rbase * W mod 4
    const float* ap = As + ty * 8;
    int i = 0;
    for (; i < nmine; ++i) {
        const int pass = first + i * step, b = i & 1;
        const bool ok = wait_parity_bounded(&bar[b], (uint32_t)((i >> 1) & 1), err);
        if (!__syncthreads_and(ok)) break;
        f32x2 acc[8][2];  // columns (0, 1) and (2, 3) of the quad
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = 0ull;
        const float* bp = Bs + b * tile + sh * K * kIRP + 4 * tx;
#pragma unroll 2
        for (int k = 0; k < K; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(ap + k * kIRM);
            const float4 a1 = *reinterpret_cast<const float4*>(ap + k * kIRM + 4);
            const ulonglong2 bb = *reinterpret_cast<const ulonglong2*>(bp + k * kIRP);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const f32x2 a2 = dup2(av[j]);
                acc[j][0] = ffma2(a2, bb.x, acc[j][0]);
                acc[j][1] = ffma2(a2, bb.y, acc[j][1]);
            }
        }
        __syncthreads();  // every thread is done with buffer b
        if (tid == 0 && i + 2 < nmine) {
            mbar_arrive_expect_tx(&bar[b], tbytes);
            bulk_load(Bs + b * tile, G + (size_t)(pass + 2 * step) * tile, tbytes, &bar[b]);
        }
        const int c = kIRP * pass + 4 * tx - sh;
        const bool whole = c >= 0 && c + 3 < W;
        float* yr = y + rbase * W;
#pragma unroll
        for (int j = 0; j < 8; ++j, yr += 4ll * W) {
            if (rbase + 4 * j >= M) break;
            const float2 lo = unpack2(acc[j][0]), hi = unpack2(acc[j][1]);
            if (whole) {
                if (FNO_DBG_OK(yr + c, 4 * sizeof(float)))
                    *reinterpret_cast<float4*>(yr + c) = make_float4(lo.x, lo.y, hi.x, hi.y);
            } else {
                const float v[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (c + u >= 0 && c + u < W && FNO_DBG_OK(yr + c + u, sizeof(float)))
                        yr[c + u] = v[u];
            }
        }
    }
    // after a timeout: the copies still in flight (iterations i and i + 1) land
    // before the CTA leaves (bounded waits, not cut short)
    if (tid == 0)
        for (int d = i; d < i + 2 && d < nmine; ++d)
            wait_parity_bounded(&bar[d & 1], (uint32_t)((d >> 1) & 1), nullptr);
}

// The forward row step for N = 2*m2 <= 32 with many rows (dft_frows_kernel):
// C[row][n] = sum_w x[row][w] F[w][n], F[w][2k2] = s cos(2 pi k2 w / W),
// F[w][2k2 + 1] = -s sin(2 pi k2 w / W) (s = 1, or 1/sqrt(L) for the 1D layer).
// The input rows (W floats, consecutive in memory) start on 16 bytes only when
// row * W = 0 (mod 4), so a CTA takes 128 rows of one residue class (rows
// 512 b + cls + 4 i, i < 128, one shift sh = cls * W mod 4) and reads the
// columns w = 64 pass + q - sh, q < 64, of every pass as aligned 16-byte
// asynchronous copies (cp.async; 16 lanes cover 256 contiguous bytes of a row)
// into one of two shared-memory buffers while the other is in use.  A quad
// that runs past the row's end copies its valid head and zero-fills the rest;
// one that starts before the row (the first quad of a row with sh > 0) is read
// element by element.  F is a plan constant: per pass and shift the tile
// Fs[q][n] = F[64 pass + q - sh][n] (zero outside [0, W) and for n >= N),
// built by dft_frows_table and streamed into one of two buffers by a bulk
// copy.  Thread t takes rows t % 64 and t % 64 + 64 and the 16 columns
// 16 (t / 64) .. + 15 of each pass (four K groups, added in shared memory at
// the end): per 4 columns two float4 loads of x, NP/4 float4 loads of F per
// column (the same address across the warp) and 8 NP fused multiply-adds
// (4 NP packed pair instructions).
constexpr int kFRM = 128;     // rows per CTA (one residue class)
constexpr int kFRP = 64;      // columns per pass
constexpr int kFRS = kFRP + 4;  // row stride of the staged x (floats)

__host__ __device__ inline int frows_passes(int W) { return (W + 3 + kFRP - 1) / kFRP; }
int frows_np(int N) { return N <= 8 ? 8 : N <= 16 ? 16 : N <= 24 ? 24 : N <= 32 ? 32 : 0; }
// two x buffers, two F buffers (or the K-group partial sums), two mbarriers
__host__ __device__ inline size_t frows_smem(int NP) {
    const size_t a = sizeof(float) * (2ull * kFRM * kFRS + 2ull * kFRP * NP);
    const size_t r = sizeof(float) * 4ull * kFRM * NP;
    return (a > r ? a : r) + 2 * sizeof(uint64_t);
}

// 16-byte asynchronous global -> shared copy of the first src_bytes (0..16)
// bytes of src, the rest of the 16 zero-filled.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int NP>
__global__ void __launch_bounds__(256, NP <= 8 ? 3 : 2)
dft_frows_kernel(const float* __restrict__ x, float* __restrict__ C, long long M, int W, int N,
                 const float* __restrict__ F, unsigned* __restrict__ err FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    extern __shared__ __align__(16) float sm_fr[];
    constexpr int tile = kFRP * NP;           // floats per pass tile
    constexpr int xbuf = kFRM * kFRS;         // floats per x buffer
    float* As = sm_fr;                        // [2][128 rows][kFRS]
    float* Fs = sm_fr + 2 * xbuf;             // [2][64 q][NP]
    float* Red = sm_fr;                       // [4 groups][128 rows][NP], after the passes
    uint64_t* bar = reinterpret_cast<uint64_t*>(
        reinterpret_cast<unsigned char*>(sm_fr) + frows_smem(NP) - 2 * sizeof(uint64_t));
    const uint32_t tbytes = (uint32_t)tile * 4u;
    const int tid = threadIdx.x;
    const int cls = blockIdx.x & 3;
    const long long rb = (long long)(blockIdx.x >> 2) * (4 * kFRM) + cls;  // row of i = 0
    const int sh = (cls * (W & 3)) & 3;
    const int npass = frows_passes(W);
    const float* Fsh = F + (size_t)sh * tile;  // this shift's tile of pass 0
    const size_t fstride = 4ull * tile;        // floats between passes

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
        for (int i = 0; i < 2 && i < npass; ++i) {
            mbar_arrive_expect_tx(&bar[i], tbytes);
            bulk_load(Fs + i * tile, Fsh + i * fstride, tbytes, &bar[i]);
        }
    }
    // staging: quad sq of rows sr + 16 j
    const int sq = tid & 15, sr = tid >> 4;
    const auto stage = [&](int pass) {
        float* dst = As + (pass & 1) * xbuf + 4 * sq;
        const int c = kFRP * pass + 4 * sq - sh;
#pragma unroll 4
        for (int j = 0; j < 8; ++j) {
            const int i = sr + 16 * j;
            const long long row = rb + 4ll * i;
            float* d = dst + i * kFRS;
            if (row < M && c >= 0 && c < W) {
                const int valid = W - c < 4 ? W - c : 4;
                cp_async16(d, x + row * W + c, 4u * (uint32_t)valid);
            } else {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (row < M && c < 0) {  // the row's first quad (sh > 0)
                    const float* xr = x + row * W;
                    if (c + 1 >= 0 && c + 1 < W) v.y = __ldg(xr + c + 1);
                    if (c + 2 >= 0 && c + 2 < W) v.z = __ldg(xr + c + 2);
                    if (c + 3 >= 0 && c + 3 < W) v.w = __ldg(xr + c + 3);
                }
                *reinterpret_cast<float4*>(d) = v;
            }
        }
        cp_async_commit();
    };
    // compute: rows r0, r0 + 64, columns 16 kg .. + 15 of the pass
    const int r0 = tid & 63, kg = tid >> 6;
    f32x2 acc0[NP / 2], acc1[NP / 2];  // output pairs (2 n, 2 n + 1)
#pragma unroll
    for (int n = 0; n < NP / 2; ++n) acc0[n] = acc1[n] = 0ull;
    stage(0);
    int pass = 0;
    for (; pass < npass; ++pass) {
        const int b = pass & 1;
        if (pass + 1 < npass) {
            stage(pass + 1);   // the buffer it fills was last read in pass - 1
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        const bool ok = wait_parity_bounded(&bar[b], (uint32_t)((pass >> 1) & 1), err);
        if (!__syncthreads_and(ok)) break;
        const float* a0p = As + b * xbuf + r0 * kFRS + 16 * kg;
        const float* a1p = a0p + 64 * kFRS;
        const float* fp = Fs + b * tile + (16 * kg) * NP;
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
            const float4 xa = *reinterpret_cast<const float4*>(a0p + k4);
            const float4 xb = *reinterpret_cast<const float4*>(a1p + k4);
            const float va[4] = {xa.x, xa.y, xa.z, xa.w};
            const float vb[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float* fr = fp + (k4 + u) * NP;
                const f32x2 a2 = dup2(va[u]), b2 = dup2(vb[u]);
#pragma unroll
                for (int n4 = 0; n4 < NP; n4 += 4) {
                    const ulonglong2 f = *reinterpret_cast<const ulonglong2*>(fr + n4);
                    acc0[n4 / 2] = ffma2(a2, f.x, acc0[n4 / 2]);
                    acc0[n4 / 2 + 1] = ffma2(a2, f.y, acc0[n4 / 2 + 1]);
                    acc1[n4 / 2] = ffma2(b2, f.x, acc1[n4 / 2]);
                    acc1[n4 / 2 + 1] = ffma2(b2, f.y, acc1[n4 / 2 + 1]);
                }
            }
        }
        __syncthreads();  // every thread is done with x buffer b and F buffer b
        if (tid == 0 && pass + 2 < npass) {
            mbar_arrive_expect_tx(&bar[b], tbytes);
            bulk_load(Fs + b * tile, Fsh + (size_t)(pass + 2) * fstride, tbytes, &bar[b]);
        }
    }
    if (pass < npass) {
        // a wait timed out (the error word is set, the output is void): the
        // copies still in flight land before the CTA leaves
        cp_async_wait<0>();
        if (tid == 0)
            for (int d = pass; d < pass + 2 && d < npass; ++d)
                wait_parity_bounded(&bar[d & 1], (uint32_t)((d >> 1) & 1), nullptr);
        return;
    }
    // the four K groups' partial sums are added in shared memory
    __syncthreads();
#pragma unroll
    for (int n = 0; n < NP / 2; ++n) {
        *reinterpret_cast<float2*>(Red + (kg * kFRM + r0) * NP + 2 * n) = unpack2(acc0[n]);
        *reinterpret_cast<float2*>(Red + (kg * kFRM + r0 + 64) * NP + 2 * n) = unpack2(acc1[n]);
    }
    __syncthreads();
    for (int e = tid; e < kFRM * N; e += 256) {
        const int i = e / N, n = e - i * N;
        const long long row = rb + 4ll * i;
        if (row >= M) continue;
        const float v = Red[i * NP + n] + Red[(kFRM + i) * NP + n] +
                        Red[(2 * kFRM + i) * NP + n] + Red[(3 * kFRM + i) * NP + n];
        if (FNO_DBG_OK(C + row * N + n, sizeof(float))) C[row * N + n] = v;
    }
}

// The column steps as complex matrix products batched over the planes q, with
// the columns c = (q, k2) of all planes side by side:
//   forward  X_q[r][k2] = s * sum_h F[r][h] T_q[h][k2],  F[r][h] = e^{-2 pi i k1(r) h / H},
//   inverse  T_q[h][k2] = sum_r G[h][r] Z_q[r][k2],      G[h][r] = e^{+2 pi i k1(r) h / H},
// i.e. C[m][c] = alpha * sum_k A[m][k] B[k][c], with B[k][(q, k2)] at
// (q*KB + k)*m2 + k2 and C[m][(q, k2)] at (q*MC + m)*m2 + k2.  A comes from a
// plan table stored as At[k][m] (dft_cols_table: forward At[h][r] =
// e^{-2 pi i k1(r) h / H}, inverse At[r][h] = e^{+2 pi i k1(r) h / H}), read
// per K chunk (consecutive lanes, consecutive m); without one (the
// allocation-free entry point) it is formed from the table e^{+2 pi i j / H} at
// the exact index (k1 * h) mod H.
// CTA: 128 threads, 32 rows x 32 complex columns; each thread 4 rows x 2
// columns (columns tx and tx + 16, so that 16 lanes store 128 contiguous
// bytes); per K step two float4 of A and two float2 of B feed 32 fused
// multiply-adds.  Chunks of 16 are double buffered.  With few tiles the K
// range is split over gridDim.y CTAs whose partial sums are added into C,
// which the launcher has zeroed.
constexpr int kCT = 128;   // threads
constexpr int kCBK = 16;   // K chunk
constexpr int kCBM = 32;   // rows per CTA
constexpr int kCBN = 32;   // complex columns per CTA

template <bool FWD>
__global__ void __launch_bounds__(kCT)
dft_cols_gemm_kernel(const float2* __restrict__ Bsrc, float2* __restrict__ Cdst, int M, int K,
                     long long ncols, int m2, int KB, int MC, int H, int m1, float alpha,
                     const float2* __restrict__ At, const float2* __restrict__ tw_h,
                     int kper FNO_DBG_PARAM) {
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
    const int kbeg = (int)blockIdx.y * kper, kend = min(K, kbeg + kper);

    float2 rb[4];
    float2 ra[4];
    const auto load_b = [&](int k0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = k0 + lk + 4 * i;
            rb[i] = bvalid && k < kend ? __ldg(&Bcol[(size_t)k * m2]) : make_float2(0.f, 0.f);
            float2 a = make_float2(0.f, 0.f);
            if (avalid && k < kend) {
                if (At) {
                    a = __ldg(&At[(size_t)k * M + am]);
                } else {
                    const int r = FWD ? am : k, h = FWD ? k : am;
                    const int k1 = r < m1 ? r : H - 2 * m1 + r;
                    a = __ldg(&tw_h[(int)(((long long)k1 * h) % H)]);
                    if (FWD) a.y = -a.y;
                }
            }
            ra[i] = a;
        }
    };
    const auto store_chunk = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            Bs[buf][lk + 4 * i][lc] = rb[i];
            As[buf][lk + 4 * i][lc] = ra[i];
        }
    };

    float2 acc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);

    load_b(kbeg);
    store_chunk(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = kbeg; k0 < kend; k0 += kCBK) {
        const bool more = k0 + kCBK < kend;
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
        if (more) store_chunk(buf ^ 1);
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
            float2* dst = &Cdst[((size_t)q * MC + m) * m2 + k2];
            if (m < M && FNO_DBG_OK(dst, sizeof(float2))) {
                if (gridDim.y == 1) *dst = cscale(acc[i][j], alpha);
                else atomicAdd(dst, cscale(acc[i][j], alpha));
            }
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
    // the forward with few retained columns, the plan's twiddle tiles and enough
    // rows for two CTAs per SM: one residue class of 128 rows per CTA, aligned
    // 16-byte copies (dft_frows_kernel; 421x421 B16 C64 m = 12: 407 us with the
    // tiles below, 291 us with it)
    // Both pass kernels below run whole passes of 64 columns: they are taken when
    // those waste at most a fifth of the row (W >= ~200; at 85 x 85 the pass
    // kernels measured slower than the tiles below: forward 55 vs 33 us).
    const bool passes_fit = 5ll * kFRP * frows_passes(W) <= 6ll * W;
    if (FWD && passes_fit && p.g_frows && frows_np(N) > 0 &&
        ((M + 4 * kFRM - 1) / (4 * kFRM)) * 4 >= kWant &&
        (reinterpret_cast<uintptr_t>(A) & 15) == 0) {
        const unsigned grid = (unsigned)(((M + 4 * kFRM - 1) / (4 * kFRM)) * 4);
        const int np = frows_np(N);
        const size_t sm = frows_smem(np);
#define FNO_FROWS(NPV)                                                                   \
    dft_frows_kernel<NPV><<<grid, 256, sm, s>>>(A, C, M, W, N, p.g_frows, p.err          \
                                                 FNO_DBG_ARG1(C, 4ull * M * N, p))
        if (np == 8) FNO_FROWS(8);
        else if (np == 16) FNO_FROWS(16);
        else if (np == 24) FNO_FROWS(24);
        else FNO_FROWS(32);
#undef FNO_FROWS
        return cudaGetLastError();
    }
    // the inverse with few retained columns, the plan's twiddle tiles and a
    // 16-byte aligned output: whole rows per CTA, aligned float4 stores
    // (dft_irows_kernel; 421x421 B16 C64 m = 12: 576 us with the tiles below,
    // 269 us with it)
    if (!FWD && passes_fit && K <= kIRKMax && p.g_irows &&
        (reinterpret_cast<uintptr_t>(C) & 15) == 0 && M > 0) {
        const long long gx = (M + kIRM - 1) / kIRM;
        const int npass = irows_passes(W);
        const long long gy = std::min<long long>(npass, (3 * 152 + gx - 1) / gx);
        dft_irows_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, irows_smem(K), s>>>(
            A, C, M, K, W, p.g_irows, p.err FNO_DBG_ARG1(C, 4ull * M * W, p));
        return cudaGetLastError();
    }
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
                             int KB, int MC, float alpha, const float2* At, const fno_plan_s& p,
                             cudaStream_t s) {
    // without the plan's matrices (the allocation-free entry point) the
    // kernel forms A from the twiddle table
    const long long ncols = planes * m2;
    const long long tiles = (long long)((M + kCBM - 1) / kCBM) * ((ncols + kCBN - 1) / kCBN);
    // with fewer than eight 4-warp CTAs per SM the K range is split (chunks of
    // at least 64) and the partial sums are added into the zeroed C; their
    // order of addition varies from run to run.  421x421 B16 C64 m = 12
    // (forward: 384 tiles, K = 421): 53 -> 50 us with the memset
    int ksplit = 1;
    constexpr long long kWantCols = 8 * 152;
    if (tiles < kWantCols && K >= 2 * 64)
        ksplit = (int)std::min<long long>((kWantCols + tiles - 1) / tiles, K / 64);
    int kper = (K + ksplit - 1) / ksplit;
    kper = (kper + kCBK - 1) / kCBK * kCBK;
    ksplit = (K + kper - 1) / kper;
    if (ksplit > 1) {
        cudaError_t e = cudaMemsetAsync(C, 0, 8ull * planes * MC * m2, s);
        if (e != cudaSuccess) return e;
    }
    dft_cols_gemm_kernel<FWD><<<dim3((unsigned)tiles, (unsigned)ksplit), kCT, 0, s>>>(
        B, C, M, K, ncols, m2, KB, MC, p.H, p.m1, alpha, At, p.tw_h, kper
        FNO_DBG_ARG1(C, 8ull * planes * MC * m2, p));
    return cudaGetLastError();
}

}  // namespace
}  // namespace fno

using namespace fno;

std::vector<float2> dft_cols_table(int H, int m1) {
    const int R2 = 2 * m1;
    std::vector<float2> t(2ull * R2 * H);
    const double two_pi = 6.283185307179586476925286766559005768;
    for (int r = 0; r < R2; ++r) {
        const int k1 = r < m1 ? r : H - R2 + r;
        for (int h = 0; h < H; ++h) {
            const long long idx = ((long long)k1 * h) % H;
            const double a = two_pi * (double)idx / (double)H;
            const float c = (float)std::cos(a), sn = (float)std::sin(a);
            t[(size_t)h * R2 + r] = make_float2(c, -sn);                 // forward At[h][r]
            t[(size_t)R2 * H + (size_t)r * H + h] = make_float2(c, sn);  // inverse At[r][h]
        }
    }
    return t;
}

std::vector<float> dft_frows_table(int W, int m2, double scale) {
    const int N = 2 * m2, NP = frows_np(N);
    if (NP == 0 || W < 1) return {};
    const int npass = frows_passes(W);
    std::vector<float> t((size_t)npass * 4 * kFRP * NP, 0.f);
    const double two_pi = 6.283185307179586476925286766559005768;
    for (int pass = 0; pass < npass; ++pass)
        for (int sh = 0; sh < 4; ++sh)
            for (int q = 0; q < kFRP; ++q) {
                const int c = kFRP * pass + q - sh;
                if (c < 0 || c >= W) continue;
                for (int n = 0; n < N; ++n) {
                    const int k2 = n >> 1;
                    const long long idx = ((long long)k2 * c) % W;
                    const double a = two_pi * (double)idx / (double)W;
                    const double v = (n & 1) ? -std::sin(a) : std::cos(a);
                    t[(((size_t)pass * 4 + sh) * kFRP + q) * NP + n] = (float)(scale * v);
                }
            }
    return t;
}

std::vector<float> dft_irows_table(int W, int m2, double scale) {
    const int K = 2 * m2;
    if (K > kIRKMax || W < 1) return {};
    const int npass = irows_passes(W);
    std::vector<float> t((size_t)npass * 4 * K * kIRP, 0.f);
    const double two_pi = 6.283185307179586476925286766559005768;
    for (int pass = 0; pass < npass; ++pass)
        for (int sh = 0; sh < 4; ++sh)
            for (int k = 0; k < K; ++k)
                for (int q = 0; q < kIRP; ++q) {
                    const int c = kIRP * pass + q - sh;
                    if (c < 0 || c >= W) continue;
                    const int k2 = k >> 1;
                    const long long idx = ((long long)k2 * c) % W;
                    const double a = two_pi * (double)idx / (double)W;
                    const double cw = (k2 == 0 || 2 * k2 == W) ? 1.0 : 2.0;
                    const double v = (k & 1) ? -std::sin(a) : std::cos(a);
                    t[(((size_t)pass * 4 + sh) * K + k) * kIRP + q] = (float)(cw * scale * v);
                }
    return t;
}

bool dft_path(int H, int W) {
    const auto pow2 = [](int v) { return v >= 1 && (v & (v - 1)) == 0; };
    return !pow2(H) || !pow2(W);
}

cudaError_t stages_dft_init() {
    cudaError_t e = cudaFuncSetAttribute(dft_irows_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)irows_smem(kIRKMax));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dft_frows_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)frows_smem(8));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dft_frows_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)frows_smem(16));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dft_frows_kernel<24>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)frows_smem(24));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(dft_frows_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)frows_smem(32));
    return e;
}

cudaError_t launch_forward_dft(const fno_plan_s& p, const float* x, float2* X, float2* T,
                               cudaStream_t s, fno_launch_ctx* ctx) {
    const long long planes = (long long)p.B * p.Cin, nrows = planes * p.H;
    cudaError_t e = launch_rows_gemm<true>(x, reinterpret_cast<float*>(T), nrows, p.W, 2 * p.m2,
                                           p.W, 1.f, p.tw_w, p, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    if (e != cudaSuccess) return e;
    e = launch_cols_gemm<true>(T, X, 2 * p.m1, p.H, planes, p.m2, p.H, 2 * p.m1, p.scale,
                               p.g_cols, p, s);  // g_cols may be null (see the launcher)
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_dft(const fno_plan_s& p, const float2* Z, float* y, float2* T,
                               cudaStream_t s, fno_launch_ctx* ctx) {
    const long long planes = (long long)p.B * p.Cout, nrows = planes * p.H;
    cudaError_t e = launch_cols_gemm<false>(Z, T, p.H, 2 * p.m1, planes, p.m2, 2 * p.m1, p.H,
                                            1.f, p.g_cols ? p.g_cols + 2ull * p.m1 * p.H : nullptr,
                                            p, s);
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
