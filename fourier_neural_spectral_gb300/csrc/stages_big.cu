// stages_big.cu -- fused transform kernels for long rows, W in {512, 1024,
// 2048, 4096}, with at most 64 kept columns (m2 <= 64).
//
// A CTA (256 threads) owns the R rows h = p + P*q of one plane, like the
// short-row kernels, and shares their column halves (fused_columns.cuh).  A row
// pair is handled by a group of L = W/16 threads (L in {32..256}):
//
// Forward row transform of the packed pair z = x_a + i x_b, pruned to the bins
// k < m2 and k > W - m2 (decimation in frequency, W = 16 * L):
//   staging: one thread of the group copies the pair's two rows into shared
//           memory with bulk asynchronous copies, one pair ahead, so that the
//           loads overlap the previous pair's arithmetic;
//   pass 1: thread n1 < L reads z[n1 + L*n2] (n2 < 16) from the staged rows,
//           16-point register DFT over n2, times e^{-2 pi i n1 kk / W}, stored
//           as S[kk][n1];
//   pass 2: for each kk, the L-point DFT over n1 is needed only at the few
//           k1 with 16*k1 + kk kept.  With n1 = a + G*b (G = L/16 lanes, b < 16),
//             Zk[k1] = sum_a e^{-2 pi i a k1 / L} D_a[k1 mod 16],
//             D_a[d] = 16-point DFT over b of S[kk][a + G*b];
//           thread (kk, a) computes D_a, forms its terms for every candidate k1
//           and the G lanes of a kk sum them with a shuffle reduce-scatter.
//   The kept bins meet in shared memory and are separated into the two rows'
//   spectra exactly as in the short-row kernels.
// Inverse (complex-to-real) row transform: the exact mirror (decimation in
// time), the kept bins of U = S_a + i S_b entering as the only nonzero inputs.
#include <algorithm>

#include "fft_reg.cuh"
#include "fused_columns.cuh"
#include "internal.h"
#include "tma.cuh"

namespace fno {
namespace {

constexpr int kBT = 256;      // threads per CTA
constexpr int kNL = 4;        // candidate k1 per side: ceil(m2 / 16) <= 4, i.e. m2 <= 64

template <int W>
struct BigCfg {
    static constexpr int L = W / 16;               // threads per row pair
    static constexpr int G = L / 16;               // lanes reduced per bin kk
    static constexpr int NK = 2 * kNL > G ? 2 * kNL : G;  // candidate slots per kk
    static constexpr int Groups = kBT / L;
    static constexpr int SStride = L + G;          // S row stride (== G mod 16)
    static constexpr int GroupScr = 16 * SStride + 16 * NK;
};

template <int W, int R>
struct BigKCfg {
    static constexpr int Scratch = BigCfg<W>::Groups * BigCfg<W>::GroupScr > ColCfg<R>::Scratch
                                       ? BigCfg<W>::Groups * BigCfg<W>::GroupScr
                                       : ColCfg<R>::Scratch;
};

// Shared memory: column/row scratch | Y or V [R][m2 + 1] (rounded to 16 bytes) |
// forward: the staged row pair of every group [Groups][2W] floats and one
// mbarrier per group; inverse: one mbarrier (the plane's Z, staged over the
// scratch and V when it fits).
constexpr size_t kStageBytesPerCta = 256 * 32 * sizeof(float);  // Groups * 2W floats

__host__ __device__ __forceinline__ size_t big_y_floats2(int R, int m2) {
    return ((size_t)R * (m2 + 1) + 1) & ~(size_t)1;
}

template <int W, int R, bool FWD>
size_t big_smem_bytes(int m2) {
    const size_t base = sizeof(float2) * ((size_t)BigKCfg<W, R>::Scratch + big_y_floats2(R, m2));
    return FWD ? base + kStageBytesPerCta + sizeof(uint64_t) * BigCfg<W>::Groups
               : base + sizeof(uint64_t);
}

// Synchronise the L threads of a row-pair group.
template <int L>
__device__ __forceinline__ void group_sync(int g) {
    if constexpr (L <= 32) {
        __syncwarp();
    } else if constexpr (L == kBT) {
        __syncthreads();
    } else {
        asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(L) : "memory");
    }
}

// Candidate k1 of slot j: the lower side 0..3, then the upper side L-4..L-1
// (every bin k < 64 and k > W - 64); slots past 8 are unused.  Candidates
// whose bin is not kept contribute zeros.
template <int L>
__device__ __forceinline__ constexpr int cand_k1(int j) { return j < kNL ? j : L - 2 * kNL + j; }

// Reduce-scatter of N complex values over the G lanes (lane bits below G) that
// share a bin: afterwards lane a holds the sums of slots a*N/G .. a*N/G + N/G - 1
// in r[0 .. N/G).
template <int N, int G>
__device__ __forceinline__ void reduce_scatter(float2 (&r)[N], int a) {
#pragma unroll
    for (int s = G / 2, c = N; s >= 1; s >>= 1, c >>= 1) {
        const bool up = (a & s) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            if (i < c / 2) {
                const float2 lo = r[i], hi = r[i + c / 2];
                const float2 send = up ? lo : hi;
                const float2 keep = up ? hi : lo;
                float2 recv;
                recv.x = __shfl_xor_sync(0xffffffffu, send.x, s);
                recv.y = __shfl_xor_sync(0xffffffffu, send.y, s);
                r[i] = cadd(keep, recv);
            }
        }
    }
}

// ---------------------------------------------------------------- forward ---
template <int W, int R>
__global__ void __launch_bounds__(kBT, 2)
fwd_big_kernel(const float* __restrict__ x, float2* __restrict__ X, int H, int m1, int m2, int P,
               float scale, const float2* __restrict__ tw_w, const float2* __restrict__ tw_h,
               unsigned* __restrict__ err FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    using B = BigCfg<W>;
    constexpr int L = B::L, G = B::G, NK = B::NK;
    constexpr uint32_t kRowBytes = W * sizeof(float);
    static_assert(B::Groups * 2 * kRowBytes == kStageBytesPerCta, "stage size");
    static_assert(BigKCfg<W, R>::Scratch % 2 == 0, "stage must start on 16 bytes");
    extern __shared__ __align__(16) float2 sm[];
    float2* scr = sm;
    float2* Y = sm + BigKCfg<W, R>::Scratch;  // [R][ys]
    float* stage = reinterpret_cast<float*>(Y + big_y_floats2(R, m2));  // [Groups][2W]
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage + B::Groups * 2 * W);
    const int ys = m2 + 1;
    const int plane = blockIdx.x / P;
    const int p = blockIdx.x - plane * P;
    const float* xp = x + (size_t)plane * H * W;

    const int g = threadIdx.x / L, t = threadIdx.x % L;
    constexpr int npairs = R / 2;
    float* stg = stage + g * 2 * W;
    uint64_t* bar = bars + g;
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < B::Groups; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    // rows p + P*2*pair and p + P*(2*pair + 1) into the group's stage
    const auto issue = [&](int pair) {
        const float* ra = xp + (size_t)(p + P * 2 * pair) * W;
        mbar_arrive_expect_tx(bar, 2 * kRowBytes);
        bulk_load(stg, ra, kRowBytes, bar);
        bulk_load(stg + W, ra + (size_t)P * W, kRowBytes, bar);
    };
    bool live = true;     // no wait of this thread has run out
    int pending = -1;     // thread t == 0: parity of a copy that was never seen to land
    if (t == 0 && g < npairs) issue(g);
    float2* S = scr + g * B::GroupScr;  // S[kk][n1], row stride L + G
    float2* Zs = S + 16 * B::SStride;   // Zs[kk][slot]
    // pass-1 twiddles e^{-2 pi i n1 kk / W} for n1 = t, and pass-2 twiddles
    // e^{-2 pi i a k1 / L} = e^{-2 pi i 16 a k1 / W} for the candidate k1
    const int kk2 = t / G, a = t % G;
    float2 tw1[16], tw2[NK];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) tw1[kk] = root<-1>(tw_w, t * kk, W);
#pragma unroll
    for (int j = 0; j < NK; ++j) tw2[j] = root<-1>(tw_w, 16 * a * cand_k1<L>(j), W);

    constexpr int iters = (npairs + B::Groups - 1) / B::Groups;
    for (int it = 0; it < iters; ++it) {
        const int pair = g + it * B::Groups;
        const bool active = pair < npairs;  // uniform over the group
        const int qa = 2 * pair;
        if (active) {
            if (live && !wait_parity_bounded(bar, (uint32_t)(it & 1), err)) {
                live = false;  // the stage holds no valid data; err is set
                if (t == 0) pending = it & 1;
            }
            float2 v[16];
#pragma unroll
            for (int n2 = 0; n2 < 16; ++n2) v[n2] = make_float2(stg[t + L * n2], stg[W + t + L * n2]);
            dft<16, -1>(v);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                S[kk * B::SStride + t] = kk == 0 ? v[0] : cmul(v[kk], tw1[kk]);
        }
        group_sync<L>(g);
        // every thread of the group has read the stage: refill it with the next pair
        if (t == 0 && live && pair + B::Groups < npairs) {
            fence_proxy_async_smem();
            issue(pair + B::Groups);
        }
        if (active) {
            float2 d[16];
#pragma unroll
            for (int b = 0; b < 16; ++b) d[b] = S[kk2 * B::SStride + a + G * b];
            dft<16, -1>(d);
            float2 r[NK];
#pragma unroll
            for (int j = 0; j < NK; ++j) {
                const int k1 = cand_k1<L>(j);
                r[j] = j < 2 * kNL ? cmul(d[k1 & 15], tw2[j]) : make_float2(0.f, 0.f);
            }
            reduce_scatter<NK, G>(r, a);
#pragma unroll
            for (int j = 0; j < NK / G; ++j) Zs[kk2 * NK + a * (NK / G) + j] = r[j];
        }
        group_sync<L>(g);
        if (active) {
            // separation of the two rows' spectra for k = 16*k1 + kk < m2
            for (int k = t; k < m2; k += L) {
                const int kk = k & 15, k1 = k >> 4;  // k1 < NL: lower slot k1
                const float2 zk = Zs[kk * NK + k1];
                float2 zm;  // Z[W - k]
                if (kk == 0) {
                    zm = k1 == 0 ? Zs[0] : Zs[0 * NK + (L - k1) - L + 2 * kNL];
                } else {
                    zm = Zs[(16 - kk) * NK + (L - 1 - k1) - L + 2 * kNL];
                }
                Y[qa * ys + k] = make_float2(0.5f * (zk.x + zm.x), 0.5f * (zk.y - zm.y));
                Y[(qa + 1) * ys + k] = make_float2(0.5f * (zk.y + zm.y), -0.5f * (zk.x - zm.x));
            }
        }
        // the next pair's pass 1 rewrites S only; S was last read before the
        // second barrier above, and Zs is rewritten only after the next first barrier
    }
    // a copy that ran out of time may still land: wait for it (bounded) before
    // the shared memory is reused or released
    if (pending >= 0) wait_parity_bounded(bar, (uint32_t)pending, nullptr);
    __syncthreads();
    columns_forward<R>(scr, Y, ys, X, (size_t)plane * 2 * m1 * m2, H, m1, m2, P, p, scale, tw_h);
}

// ---------------------------------------------------------------- inverse ---
// Whether the plane's Z (16*m1*m2 bytes, contiguous) is brought into shared
// memory with one bulk copy: the column transform must take a single pass and
// Z must fit over the scratch and V, which it overwrites only after it is read.
template <int W, int R>
__host__ __device__ bool big_z_staged(int m1, int m2) {
    return m2 <= ColCfg<R>::CP &&
           16ull * m1 * m2 <= sizeof(float2) * (BigKCfg<W, R>::Scratch + big_y_floats2(R, m2));
}

template <int W, int R, bool ZS>
__global__ void __launch_bounds__(kBT, 2)
inv_big_kernel(const float2* __restrict__ Z, float* __restrict__ y, int H, int m1, int m2, int P,
               float scale, const float2* __restrict__ tw_w, const float2* __restrict__ tw_h,
               unsigned* __restrict__ err FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    using B = BigCfg<W>;
    constexpr int L = B::L, G = B::G, NK = B::NK;
    constexpr int half = W / 2;
    extern __shared__ __align__(16) float2 sm[];
    float2* scr = sm;
    float2* V = sm + BigKCfg<W, R>::Scratch;  // [R][ys]
    const int ys = m2 + 1;
    const int plane = blockIdx.x / P;
    const int p = blockIdx.x - plane * P;
    const float2* Zp = Z + (size_t)plane * 2 * m1 * m2;
    griddep_wait();
    griddep_launch_dependents();

    // ZS (big_z_staged): the plane's Z comes into shared memory with one bulk copy
    uint64_t* zbar = reinterpret_cast<uint64_t*>(V + big_y_floats2(R, m2));
    const uint32_t zbytes = 16u * (uint32_t)m1 * (uint32_t)m2;
    if constexpr (ZS) {
        if (threadIdx.x == 0) {
            mbar_init(zbar, 1);
            fence_barrier_init();
            mbar_arrive_expect_tx(zbar, zbytes);
            bulk_load(sm, Zp, zbytes, zbar);
        }
        __syncthreads();
    }

    if constexpr (ZS) {
        const bool zok = wait_parity_bounded(zbar, 0, err);
        // on a timeout err is set and the output is void; thread 0 still waits
        // (bounded) for the copy, and every thread for thread 0, before the
        // shared memory is rewritten
        if (!zok && threadIdx.x == 0) wait_parity_bounded(zbar, 0, nullptr);
        __syncthreads();
        columns_inverse<R, 0, true>(scr, V, ys, sm, H, m1, m2, P, p, tw_h);
    } else {
        columns_inverse<R>(scr, V, ys, Zp, H, m1, m2, P, p, tw_h);
    }
    __syncthreads();

    const int g = threadIdx.x / L, t = threadIdx.x % L;
    const int kk2 = t / G, a = t % G;
    // second-pass twiddles times the output scale 1/sqrt(HW) (the transform is
    // linear, so scaling its inputs scales the rows it writes)
    float2 tw1[16], tw2[NK];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) tw1[kk] = cscale(root<1>(tw_w, t * kk, W), scale);
#pragma unroll
    for (int j = 0; j < NK; ++j) tw2[j] = root<1>(tw_w, 16 * a * cand_k1<L>(j), W);
    float2* S = scr + g * B::GroupScr;  // S[kk][n1], row stride L + G
    float* yp = y + (size_t)plane * H * W;

    constexpr int npairs = R / 2;
    constexpr int iters = (npairs + B::Groups - 1) / B::Groups;
    for (int it = 0; it < iters; ++it) {
        const int pair = g + it * B::Groups;
        const bool active = pair < npairs;
        const int qa = 2 * pair;
        if (active) {
            const float2* Va = V + qa * ys;
            const float2* Vb = Va + ys;
            // E_a[d] = sum over candidates k1 == d (mod 16) of e^{+2 pi i a k1 / L} U[16 k1 + kk]
            float2 e[16];
#pragma unroll
            for (int d = 0; d < 16; ++d) e[d] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 2 * kNL; ++j) {
                const int k1 = cand_k1<L>(j);
                const int k = 16 * k1 + kk2;
                const int kr = k <= half ? k : W - k;
                if (kr >= m2) continue;
                float2 uk, um;
                packed_bin(Va[kr], Vb[kr], kr == 0 || kr == half, &uk, &um);
                const float2 u = k <= half ? uk : um;
                e[k1 & 15] = cmul(u, tw2[j]);
            }
            // the candidates k1 = 0..3 and L-4..L-1 fill e[0..3] and e[12..15] only
            static_assert(L % 16 == 0 && 2 * kNL == 8, "candidate residues 0..3, 12..15");
            dft16_in8<1>(e);
#pragma unroll
            for (int b = 0; b < 16; ++b) S[kk2 * B::SStride + a + G * b] = e[b];
        }
        group_sync<L>(g);
        if (active) {
            float2 v[16];
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                v[kk] = kk == 0 ? cscale(S[t], scale) : cmul(S[kk * B::SStride + t], tw1[kk]);
            dft<16, 1>(v);
            float* ya = yp + (size_t)(p + P * qa) * W;
            float* yb = ya + (size_t)P * W;
#pragma unroll
            for (int n2 = 0; n2 < 16; ++n2) {
                if (FNO_DBG_OK(&ya[t + L * n2], sizeof(float))) ya[t + L * n2] = v[n2].x;
                if (FNO_DBG_OK(&yb[t + L * n2], sizeof(float))) yb[t + L * n2] = v[n2].y;
            }
        }
        group_sync<L>(g);
    }
}

// ---------------------------------------------------------------- 1D rows ---
// The 1D layer for power-of-two lengths W = L in {512, ..., 4096} with m2 = m <= 64:
// the long-row transforms above without a column step.  Group g of CTA c takes
// the sequences qa = 2*(c*Groups + g) and qa + 1 (a zero row when the count is
// odd), read straight from global memory, and writes their kept bins times
// `scale` to X[seq][k] (forward), or rebuilds their two rows from Z[seq][k]
// (inverse).  The arithmetic is that of fwd_big_kernel / inv_big_kernel for one
// row pair per group.
template <int W>
__global__ void __launch_bounds__(kBT, 2)
fwd_rows1d_kernel(const float* __restrict__ x, float2* __restrict__ X, int S, int m2,
                  float scale, const float2* __restrict__ tw_w FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    using B = BigCfg<W>;
    constexpr int L = B::L, G = B::G, NK = B::NK;
    __shared__ __align__(16) float2 scr[B::Groups * B::GroupScr];
    const int g = threadIdx.x / L, t = threadIdx.x % L;
    const int qa = 2 * (blockIdx.x * B::Groups + g);
    const bool active = qa < S;  // uniform over the group
    const bool has_b = qa + 1 < S;
    griddep_wait();  // x may be the previous kernel's output
    griddep_launch_dependents();
    float2* Sm = scr + g * B::GroupScr;  // S[kk][n1], row stride L + G
    float2* Zs = Sm + 16 * B::SStride;   // Zs[kk][slot]
    const int kk2 = t / G, a = t % G;
    float2 tw1[16], tw2[NK];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) tw1[kk] = root<-1>(tw_w, t * kk, W);
#pragma unroll
    for (int j = 0; j < NK; ++j) tw2[j] = root<-1>(tw_w, 16 * a * cand_k1<L>(j), W);

    if (active) {
        const float* ra = x + (size_t)qa * W;
        const float* rb = ra + W;
        float2 v[16];
#pragma unroll
        for (int n2 = 0; n2 < 16; ++n2)
            v[n2] = make_float2(__ldg(ra + t + L * n2), has_b ? __ldg(rb + t + L * n2) : 0.f);
        dft<16, -1>(v);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            Sm[kk * B::SStride + t] = kk == 0 ? v[0] : cmul(v[kk], tw1[kk]);
    }
    group_sync<L>(g);
    if (active) {
        float2 d[16];
#pragma unroll
        for (int b = 0; b < 16; ++b) d[b] = Sm[kk2 * B::SStride + a + G * b];
        dft<16, -1>(d);
        float2 r[NK];
#pragma unroll
        for (int j = 0; j < NK; ++j) {
            const int k1 = cand_k1<L>(j);
            r[j] = j < 2 * kNL ? cmul(d[k1 & 15], tw2[j]) : make_float2(0.f, 0.f);
        }
        reduce_scatter<NK, G>(r, a);
#pragma unroll
        for (int j = 0; j < NK / G; ++j) Zs[kk2 * NK + a * (NK / G) + j] = r[j];
    }
    group_sync<L>(g);
    if (active) {
        // separation of the two rows' spectra for k = 16*k1 + kk < m2
        const float hs = 0.5f * scale;
        for (int k = t; k < m2; k += L) {
            const int kk = k & 15, k1 = k >> 4;
            const float2 zk = Zs[kk * NK + k1];
            float2 zm;  // Z[W - k]
            if (kk == 0) {
                zm = k1 == 0 ? Zs[0] : Zs[0 * NK + (L - k1) - L + 2 * kNL];
            } else {
                zm = Zs[(16 - kk) * NK + (L - 1 - k1) - L + 2 * kNL];
            }
            if (FNO_DBG_OK(&X[(size_t)qa * m2 + k], sizeof(float2)))
                X[(size_t)qa * m2 + k] = make_float2(hs * (zk.x + zm.x), hs * (zk.y - zm.y));
            if (has_b && FNO_DBG_OK(&X[(size_t)(qa + 1) * m2 + k], sizeof(float2)))
                X[(size_t)(qa + 1) * m2 + k] = make_float2(hs * (zk.y + zm.y), -hs * (zk.x - zm.x));
        }
    }
}

template <int W>
__global__ void __launch_bounds__(kBT, 2)
inv_rows1d_kernel(const float2* __restrict__ Z, float* __restrict__ y, int S, int m2,
                  float scale, const float2* __restrict__ tw_w FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    using B = BigCfg<W>;
    constexpr int L = B::L, G = B::G, NK = B::NK;
    constexpr int half = W / 2;
    __shared__ __align__(16) float2 scr[B::Groups * B::GroupScr];
    const int g = threadIdx.x / L, t = threadIdx.x % L;
    const int qa = 2 * (blockIdx.x * B::Groups + g);
    const bool active = qa < S;
    const bool has_b = qa + 1 < S;
    griddep_wait();  // Z is the previous kernel's output; y may still be read before it
    griddep_launch_dependents();
    float2* Sm = scr + g * B::GroupScr;
    const int kk2 = t / G, a = t % G;
    float2 tw1[16], tw2[NK];
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) tw1[kk] = cscale(root<1>(tw_w, t * kk, W), scale);
#pragma unroll
    for (int j = 0; j < NK; ++j) tw2[j] = root<1>(tw_w, 16 * a * cand_k1<L>(j), W);

    if (active) {
        const float2* Va = Z + (size_t)qa * m2;
        const float2* Vb = Va + m2;
        float2 e[16];
#pragma unroll
        for (int d = 0; d < 16; ++d) e[d] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 2 * kNL; ++j) {
            const int k1 = cand_k1<L>(j);
            const int k = 16 * k1 + kk2;
            const int kr = k <= half ? k : W - k;
            if (kr >= m2) continue;
            const float2 va = __ldg(&Va[kr]);
            const float2 vb = has_b ? __ldg(&Vb[kr]) : make_float2(0.f, 0.f);
            float2 uk, um;
            packed_bin(va, vb, kr == 0 || kr == half, &uk, &um);
            e[k1 & 15] = cmul(k <= half ? uk : um, tw2[j]);
        }
        static_assert(L % 16 == 0 && 2 * kNL == 8, "candidate residues 0..3, 12..15");
        dft16_in8<1>(e);
#pragma unroll
        for (int b = 0; b < 16; ++b) Sm[kk2 * B::SStride + a + G * b] = e[b];
    }
    group_sync<L>(g);
    if (active) {
        float2 v[16];
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            v[kk] = kk == 0 ? cscale(Sm[t], scale) : cmul(Sm[kk * B::SStride + t], tw1[kk]);
        dft<16, 1>(v);
        float* ya = y + (size_t)qa * W;
        float* yb = ya + W;
#pragma unroll
        for (int n2 = 0; n2 < 16; ++n2) {
            if (FNO_DBG_OK(&ya[t + L * n2], sizeof(float))) ya[t + L * n2] = v[n2].x;
            if (has_b && FNO_DBG_OK(&yb[t + L * n2], sizeof(float))) yb[t + L * n2] = v[n2].y;
        }
    }
}

template <bool FWD, int W>
cudaError_t launch_rows1d_w(const fno_plan_s& p, const float* x, float2* X, const float2* Z,
                            float* y, cudaStream_t s) {
    const int S = p.B * (FWD ? p.Cin : p.Cout);
    const int pairs = (S + 1) / 2;
    const unsigned grid = (unsigned)((pairs + BigCfg<W>::Groups - 1) / BigCfg<W>::Groups);
    if (FWD)
        return launch_pdl(fwd_rows1d_kernel<W>, grid, kBT, 0, s, x, X, S, p.m2, p.scale, p.tw_w
                          FNO_DBG_ARG1(X, 8ull * S * p.m2, p));
    return launch_pdl(inv_rows1d_kernel<W>, grid, kBT, 0, s, Z, y, S, p.m2, p.scale, p.tw_w
                      FNO_DBG_ARG1(y, 4ull * S * p.W, p));
}

template <bool FWD>
cudaError_t launch_rows1d(const fno_plan_s& p, const float* x, float2* X, const float2* Z,
                          float* y, cudaStream_t s) {
    switch (p.W) {
        case 512: return launch_rows1d_w<FWD, 512>(p, x, X, Z, y, s);
        case 1024: return launch_rows1d_w<FWD, 1024>(p, x, X, Z, y, s);
        case 2048: return launch_rows1d_w<FWD, 2048>(p, x, X, Z, y, s);
        case 4096: return launch_rows1d_w<FWD, 4096>(p, x, X, Z, y, s);
    }
    return cudaErrorInvalidValue;
}

template <int W, int R>
cudaError_t set_attrs() {
    const int fb = (int)std::min<size_t>(big_smem_bytes<W, R, true>(64), kMaxDynSmem);
    const int ib = (int)std::min<size_t>(big_smem_bytes<W, R, false>(64), kMaxDynSmem);
    cudaError_t e =
        cudaFuncSetAttribute(fwd_big_kernel<W, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, fb);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inv_big_kernel<W, R, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, ib);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inv_big_kernel<W, R, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, ib);
    return e;
}

template <int W>
cudaError_t set_attrs_w() {
    cudaError_t e = set_attrs<W, 32>();
    if (e == cudaSuccess) e = set_attrs<W, 64>();
    if (e == cudaSuccess) e = set_attrs<W, 128>();
    if (e == cudaSuccess) e = set_attrs<W, 256>();
    return e;
}

template <bool FWD, int W, int R>
cudaError_t launch(const fno_plan_s& p, const float* x, float2* X, const float2* Z, float* y,
                   cudaStream_t s) {
    if (FWD) {
        const size_t smem = big_smem_bytes<W, R, true>(p.m2);
        const unsigned grid = (unsigned)((size_t)p.B * p.Cin * p.P);
        return launch_pdl(fwd_big_kernel<W, R>, grid, kBT, smem, s, x, X, p.H, p.m1, p.m2, p.P,
                          p.scale, p.tw_w, p.tw_h, p.err
                          FNO_DBG_ARG1(X, 8ull * p.B * p.Cin * p.nm, p));
    } else {
        const size_t smem = big_smem_bytes<W, R, false>(p.m2);
        const unsigned grid = (unsigned)((size_t)p.B * p.Cout * p.Pi);
        if (big_z_staged<W, R>(p.m1, p.m2))
            return launch_pdl(inv_big_kernel<W, R, true>, grid, kBT, smem, s, Z, y, p.H, p.m1,
                              p.m2, p.Pi, p.scale, p.tw_w, p.tw_h, p.err
                              FNO_DBG_ARG1(y, 4ull * p.B * p.Cout * p.H * p.W, p));
        return launch_pdl(inv_big_kernel<W, R, false>, grid, kBT, smem, s, Z, y, p.H, p.m1, p.m2,
                          p.Pi, p.scale, p.tw_w, p.tw_h, p.err
                          FNO_DBG_ARG1(y, 4ull * p.B * p.Cout * p.H * p.W, p));
    }
}

template <bool FWD, int W>
cudaError_t dispatch_r(const fno_plan_s& p, const float* x, float2* X, const float2* Z, float* y,
                       cudaStream_t s) {
    switch (FWD ? p.R : p.Ri) {
        case 32: return launch<FWD, W, 32>(p, x, X, Z, y, s);
        case 64: return launch<FWD, W, 64>(p, x, X, Z, y, s);
        case 128: return launch<FWD, W, 128>(p, x, X, Z, y, s);
        case 256: return launch<FWD, W, 256>(p, x, X, Z, y, s);
    }
    return cudaErrorInvalidValue;
}

template <bool FWD>
cudaError_t dispatch(const fno_plan_s& p, const float* x, float2* X, const float2* Z, float* y,
                     cudaStream_t s) {
    switch (p.W) {
        case 512: return dispatch_r<FWD, 512>(p, x, X, Z, y, s);
        case 1024: return dispatch_r<FWD, 1024>(p, x, X, Z, y, s);
        case 2048: return dispatch_r<FWD, 2048>(p, x, X, Z, y, s);
        case 4096: return dispatch_r<FWD, 4096>(p, x, X, Z, y, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t stages_big_init() {
    cudaError_t e = set_attrs_w<512>();
    if (e == cudaSuccess) e = set_attrs_w<1024>();
    if (e == cudaSuccess) e = set_attrs_w<2048>();
    if (e == cudaSuccess) e = set_attrs_w<4096>();
    return e;
}

size_t big_smem_bytes_any(int W, int R, int m2, bool fwd) {
    switch (W * 1000 + R) {
#define CASE(w, r) \
    case w * 1000 + r: return fwd ? big_smem_bytes<w, r, true>(m2) : big_smem_bytes<w, r, false>(m2);
        CASE(512, 32) CASE(512, 64) CASE(512, 128) CASE(512, 256)
        CASE(1024, 32) CASE(1024, 64) CASE(1024, 128) CASE(1024, 256)
        CASE(2048, 32) CASE(2048, 64) CASE(2048, 128) CASE(2048, 256)
        CASE(4096, 32) CASE(4096, 64) CASE(4096, 128) CASE(4096, 256)
#undef CASE
    }
    return (size_t)-1;
}

bool big_z_staged_any(int W, int R, int m1, int m2) {
    switch (W * 1000 + R) {
#define CASE(w, r) \
    case w * 1000 + r: return big_z_staged<w, r>(m1, m2);
        CASE(512, 32) CASE(512, 64) CASE(512, 128) CASE(512, 256)
        CASE(1024, 32) CASE(1024, 64) CASE(1024, 128) CASE(1024, 256)
        CASE(2048, 32) CASE(2048, 64) CASE(2048, 128) CASE(2048, 256)
        CASE(4096, 32) CASE(4096, 64) CASE(4096, 128) CASE(4096, 256)
#undef CASE
    }
    return false;
}

cudaError_t launch_forward_big(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s) {
    return dispatch<true>(p, x, X, nullptr, nullptr, s);
}

cudaError_t launch_inverse_big(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s) {
    return dispatch<false>(p, nullptr, nullptr, Z, y, s);
}

bool rows1d_supported(int W, int m2) {
    return (W == 512 || W == 1024 || W == 2048 || W == 4096) && m2 <= 16 * kNL;
}

cudaError_t launch_forward_rows1d(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s,
                                  fno_launch_ctx* ctx) {
    cudaError_t e = launch_rows1d<true>(p, x, X, nullptr, nullptr, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_rows1d(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s,
                                  fno_launch_ctx* ctx) {
    cudaError_t e = launch_rows1d<false>(p, nullptr, nullptr, Z, y, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
