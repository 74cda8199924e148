// fused_rows.cuh -- the row halves of the fused transform kernels for row
// lengths W and column lengths R in {32, 64, 128, 256} (the algorithm is
// described at the top of stages_fused.cu), shared by the standalone kernels
// (stages_fused.cu) and the single-launch layer (layer_persistent.cu), and the
// per-plane forward and inverse bodies that the single-launch layer loops
// over.  The standalone kernels spell the same per-plane steps out inline: the
// register allocation of their tuned versions depends on it.
#pragma once

#include "fft_reg.cuh"
#include "fused_columns.cuh"
#include "internal.h"
#include "tma.cuh"

namespace fno {
namespace {

constexpr int kFT = 256;  // threads per CTA

// Row-pass scratch of one row-pair group: forward S[kk][n1] (row stride Bq+1),
// inverse S[n1][kk] (row stride 17), plus for Bq = 16 the W outputs of the
// pair.  The group stride is == Bq (mod 16) complex elements so that the
// 16/Bq groups sharing a half-warp fall on different shared-memory banks.
template <int W>
struct RowCfg {
    static constexpr int Bq = W / 16;
    static constexpr int need0 = 16 * (Bq + 1) > 17 * Bq ? 16 * (Bq + 1) : 17 * Bq;
    static constexpr int need = need0 + (Bq == 16 ? W : 0);
    static constexpr int Scr = need + ((Bq % 16) - need % 16 + 16) % 16;
};

template <int W, int R>
struct FusedCfg {
    static constexpr int BqW = W / 16;           // threads per row pair
    static constexpr int BqR = R / 16;           // threads per column
    static constexpr int RowGroups = kFT / BqW;  // row pairs in flight
    static constexpr int ColsPerPass = kFT / BqR;
    static_assert(kFT == kColThreads, "column passes assume 256 threads");
    static constexpr int RowScr = RowCfg<W>::Scr;
    // Column-pass scratch: S[col][kk][n1], per column stride R + 17 (== 1 mod 16,
    // lanes run over columns).
    static constexpr int ColScr = R + 17;
    static constexpr int ScratchA = RowGroups * RowScr;
    static constexpr int ScratchB = ColsPerPass * ColScr;
    static constexpr int Scratch = ScratchA > ScratchB ? ScratchA : ScratchB;
    // CTAs per SM the register allocation is sized for (shared memory allows
    // three for planes up to 128 x 128, fewer above)
    static constexpr int MinBlocks = W * R <= 128 * 128 ? 3 : (W * R <= 256 * 128 ? 2 : 1);
};

// Row stride of the kept-column array Y / V: m2 rounded up to == 4 (mod 8)
// complex elements, so that the rows written (read) by neighbouring row-pair
// groups fall on different shared-memory banks.
__host__ __device__ inline int kept_stride(int m2) { return m2 + ((4 - m2 % 8) + 8) % 8; }

// The inverse of 128- and 256-point rows can bring the plane's Z into shared
// memory with one bulk copy (fused_z_staged).  Staging the forward's row pairs
// and the inverse's output rows through shared memory by bulk copies was
// measured too (128 x 128: no gain; 256 x 256: forward 76 -> 111 us, inverse
// 87 -> 94 us) and is not used.
template <int W>
constexpr bool staged_z() { return W >= 128; }

// Shared memory: scratch | Y or V [R][ys] | one mbarrier (staged Z).
template <int W, int R>
size_t fused_smem_bytes(int m2) {
    using C = FusedCfg<W, R>;
    return sizeof(float2) * ((size_t)C::Scratch + (size_t)R * kept_stride(m2)) + sizeof(uint64_t);
}

// Streaming accesses of data that one kernel touches once (the layer's x and
// y): an L2 cache policy with evict-first priority, so that they do not push
// the workspaces X and Z, which the next kernel reads, out of L2.
__device__ __forceinline__ unsigned long long l2_evict_first() {
    unsigned long long pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ float ld_stream(const float* p, unsigned long long pol) {
    float v;
    asm("ld.global.nc.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_stream(float* p, float v, unsigned long long pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

// Mirror partner of bin kk of the 16-point first pass: kk and (16 - kk) mod 16
// are handled by the same thread so that Z[k] and Z[W - k] meet in registers.
// Pair p (p in [0, 8)) is {0, 8} for p = 0 and {p, 16 - p} otherwise.
__device__ __forceinline__ int pair_a(int p) { return p; }
__device__ __forceinline__ int pair_b(int p) { return p == 0 ? 8 : 16 - p; }

// One packed row pair through the forward row transform.  Called by every lane
// of the warp (the group of Bq lanes is inside one warp); `active` lanes do work.
// Writes the separated spectra of the two rows, bins k < m2, to Ya and Yb.
// tw1[kk] = e^{-2 pi i t kk / W}: the thread's first-pass twiddles, loaded once
// per kernel and reused for every row pair.
template <int W, int M2S = 0>
__device__ __forceinline__ void row_pair_forward(const float* __restrict__ ra,
                                                 const float* __restrict__ rb, float2* S,
                                                 float2* Ya, float2* Yb, int t, int m2,
                                                 const float2 (&tw1)[16], bool active) {
    constexpr int Bq = W / 16;
    constexpr int RS = Bq + 1;
    // k1 blocks that can hold a kept bin k < m2 (all of them when m2 is known
    // only at run time)
    constexpr int KH = M2S > 0 ? (M2S + 15) / 16 : Bq;
    if (M2S) m2 = M2S;
    if (active) {
        // x with an evict-first L2 policy for rows up to 128 points (16 x 64 x
        // 128 x 128: forward 33.8 -> 32.0 us, the workspaces stay in L2); at 256
        // points it slowed the contraction that follows (180 -> 186 us)
        const unsigned long long pol = W <= 128 ? l2_evict_first() : 0ull;
        float2 v[16];
#pragma unroll
        for (int n2 = 0; n2 < 16; ++n2) {
            const float* pa = ra + t + Bq * n2;
            const float* pb = rb + t + Bq * n2;
            v[n2] = W <= 128 ? make_float2(ld_stream(pa, pol), ld_stream(pb, pol))
                             : make_float2(__ldg(pa), __ldg(pb));
        }
        dft<16, -1>(v);
#pragma unroll
        for (int kk = 1; kk < 16; ++kk) v[kk] = cmul(v[kk], tw1[kk]);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) S[kk * RS + t] = v[kk];
    }
    __syncwarp();
    if constexpr (Bq == 16) {
        // one bin kk = t per thread; the outputs meet in shared memory
        float2* Zs = S + 16 * RS;
        if (active) {
            float2 u[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) u[j] = S[t * RS + j];
            dft<16, -1>(u);
#pragma unroll
            for (int k1 = 0; k1 < 16; ++k1) {
                const int k = 16 * k1 + t;
                if (k < m2 || k > W - m2) Zs[k] = u[k1];
            }
        }
        __syncwarp();
        if (active) {
            for (int k = t; k < m2; k += Bq) {
                const float2 zk = Zs[k], zm = Zs[(W - k) & (W - 1)];
                Ya[k] = make_float2(0.5f * (zk.x + zm.x), 0.5f * (zk.y - zm.y));
                Yb[k] = make_float2(0.5f * (zk.y + zm.y), -0.5f * (zk.x - zm.x));
            }
        }
        __syncwarp();
    } else {
        constexpr int NP = 8 / Bq;  // mirror pairs per thread
        float2 za[NP][Bq], zb[NP][Bq];
        if (active) {
#pragma unroll
            for (int ps = 0; ps < NP; ++ps) {
                const int p = t + Bq * ps;
                const int ka = pair_a(p), kb = pair_b(p);
#pragma unroll
                for (int j = 0; j < Bq; ++j) {
                    za[ps][j] = S[ka * RS + j];
                    zb[ps][j] = S[kb * RS + j];
                }
                dft<Bq, -1>(za[ps]);
                dft<Bq, -1>(zb[ps]);
            }
        }
        __syncwarp();  // S may be overwritten by the next pair from here on
        if (active) {
#pragma unroll
            for (int ps = 0; ps < NP; ++ps) {
                const int p = t + Bq * ps;
                const int ka = pair_a(p), kb = pair_b(p);
#pragma unroll
                for (int k1 = 0; k1 < Bq; ++k1) {
                    if (k1 >= KH) continue;
                    // X_a[k] = (Z[k] + conj Z[W-k]) / 2,  X_b[k] = (Z[k] - conj Z[W-k]) / 2i
                    const int k = 16 * k1 + ka;
                    if (k < m2) {
                        const float2 zk = za[ps][k1];
                        const float2 zm = p == 0 ? za[ps][(Bq - k1) % Bq] : zb[ps][Bq - 1 - k1];
                        Ya[k] = make_float2(0.5f * (zk.x + zm.x), 0.5f * (zk.y - zm.y));
                        Yb[k] = make_float2(0.5f * (zk.y + zm.y), -0.5f * (zk.x - zm.x));
                    }
                    const int k2 = 16 * k1 + kb;
                    if (k2 < m2) {
                        const float2 zk = zb[ps][k1];
                        const float2 zm = p == 0 ? zb[ps][Bq - 1 - k1] : za[ps][Bq - 1 - k1];
                        Ya[k2] = make_float2(0.5f * (zk.x + zm.x), 0.5f * (zk.y - zm.y));
                        Yb[k2] = make_float2(0.5f * (zk.y + zm.y), -0.5f * (zk.x - zm.x));
                    }
                }
            }
        }
    }
}

// One row pair through the inverse (complex-to-real) row transform: reads the
// kept bins of rows a and b from Va, Vb and writes the two output rows.
// The thread's first-pass twiddles e^{+2 pi i n1 kk / W} for its bins kk,
// loaded once per kernel: twi[(ps * 2 + side) * Bq + n1] with side 0 for bin
// pair_a(p), 1 for pair_b(p) (and twi[n1] = e^{+2 pi i n1 t / W} when Bq = 16).
// The twiddles carry the output scale 1/sqrt(HW) (the row transform is linear,
// so scaling the first pass's outputs scales the rows); the n1 = 0 terms, which
// take no twiddle, are scaled where they are stored.
template <int W>
__device__ __forceinline__ void inverse_twiddles(float2 (&twi)[16], int t,
                                                 const float2* __restrict__ tw, float scale) {
    constexpr int Bq = W / 16;
    if constexpr (Bq == 16) {
#pragma unroll
        for (int n1 = 0; n1 < 16; ++n1) twi[n1] = cscale(root<1>(tw, n1 * t, W), scale);
    } else {
        constexpr int NP = 8 / Bq;
#pragma unroll
        for (int ps = 0; ps < NP; ++ps) {
            const int p = t + Bq * ps;
#pragma unroll
            for (int n1 = 0; n1 < Bq; ++n1) {
                twi[(ps * 2) * Bq + n1] = cscale(root<1>(tw, n1 * pair_a(p), W), scale);
                twi[(ps * 2 + 1) * Bq + n1] = cscale(root<1>(tw, n1 * pair_b(p), W), scale);
            }
        }
    }
}

template <int W, int M2S = 0>
__device__ __forceinline__ void row_pair_inverse(const float2* Va, const float2* Vb, float2* S,
                                                 float* __restrict__ ya, float* __restrict__ yb,
                                                 int t, int m2, const float2 (&twi)[16],
                                                 float scale, bool active) {
    constexpr int Bq = W / 16;
    constexpr int RS = 17;
    constexpr int half = W / 2;
    constexpr int KH = M2S > 0 ? (M2S + 15) / 16 : Bq;  // k1 blocks holding bins k < m2
    if (M2S) m2 = M2S;
    if (active) {
        if constexpr (Bq == 16) {
            const int kk = t;
            float2 u[16];
#pragma unroll
            for (int k1 = 0; k1 < 16; ++k1) {
                const int k = 16 * k1 + kk;
                float2 val = make_float2(0.f, 0.f);
                const int kr = k <= half ? k : W - k;
                if (kr < m2) {
                    float2 uk, um;
                    packed_bin(Va[kr], Vb[kr], kr == 0 || kr == half, &uk, &um);
                    val = k <= half ? uk : um;
                }
                u[k1] = val;
            }
            dft<16, 1>(u);
#pragma unroll
            for (int n1 = 0; n1 < 16; ++n1)
                S[n1 * RS + kk] = n1 == 0 ? cscale(u[0], scale) : cmul(u[n1], twi[n1]);
        } else {
            constexpr int NP = 8 / Bq;
#pragma unroll
            for (int ps = 0; ps < NP; ++ps) {
                const int p = t + Bq * ps;
                const int ka = pair_a(p), kb = pair_b(p);
                float2 ua[Bq], ub[Bq];
#pragma unroll
                for (int j = 0; j < Bq; ++j) ua[j] = ub[j] = make_float2(0.f, 0.f);
#pragma unroll
                for (int k1 = 0; k1 < Bq; ++k1) {
                    if (k1 >= KH) continue;      // only bins k < m2 carry data (mirrors below)
                    const int k = 16 * k1 + ka;  // its mirror W - k is bin kb (ka if p = 0)
                    if (k <= half && k < m2) {
                        float2 uk, um;
                        packed_bin(Va[k], Vb[k], k == 0 || k == half, &uk, &um);
                        ua[k1] = uk;
                        if (k != 0 && k != half) {
                            if (p == 0) ua[(Bq - k1) % Bq] = um;
                            else ub[Bq - 1 - k1] = um;
                        }
                    }
                    const int k2 = 16 * k1 + kb;
                    if (k2 <= half && k2 < m2) {
                        float2 uk, um;
                        packed_bin(Va[k2], Vb[k2], k2 == half, &uk, &um);
                        ub[k1] = uk;
                        if (k2 != half) {
                            if (p == 0) ub[Bq - 1 - k1] = um;
                            else ua[Bq - 1 - k1] = um;
                        }
                    }
                }
                dft<Bq, 1>(ua);
                dft<Bq, 1>(ub);
#pragma unroll
                for (int n1 = 0; n1 < Bq; ++n1) {
                    S[n1 * RS + ka] =
                        n1 == 0 ? cscale(ua[0], scale) : cmul(ua[n1], twi[(ps * 2) * Bq + n1]);
                    S[n1 * RS + kb] =
                        n1 == 0 ? cscale(ub[0], scale) : cmul(ub[n1], twi[(ps * 2 + 1) * Bq + n1]);
                }
            }
        }
    }
    __syncwarp();
    if (active) {
        float2 v[16];
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) v[kk] = S[t * RS + kk];
        dft<16, 1>(v);
        // y with an evict-first L2 policy for rows up to 128 points, as x in the
        // forward (16 x 64 x 128 x 128: layer 80.2 -> 79.6 us with both)
        const unsigned long long pol = W <= 128 ? l2_evict_first() : 0ull;
#pragma unroll
        for (int n2 = 0; n2 < 16; ++n2) {
            float* pa = &ya[t + Bq * n2];
            float* pb = &yb[t + Bq * n2];
            if (W <= 128) {
                if (FNO_DBG_OK(pa, sizeof(float))) st_stream(pa, v[n2].x, pol);
                if (FNO_DBG_OK(pb, sizeof(float))) st_stream(pb, v[n2].y, pol);
            } else {
                if (FNO_DBG_OK(pa, sizeof(float))) *pa = v[n2].x;
                if (FNO_DBG_OK(pb, sizeof(float))) *pb = v[n2].y;
            }
        }
    }
    __syncwarp();
}

// Forward transform of one plane (rows h = p + P*q of plane `plane`): rows into
// Y in shared memory, then the column transform into X.  256 threads; ends
// with a CTA barrier, after which the shared memory may be reused.  scr: the
// scratch (FusedCfg::Scratch elements), Y: the kept columns [R][ys] after it,
// ys = kept_stride(m2), xp: the plane's first element, x + plane * H * W.
template <int W, int R, int M1S = 0, int M2S = 0>
__device__ __forceinline__ void fwd_fused_plane(float2* scr, float2* Y, int ys, const float* xp,
                                                float2* X, int H, int m1, int m2, int P,
                                                int plane, int p, float scale,
                                                const float2* tw_w, const float2* tw_h) {
    using C = FusedCfg<W, R>;
    {
        constexpr int Bq = C::BqW;
        const int g = threadIdx.x / Bq, t = threadIdx.x % Bq;
        float2* S = scr + g * C::RowScr;
        float2 tw1[16];
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) tw1[kk] = root<-1>(tw_w, t * kk, W);
        constexpr int npairs = R / 2;
        constexpr int iters = (npairs + C::RowGroups - 1) / C::RowGroups;
        for (int it = 0; it < iters; ++it) {
            const int pair = g + it * C::RowGroups;
            const bool active = pair < npairs;
            const int qa = 2 * pair;
            const float* ra = xp + (size_t)(p + P * qa) * W;
            row_pair_forward<W, M2S>(ra, ra + (size_t)P * W, S, Y + qa * ys, Y + (qa + 1) * ys, t,
                                     m2, tw1, active);
        }
    }
    __syncthreads();
    columns_forward<R, M1S>(scr, Y, ys, X, (size_t)plane * 2 * m1 * m2, H, m1, m2, P, p, scale,
                            tw_h);
}

// Row half of the inverse of one plane: pairs of V rows (shared memory, after
// the column transform) -> two real output rows each.  256 threads.
template <int W, int R, int M2S = 0>
__device__ __forceinline__ void inv_rows_plane(float2* scr, const float2* V, int ys,
                                               float* __restrict__ y, int H, int m2, int P,
                                               int plane, int p, float scale,
                                               const float2* __restrict__ tw_w) {
    using C = FusedCfg<W, R>;
    constexpr int Bq = C::BqW;
    const int g = threadIdx.x / Bq, t = threadIdx.x % Bq;
    float2* S = scr + g * C::RowScr;
    float2 twi[16];
    inverse_twiddles<W>(twi, t, tw_w, scale);
    float* yp = y + (size_t)plane * H * W;
    constexpr int npairs = R / 2;
    constexpr int iters = (npairs + C::RowGroups - 1) / C::RowGroups;
    for (int it = 0; it < iters; ++it) {
        const int pair = g + it * C::RowGroups;
        const bool active = pair < npairs;
        const int qa = 2 * pair;
        float* ya = yp + (size_t)(p + P * qa) * W;
        row_pair_inverse<W, M2S>(V + qa * ys, V + (qa + 1) * ys, S, ya, ya + (size_t)P * W, t,
                                 m2, twi, scale, active);
    }
}

}  // namespace
}  // namespace fno
