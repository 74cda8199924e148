// fused_columns.cuh -- the column halves of the fused transform kernels,
// shared by the kernels for short rows (stages_fused.cu) and long rows
// (stages_big.cu).  256 threads; R is the column length (32..256).
//
// Forward: every kept column k2 of Y[q][k2] (q in [0, R)) is transformed with an
// R-point DFT split as R = 16 * (R/16): a 16-point register DFT over the rows
// q = n1 + (R/16)*n2, twiddle e^{-2 pi i n1 kk / R}, shared-memory transpose,
// then (R/16)-point DFTs.  With P = 1 (R = H) output residue f is the
// frequency itself and is scaled by 1/sqrt(HW) and stored to X.  With P > 1 the
// rows are h = p + P*q and, since H = P*R,
//   X[k1] = sum_h Y[h] e^{-2 pi i k1 h / H}
//         = e^{-2 pi i k1 p / H} * (R-point DFT over q)[k1 mod R],
// so every retained k1 takes residue k1 mod R times its own twiddle and adds it
// into X (R need not reach 2*m1: frequencies sharing a residue simply read the
// same value).  Inverse: the mirror (decimation in time); with P > 1 the inputs
// of a residue are the sum of its retained frequencies times e^{+2 pi i k1 p / H}.
#pragma once

#include "fft_reg.cuh"

namespace fno {

constexpr int kColThreads = 256;

template <int R>
struct ColCfg {
    static constexpr int Bq = R / 16;
    static constexpr int CP = kColThreads / Bq;  // columns per pass
    static constexpr int Scr = R + 17;           // per-column scratch (== 1 mod 16)
    static constexpr int Scratch = CP * Scr;
};

// Whether output residue block k1 (residues 16*k1 .. 16*k1 + 15) can hold a
// retained frequency when m1 is the compile-time constant M1S (> 0); always
// true when M1S = 0 (m1 known only at run time).
template <int R, int M1S>
__device__ __forceinline__ constexpr bool k1_live(int k1) {
    return M1S == 0 || 16 * k1 < M1S || 16 * k1 + 15 >= R - M1S;
}

template <int R, int M1S = 0>
__device__ __forceinline__ void columns_forward(float2* scr, const float2* Y, int ys,
                                                float2* __restrict__ X, size_t xbase, int H,
                                                int m1, int m2, int P, int p, float scale,
                                                const float2* __restrict__ tw_h) {
    if (M1S) m1 = M1S;
    constexpr int Bq = ColCfg<R>::Bq;
    constexpr int J = 16 / Bq;
    constexpr int CP = ColCfg<R>::CP;
    const int cs = threadIdx.x % CP;   // column within the pass
    const int n1 = threadIdx.x / CP;   // position within the column transform
    float2* S = scr + cs * ColCfg<R>::Scr;  // S[kk][n1] with row stride Bq
    const float2 cdn = root<-1>(tw_h, (H - R) * p, H);  // e^{-2 pi i (H - R) p / H}
    for (int c0 = 0; c0 < m2; c0 += CP) {
        const int col = c0 + cs;
        const bool active = col < m2;
        if (active) {
            float2 v[16];
#pragma unroll
            for (int n2 = 0; n2 < 16; ++n2) v[n2] = Y[(n1 + Bq * n2) * ys + col];
            dft<16, -1>(v);
#pragma unroll
            for (int kk = 1; kk < 16; ++kk) v[kk] = cmul(v[kk], root<-1>(tw_h, n1 * kk * P, H));
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) S[kk * Bq + n1] = v[kk];
        }
        __syncthreads();
        if (active) {
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int kk = n1 + Bq * j;
                float2 u[Bq];
#pragma unroll
                for (int t = 0; t < Bq; ++t) u[t] = S[kk * Bq + t];
                dft<Bq, -1>(u);
#pragma unroll
                for (int k1 = 0; k1 < Bq; ++k1) {
                    if (!k1_live<R, M1S>(k1)) continue;
                    const int f = 16 * k1 + kk;  // residue of the retained frequencies
                    const float2 val = cscale(u[k1], scale);
                    if (P == 1) {
                        int kf;
                        const int r = row_of_residue(f, R, H, m1, &kf);
                        if (r >= 0 && FNO_DBG_OK(&X[xbase + (size_t)r * m2 + col], sizeof(float2)))
                            X[xbase + (size_t)r * m2 + col] = val;
                    } else if (m1 <= R) {
                        // at most one retained frequency per side: lower k1 = f, upper
                        // k1 = H - R + f, whose twiddle is the lower one times cdn
                        const bool lo = f < m1, hi = f >= R - m1;
                        if (!lo && !hi) continue;
                        const float2 a = cmul(val, root<-1>(tw_h, f * p, H));
                        float2* xl = X + xbase + (size_t)f * m2 + col;
                        float2* xh = X + xbase + (size_t)(f - R + 2 * m1) * m2 + col;
                        if (lo && FNO_DBG_OK(xl, sizeof(float2))) atomicAdd(xl, a);
                        if (hi && FNO_DBG_OK(xh, sizeof(float2))) atomicAdd(xh, cmul(a, cdn));
                    } else {
                        // every retained k1 == f (mod R): lower side f, f + R, ... < m1,
                        // upper side H - R + f, H - 2R + f, ... >= H - m1
                        for (int kf = f; kf < m1; kf += R) {
                            float2* xa = X + xbase + (size_t)kf * m2 + col;
                            if (FNO_DBG_OK(xa, sizeof(float2)))
                                atomicAdd(xa, cmul(val, root<-1>(tw_h, kf * p, H)));
                        }
                        for (int kf = H - R + f; kf >= H - m1; kf -= R) {
                            float2* xa = X + xbase + (size_t)(kf - H + 2 * m1) * m2 + col;
                            if (FNO_DBG_OK(xa, sizeof(float2)))
                                atomicAdd(xa, cmul(val, root<-1>(tw_h, kf * p, H)));
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
}

// Input residue f of the inverse column transform of the row group p: the
// sum of Z over the retained k1 == f (mod R), each times e^{+2 pi i k1 p / H}
// (P = 1: the single retained frequency k1 = f, if any).  `cup` is
// e^{+2 pi i (H - R) p / H}, the ratio of the upper-side twiddle to the lower.
// ZS: Z is in shared memory (plain loads) rather than global memory.  COH: Z
// in global memory was written earlier in the same launch by other CTAs, so it
// is read through L2 (ld.global.cg) instead of the read-only path.
template <int R, bool ZS, bool COH = false>
__device__ __forceinline__ float2 gather_residue(const float2* Zp, int f, int col, int H, int m1,
                                                 int m2, int P, int p, float2 cup,
                                                 const float2* __restrict__ tw_h) {
    const auto ld = [&](size_t i) {
        return ZS ? Zp[i] : (COH ? __ldcg(&Zp[i]) : __ldg(&Zp[i]));
    };
    float2 val = make_float2(0.f, 0.f);
    if (P == 1) {
        int kf;
        const int r = row_of_residue(f, R, H, m1, &kf);
        if (r >= 0) val = ld((size_t)r * m2 + col);
    } else if (m1 <= R) {
        // at most one retained frequency per side: lower k1 = f, upper k1 = H - R + f
        const bool lo = f < m1, hi = f >= R - m1;
        float2 s = lo ? ld((size_t)f * m2 + col) : make_float2(0.f, 0.f);
        if (hi) s = cadd(s, cmul(ld((size_t)(f - R + 2 * m1) * m2 + col), cup));
        if (lo || hi) val = cmul(s, root<1>(tw_h, f * p, H));
    } else {
        for (int kf = f; kf < m1; kf += R)
            val = cadd(val, cmul(ld((size_t)kf * m2 + col), root<1>(tw_h, kf * p, H)));
        for (int kf = H - R + f; kf >= H - m1; kf -= R)
            val = cadd(val, cmul(ld((size_t)(kf - H + 2 * m1) * m2 + col), root<1>(tw_h, kf * p, H)));
    }
    return val;
}

// ZS = true: Zp points to the plane's Z in shared memory, overlapping scr and V;
// requires a single pass (m2 <= ColCfg<R>::CP).  Every thread reads its inputs
// before the first barrier, after which the scratch and V may be rewritten.
template <int R, int M1S = 0, bool ZS = false, bool COH = false>
__device__ __forceinline__ void columns_inverse(float2* scr, float2* V, int ys, const float2* Zp,
                                                int H, int m1, int m2, int P, int p,
                                                const float2* __restrict__ tw_h) {
    if (M1S) m1 = M1S;
    constexpr int Bq = ColCfg<R>::Bq;
    constexpr int J = 16 / Bq;
    constexpr int CP = ColCfg<R>::CP;
    const int cs = threadIdx.x % CP;
    const int t = threadIdx.x / CP;
    float2* S = scr + cs * ColCfg<R>::Scr;  // S[n1][kk] with row stride 16
    const float2 cup = root<1>(tw_h, (H - R) * p, H);
    for (int c0 = 0; c0 < m2; c0 += CP) {
        const int col = c0 + cs;
        const bool active = col < m2;
        // the inputs U[16*k1 + kk] for kk = t + Bq*j; from shared memory all of
        // them are read before the barrier that frees the scratch
        const auto gather = [&](float2 (&u)[Bq], int j) {
#pragma unroll
            for (int k1 = 0; k1 < Bq; ++k1)
                u[k1] = k1_live<R, M1S>(k1)
                            ? gather_residue<R, ZS, COH>(Zp, 16 * k1 + t + Bq * j, col, H, m1, m2, P, p,
                                                    cup, tw_h)
                            : make_float2(0.f, 0.f);
        };
        float2 ug[ZS ? J : 1][Bq];
        if (ZS) {
            if (active) {
#pragma unroll
                for (int j = 0; j < J; ++j) gather(ug[ZS ? j : 0], j);
            }
            __syncthreads();
        }
        if (active) {
            // pass 1 (transposed): for kk = t + Bq*j, inverse Bq-point DFT over
            // k1, then times e^{+2 pi i n1 kk / R}
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int kk = t + Bq * j;
                float2 u[Bq];
                if (ZS) {
#pragma unroll
                    for (int k1 = 0; k1 < Bq; ++k1) u[k1] = ug[ZS ? j : 0][k1];
                } else {
                    gather(u, j);
                }
                dft<Bq, 1>(u);
#pragma unroll
                for (int n1 = 0; n1 < Bq; ++n1) {
                    const float2 w = n1 == 0 ? u[n1] : cmul(u[n1], root<1>(tw_h, n1 * kk * P, H));
                    S[n1 * 16 + kk] = w;
                }
            }
        }
        __syncthreads();
        if (active) {
            // pass 2: thread n1 = t, inverse 16-point DFT over kk
            const int n1 = t;
            float2 v[16];
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) v[kk] = S[n1 * 16 + kk];
            dft<16, 1>(v);
#pragma unroll
            for (int n2 = 0; n2 < 16; ++n2) V[(n1 + Bq * n2) * ys + col] = v[n2];
        }
        __syncthreads();
    }
}

}  // namespace fno
