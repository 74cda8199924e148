// stages_fused.cu -- fused transform kernels for row lengths W and column
// lengths R in {32, 64, 128, 256}.
//
// Forward (stages a1 + a2 in one kernel).  A CTA owns the R rows
// h = p + P*q (q in [0, R), H = P*R, R >= 2*m1) of one (b, i) plane:
//   rows:    pairs of rows are packed as z = x_a + i x_b and transformed by a
//            W-point DFT split as W = 16 * Bq (decimation in frequency):
//              pass 1: thread n1 < Bq loads z[n1 + Bq*n2], n2 < 16, straight
//                      from global memory, does a 16-point DFT in registers and
//                      multiplies output kk by e^{-2 pi i n1 kk / W};
//              pass 2: after a shared-memory transpose, Bq-point DFTs over n1
//                      give Z[16*k1 + kk]; only k2 < m2 and its mirror are kept.
//            The two real-input spectra are separated,
//              X_a[k] = (Z[k] + conj Z[-k]) / 2,  X_b[k] = (Z[k] - conj Z[-k]) / 2i,
//            and the m2 kept columns of every row stay in shared memory (Y).
//   columns: the same two-pass scheme of length R runs down each kept column.
//            Output residue f holds the retained frequency k1 with k1 = f mod R.
//            With P = 1 the result times 1/sqrt(HW) is stored to X; with P > 1
//            it is multiplied by e^{-2 pi i k1 p / H} (the rows start at p) and
//            added into X, which the launcher has zeroed.
// Inverse (stages a4 + a5 in one kernel) is the exact mirror: the column
// transform reads the retained rows of Z (times e^{+2 pi i k1 p / H} when
// P > 1), runs the input-pruned inverse (decimation in time) into shared
// memory, then every pair of rows is rebuilt as U = S_a + i S_b from the
// Hermitian extension of its kept bins (imaginary parts of k2 = 0 and of
// k2 = W/2 dropped), inverse transformed, and the real and imaginary parts are
// written as the two output rows times 1/sqrt(HW).
//
// The split of a DFT into a 16-point register pass and a second pass is the
// textbook Cooley-Tukey factorisation; the packing of two real rows into one
// complex transform and the Hermitian separation are the standard real-input
// identities.
#include <algorithm>

#include "fft_reg.cuh"
#include "internal.h"

namespace fno {
namespace {

constexpr int kFT = 256;  // threads per CTA

template <int W, int R>
struct FusedCfg {
    static constexpr int BqW = W / 16;           // threads per row pair
    static constexpr int BqR = R / 16;           // threads per column
    static constexpr int RowGroups = kFT / BqW;  // row pairs in flight
    static constexpr int ColsPerPass = kFT / BqR;
    // Row-pass scratch per group: S[kk][n1] with row stride Bq+1; the group
    // stride is 1 mod 16 complex so that neighbouring groups use other banks.
    static constexpr int RowStride = BqW + 1;
    static constexpr int RowScr = ((16 * RowStride + W + 15) / 16) * 16 + 1;
    // Column-pass scratch: S[col][kk][n1], per column stride R + 16 + 1.
    static constexpr int ColScr = R + 17;
    static constexpr int ScratchA = RowGroups * RowScr;
    static constexpr int ScratchB = ColsPerPass * ColScr;
    static constexpr int Scratch = ScratchA > ScratchB ? ScratchA : ScratchB;
};

template <int W, int R>
size_t fused_smem_bytes(int m2) {
    using C = FusedCfg<W, R>;
    return sizeof(float2) * ((size_t)C::Scratch + (size_t)R * (m2 + 1));
}

// ---------------------------------------------------------------- forward ---
template <int W, int R>
__global__ void __launch_bounds__(kFT)
fwd_fused_kernel(const float* __restrict__ x, float2* __restrict__ X, int H, int m1, int m2,
                 int P, float scale, const float2* __restrict__ tw_w,
                 const float2* __restrict__ tw_h) {
    using C = FusedCfg<W, R>;
    extern __shared__ float2 sm[];
    float2* scr = sm;
    float2* Y = sm + C::Scratch;  // [R][ys]
    const int ys = m2 + 1;
    const int plane = blockIdx.x / P;
    const int p = blockIdx.x - plane * P;
    const float* xp = x + (size_t)plane * H * W;

    // ---- rows -----------------------------------------------------------
    {
        constexpr int Bq = C::BqW;
        constexpr int J = 16 / Bq;
        const int g = threadIdx.x / Bq, n1 = threadIdx.x % Bq;
        float2* S = scr + g * C::RowScr;
        float2* Zs = S + 16 * C::RowStride;  // W kept outputs of this pair
        constexpr int npairs = R / 2;
        constexpr int iters = (npairs + C::RowGroups - 1) / C::RowGroups;
        for (int it = 0; it < iters; ++it) {
            const int pair = g + it * C::RowGroups;
            const bool active = pair < npairs;
            const int qa = 2 * pair;
            if (active) {
                const float* ra = xp + (size_t)(p + P * qa) * W;
                const float* rb = xp + (size_t)(p + P * (qa + 1)) * W;
                float2 v[16];
#pragma unroll
                for (int n2 = 0; n2 < 16; ++n2)
                    v[n2] = make_float2(__ldg(ra + n1 + Bq * n2), __ldg(rb + n1 + Bq * n2));
                dft<16, -1>(v);
#pragma unroll
                for (int kk = 1; kk < 16; ++kk) v[kk] = cmul(v[kk], root<-1>(tw_w, n1 * kk, W));
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) S[kk * C::RowStride + n1] = v[kk];
            }
            __syncwarp();
            float2 u[J][Bq];
            if (active) {
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    const int kk = n1 + Bq * j;
#pragma unroll
                    for (int t = 0; t < Bq; ++t) u[j][t] = S[kk * C::RowStride + t];
                    dft<Bq, -1>(u[j]);
                }
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    const int kk = n1 + Bq * j;
#pragma unroll
                    for (int k1 = 0; k1 < Bq; ++k1) {
                        const int k = 16 * k1 + kk;
                        if (k < m2 || k > W - m2) Zs[k] = u[j][k1];
                    }
                }
            }
            __syncwarp();
            if (active) {
                for (int k = n1; k < m2; k += Bq) {
                    const float2 zk = Zs[k], zm = Zs[(W - k) & (W - 1)];
                    Y[qa * ys + k] = make_float2(0.5f * (zk.x + zm.x), 0.5f * (zk.y - zm.y));
                    Y[(qa + 1) * ys + k] = make_float2(0.5f * (zk.y + zm.y), -0.5f * (zk.x - zm.x));
                }
            }
            __syncwarp();
        }
    }
    __syncthreads();

    // ---- columns --------------------------------------------------------
    {
        constexpr int Bq = C::BqR;
        constexpr int J = 16 / Bq;
        constexpr int CP = C::ColsPerPass;
        const int cs = threadIdx.x % CP;   // column within the pass
        const int n1 = threadIdx.x / CP;   // position within the column transform
        float2* S = scr + cs * C::ColScr;  // S[kk][n1] with row stride Bq
        const int R2 = 2 * m1;
        const size_t xbase = (size_t)plane * R2 * m2;
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
                        int kf;
                        const int r = row_of_residue(16 * k1 + kk, R, H, m1, &kf);
                        if (r < 0) continue;
                        float2 val = cscale(u[k1], scale);
                        float2* dst = X + xbase + (size_t)r * m2 + col;
                        if (P == 1) {
                            *dst = val;
                        } else {
                            val = cmul(val, root<-1>(tw_h, kf * p, H));
                            atomicAdd(&dst->x, val.x);
                            atomicAdd(&dst->y, val.y);
                        }
                    }
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------- inverse ---
template <int W, int R>
__global__ void __launch_bounds__(kFT)
inv_fused_kernel(const float2* __restrict__ Z, float* __restrict__ y, int H, int m1, int m2,
                 int P, float scale, const float2* __restrict__ tw_w,
                 const float2* __restrict__ tw_h) {
    using C = FusedCfg<W, R>;
    extern __shared__ float2 sm[];
    float2* scr = sm;
    float2* V = sm + C::Scratch;  // [R][ys]
    const int ys = m2 + 1;
    const int plane = blockIdx.x / P;
    const int p = blockIdx.x - plane * P;
    const int R2 = 2 * m1;
    const float2* Zp = Z + (size_t)plane * R2 * m2;

    // ---- columns: retained rows of Z -> V[q][col], q in [0, R) ----------
    {
        constexpr int Bq = C::BqR;
        constexpr int J = 16 / Bq;
        constexpr int CP = C::ColsPerPass;
        const int cs = threadIdx.x % CP;
        const int t = threadIdx.x / CP;
        float2* S = scr + cs * C::ColScr;  // S[n1][kk] with row stride 16
        for (int c0 = 0; c0 < m2; c0 += CP) {
            const int col = c0 + cs;
            const bool active = col < m2;
            if (active) {
                // pass 1 (transposed): for kk = t + Bq*j, inverse Bq-point DFT over
                // k1 of U[16*k1 + kk], then times e^{+2 pi i n1 kk / R}
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    const int kk = t + Bq * j;
                    float2 u[Bq];
#pragma unroll
                    for (int k1 = 0; k1 < Bq; ++k1) {
                        int kf;
                        const int r = row_of_residue(16 * k1 + kk, R, H, m1, &kf);
                        float2 val = make_float2(0.f, 0.f);
                        if (r >= 0) {
                            val = __ldg(&Zp[(size_t)r * m2 + col]);
                            if (P > 1) val = cmul(val, root<1>(tw_h, kf * p, H));
                        }
                        u[k1] = val;
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

    // ---- rows: pairs of V rows -> two real output rows ------------------
    {
        constexpr int Bq = C::BqW;
        constexpr int J = 16 / Bq;
        const int g = threadIdx.x / Bq, t = threadIdx.x % Bq;
        float2* S = scr + g * C::RowScr;  // S[n1][kk] with row stride 17
        float* yp = y + (size_t)plane * H * W;
        constexpr int npairs = R / 2;
        constexpr int iters = (npairs + C::RowGroups - 1) / C::RowGroups;
        const int half = W / 2;
        for (int it = 0; it < iters; ++it) {
            const int pair = g + it * C::RowGroups;
            const bool active = pair < npairs;
            const int qa = 2 * pair;
            if (active) {
                const float2* Va = V + qa * ys;
                const float2* Vb = Va + ys;
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    const int kk = t + Bq * j;
                    float2 u[Bq];
#pragma unroll
                    for (int k1 = 0; k1 < Bq; ++k1) {
                        const int k = 16 * k1 + kk;  // bin of the packed spectrum U
                        float2 val = make_float2(0.f, 0.f);
                        if (k == 0 || k == half) {
                            if (k < m2) val = make_float2(Va[k].x, Vb[k].x);
                        } else if (k < half) {
                            if (k < m2) {
                                const float2 a = Va[k], b = Vb[k];
                                val = make_float2(a.x - b.y, a.y + b.x);
                            }
                        } else {
                            const int kr = W - k;
                            if (kr < m2) {
                                const float2 a = Va[kr], b = Vb[kr];
                                val = make_float2(a.x + b.y, b.x - a.y);
                            }
                        }
                        u[k1] = val;
                    }
                    dft<Bq, 1>(u);
#pragma unroll
                    for (int n1 = 0; n1 < Bq; ++n1) {
                        const float2 w = n1 == 0 ? u[n1] : cmul(u[n1], root<1>(tw_w, n1 * kk, W));
                        S[n1 * 17 + kk] = w;
                    }
                }
            }
            __syncwarp();
            if (active) {
                const int n1 = t;
                float2 v[16];
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) v[kk] = S[n1 * 17 + kk];
                dft<16, 1>(v);
                float* ya = yp + (size_t)(p + P * qa) * W;
                float* yb = yp + (size_t)(p + P * (qa + 1)) * W;
#pragma unroll
                for (int n2 = 0; n2 < 16; ++n2) {
                    ya[n1 + Bq * n2] = v[n2].x * scale;
                    yb[n1 + Bq * n2] = v[n2].y * scale;
                }
            }
            __syncwarp();
        }
    }
}

__global__ void zero_kernel(float4* __restrict__ p, size_t n4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

template <int W, int R>
cudaError_t set_attrs() {
    const int bytes = (int)std::min<size_t>(fused_smem_bytes<W, R>(W / 2 + 1), 227 * 1024);
    cudaError_t e = cudaFuncSetAttribute(fwd_fused_kernel<W, R>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inv_fused_kernel<W, R>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
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

template <int W, int R>
cudaError_t launch_fwd(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s) {
    const size_t smem = fused_smem_bytes<W, R>(p.m2);
    const unsigned grid = (unsigned)((size_t)p.B * p.Cin * p.P);
    fwd_fused_kernel<W, R><<<grid, kFT, smem, s>>>(x, X, p.H, p.m1, p.m2, p.P, p.scale, p.tw_w,
                                                   p.tw_h);
    return cudaGetLastError();
}

template <int W, int R>
cudaError_t launch_inv(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s) {
    const size_t smem = fused_smem_bytes<W, R>(p.m2);
    const unsigned grid = (unsigned)((size_t)p.B * p.Cout * p.P);
    inv_fused_kernel<W, R><<<grid, kFT, smem, s>>>(Z, y, p.H, p.m1, p.m2, p.P, p.scale, p.tw_w,
                                                   p.tw_h);
    return cudaGetLastError();
}

template <bool FWD, int W>
cudaError_t dispatch_r(const fno_plan_s& p, const float* x, float2* X, const float2* Z, float* y,
                       cudaStream_t s) {
    switch (p.R) {
        case 32: return FWD ? launch_fwd<W, 32>(p, x, X, s) : launch_inv<W, 32>(p, Z, y, s);
        case 64: return FWD ? launch_fwd<W, 64>(p, x, X, s) : launch_inv<W, 64>(p, Z, y, s);
        case 128: return FWD ? launch_fwd<W, 128>(p, x, X, s) : launch_inv<W, 128>(p, Z, y, s);
        case 256: return FWD ? launch_fwd<W, 256>(p, x, X, s) : launch_inv<W, 256>(p, Z, y, s);
    }
    return cudaErrorInvalidValue;
}

template <bool FWD>
cudaError_t dispatch(const fno_plan_s& p, const float* x, float2* X, const float2* Z, float* y,
                     cudaStream_t s) {
    switch (p.W) {
        case 32: return dispatch_r<FWD, 32>(p, x, X, Z, y, s);
        case 64: return dispatch_r<FWD, 64>(p, x, X, Z, y, s);
        case 128: return dispatch_r<FWD, 128>(p, x, X, Z, y, s);
        case 256: return dispatch_r<FWD, 256>(p, x, X, Z, y, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace fno

using namespace fno;

cudaError_t stages_fused_init() {
    cudaError_t e = set_attrs_w<32>();
    if (e == cudaSuccess) e = set_attrs_w<64>();
    if (e == cudaSuccess) e = set_attrs_w<128>();
    if (e == cudaSuccess) e = set_attrs_w<256>();
    return e;
}

size_t fused_smem_bytes_any(int W, int R, int m2);

bool fused_supported(int W, int H, int m1, int m2, int* R_out) {
    if (W < 32 || W > 256 || H < 32) return false;
    // the column length R: the whole column when it fits, else the smallest
    // power of two >= max(2*m1, 32) that divides H, at most 256
    int R = H <= 256 ? H : 0;
    if (!R) {
        R = 32;
        while (R < 2 * m1) R <<= 1;
        if (R > 256) return false;
    }
    if (R < 2 * m1 || R > H) return false;
    if (fused_smem_bytes_any(W, R, m2) > 227 * 1024) return false;
    *R_out = R;
    return true;
}

size_t fused_smem_bytes_any(int W, int R, int m2) {
    switch (W * 1000 + R) {
#define CASE(w, r) case w * 1000 + r: return fused_smem_bytes<w, r>(m2);
        CASE(32, 32) CASE(32, 64) CASE(32, 128) CASE(32, 256)
        CASE(64, 32) CASE(64, 64) CASE(64, 128) CASE(64, 256)
        CASE(128, 32) CASE(128, 64) CASE(128, 128) CASE(128, 256)
        CASE(256, 32) CASE(256, 64) CASE(256, 128) CASE(256, 256)
#undef CASE
    }
    return (size_t)-1;
}

cudaError_t launch_forward_fused(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s,
                                 fno_launch_ctx* ctx) {
    cudaError_t e = cudaSuccess;
    if (p.P > 1) {
        const size_t n4 = (size_t)p.B * p.Cin * p.nm / 2;  // complex pairs -> float4
        zero_kernel<<<std::min<size_t>((n4 + 255) / 256, 4096), 256, 0, s>>>(
            reinterpret_cast<float4*>(X), n4);
        e = cudaGetLastError();
        if (e == cudaSuccess && ctx) e = ctx->mark(s);
        if (e != cudaSuccess) return e;
    }
    e = dispatch<true>(p, x, X, nullptr, nullptr, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_fused(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s,
                                 fno_launch_ctx* ctx) {
    cudaError_t e = dispatch<false>(p, nullptr, nullptr, Z, y, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
