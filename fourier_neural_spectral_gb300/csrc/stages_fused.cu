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

#include "fused_rows.cuh"


namespace fno {
namespace {

// ---------------------------------------------------------------- forward ---
template <int W, int R, int M1S = 0, int M2S = 0>
__global__ void __launch_bounds__(kFT, (FusedCfg<W, R>::MinBlocks))
fwd_fused_kernel(const float* __restrict__ x, float2* __restrict__ X, int H, int m1, int m2,
                 int P, float scale, const float2* __restrict__ tw_w,
                 const float2* __restrict__ tw_h FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    using C = FusedCfg<W, R>;
    extern __shared__ float2 sm[];
    float2* scr = sm;
    float2* Y = sm + C::Scratch;  // [R][ys]
    const int ys = kept_stride(M2S ? M2S : m2);
    const int plane = blockIdx.x / P;
    const int p = blockIdx.x - plane * P;
    const float* xp = x + (size_t)plane * H * W;
    griddep_wait();
    griddep_launch_dependents();

    // ---- rows -----------------------------------------------------------
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

    // ---- columns --------------------------------------------------------
    columns_forward<R, M1S>(scr, Y, ys, X, (size_t)plane * 2 * m1 * m2, H, m1, m2, P, p, scale,
                            tw_h);
}

// ---------------------------------------------------------------- inverse ---
// Whether the inverse brings the plane's Z (16*m1*m2 bytes, contiguous) into
// shared memory with one bulk copy: rows of 128 or 256 points, a single column
// pass, and Z fitting over the scratch and V (overwritten only after Z is read).
template <int W, int R>
bool fused_z_staged(int m1, int m2) {
    using C = FusedCfg<W, R>;
    return staged_z<W>() && m2 <= ColCfg<R>::CP &&
           16ull * m1 * m2 <= sizeof(float2) * ((size_t)C::Scratch + (size_t)R * kept_stride(m2));
}

// Z staging is compiled where the register budget holds it without spills:
// the kernels specialised for (m1, m2), or those sized for <= 2 CTAs per SM.
template <int W, int R, int M2S>
constexpr bool zs_compiled() {
    return staged_z<W>() && (M2S > 0 || FusedCfg<W, R>::MinBlocks <= 2);
}

template <int W, int R, int M1S = 0, int M2S = 0, bool ZS = false>
__global__ void __launch_bounds__(kFT, (FusedCfg<W, R>::MinBlocks))
inv_fused_kernel(const float2* __restrict__ Z, float* __restrict__ y, int H, int m1, int m2,
                 int P, float scale, const float2* __restrict__ tw_w,
                 const float2* __restrict__ tw_h, unsigned* __restrict__ err FNO_DBG_PARAM) {
    FNO_DBG_BEGIN();
    using C = FusedCfg<W, R>;
    extern __shared__ __align__(16) float2 sm[];
    float2* scr = sm;
    float2* V = sm + C::Scratch;  // [R][ys]
    const int ys = kept_stride(M2S ? M2S : m2);
    uint64_t* zbar = reinterpret_cast<uint64_t*>(V + R * ys);
    const int plane = blockIdx.x / P;
    const int p = blockIdx.x - plane * P;
    const int R2 = 2 * m1;
    const float2* Zp = Z + (size_t)plane * R2 * m2;
    griddep_wait();
    griddep_launch_dependents();

    // ---- columns: retained rows of Z -> V[q][col], q in [0, R) ----------
    // ZS (fused_z_staged): the plane's Z comes into shared memory first
    if constexpr (ZS) {
        const uint32_t zbytes = 16u * (uint32_t)(M1S ? M1S : m1) * (uint32_t)(M2S ? M2S : m2);
        if (threadIdx.x == 0) {
            mbar_init(zbar, 1);
            fence_barrier_init();
            mbar_arrive_expect_tx(zbar, zbytes);
            bulk_load(sm, Zp, zbytes, zbar);
        }
        __syncthreads();
        const bool zok = wait_parity_bounded(zbar, 0, err);
        // on a timeout err is set and the output is void; thread 0 still waits
        // (bounded) for the copy, and every thread for thread 0, before the
        // shared memory is rewritten
        if (!zok && threadIdx.x == 0) wait_parity_bounded(zbar, 0, nullptr);
        __syncthreads();
        columns_inverse<R, M1S, true>(scr, V, ys, sm, H, m1, m2, P, p, tw_h);
    } else {
        columns_inverse<R, M1S>(scr, V, ys, Zp, H, m1, m2, P, p, tw_h);
    }
    __syncthreads();

    // ---- rows: pairs of V rows -> two real output rows ------------------
    {
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
}

// Shapes with a kernel compiled for their (m1, m2): square planes with
// m1 = m2 = W/4 (the retained block of the 64-, 128- and 256-point workloads).
template <int W, int R>
constexpr bool has_static() { return W == R && (W == 64 || W == 128 || W == 256); }

__global__ void zero_kernel(float4* __restrict__ p, size_t n4) {
    griddep_wait();
    griddep_launch_dependents();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

template <int W, int R>
cudaError_t set_attrs() {
    const int bytes = (int)std::min<size_t>(fused_smem_bytes<W, R>(W / 2 + 1), kMaxDynSmem);
    cudaError_t e = cudaFuncSetAttribute(fwd_fused_kernel<W, R>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(inv_fused_kernel<W, R>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && zs_compiled<W, R, 0>())
        e = cudaFuncSetAttribute(inv_fused_kernel<W, R, 0, 0, zs_compiled<W, R, 0>()>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if constexpr (has_static<W, R>()) {
        const int sb = (int)std::min<size_t>(fused_smem_bytes<W, R>(W / 4), kMaxDynSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fwd_fused_kernel<W, R, W / 4, W / 4>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, sb);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(inv_fused_kernel<W, R, W / 4, W / 4>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, sb);
        if (e == cudaSuccess && zs_compiled<W, R, W / 4>())
            e = cudaFuncSetAttribute(inv_fused_kernel<W, R, W / 4, W / 4, zs_compiled<W, R, W / 4>()>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, sb);
    }
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
    if constexpr (has_static<W, R>()) {
        if (p.m1 == W / 4 && p.m2 == W / 4) {
            return launch_pdl(fwd_fused_kernel<W, R, W / 4, W / 4>, grid, kFT, smem, s, x, X, p.H,
                              p.m1, p.m2, p.P, p.scale, p.tw_w, p.tw_h
                              FNO_DBG_ARG1(X, 8ull * p.B * p.Cin * p.nm, p));
        }
    }
    return launch_pdl(fwd_fused_kernel<W, R>, grid, kFT, smem, s, x, X, p.H, p.m1, p.m2, p.P,
                      p.scale, p.tw_w, p.tw_h FNO_DBG_ARG1(X, 8ull * p.B * p.Cin * p.nm, p));
}

template <int W, int R, int M1S, int M2S>
cudaError_t launch_inv_zs(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s) {
    const size_t smem = fused_smem_bytes<W, R>(p.m2);
    const unsigned grid = (unsigned)((size_t)p.B * p.Cout * p.Pi);
    if (zs_compiled<W, R, M2S>() && fused_z_staged<W, R>(p.m1, p.m2))
        return launch_pdl(inv_fused_kernel<W, R, M1S, M2S, zs_compiled<W, R, M2S>()>, grid, kFT,
                          smem, s, Z, y, p.H, p.m1, p.m2, p.Pi, p.scale, p.tw_w, p.tw_h, p.err
                          FNO_DBG_ARG1(y, 4ull * p.B * p.Cout * p.H * p.W, p));
    return launch_pdl(inv_fused_kernel<W, R, M1S, M2S, false>, grid, kFT, smem, s, Z, y, p.H,
                      p.m1, p.m2, p.Pi, p.scale, p.tw_w, p.tw_h, p.err
                      FNO_DBG_ARG1(y, 4ull * p.B * p.Cout * p.H * p.W, p));
}

template <int W, int R>
cudaError_t launch_inv(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s) {
    if constexpr (has_static<W, R>()) {
        if (p.m1 == W / 4 && p.m2 == W / 4) return launch_inv_zs<W, R, W / 4, W / 4>(p, Z, y, s);
    }
    return launch_inv_zs<W, R, 0, 0>(p, Z, y, s);
}

template <bool FWD, int W>
cudaError_t dispatch_r(const fno_plan_s& p, const float* x, float2* X, const float2* Z, float* y,
                       cudaStream_t s) {
    switch (FWD ? p.R : p.Ri) {
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

bool fused_supported(int W, int H, int m1, int m2, int* R_fwd, int* R_inv) {
    if (W < 32 || H < 32) return false;
    if (W > 256 && m2 > 64) return false;  // long rows keep at most 64 columns
    // the column length R: the whole column when it fits (P = 1), else strided
    // row groups h = p + P*q of R rows per CTA (the forward adds its groups into
    // X with atomics; retained frequencies sharing a residue mod R read the
    // same value, so R need not reach 2*m1).  Long rows take R = 64 for the
    // inverse too when the plane's Z can be staged in shared memory.  Measured
    // at 2048 x 2048, m1 = m2 = 64: forward R = 32 / 64 / 128 -> 379 / 259 /
    // 318 us; inverse R = 64 / 128 -> 289 / 302 us with Z staged, 336 / 296
    // without.
    int Rf = H, Ri = H;
    if (H > 256) {
        Rf = 64;
        if (W > 256 && big_z_staged_any(W, 64, m1, m2)) {
            Ri = 64;
        } else {
            Ri = 32;
            while (Ri < 2 * m1 && Ri < 128) Ri <<= 1;
        }
    }
    if (H <= 256 && H < 2 * m1) return false;
    const auto smem = [&](int R, bool fwd) {
        return W <= 256 ? fused_smem_bytes_any(W, R, m2) : big_smem_bytes_any(W, R, m2, fwd);
    };
    if (smem(Rf, true) > kMaxDynSmem || smem(Ri, false) > kMaxDynSmem) return false;
    *R_fwd = Rf;
    *R_inv = Ri;
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
        e = launch_pdl(zero_kernel, dim3((unsigned)std::min<size_t>((n4 + 255) / 256, 4096)),
                       dim3(256), 0, s, reinterpret_cast<float4*>(X), n4);
        if (e == cudaSuccess && ctx) e = ctx->mark(s);
        if (e != cudaSuccess) return e;
    }
    e = p.W <= 256 ? dispatch<true>(p, x, X, nullptr, nullptr, s) : launch_forward_big(p, x, X, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}

cudaError_t launch_inverse_fused(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s,
                                 fno_launch_ctx* ctx) {
    cudaError_t e = p.W <= 256 ? dispatch<false>(p, nullptr, nullptr, Z, y, s)
                               : launch_inverse_big(p, Z, y, s);
    if (e == cudaSuccess && ctx) e = ctx->mark(s);
    return e;
}
