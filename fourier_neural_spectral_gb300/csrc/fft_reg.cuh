// fft_reg.cuh -- small DFTs held entirely in registers, and the pieces the
// fused transform kernels build on.
//
// dft<N, SGN>(v): v[k] <- sum_n v[n] * e^{SGN * 2 pi i n k / N} for N in
// {1, 2, 4, 8, 16}, natural order in and out (radix-2 decimation in time,
// fully unrolled; a butterfly with a twiddle other than 1 or +-i takes six
// fused multiply-adds).  SGN = -1 is the forward transform, +1 the inverse
// (unnormalised).  The twiddles inside are the exact angles k*pi/8; their
// cosines and sines are written out below as float literals.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace fno {

// cos and sin of j*pi/8 for j = 0..15 (values of cos(pi/8), sin(pi/8) and
// sqrt(2)/2 rounded to float).
__device__ __forceinline__ float2 unit16(int j) {
    constexpr float c1 = 0.923879532511286756128f;  // cos(pi/8)
    constexpr float s1 = 0.382683432365089771728f;  // sin(pi/8)
    constexpr float r2 = 0.707106781186547524401f;  // sqrt(2)/2
    switch (j & 15) {
        case 0: return make_float2(1.f, 0.f);
        case 1: return make_float2(c1, s1);
        case 2: return make_float2(r2, r2);
        case 3: return make_float2(s1, c1);
        case 4: return make_float2(0.f, 1.f);
        case 5: return make_float2(-s1, c1);
        case 6: return make_float2(-r2, r2);
        case 7: return make_float2(-c1, s1);
        case 8: return make_float2(-1.f, 0.f);
        case 9: return make_float2(-c1, -s1);
        case 10: return make_float2(-r2, -r2);
        case 11: return make_float2(-s1, -c1);
        case 12: return make_float2(0.f, -1.f);
        case 13: return make_float2(s1, -c1);
        case 14: return make_float2(r2, -r2);
        default: return make_float2(c1, -s1);
    }
}

// a * e^{SGN * i * pi * j / 8}; j is a compile-time constant after unrolling,
// so the multiplications by 1 and by +-i fold away.
template <int SGN>
__device__ __forceinline__ float2 rot16(float2 a, int j) {
    j &= 15;
    if (j == 0) return a;
    if (j == 8) return make_float2(-a.x, -a.y);
    if (j == 4) return SGN < 0 ? make_float2(a.y, -a.x) : make_float2(-a.y, a.x);
    if (j == 12) return SGN < 0 ? make_float2(-a.y, a.x) : make_float2(a.y, -a.x);
    float2 w = unit16(j);
    if (SGN < 0) w.y = -w.y;
    return cmul(a, w);
}

template <int N, int SGN>
struct Dft {
    static __device__ __forceinline__ void run(float2 (&v)[N]) {
        float2 e[N / 2], o[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            e[i] = v[2 * i];
            o[i] = v[2 * i + 1];
        }
        Dft<N / 2, SGN>::run(e);
        Dft<N / 2, SGN>::run(o);
#pragma unroll
        for (int k = 0; k < N / 2; ++k) {
            const int j = (16 / N) * k;  // in [0, 8): rotation by 1 (j = 0) or +-i (j = 4)
            if (j == 0 || j == 4) {
                const float2 t = rot16<SGN>(o[k], j);
                v[k] = cadd(e[k], t);
                v[k + N / 2] = csub(e[k], t);
            } else {
                // e + w*o as four fused multiply-adds, and e - w*o = 2e - (e + w*o)
                // as two more (instead of a complex product and four additions)
                float2 w = unit16(j);
                if (SGN < 0) w.y = -w.y;
                const float2 a = o[k], b = e[k];
                float2 p;
                p.x = fmaf(a.x, w.x, fmaf(-a.y, w.y, b.x));
                p.y = fmaf(a.x, w.y, fmaf(a.y, w.x, b.y));
                v[k] = p;
                v[k + N / 2] = make_float2(fmaf(2.f, b.x, -p.x), fmaf(2.f, b.y, -p.y));
            }
        }
    }
};

template <int SGN>
struct Dft<2, SGN> {
    static __device__ __forceinline__ void run(float2 (&v)[2]) {
        const float2 a = v[0], b = v[1];
        v[0] = cadd(a, b);
        v[1] = csub(a, b);
    }
};

template <int SGN>
struct Dft<1, SGN> {
    static __device__ __forceinline__ void run(float2 (&)[1]) {}
};

template <int N, int SGN>
__device__ __forceinline__ void dft(float2 (&v)[N]) {
    Dft<N, SGN>::run(v);
}

// The 16-point DFT of a sequence whose only nonzero entries are e[0..3] and
// e[12..15] (indices m = -4..3 mod 16), e[4..11] being ignored.  Splitting the
// outputs by parity,
//   X[2k]     = sum_m e_m w8^{mk},              w8 = e^{SGN 2 pi i / 8},
//   X[2k + 1] = sum_m (e_m w16^m) w8^{mk},       w16 = e^{SGN 2 pi i / 16},
// i.e. two 8-point DFTs over m mod 8, which skips the additions of the zero
// entries that a full 16-point transform would perform.
template <int SGN>
__device__ __forceinline__ void dft16_in8(float2 (&e)[16]) {
    float2 a[8], b[8];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        a[r] = e[r];
        a[4 + r] = e[12 + r];
        b[r] = rot16<SGN>(e[r], r);
        b[4 + r] = rot16<SGN>(e[12 + r], 12 + r);
    }
    dft<8, SGN>(a);
    dft<8, SGN>(b);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        e[2 * k] = a[k];
        e[2 * k + 1] = b[k];
    }
}

// e^{SGN * 2 pi i * j / N} from a table tab[j] = e^{+2 pi i j / N}, j reduced mod N.
template <int SGN>
__device__ __forceinline__ float2 root(const float2* __restrict__ tab, int j, int N) {
    float2 w = __ldg(&tab[j & (N - 1)]);
    if (SGN < 0) w.y = -w.y;
    return w;
}

// Retained row r of the weight layout for true frequency k1, and back.
__device__ __forceinline__ int freq_of_row(int r, int H, int m1) { return r < m1 ? r : H - 2 * m1 + r; }

// For a column transform of length R over the rows p + P*q (H = P*R) with
// R >= 2*m1, at most one retained frequency k1 has k1 mod R == f for an output
// residue f in [0, R).  Returns the retained row r of that frequency, or -1 if
// there is none.  *k1 receives the true frequency.
__device__ __forceinline__ int row_of_residue(int f, int R, int H, int m1, int* k1) {
    if (f < m1) {
        *k1 = f;
        return f;
    }
    if (f >= R - m1) {
        *k1 = H - R + f;
        return f - R + 2 * m1;
    }
    return -1;
}

// Packed spectrum bin k of U = S_a + i S_b (the Hermitian extensions of the kept
// bins of rows a and b, imaginary parts of k = 0 and k = W/2 dropped), for
// k <= W/2, and the value of its mirror bin W - k.
__device__ __forceinline__ void packed_bin(float2 a, float2 b, bool self_mirror, float2* uk,
                                           float2* um) {
    if (self_mirror) {
        *uk = make_float2(a.x, b.x);
        *um = *uk;
    } else {
        *uk = make_float2(a.x - b.y, a.y + b.x);  // Va + i Vb
        *um = make_float2(a.x + b.y, b.x - a.y);  // conj Va + i conj Vb
    }
}

}  // namespace fno
