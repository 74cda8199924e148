// fno_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded, double-precision statement of the FNO 2D
// spectral-convolution layer.  Only tests/, __graft_entry__.smoke() and the
// CPU-baseline leg of bench.py may load this library; the product path
// (libfnospec) shares no code, header, table or helper with it.
//
// What it computes (every DFT is a direct O(N^2)-style sum, no FFT):
//
//   X = rfft2(x, norm="ortho") restricted to the retained modes
//       k1 in R1 = {0..m1-1} U {H-m1..H-1},  k2 in R2 = {0..m2-1}
//   Z[b,o,k1,k2] = sum_i X[b,i,k1,k2] * W[i,o,r(k1),k2]      (complex product)
//   y = irfft2(Z zero-filled outside R1 x R2, s=(H,W), norm="ortho")
//
// Sources: "TurboFNO: FFT-GEMM-iFFT fused operator" page, section 2.2 (only the
// low-frequency block is transformed, everything else is set to zero; the
// per-mode complex product (a+bi)(c+di) = (ac-bd) + (ad+bc)i) and section 3.1
// (orthonormal normalisation); the FFT operator-optimisation page
// (lpnh.cn/news/2688017), section 2.2 (the real-to-complex half spectrum is
// W/2+1 wide and the complex-to-real step is the Hermitian inverse).
//
// Readings taken where the pages are silent or garbled:
//   * Row order of the 2*m1 retained rows: r < m1 is k1 = r, r >= m1 is
//     k1 = H - 2*m1 + r (top rows, then bottom rows).
//   * The complex-to-real row step keeps only the real part of the k2 = 0 bin
//     and, when it is retained (m2 = W/2 + 1), of the k2 = W/2 bin; every other
//     retained bin counts twice (it stands for itself and its Hermitian mirror).
//   * Angles are formed from the integer product reduced modulo N before the
//     conversion to radians, so cos/sin see an argument in [0, 2*pi).
//
// Parity is pinned in tests/test_oracle.py against closed forms (delta,
// constant, single cosine), Parseval, the identity layer, the convolution
// theorem (brute-force circular convolution), shift equivariance, linearity and
// numpy's pocketfft rfft2/irfft2 on small inputs.
//
// Data layout (all arrays dense, row-major, complex values stored re,im):
//   x : double [B][C][H][W]
//   X : double [B][C][2*m1][m2][2]
//   w : double [Cin][Cout][2*m1][m2][2]
//   Z : double [B][Cout][2*m1][m2][2]
//   y : double [B][Cout][H][W]
//
// Backward (gradients of a real loss L given g = dL/dy, with the complex
// gradient convention dL/dRe(z) + i dL/dIm(z)), derived by differentiating the
// sums above:
//   G[b,o,k1,k2]  = c(k2) / sqrt(HW) * sum_{h,w} g[b,o,h,w] exp(-2 pi i (k1 h/H + k2 w/W))
//                   (c = 1 for k2 = 0 and k2 = W/2, else 2: the weights of the
//                   complex-to-real step)
//   GX[b,i,k1,k2] = sum_o G[b,o,k1,k2] * conj(W[i,o,r(k1),k2])
//   gx[b,i,h,w]   = 1/sqrt(HW) * Re sum_{k1 in R1, k2 in R2} GX[b,i,k1,k2]
//                   * exp(+2 pi i (k1 h/H + k2 w/W))
//   gW[i,o,r,k2]  = sum_b conj(X[b,i,r,k2]) * G[b,o,r,k2]
// Pinned in tests/test_oracle.py by the adjoint identity <J x, g> = <x, gx>,
// the weight identity <y(x, v), g> = Re sum conj(gW) v, and finite differences.
//
// Return value of every entry point: 0 on success, -1 on an invalid argument.

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <vector>

namespace {

const double kTwoPi = 6.283185307179586476925286766559005768;

// Table of exp(sign * 2*pi*i * j / N) for j in [0, N).  The angle is formed from
// the exact integer j, so every entry is accurate to double rounding.
std::vector<double> root_table(long long N, int sign) {
    std::vector<double> t(2 * (size_t)N);
    for (long long j = 0; j < N; ++j) {
        double ang = kTwoPi * (double)j / (double)N;
        t[2 * j] = std::cos(ang);
        t[2 * j + 1] = sign * std::sin(ang);
    }
    return t;
}

// Index into a root table for the product k*n, reduced modulo N.
inline long long red(long long k, long long n, long long N) {
    long long r = (k * n) % N;
    return r < 0 ? r + N : r;
}

// Frequency row k1 held in retained row r (top rows then bottom rows).
inline long long row_of(long long r, long long H, long long m1) {
    return r < m1 ? r : H - 2 * m1 + r;
}

bool shape_ok(int B, int C, int H, int W, int m1, int m2) {
    if (B <= 0 || C <= 0 || H < 2 || W < 2 || m1 <= 0 || m2 <= 0) return false;
    if (2 * (long long)m1 > H) return false;
    if ((long long)m2 > W / 2 + 1) return false;
    return true;
}

}  // namespace

extern "C" {

// Forward truncated 2D DFT with orthonormal scale (steps: row DFT over w for
// the retained k2, then column DFT over h for the retained k1).
int oracle_forward_modes(const double* x, int B, int C, int H, int W, int m1, int m2,
                         double* X) {
    if (!x || !X || !shape_ok(B, C, H, W, m1, m2)) return -1;
    const std::vector<double> tw_w = root_table(W, -1);
    const std::vector<double> tw_h = root_table(H, -1);
    const double scale = 1.0 / std::sqrt((double)H * (double)W);
    const int R = 2 * m1;
    std::vector<double> rowdft(2 * (size_t)H * m2);
    for (long long p = 0; p < (long long)B * C; ++p) {
        const double* xp = x + p * (long long)H * W;
        // Y[h][k2] = sum_w x[h][w] * exp(-2*pi*i*k2*w/W)
        for (int h = 0; h < H; ++h) {
            for (int k2 = 0; k2 < m2; ++k2) {
                double re = 0.0, im = 0.0;
                for (int w = 0; w < W; ++w) {
                    long long j = red(k2, w, W);
                    double v = xp[(long long)h * W + w];
                    re += v * tw_w[2 * j];
                    im += v * tw_w[2 * j + 1];
                }
                rowdft[2 * ((size_t)h * m2 + k2)] = re;
                rowdft[2 * ((size_t)h * m2 + k2) + 1] = im;
            }
        }
        // X[r][k2] = scale * sum_h Y[h][k2] * exp(-2*pi*i*k1*h/H)
        double* Xp = X + p * (long long)R * m2 * 2;
        for (int r = 0; r < R; ++r) {
            long long k1 = row_of(r, H, m1);
            for (int k2 = 0; k2 < m2; ++k2) {
                double re = 0.0, im = 0.0;
                for (int h = 0; h < H; ++h) {
                    long long j = red(k1, h, H);
                    double a = rowdft[2 * ((size_t)h * m2 + k2)];
                    double b = rowdft[2 * ((size_t)h * m2 + k2) + 1];
                    double c = tw_h[2 * j], d = tw_h[2 * j + 1];
                    re += a * c - b * d;
                    im += a * d + b * c;
                }
                Xp[2 * ((size_t)r * m2 + k2)] = scale * re;
                Xp[2 * ((size_t)r * m2 + k2) + 1] = scale * im;
            }
        }
    }
    return 0;
}

// Per-mode complex channel contraction: Z[b,o,m] = sum_i X[b,i,m] * w[i,o,m].
int oracle_mix_modes(const double* X, const double* w, int B, int Cin, int Cout, int nmodes,
                     double* Z) {
    if (!X || !w || !Z || B <= 0 || Cin <= 0 || Cout <= 0 || nmodes <= 0) return -1;
    for (long long b = 0; b < B; ++b) {
        for (long long o = 0; o < Cout; ++o) {
            for (long long m = 0; m < nmodes; ++m) {
                double re = 0.0, im = 0.0;
                for (long long i = 0; i < Cin; ++i) {
                    const double* xv = X + 2 * ((b * Cin + i) * nmodes + m);
                    const double* wv = w + 2 * ((i * Cout + o) * nmodes + m);
                    re += xv[0] * wv[0] - xv[1] * wv[1];
                    im += xv[0] * wv[1] + xv[1] * wv[0];
                }
                Z[2 * ((b * Cout + o) * nmodes + m)] = re;
                Z[2 * ((b * Cout + o) * nmodes + m) + 1] = im;
            }
        }
    }
    return 0;
}

// Inverse: column inverse DFT over the retained rows (all other rows are zero),
// then the complex-to-real row inverse over the retained columns, orthonormal.
int oracle_inverse_modes(const double* Z, int B, int C, int H, int W, int m1, int m2,
                         double* y) {
    if (!Z || !y || !shape_ok(B, C, H, W, m1, m2)) return -1;
    const std::vector<double> tw_w = root_table(W, +1);
    const std::vector<double> tw_h = root_table(H, +1);
    const double scale = 1.0 / std::sqrt((double)H * (double)W);
    const int R = 2 * m1;
    std::vector<double> V(2 * (size_t)H * m2);
    for (long long p = 0; p < (long long)B * C; ++p) {
        const double* Zp = Z + p * (long long)R * m2 * 2;
        // V[h][k2] = sum_r Z[r][k2] * exp(+2*pi*i*k1(r)*h/H)
        for (int h = 0; h < H; ++h) {
            for (int k2 = 0; k2 < m2; ++k2) {
                double re = 0.0, im = 0.0;
                for (int r = 0; r < R; ++r) {
                    long long j = red(row_of(r, H, m1), h, H);
                    double a = Zp[2 * ((size_t)r * m2 + k2)];
                    double b = Zp[2 * ((size_t)r * m2 + k2) + 1];
                    double c = tw_h[2 * j], d = tw_h[2 * j + 1];
                    re += a * c - b * d;
                    im += a * d + b * c;
                }
                V[2 * ((size_t)h * m2 + k2)] = re;
                V[2 * ((size_t)h * m2 + k2) + 1] = im;
            }
        }
        // y[h][w] = scale * sum_k2 c(k2) * Re(V'[h][k2] * exp(+2*pi*i*k2*w/W))
        double* yp = y + p * (long long)H * W;
        for (int h = 0; h < H; ++h) {
            for (int w = 0; w < W; ++w) {
                double acc = 0.0;
                for (int k2 = 0; k2 < m2; ++k2) {
                    long long j = red(k2, w, W);
                    double a = V[2 * ((size_t)h * m2 + k2)];
                    double b = V[2 * ((size_t)h * m2 + k2) + 1];
                    bool self_mirror = (k2 == 0) || (2LL * k2 == W);
                    if (self_mirror) {
                        // imaginary part of this bin is discarded
                        acc += a * tw_w[2 * j];
                    } else {
                        acc += 2.0 * (a * tw_w[2 * j] - b * tw_w[2 * j + 1]);
                    }
                }
                yp[(size_t)h * W + w] = scale * acc;
            }
        }
    }
    return 0;
}

// Selected outputs of the inverse step: out[s] = y[b,o,h,w] for the s-th
// quadruple (b, o, h, w) in idx (4 ints per sample).  Same sums as above.
int oracle_inverse_modes_at(const double* Z, int B, int C, int H, int W, int m1, int m2,
                            const int* idx, int nsamples, double* out) {
    if (!Z || !out || (nsamples > 0 && !idx) || nsamples < 0 ||
        !shape_ok(B, C, H, W, m1, m2))
        return -1;
    const std::vector<double> tw_w = root_table(W, +1);
    const std::vector<double> tw_h = root_table(H, +1);
    const double scale = 1.0 / std::sqrt((double)H * (double)W);
    const int R = 2 * m1;
    for (int s = 0; s < nsamples; ++s) {
        int b = idx[4 * s], o = idx[4 * s + 1], h = idx[4 * s + 2], w = idx[4 * s + 3];
        if (b < 0 || b >= B || o < 0 || o >= C || h < 0 || h >= H || w < 0 || w >= W)
            return -1;
        const double* Zp = Z + ((long long)b * C + o) * R * m2 * 2;
        double acc = 0.0;
        for (int k2 = 0; k2 < m2; ++k2) {
            double vre = 0.0, vim = 0.0;
            for (int r = 0; r < R; ++r) {
                long long j = red(row_of(r, H, m1), h, H);
                double a = Zp[2 * ((size_t)r * m2 + k2)];
                double bb = Zp[2 * ((size_t)r * m2 + k2) + 1];
                vre += a * tw_h[2 * j] - bb * tw_h[2 * j + 1];
                vim += a * tw_h[2 * j + 1] + bb * tw_h[2 * j];
            }
            long long j = red(k2, w, W);
            bool self_mirror = (k2 == 0) || (2LL * k2 == W);
            if (self_mirror)
                acc += vre * tw_w[2 * j];
            else
                acc += 2.0 * (vre * tw_w[2 * j] - vim * tw_w[2 * j + 1]);
        }
        out[s] = scale * acc;
    }
    return 0;
}

// dL/dZ from g = dL/dy: c(k2) times the orthonormal truncated forward DFT of g.
int oracle_backward_modes(const double* g, int B, int C, int H, int W, int m1, int m2,
                          double* G) {
    int rc = oracle_forward_modes(g, B, C, H, W, m1, m2, G);
    if (rc) return rc;
    const long long R = 2LL * m1;
    for (long long p = 0; p < (long long)B * C; ++p)
        for (long long r = 0; r < R; ++r)
            for (long long k2 = 0; k2 < m2; ++k2) {
                const bool self_mirror = (k2 == 0) || (2LL * k2 == W);
                const double c = self_mirror ? 1.0 : 2.0;
                double* v = G + 2 * ((p * R + r) * m2 + k2);
                v[0] *= c;
                v[1] *= c;
            }
    return 0;
}

// GX[b,i,m] = sum_o G[b,o,m] * conj(w[i,o,m]).
int oracle_mix_adjoint(const double* G, const double* w, int B, int Cin, int Cout, int nmodes,
                       double* GX) {
    if (!G || !w || !GX || B <= 0 || Cin <= 0 || Cout <= 0 || nmodes <= 0) return -1;
    for (long long b = 0; b < B; ++b) {
        for (long long i = 0; i < Cin; ++i) {
            for (long long m = 0; m < nmodes; ++m) {
                double re = 0.0, im = 0.0;
                for (long long o = 0; o < Cout; ++o) {
                    const double* gv = G + 2 * ((b * Cout + o) * nmodes + m);
                    const double* wv = w + 2 * ((i * Cout + o) * nmodes + m);
                    // (a + bi) * (c - di) = (ac + bd) + (bc - ad) i
                    re += gv[0] * wv[0] + gv[1] * wv[1];
                    im += gv[1] * wv[0] - gv[0] * wv[1];
                }
                GX[2 * ((b * Cin + i) * nmodes + m)] = re;
                GX[2 * ((b * Cin + i) * nmodes + m) + 1] = im;
            }
        }
    }
    return 0;
}

// gx = 1/sqrt(HW) * Re sum over the retained bins of GX * exp(+2 pi i (...)),
// every retained bin with weight 1 (the transpose of the truncated forward DFT).
int oracle_backward_input(const double* GX, int B, int C, int H, int W, int m1, int m2,
                          double* gx) {
    if (!GX || !gx || !shape_ok(B, C, H, W, m1, m2)) return -1;
    const std::vector<double> tw_w = root_table(W, +1);
    const std::vector<double> tw_h = root_table(H, +1);
    const double scale = 1.0 / std::sqrt((double)H * (double)W);
    const int R = 2 * m1;
    std::vector<double> V(2 * (size_t)H * m2);
    for (long long p = 0; p < (long long)B * C; ++p) {
        const double* Gp = GX + p * (long long)R * m2 * 2;
        // V[h][k2] = sum_r GX[r][k2] * exp(+2*pi*i*k1(r)*h/H)
        for (int h = 0; h < H; ++h) {
            for (int k2 = 0; k2 < m2; ++k2) {
                double re = 0.0, im = 0.0;
                for (int r = 0; r < R; ++r) {
                    long long j = red(row_of(r, H, m1), h, H);
                    double a = Gp[2 * ((size_t)r * m2 + k2)];
                    double b = Gp[2 * ((size_t)r * m2 + k2) + 1];
                    re += a * tw_h[2 * j] - b * tw_h[2 * j + 1];
                    im += a * tw_h[2 * j + 1] + b * tw_h[2 * j];
                }
                V[2 * ((size_t)h * m2 + k2)] = re;
                V[2 * ((size_t)h * m2 + k2) + 1] = im;
            }
        }
        // gx[h][w] = scale * sum_k2 Re(V[h][k2] * exp(+2*pi*i*k2*w/W))
        double* gp = gx + p * (long long)H * W;
        for (int h = 0; h < H; ++h) {
            for (int w = 0; w < W; ++w) {
                double acc = 0.0;
                for (int k2 = 0; k2 < m2; ++k2) {
                    long long j = red(k2, w, W);
                    acc += V[2 * ((size_t)h * m2 + k2)] * tw_w[2 * j] -
                           V[2 * ((size_t)h * m2 + k2) + 1] * tw_w[2 * j + 1];
                }
                gp[(size_t)h * W + w] = scale * acc;
            }
        }
    }
    return 0;
}

// gw[i,o,m] = sum_b conj(X[b,i,m]) * G[b,o,m].
int oracle_weight_grad(const double* X, const double* G, int B, int Cin, int Cout, int nmodes,
                       double* gw) {
    if (!X || !G || !gw || B <= 0 || Cin <= 0 || Cout <= 0 || nmodes <= 0) return -1;
    for (long long i = 0; i < Cin; ++i) {
        for (long long o = 0; o < Cout; ++o) {
            for (long long m = 0; m < nmodes; ++m) {
                double re = 0.0, im = 0.0;
                for (long long b = 0; b < B; ++b) {
                    const double* xv = X + 2 * ((b * Cin + i) * nmodes + m);
                    const double* gv = G + 2 * ((b * Cout + o) * nmodes + m);
                    // (a - bi) * (c + di) = (ac + bd) + (ad - bc) i
                    re += xv[0] * gv[0] + xv[1] * gv[1];
                    im += xv[0] * gv[1] - xv[1] * gv[0];
                }
                gw[2 * ((i * Cout + o) * nmodes + m)] = re;
                gw[2 * ((i * Cout + o) * nmodes + m) + 1] = im;
            }
        }
    }
    return 0;
}

// The whole backward: gx and gw from x, w and g = dL/dy.
int oracle_spectral_conv2d_backward(const double* x, const double* w, const double* g, int B,
                                    int Cin, int Cout, int H, int W, int m1, int m2,
                                    double* gx, double* gw) {
    if (!x || !w || !g || !gx || !gw || Cout <= 0 || !shape_ok(B, Cin, H, W, m1, m2)) return -1;
    const long long nm = 2LL * m1 * m2;
    std::vector<double> X(2 * (size_t)B * Cin * nm), G(2 * (size_t)B * Cout * nm),
        GX(2 * (size_t)B * Cin * nm);
    int rc = oracle_forward_modes(x, B, Cin, H, W, m1, m2, X.data());
    if (!rc) rc = oracle_backward_modes(g, B, Cout, H, W, m1, m2, G.data());
    if (!rc) rc = oracle_mix_adjoint(G.data(), w, B, Cin, Cout, (int)nm, GX.data());
    if (!rc) rc = oracle_backward_input(GX.data(), B, Cin, H, W, m1, m2, gx);
    if (!rc) rc = oracle_weight_grad(X.data(), G.data(), B, Cin, Cout, (int)nm, gw);
    return rc;
}

// The whole layer: inverse(mix(forward(x), w)).
int oracle_spectral_conv2d(const double* x, const double* w, int B, int Cin, int Cout, int H,
                           int W, int m1, int m2, double* y) {
    if (!x || !w || !y || Cout <= 0 || !shape_ok(B, Cin, H, W, m1, m2)) return -1;
    const long long nm = 2LL * m1 * m2;
    std::vector<double> X(2 * (size_t)B * Cin * nm), Z(2 * (size_t)B * Cout * nm);
    int rc = oracle_forward_modes(x, B, Cin, H, W, m1, m2, X.data());
    if (rc) return rc;
    rc = oracle_mix_modes(X.data(), w, B, Cin, Cout, (int)nm, Z.data());
    if (rc) return rc;
    return oracle_inverse_modes(Z.data(), B, Cout, H, W, m1, m2, y);
}

}  // extern "C"
