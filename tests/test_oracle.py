"""Pins for the double-precision oracle (CPU only).

Each test checks the oracle against something other than itself: a closed
form, an invariant of the DFT, a brute-force definition written differently
(2D double sums, circular convolution), or numpy's pocketfft rfft2/irfft2, which
computes exactly the orthonormal irfft2(Z, s=(H, W)) of the layer's
definition.  Together they fail on a dropped term, a wrong sign or index, a
transposed operand, a wrong scale or a wrong retained-row order.
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(12345)


def kept_rows(H, m1):
    return list(range(m1)) + list(range(H - m1, H))


def numpy_layer(x, w, m1, m2):
    """The layer through numpy's FFT library (independent of the oracle)."""
    B, Cin, H, W = x.shape
    F = np.fft.rfft2(x, norm="ortho")
    rows = kept_rows(H, m1)
    Z = np.einsum("bixy,ioxy->boxy", F[:, :, rows, :m2], w)
    full = np.zeros((B, w.shape[1], H, W // 2 + 1), dtype=complex)
    full[:, :, rows, :m2] = Z
    return np.fft.irfft2(full, s=(H, W), norm="ortho")


def rand_w(Cin, Cout, m1, m2):
    return RNG.standard_normal((Cin, Cout, 2 * m1, m2)) + 1j * RNG.standard_normal(
        (Cin, Cout, 2 * m1, m2))


# ---------------------------------------------------------------- forward ---

@pytest.mark.parametrize("H,W,h0,w0", [(8, 8, 3, 5), (16, 4, 0, 1), (4, 32, 2, 31)])
def test_forward_delta_is_flat_phase(H, W, h0, w0):
    x = np.zeros((1, 1, H, W))
    x[0, 0, h0, w0] = 1.0
    m1, m2 = H // 2, W // 2 + 1
    X = oracle.forward_modes(x, m1, m2)[0, 0]
    for r, k1 in enumerate(kept_rows(H, m1)):
        for k2 in range(m2):
            ref = np.exp(-2j * np.pi * (k1 * h0 / H + k2 * w0 / W)) / np.sqrt(H * W)
            assert abs(X[r, k2] - ref) < 1e-14
    assert np.allclose(np.abs(X), 1 / np.sqrt(H * W), atol=1e-15)


def test_forward_constant_is_dc_only():
    H, W, c = 16, 8, 2.5
    x = np.full((1, 1, H, W), c)
    X = oracle.forward_modes(x, 4, 3)[0, 0]
    assert abs(X[0, 0] - np.sqrt(H * W) * c) < 1e-12
    X[0, 0] = 0
    assert np.abs(X).max() < 1e-12


@pytest.mark.parametrize("p,q", [(2, 0), (1, 3), (-3, 2)])
def test_forward_single_cosine(p, q):
    H, W = 16, 16
    h = np.arange(H)[:, None]
    w = np.arange(W)[None, :]
    x = np.cos(2 * np.pi * (p * h / H + q * w / W))[None, None]
    m1, m2 = 4, 5
    X = oracle.forward_modes(x, m1, m2)[0, 0]
    expect = np.zeros_like(X)
    rows = kept_rows(H, m1)
    half = np.sqrt(H * W) / 2
    for (kp, kq) in [(p % H, q), ((-p) % H, -q)]:
        if 0 <= kq < m2 and kp in rows:
            expect[rows.index(kp), kq] += half
    assert np.abs(X - expect).max() < 1e-12


@pytest.mark.parametrize("H,W", [(8, 8), (4, 16), (16, 2)])
def test_forward_parseval_full_modes(H, W):
    x = RNG.standard_normal((2, 3, H, W))
    X = oracle.forward_modes(x, H // 2, W // 2 + 1)
    # half spectrum: bins 1..W/2-1 stand for themselves and their mirrors
    wgt = np.full(W // 2 + 1, 2.0)
    wgt[0] = 1.0
    wgt[W // 2] = 1.0
    energy_X = (np.abs(X) ** 2 * wgt).sum(axis=(2, 3))
    energy_x = (x ** 2).sum(axis=(2, 3))
    assert np.allclose(energy_X, energy_x, rtol=1e-13)


def test_forward_brute_force_2d_sum():
    H, W, m1, m2 = 4, 8, 1, 3
    x = RNG.standard_normal((1, 2, H, W))
    X = oracle.forward_modes(x, m1, m2)
    for c in range(2):
        for r, k1 in enumerate(kept_rows(H, m1)):
            for k2 in range(m2):
                s = 0j
                for h in range(H):
                    for w in range(W):
                        s += x[0, c, h, w] * np.exp(-2j * np.pi * (k1 * h / H + k2 * w / W))
                assert abs(X[0, c, r, k2] - s / np.sqrt(H * W)) < 1e-13


@pytest.mark.parametrize("H,W,m1,m2", [(16, 16, 4, 4), (8, 32, 4, 17), (32, 8, 3, 2)])
def test_forward_matches_numpy_rfft2(H, W, m1, m2):
    x = RNG.standard_normal((2, 3, H, W))
    X = oracle.forward_modes(x, m1, m2)
    F = np.fft.rfft2(x, norm="ortho")[:, :, kept_rows(H, m1), :m2]
    assert np.abs(X - F).max() < 1e-13


# -------------------------------------------------------------------- mix ---

def test_mix_matches_numpy_complex_matmul():
    B, Cin, Cout, nm = 3, 5, 4, 7
    X = RNG.standard_normal((B, Cin, nm)) + 1j * RNG.standard_normal((B, Cin, nm))
    w = RNG.standard_normal((Cin, Cout, nm)) + 1j * RNG.standard_normal((Cin, Cout, nm))
    Z = oracle.mix_modes(X, w)
    for m in range(nm):
        assert np.abs(Z[:, :, m] - X[:, :, m] @ w[:, :, m]).max() < 1e-13


def test_mix_not_transposed():
    # Cin != Cout and B != Cin: a transposed operand would not even type-check
    X = np.zeros((2, 3, 1), complex)
    X[1, 2, 0] = 1j
    w = np.zeros((3, 5, 1), complex)
    w[2, 4, 0] = 2 + 1j
    Z = oracle.mix_modes(X, w)
    expect = np.zeros((2, 5, 1), complex)
    expect[1, 4, 0] = 1j * (2 + 1j)
    assert np.abs(Z - expect).max() == 0


# ---------------------------------------------------------------- inverse ---

@pytest.mark.parametrize("H,W,m1,m2", [(16, 16, 4, 4), (8, 32, 4, 17), (32, 8, 3, 2),
                                       (16, 16, 8, 9), (2, 2, 1, 2)])
def test_inverse_matches_numpy_irfft2(H, W, m1, m2):
    Z = RNG.standard_normal((2, 3, 2 * m1, m2)) + 1j * RNG.standard_normal((2, 3, 2 * m1, m2))
    y = oracle.inverse_modes(Z, H, W)
    full = np.zeros((2, 3, H, W // 2 + 1), complex)
    full[:, :, kept_rows(H, m1), :m2] = Z
    assert np.abs(y - np.fft.irfft2(full, s=(H, W), norm="ortho")).max() < 1e-13


def test_inverse_discards_imaginary_dc_and_nyquist():
    H, W = 8, 8
    Z = np.zeros((1, 1, 8, 5), complex)
    Z[0, 0, 0, 0] = 3j          # k1 = 0, k2 = 0: purely imaginary DC
    Z[0, 0, 0, 4] = -2j         # k1 = 0, k2 = W/2: purely imaginary Nyquist
    y = oracle.inverse_modes(Z, H, W)
    assert np.abs(y).max() < 1e-15


def test_inverse_at_matches_full():
    H, W, m1, m2 = 16, 8, 3, 4
    Z = RNG.standard_normal((2, 3, 2 * m1, m2)) + 1j * RNG.standard_normal((2, 3, 2 * m1, m2))
    y = oracle.inverse_modes(Z, H, W)
    idx = np.array([[0, 0, 0, 0], [1, 2, 15, 7], [1, 0, 9, 3], [0, 1, 4, 6]])
    assert np.abs(oracle.inverse_modes_at(Z, H, W, idx) - y[tuple(idx.T)]).max() < 1e-14


# ------------------------------------------------------------------ layer ---

@pytest.mark.parametrize("B,Cin,Cout,H,W,m1,m2", [
    (2, 4, 4, 16, 16, 4, 4),
    (1, 3, 5, 8, 32, 2, 17),
    (3, 2, 1, 32, 8, 16, 5),
    (1, 1, 1, 2, 2, 1, 2),
    (2, 6, 3, 16, 4, 1, 1),
])
def test_layer_matches_numpy(B, Cin, Cout, H, W, m1, m2):
    x = RNG.standard_normal((B, Cin, H, W))
    w = rand_w(Cin, Cout, m1, m2)
    y = oracle.spectral_conv2d(x, w, m1, m2)
    assert np.abs(y - numpy_layer(x, w, m1, m2)).max() < 1e-12 * max(1, np.abs(y).max())


@pytest.mark.parametrize("H,W", [(8, 8), (16, 4), (4, 16)])
def test_identity_weights_full_modes_give_identity(H, W):
    C = 3
    m1, m2 = H // 2, W // 2 + 1
    w = np.zeros((C, C, 2 * m1, m2), complex)
    for i in range(C):
        w[i, i] = 1.0
    x = RNG.standard_normal((2, C, H, W))
    y = oracle.spectral_conv2d(x, w, m1, m2)
    assert np.abs(y - x).max() < 1e-13


@pytest.mark.parametrize("H,W", [(8, 8), (4, 16)])
def test_convolution_theorem(H, W):
    """Cin = Cout = 1, all modes, w = unnormalised DFT of g: y = x (*) g (circular)."""
    x = RNG.standard_normal((1, 1, H, W))
    g = RNG.standard_normal((H, W))
    G = np.zeros((H, W), complex)
    hh = np.arange(H)[:, None]
    ww = np.arange(W)[None, :]
    for k1 in range(H):
        for k2 in range(W):
            G[k1, k2] = (g * np.exp(-2j * np.pi * (k1 * hh / H + k2 * ww / W))).sum()
    m1, m2 = H // 2, W // 2 + 1
    w = G[kept_rows(H, m1), :m2][None, None]
    y = oracle.spectral_conv2d(x, w, m1, m2)[0, 0]
    conv = np.zeros((H, W))
    for h in range(H):
        for wv in range(W):
            s = 0.0
            for a in range(H):
                for b in range(W):
                    s += x[0, 0, a, b] * g[(h - a) % H, (wv - b) % W]
            conv[h, wv] = s
    assert np.abs(y - conv).max() < 1e-12


def test_shift_equivariance_truncated():
    B, C, H, W, m1, m2 = 1, 2, 16, 8, 3, 3
    x = RNG.standard_normal((B, C, H, W))
    w = rand_w(C, C, m1, m2)
    y = oracle.spectral_conv2d(x, w, m1, m2)
    ys = oracle.spectral_conv2d(np.roll(x, (5, 3), axis=(2, 3)), w, m1, m2)
    assert np.abs(ys - np.roll(y, (5, 3), axis=(2, 3))).max() < 1e-12


def test_linearity_in_x_and_w():
    B, C, H, W, m1, m2 = 2, 3, 8, 8, 2, 3
    x1, x2 = RNG.standard_normal((2, B, C, H, W))
    w1, w2 = rand_w(C, C, m1, m2), rand_w(C, C, m1, m2)
    a, b = 0.7, -1.3
    f = oracle.spectral_conv2d
    assert np.abs(f(a * x1 + b * x2, w1, m1, m2) - a * f(x1, w1, m1, m2)
                  - b * f(x2, w1, m1, m2)).max() < 1e-12
    assert np.abs(f(x1, a * w1 + b * w2, m1, m2) - a * f(x1, w1, m1, m2)
                  - b * f(x1, w2, m1, m2)).max() < 1e-12


def test_zero_input_zero_output():
    w = rand_w(2, 2, 2, 2)
    y = oracle.spectral_conv2d(np.zeros((1, 2, 8, 8)), w, 2, 2)
    assert np.abs(y).max() == 0


def test_truncation_is_not_idempotent():
    """The retained row set keeps k1 = H - m1 but not its mirror m1, so the
    identity-weight layer with truncation is not a projection (reading c.4)."""
    H, W, m1, m2, C = 8, 8, 2, 2, 1
    w = np.ones((C, C, 2 * m1, m2), complex)
    x = RNG.standard_normal((1, C, H, W))
    y1 = oracle.spectral_conv2d(x, w, m1, m2)
    y2 = oracle.spectral_conv2d(y1, w, m1, m2)
    assert np.abs(y2 - y1).max() > 1e-3


@pytest.mark.parametrize("args", [
    (0, 1, 8, 8, 2, 2), (1, 1, 8, 8, 5, 2), (1, 1, 8, 8, 2, 6), (1, 1, 12, 8, 7, 2),
    (1, 1, 8, 8, 0, 2), (1, 1, 1, 8, 1, 2)])
def test_invalid_shapes_rejected(args):
    B, C, H, W, m1, m2 = args
    x = np.zeros((max(B, 1), C, H, W))
    with pytest.raises((ValueError, AssertionError)):
        if B == 0:
            oracle.forward_modes(np.zeros((0, C, H, W)), m1, m2)
        else:
            oracle.forward_modes(x, m1, m2)


# --------------------------------------------------------------- backward ---
# The gradients of L = <y, g> for g = dL/dy, with the complex convention
# dL/dRe(w) + i dL/dIm(w).  Pinned against the (already pinned) forward by
# identities that hold for any correct gradient of a linear map, and by finite
# differences; a wrong conjugation, a missing c(k2) weight, a transposed
# weight or a dropped Nyquist/DC term breaks one of them.

BACKWARD_SHAPES = [
    # B, Cin, Cout, H, W, m1, m2
    (2, 3, 2, 8, 8, 2, 3),       # interior columns only
    (1, 2, 3, 8, 8, 4, 5),       # 2*m1 = H, Nyquist column kept (m2 = W/2 + 1)
    (2, 1, 2, 16, 4, 3, 2),      # tall, k2 = 0 and the last-but-Nyquist column
    (1, 2, 2, 4, 16, 1, 9),      # wide, every column incl. Nyquist
]


@pytest.mark.parametrize("shape", BACKWARD_SHAPES)
def test_backward_input_is_the_adjoint(shape):
    B, Cin, Cout, H, W, m1, m2 = shape
    x = RNG.standard_normal((B, Cin, H, W))
    g = RNG.standard_normal((B, Cout, H, W))
    w = rand_w(Cin, Cout, m1, m2)
    y = oracle.spectral_conv2d(x, w, m1, m2)
    gx, _ = oracle.spectral_conv2d_backward(x, w, g, m1, m2)
    lhs, rhs = np.sum(y * g), np.sum(x * gx)
    assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + np.abs(y * g).sum())


@pytest.mark.parametrize("shape", BACKWARD_SHAPES)
def test_weight_gradient_identity(shape):
    # y is linear in w, so <y(x, v), g> = Re sum conj(gw) * v for every v
    B, Cin, Cout, H, W, m1, m2 = shape
    x = RNG.standard_normal((B, Cin, H, W))
    g = RNG.standard_normal((B, Cout, H, W))
    w = rand_w(Cin, Cout, m1, m2)
    v = rand_w(Cin, Cout, m1, m2)
    _, gw = oracle.spectral_conv2d_backward(x, w, g, m1, m2)
    lhs = np.sum(oracle.spectral_conv2d(x, v, m1, m2) * g)
    rhs = np.real(np.sum(np.conj(gw) * v))
    assert abs(lhs - rhs) <= 1e-12 * np.abs(np.conj(gw) * v).sum()


def test_backward_finite_differences():
    # central differences of L = <y, g> in one element of x, and in the real and
    # imaginary parts of one weight of each column kind (k2 = 0, interior, Nyquist)
    B, Cin, Cout, H, W, m1, m2 = 1, 2, 2, 8, 8, 2, 5
    x = RNG.standard_normal((B, Cin, H, W))
    g = RNG.standard_normal((B, Cout, H, W))
    w = rand_w(Cin, Cout, m1, m2)
    gx, gw = oracle.spectral_conv2d_backward(x, w, g, m1, m2)
    L = lambda xx, ww: np.sum(oracle.spectral_conv2d(xx, ww, m1, m2) * g)  # noqa: E731
    eps = 1e-4
    for idx in [(0, 1, 3, 5), (0, 0, 0, 0), (0, 1, 7, 2)]:
        dx = np.zeros_like(x)
        dx[idx] = eps
        fd = (L(x + dx, w) - L(x - dx, w)) / (2 * eps)
        assert abs(fd - gx[idx]) < 1e-7 * max(1.0, abs(fd))
    for widx in [(1, 0, 1, 0), (0, 1, 2, 3), (1, 1, 3, 4)]:
        for unit in (1.0, 1j):
            dw = np.zeros_like(w)
            dw[widx] = eps * unit
            fd = (L(x, w + dw) - L(x, w - dw)) / (2 * eps)
            want = gw[widx].real if unit == 1.0 else gw[widx].imag
            assert abs(fd - want) < 1e-7 * max(1.0, abs(fd))


def test_backward_modes_weights_columns():
    # dL/dZ is c(k2) times the truncated DFT of g: c = 1 for k2 = 0 and k2 = W/2
    g = RNG.standard_normal((1, 1, 8, 8))
    G = oracle.backward_modes(g, 2, 5)
    F = np.fft.rfft2(g, norm="ortho")[:, :, kept_rows(8, 2), :5]
    c = np.array([1.0, 2.0, 2.0, 2.0, 1.0])
    assert np.allclose(G, F * c, rtol=1e-12, atol=1e-12)


def test_mix_adjoint_and_weight_grad_match_numpy():
    B, Cin, Cout, nm = 3, 4, 5, 7
    G = RNG.standard_normal((B, Cout, nm)) + 1j * RNG.standard_normal((B, Cout, nm))
    X = RNG.standard_normal((B, Cin, nm)) + 1j * RNG.standard_normal((B, Cin, nm))
    w = RNG.standard_normal((Cin, Cout, nm)) + 1j * RNG.standard_normal((Cin, Cout, nm))
    assert np.allclose(oracle.mix_adjoint(G, w), np.einsum("bom,iom->bim", G, np.conj(w)),
                       rtol=1e-12, atol=1e-12)
    assert np.allclose(oracle.weight_grad(X, G), np.einsum("bim,bom->iom", np.conj(X), G),
                       rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ block epilogue ---

def test_gelu_closed_forms():
    import math
    v = np.array([-3.0, -1.0, -0.25, 0.0, 0.5, 2.0, 6.0])
    g = oracle.gelu(v)
    # scalar definition with the standard library's erf (independent of scipy)
    ref = np.array([0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0))) for t in v])
    assert np.allclose(g, ref, rtol=1e-15, atol=1e-15)
    # Phi(t) + Phi(-t) = 1  =>  gelu(t) - gelu(-t) = t
    t = RNG.standard_normal(1000) * 3
    assert np.allclose(oracle.gelu(t) - oracle.gelu(-t), t, rtol=0, atol=1e-13)
    assert oracle.gelu(0.0) == 0.0 and abs(oracle.gelu(40.0) - 40.0) < 1e-12


def test_pointwise_brute_force():
    B, Cin, Cout, H, W = 2, 3, 4, 5, 6
    x = RNG.standard_normal((B, Cin, H, W))
    wpw = RNG.standard_normal((Cout, Cin))
    bias = RNG.standard_normal(Cout)
    out = oracle.pointwise(x, wpw, bias)
    for b in range(B):
        for o in range(Cout):
            for h in range(H):
                for w_ in range(W):
                    want = bias[o] + sum(wpw[o, i] * x[b, i, h, w_] for i in range(Cin))
                    assert abs(out[b, o, h, w_] - want) < 1e-12


def test_block_special_cases():
    B, Cin, Cout, H, W, m1, m2 = 2, 3, 2, 8, 8, 2, 3
    x = RNG.standard_normal((B, Cin, H, W))
    w = rand_w(Cin, Cout, m1, m2)
    zero_pw = np.zeros((Cout, Cin))
    # no pointwise branch, no bias, no activation: the spectral layer itself
    assert np.allclose(oracle.block(x, w, zero_pw, np.zeros(Cout), m1, m2, "none"),
                       oracle.spectral_conv2d(x, w, m1, m2), rtol=1e-13, atol=1e-13)
    # no spectral weights: the pointwise branch through GELU
    wpw = RNG.standard_normal((Cout, Cin))
    bias = RNG.standard_normal(Cout)
    assert np.allclose(oracle.block(x, np.zeros_like(w), wpw, bias, m1, m2),
                       oracle.gelu(np.einsum("oi,bihw->bohw", wpw, x) + bias[None, :, None, None]),
                       rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("B,Cin,Cout,H,W,m1,m2", [
    (1, 2, 3, 12, 10, 3, 4),     # neither a power of two, even W (Nyquist at 5)
    (2, 1, 2, 9, 7, 2, 4),       # odd H and W (no Nyquist column)
    (1, 2, 2, 30, 50, 15, 26),   # 2*m1 = H, m2 = W/2 + 1
    (1, 1, 1, 3, 5, 1, 3),       # smallest odd grid, every column kept
])
def test_layer_matches_numpy_any_size(B, Cin, Cout, H, W, m1, m2):
    # the layer's definition holds for any H, W; numpy's pocketfft is independent
    x = RNG.standard_normal((B, Cin, H, W))
    w = rand_w(Cin, Cout, m1, m2)
    assert np.allclose(oracle.spectral_conv2d(x, w, m1, m2), numpy_layer(x, w, m1, m2),
                       rtol=1e-11, atol=1e-11)


# -------------------------------------------------------------------- 1D ---

def numpy_layer_1d(x, w, m):
    """The 1D layer through numpy's FFT library (independent of the oracle)."""
    B, Cin, L = x.shape
    F = np.fft.rfft(x, norm="ortho")[:, :, :m]
    Z = np.einsum("bik,iok->bok", F, w)
    full = np.zeros((B, w.shape[1], L // 2 + 1), dtype=complex)
    full[:, :, :m] = Z
    return np.fft.irfft(full, n=L, norm="ortho")


@pytest.mark.parametrize("B,Cin,Cout,L,m", [
    (2, 3, 2, 16, 5), (1, 2, 2, 16, 9),   # Nyquist kept (m = L/2 + 1)
    (2, 1, 3, 15, 8), (1, 2, 1, 100, 12),  # odd and non-power-of-two lengths
])
def test_layer_1d_matches_numpy(B, Cin, Cout, L, m):
    x = RNG.standard_normal((B, Cin, L))
    w = RNG.standard_normal((Cin, Cout, m)) + 1j * RNG.standard_normal((Cin, Cout, m))
    assert np.allclose(oracle.spectral_conv1d(x, w, m), numpy_layer_1d(x, w, m),
                       rtol=1e-12, atol=1e-12)


def test_layer_1d_convolution_theorem():
    # all modes kept, Cin = Cout = 1, w = unnormalised DFT of g: circular convolution
    L = 12
    x = RNG.standard_normal((1, 1, L))
    g = RNG.standard_normal(L)
    w = np.fft.rfft(g)[None, None, :]
    y = oracle.spectral_conv1d(x, w, L // 2 + 1)
    ref = np.array([sum(x[0, 0, j] * g[(n - j) % L] for j in range(L)) for n in range(L)])
    assert np.allclose(y[0, 0], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("L,m", [(16, 9), (15, 6)])
def test_backward_1d_identities(L, m):
    B, Cin, Cout = 2, 3, 2
    x = RNG.standard_normal((B, Cin, L))
    g = RNG.standard_normal((B, Cout, L))
    w = RNG.standard_normal((Cin, Cout, m)) + 1j * RNG.standard_normal((Cin, Cout, m))
    v = RNG.standard_normal((Cin, Cout, m)) + 1j * RNG.standard_normal((Cin, Cout, m))
    gx, gw = oracle.spectral_conv1d_backward(x, w, g, m)
    lhs = np.sum(oracle.spectral_conv1d(x, w, m) * g)
    assert abs(lhs - np.sum(x * gx)) <= 1e-12 * np.abs(x * gx).sum()
    lhs = np.sum(oracle.spectral_conv1d(x, v, m) * g)
    assert abs(lhs - np.real(np.sum(np.conj(gw) * v))) <= 1e-12 * np.abs(np.conj(gw) * v).sum()


def test_block_1d_special_cases():
    B, Cin, Cout, L, m = 2, 3, 2, 12, 5
    x = RNG.standard_normal((B, Cin, L))
    w = RNG.standard_normal((Cin, Cout, m)) + 1j * RNG.standard_normal((Cin, Cout, m))
    # no pointwise branch, bias or activation: the 1D layer itself
    assert np.allclose(oracle.block1d(x, w, np.zeros((Cout, Cin)), np.zeros(Cout), m, "none"),
                       oracle.spectral_conv1d(x, w, m), rtol=1e-13, atol=1e-13)
    # no spectral weights: each output point is GELU(bias + sum_i w_pw x), by hand
    wpw = RNG.standard_normal((Cout, Cin))
    bias = RNG.standard_normal(Cout)
    out = oracle.block1d(x, np.zeros_like(w), wpw, bias, m)
    for b in range(B):
        for o in range(Cout):
            for n in range(L):
                v = bias[o] + sum(wpw[o, i] * x[b, i, n] for i in range(Cin))
                want = 0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0)))
                assert abs(out[b, o, n] - want) < 1e-12


# ------------------------------------------- threaded wrappers (full-size) ---
# forward_modes_parallel / inverse_modes_parallel re-slice the planes over host
# threads to build the references of the large parity cases.  The arithmetic
# per plane is the serial oracle's, so the results must be bit-identical to it;
# they are also compared with numpy's pocketfft directly, so that a plane-order
# or reshape mistake (planes swapped, batch and channel transposed, a plane
# skipped by the striding) fails even where the serial path would too.

PARALLEL_SHAPES = [
    # B, C, H, W, m1, m2, threads
    (2, 3, 8, 16, 2, 5, 4),      # 6 planes over 4 threads (uneven stride)
    (3, 2, 16, 8, 4, 3, 16),     # more threads than planes
    (1, 5, 12, 10, 3, 6, 2),     # sizes that are not powers of two, Nyquist column kept
    (4, 1, 4, 32, 2, 17, 1),     # one thread, full half spectrum along W
    (2, 4, 16, 16, 8, 9, 3),     # 2*m1 = H, full modes
]


@pytest.mark.parametrize("B,C,H,W,m1,m2,threads", PARALLEL_SHAPES)
def test_forward_modes_parallel_equals_serial(B, C, H, W, m1, m2, threads):
    x = RNG.standard_normal((B, C, H, W))
    Xp = oracle.forward_modes_parallel(x, m1, m2, threads=threads)
    Xs = oracle.forward_modes(x, m1, m2)
    assert Xp.shape == (B, C, 2 * m1, m2)
    assert np.array_equal(Xp, Xs)
    F = np.fft.rfft2(x, norm="ortho")[:, :, kept_rows(H, m1), :m2]
    assert np.abs(Xp - F).max() < 1e-13


@pytest.mark.parametrize("B,C,H,W,m1,m2,threads", PARALLEL_SHAPES)
def test_inverse_modes_parallel_equals_serial(B, C, H, W, m1, m2, threads):
    Z = RNG.standard_normal((B, C, 2 * m1, m2)) + 1j * RNG.standard_normal((B, C, 2 * m1, m2))
    yp = oracle.inverse_modes_parallel(Z, H, W, threads=threads)
    ys = oracle.inverse_modes(Z, H, W)
    assert yp.shape == (B, C, H, W)
    assert np.array_equal(yp, ys)
    full = np.zeros((B, C, H, W // 2 + 1), complex)
    full[:, :, kept_rows(H, m1), :m2] = Z
    assert np.abs(yp - np.fft.irfft2(full, s=(H, W), norm="ortho")).max() < 1e-13


def test_parallel_wrappers_keep_plane_identity():
    """Each plane carries a distinct constant: the DC bin of plane (b, c) must
    come back at (b, c), and the inverse of a DC-only spectrum is that constant
    over the plane (orthonormal scale: DC = sqrt(HW) * value)."""
    B, C, H, W = 3, 4, 8, 8
    vals = np.arange(1, B * C + 1, dtype=np.float64).reshape(B, C)
    x = np.broadcast_to(vals[:, :, None, None], (B, C, H, W)).copy()
    X = oracle.forward_modes_parallel(x, 2, 2, threads=5)
    assert np.abs(X[:, :, 0, 0] - vals * np.sqrt(H * W)).max() < 1e-12
    X[:, :, 0, 0] = 0
    assert np.abs(X).max() < 1e-12
    Z = np.zeros((B, C, 4, 2), complex)
    Z[:, :, 0, 0] = vals * np.sqrt(H * W)
    y = oracle.inverse_modes_parallel(Z, H, W, threads=7)
    assert np.abs(y - x).max() < 1e-12
