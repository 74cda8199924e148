"""Double-precision oracle for the FNO 2D spectral-convolution layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library: it is plain single-threaded C++ (``fno_oracle.cpp``)
computing every DFT by direct sums, reached here through ctypes.

All functions take numpy arrays (converted to float64, C-contiguous) and return
float64 arrays.  Complex arrays use numpy complex128.  Layouts:

  x : [B, C, H, W] real
  X : [B, C, 2*m1, m2] complex (retained rows: k1 = 0..m1-1, then H-m1..H-1)
  w : [Cin, Cout, 2*m1, m2] complex
  Z : [B, Cout, 2*m1, m2] complex
  y : [B, Cout, H, W] real
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fno_oracle.cpp")
_LIB = os.path.join(_HERE, "libfno_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no fast-math, no OpenMP) if it is stale."""
    with _lock:
        stale = force or not os.path.exists(_LIB) or (
            os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
        if stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["g++", "-std=c++17", "-O2", "-fPIC", "-shared",
                                   "-fno-fast-math", "-ffp-contract=off",
                                   "-o", tmp, _SRC])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        i = ctypes.c_int
        lib.oracle_forward_modes.argtypes = [dp, i, i, i, i, i, i, dp]
        lib.oracle_mix_modes.argtypes = [dp, dp, i, i, i, i, dp]
        lib.oracle_inverse_modes.argtypes = [dp, i, i, i, i, i, i, dp]
        lib.oracle_inverse_modes_at.argtypes = [dp, i, i, i, i, i, i, ip, i, dp]
        lib.oracle_spectral_conv2d.argtypes = [dp, dp, i, i, i, i, i, i, i, dp]
        lib.oracle_backward_modes.argtypes = [dp, i, i, i, i, i, i, dp]
        lib.oracle_mix_adjoint.argtypes = [dp, dp, i, i, i, i, dp]
        lib.oracle_backward_input.argtypes = [dp, i, i, i, i, i, i, dp]
        lib.oracle_weight_grad.argtypes = [dp, dp, i, i, i, i, dp]
        lib.oracle_spectral_conv2d_backward.argtypes = [dp, dp, dp, i, i, i, i, i, i, i, dp, dp]
        for f in (lib.oracle_forward_modes, lib.oracle_mix_modes, lib.oracle_inverse_modes,
                  lib.oracle_inverse_modes_at, lib.oracle_spectral_conv2d,
                  lib.oracle_backward_modes, lib.oracle_mix_adjoint, lib.oracle_backward_input,
                  lib.oracle_weight_grad, lib.oracle_spectral_conv2d_backward):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _real(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _cplx(a) -> np.ndarray:
    """complex array [...] -> contiguous float64 [..., 2] view-compatible buffer."""
    a = np.asarray(a)
    if np.iscomplexobj(a):
        return np.ascontiguousarray(a.astype(np.complex128))
    # interleaved real pairs [..., 2]
    a = np.ascontiguousarray(a, dtype=np.float64)
    assert a.shape[-1] == 2
    return a.view(np.complex128)[..., 0]


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle: invalid arguments to {what}")


def forward_modes(x, m1: int, m2: int) -> np.ndarray:
    """X = orthonormal rfft2(x) on the retained modes, by direct sums."""
    x = _real(x)
    B, C, H, W = x.shape
    X = np.zeros((B, C, 2 * m1, m2), dtype=np.complex128)
    _check(_load().oracle_forward_modes(_dptr(x), B, C, H, W, m1, m2,
                                        _dptr(X.view(np.float64))), "forward_modes")
    return X


def mix_modes(X, w) -> np.ndarray:
    """Z[b,o,m] = sum_i X[b,i,m] w[i,o,m] (complex), modes flattened."""
    X = _cplx(X)
    w = _cplx(w)
    B, Cin = X.shape[:2]
    Cin2, Cout = w.shape[:2]
    assert Cin == Cin2 and X.shape[2:] == w.shape[2:]
    nm = int(np.prod(X.shape[2:]))
    Z = np.zeros((B, Cout) + X.shape[2:], dtype=np.complex128)
    _check(_load().oracle_mix_modes(_dptr(X.view(np.float64)), _dptr(w.view(np.float64)),
                                    B, Cin, Cout, nm, _dptr(Z.view(np.float64))), "mix_modes")
    return Z


def inverse_modes(Z, H: int, W: int) -> np.ndarray:
    """y = orthonormal irfft2 of Z zero-filled outside the retained modes."""
    Z = _cplx(Z)
    B, C, R, m2 = Z.shape
    m1 = R // 2
    y = np.zeros((B, C, H, W), dtype=np.float64)
    _check(_load().oracle_inverse_modes(_dptr(Z.view(np.float64)), B, C, H, W, m1, m2,
                                        _dptr(y)), "inverse_modes")
    return y


def inverse_modes_at(Z, H: int, W: int, idx) -> np.ndarray:
    """y[b,o,h,w] for each row (b,o,h,w) of idx (int array [n,4])."""
    Z = _cplx(Z)
    B, C, R, m2 = Z.shape
    m1 = R // 2
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32).reshape(-1, 4))
    out = np.zeros(idx.shape[0], dtype=np.float64)
    _check(_load().oracle_inverse_modes_at(
        _dptr(Z.view(np.float64)), B, C, H, W, m1, m2,
        idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), idx.shape[0], _dptr(out)),
        "inverse_modes_at")
    return out


def spectral_conv2d(x, w, m1: int, m2: int) -> np.ndarray:
    """The whole layer y = inverse(mix(forward(x), w)) in double."""
    x = _real(x)
    w = _cplx(w)
    B, Cin, H, W = x.shape
    Cout = w.shape[1]
    assert w.shape == (Cin, Cout, 2 * m1, m2)
    y = np.zeros((B, Cout, H, W), dtype=np.float64)
    _check(_load().oracle_spectral_conv2d(_dptr(x), _dptr(w.view(np.float64)), B, Cin, Cout,
                                          H, W, m1, m2, _dptr(y)), "spectral_conv2d")
    return y


def backward_modes(g, m1: int, m2: int) -> np.ndarray:
    """dL/dZ = c(k2) * orthonormal truncated DFT of g = dL/dy (c = 1 at k2 = 0 and
    k2 = W/2, else 2)."""
    g = _real(g)
    B, C, H, W = g.shape
    G = np.zeros((B, C, 2 * m1, m2), dtype=np.complex128)
    _check(_load().oracle_backward_modes(_dptr(g), B, C, H, W, m1, m2,
                                         _dptr(G.view(np.float64))), "backward_modes")
    return G


def mix_adjoint(G, w) -> np.ndarray:
    """GX[b,i,m] = sum_o G[b,o,m] conj(w[i,o,m])."""
    G = _cplx(G)
    w = _cplx(w)
    B, Cout = G.shape[:2]
    Cin, Cout2 = w.shape[:2]
    assert Cout == Cout2 and G.shape[2:] == w.shape[2:]
    nm = int(np.prod(G.shape[2:]))
    GX = np.zeros((B, Cin) + G.shape[2:], dtype=np.complex128)
    _check(_load().oracle_mix_adjoint(_dptr(G.view(np.float64)), _dptr(w.view(np.float64)),
                                      B, Cin, Cout, nm, _dptr(GX.view(np.float64))),
           "mix_adjoint")
    return GX


def backward_input(GX, H: int, W: int) -> np.ndarray:
    """gx = transpose of the truncated forward DFT applied to GX."""
    GX = _cplx(GX)
    B, C, R, m2 = GX.shape
    gx = np.zeros((B, C, H, W), dtype=np.float64)
    _check(_load().oracle_backward_input(_dptr(GX.view(np.float64)), B, C, H, W, R // 2, m2,
                                         _dptr(gx)), "backward_input")
    return gx


def weight_grad(X, G) -> np.ndarray:
    """gw[i,o,m] = sum_b conj(X[b,i,m]) G[b,o,m]."""
    X = _cplx(X)
    G = _cplx(G)
    B, Cin = X.shape[:2]
    B2, Cout = G.shape[:2]
    assert B == B2 and X.shape[2:] == G.shape[2:]
    nm = int(np.prod(X.shape[2:]))
    gw = np.zeros((Cin, Cout) + X.shape[2:], dtype=np.complex128)
    _check(_load().oracle_weight_grad(_dptr(X.view(np.float64)), _dptr(G.view(np.float64)),
                                      B, Cin, Cout, nm, _dptr(gw.view(np.float64))),
           "weight_grad")
    return gw


def spectral_conv2d_backward(x, w, g, m1: int, m2: int):
    """(gx, gw): gradients of a real loss with dL/dy = g, in double.  The
    complex gradient is dL/dRe(w) + i dL/dIm(w)."""
    x = _real(x)
    g = _real(g)
    w = _cplx(w)
    B, Cin, H, W = x.shape
    Cout = w.shape[1]
    assert w.shape == (Cin, Cout, 2 * m1, m2) and g.shape == (B, Cout, H, W)
    gx = np.zeros((B, Cin, H, W), dtype=np.float64)
    gw = np.zeros((Cin, Cout, 2 * m1, m2), dtype=np.complex128)
    _check(_load().oracle_spectral_conv2d_backward(
        _dptr(x), _dptr(w.view(np.float64)), _dptr(g), B, Cin, Cout, H, W, m1, m2, _dptr(gx),
        _dptr(gw.view(np.float64))), "spectral_conv2d_backward")
    return gx, gw


def _roots(L: int, sign: int) -> np.ndarray:
    """exp(sign * 2 pi i j / L) for j in [0, L), angles from the exact integer j."""
    j = np.arange(L, dtype=np.float64)
    return np.exp(sign * 2j * np.pi * j / L)


def spectral_conv1d(x, w, m: int) -> np.ndarray:
    """The 1D layer in double, by direct sums:
      X[b,i,k] = 1/sqrt(L) sum_n x[b,i,n] exp(-2 pi i k n / L),   k < m
      Z[b,o,k] = sum_i X[b,i,k] w[i,o,k]
      y[b,o,n] = 1/sqrt(L) sum_{k<m} c(k) Re(Z[b,o,k] exp(+2 pi i k n / L))
    with c = 1 for k = 0 and k = L/2, else 2 (the irfft of the truncated half
    spectrum, norm="ortho")."""
    x = _real(x)
    w = np.asarray(w, dtype=np.complex128)
    B, Cin, L = x.shape
    assert w.shape[0] == Cin and w.shape[2] == m and 1 <= m <= L // 2 + 1
    k = np.arange(m)
    n = np.arange(L)
    kn = np.outer(k, n) % L                        # exact integer products, reduced
    F = _roots(L, -1)[kn] / np.sqrt(L)             # [m, L]
    X = np.einsum("bin,kn->bik", x, F)
    Z = np.einsum("bik,iok->bok", X, w)
    c = np.where((k == 0) | (2 * k == L), 1.0, 2.0)
    G = _roots(L, +1)[kn] / np.sqrt(L)             # [m, L]
    return np.real(np.einsum("bok,kn->bon", Z * c, G))


def spectral_conv1d_backward(x, w, g, m: int):
    """(gx, gw) of the 1D layer for dL/dy = g, by the same derivation as the 2D
    backward: dL/dZ = c(k) G with G the truncated DFT of g; dL/dx is the
    transpose of the truncated DFT applied to sum_o dL/dZ conj(w); dL/dw =
    sum_b conj(X) dL/dZ."""
    x = _real(x)
    g = _real(g)
    w = np.asarray(w, dtype=np.complex128)
    B, Cin, L = x.shape
    k = np.arange(m)
    n = np.arange(L)
    kn = np.outer(k, n) % L
    F = _roots(L, -1)[kn] / np.sqrt(L)
    c = np.where((k == 0) | (2 * k == L), 1.0, 2.0)
    X = np.einsum("bin,kn->bik", x, F)
    GZ = np.einsum("bon,kn->bok", g, F) * c
    GX = np.einsum("bok,iok->bik", GZ, np.conj(w))
    gx = np.real(np.einsum("bik,kn->bin", GX, _roots(L, +1)[kn] / np.sqrt(L)))
    gw = np.einsum("bik,bok->iok", np.conj(X), GZ)
    return gx, gw


def gelu(v) -> np.ndarray:
    """GELU in its erf form, v * Phi(v) = v/2 * (1 + erf(v / sqrt(2))), in double."""
    from scipy.special import erf
    v = np.asarray(v, dtype=np.float64)
    return 0.5 * v * (1.0 + erf(v / np.sqrt(2.0)))


def pointwise(x, w_pw, bias=None) -> np.ndarray:
    """The 1x1 convolution of the FNO block: out[b,o,h,w] = sum_i w_pw[o,i] x[b,i,h,w]
    (+ bias[o]), in double."""
    x = _real(x)
    w_pw = _real(w_pw)
    out = np.einsum("oi,bihw->bohw", w_pw, x)
    if bias is not None:
        out = out + _real(bias)[None, :, None, None]
    return out


def block(x, w, w_pw, bias, m1: int, m2: int, activation: str = "gelu") -> np.ndarray:
    """One FNO block: act(spectral_conv2d(x, w) + w_pw x + bias), act in
    {"gelu", "none"} (the spectral layer plus the pointwise branch and the
    activation that follows it in the neural-operator block)."""
    y = spectral_conv2d(x, w, m1, m2) + pointwise(x, w_pw, bias)
    if activation == "gelu":
        return gelu(y)
    assert activation == "none"
    return y


def block1d(x, w, w_pw, bias, m: int, activation: str = "gelu") -> np.ndarray:
    """The block around the 1D layer: act(spectral_conv1d(x, w) + w_pw x + bias),
    x [B, Cin, L]; the pointwise branch is the 2D one over a 1 x L grid."""
    x = _real(x)
    B, Cin, L = x.shape
    y = spectral_conv1d(x, w, m) + pointwise(x.reshape(B, Cin, 1, L), w_pw, bias)[:, :, 0, :]
    if activation == "gelu":
        return gelu(y)
    assert activation == "none"
    return y


def forward_modes_parallel(x, m1: int, m2: int, threads: int | None = None) -> np.ndarray:
    """forward_modes over independent planes on several host threads.

    ctypes releases the GIL during the call, so each thread runs the same
    single-threaded oracle on its own planes; the arithmetic per plane is
    unchanged.  Used only to keep full-size parity checks fast.
    """
    x = _real(x)
    B, C, H, W = x.shape
    flat = x.reshape(B * C, 1, H, W)
    X = np.zeros((B * C, 1, 2 * m1, m2), dtype=np.complex128)
    n = threads or min(16, os.cpu_count() or 1)
    lib = _load()

    def work(t):
        for p in range(t, B * C, n):
            xp = np.ascontiguousarray(flat[p])
            Xp = np.zeros((1, 2 * m1, m2), dtype=np.complex128)
            _check(lib.oracle_forward_modes(_dptr(xp), 1, 1, H, W, m1, m2,
                                            _dptr(Xp.view(np.float64))), "forward_modes")
            X[p] = Xp

    ts = [threading.Thread(target=work, args=(t,)) for t in range(n)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return X.reshape(B, C, 2 * m1, m2)


def inverse_modes_parallel(Z, H: int, W: int, threads: int | None = None) -> np.ndarray:
    """inverse_modes over independent planes on several host threads."""
    Z = _cplx(Z)
    B, C, R, m2 = Z.shape
    flat = Z.reshape(B * C, 1, R, m2)
    y = np.zeros((B * C, 1, H, W), dtype=np.float64)
    n = threads or min(16, os.cpu_count() or 1)
    lib = _load()

    def work(t):
        for p in range(t, B * C, n):
            Zp = np.ascontiguousarray(flat[p])
            yp = np.zeros((1, 1, H, W), dtype=np.float64)
            _check(lib.oracle_inverse_modes(_dptr(Zp.view(np.float64)), 1, 1, H, W, R // 2,
                                            m2, _dptr(yp)), "inverse_modes")
            y[p] = yp[0]

    ts = [threading.Thread(target=work, args=(t,)) for t in range(n)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return y.reshape(B, C, H, W)
