"""Seeded synthetic inputs for the FNO spectral-convolution layer.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds no arithmetic of the layer: only a counter-based generator (SplitMix64,
see ``synth.c``) and the recipes that turn its draws into the inputs.

Recipes (seed 0 unless a caller says otherwise):
  * x ~ N(0, 1) float32, stream 1, flat index order [B][Cin][H][W].
  * "smooth" x: per plane, 8 random low-frequency cosines (integer wave numbers
    in [-4, 4], amplitude ~ N(0, 1/4), phase ~ U[0, 2 pi)) plus 0.1 * N(0, 1)
    noise; sinusoid parameters from stream 3, noise from stream 1.
  * w complex64 [Cin][Cout][2*m1][m2] stored as float32 (re, im) pairs with
    re, im ~ U[0, 1) / (Cin * Cout), stream 2, re drawn before im.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libfno_synth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    with _lock:
        stale = force or not os.path.exists(_LIB) or (
            os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
        if stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
                                   "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int
        fp = ctypes.POINTER(ctypes.c_float)
        lib.synth_draw.argtypes = [u64, u64, u64]
        lib.synth_draw.restype = u64
        lib.synth_uniform.argtypes = [u64, u64, u64]
        lib.synth_uniform.restype = ctypes.c_double
        lib.synth_normal.argtypes = [u64, u64, u64]
        lib.synth_normal.restype = ctypes.c_double
        lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, fp]
        lib.synth_uniform_f32.argtypes = [u64, u64, u64, i64, ctypes.c_double, fp]
        lib.synth_smooth_f32.argtypes = [u64, i32, i32, i32, i32, fp]
        for f in (lib.synth_normal_f32, lib.synth_uniform_f32, lib.synth_smooth_f32):
            f.restype = None
        _lib = lib
    return _lib


def _fp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def draw(seed: int, stream: int, j: int) -> int:
    return int(_load().synth_draw(seed, stream, j))


def uniform(seed: int, stream: int, j: int) -> float:
    return float(_load().synth_uniform(seed, stream, j))


def normal(seed: int, stream: int, j: int) -> float:
    return float(_load().synth_normal(seed, stream, j))


def normal_f32(shape, seed: int = 0, stream: int = 1, offset: int = 0,
               out: np.ndarray | None = None) -> np.ndarray:
    n = int(np.prod(shape))
    a = np.empty(n, dtype=np.float32) if out is None else out.reshape(-1)
    _load().synth_normal_f32(seed, stream, offset, n, _fp(a))
    return a.reshape(shape)


def uniform_f32(shape, scale: float = 1.0, seed: int = 0, stream: int = 2,
                offset: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    n = int(np.prod(shape))
    a = np.empty(n, dtype=np.float32) if out is None else out.reshape(-1)
    _load().synth_uniform_f32(seed, stream, offset, n, float(scale), _fp(a))
    return a.reshape(shape)


def smooth_f32(B: int, C: int, H: int, W: int, seed: int = 0,
               out: np.ndarray | None = None) -> np.ndarray:
    a = np.empty((B, C, H, W), dtype=np.float32) if out is None else out
    _load().synth_smooth_f32(seed, B, C, H, W, _fp(a))
    return a


@dataclass(frozen=True)
class LayerConfig:
    name: str
    B: int
    Cin: int
    Cout: int
    H: int
    W: int
    m1: int
    m2: int
    smooth: bool = False

    @property
    def nmodes(self) -> int:
        return 2 * self.m1 * self.m2

    def x_bytes(self) -> int:
        return 4 * self.B * self.Cin * self.H * self.W

    def y_bytes(self) -> int:
        return 4 * self.B * self.Cout * self.H * self.W

    def w_bytes(self) -> int:
        return 8 * self.Cin * self.Cout * self.nmodes

    def algorithmic_bytes(self) -> int:
        """x read once + y written once + w read once."""
        return self.x_bytes() + self.y_bytes() + self.w_bytes()

    def gemm_flops(self) -> int:
        """Real flops of the per-mode complex contraction (8 per complex MAC)."""
        return 8 * self.B * self.Cin * self.Cout * self.nmodes


# The five workloads: a tiny case, a smooth 64x64 case, the 128x128 C=64 case
# (the 128x128 resolution the fused-operator page measures, batch 16), a wide
# 256x256 C=128 case whose weight tensor dominates, and the 2048x2048 grid
# with 64x64 retained modes.
CONFIGS = {
    c.name: c for c in (
        LayerConfig("B2_C4_16x16_m4", 2, 4, 4, 16, 16, 4, 4),
        LayerConfig("B8_C32_64x64_m16_smooth", 8, 32, 32, 64, 64, 16, 16, smooth=True),
        LayerConfig("B16_C64_128x128_m32", 16, 64, 64, 128, 128, 32, 32),
        LayerConfig("B4_C128_256x256_m64", 4, 128, 128, 256, 256, 64, 64),
        LayerConfig("B2_C32_2048x2048_m64", 2, 32, 32, 2048, 2048, 64, 64),
    )
}
CONFIG_ORDER = list(CONFIGS)
HEADLINE = "B16_C64_128x128_m32"


def make_x(cfg: LayerConfig, seed: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    if cfg.smooth:
        return smooth_f32(cfg.B, cfg.Cin, cfg.H, cfg.W, seed=seed, out=out)
    return normal_f32((cfg.B, cfg.Cin, cfg.H, cfg.W), seed=seed, stream=1, out=out)


def make_w(cfg: LayerConfig, seed: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """float32 [Cin, Cout, 2*m1, m2, 2] (re, im interleaved)."""
    return uniform_f32((cfg.Cin, cfg.Cout, 2 * cfg.m1, cfg.m2, 2),
                       scale=1.0 / (cfg.Cin * cfg.Cout), seed=seed, stream=2, out=out)


def make_inputs(cfg: LayerConfig, seed: int = 0):
    return make_x(cfg, seed), make_w(cfg, seed)
