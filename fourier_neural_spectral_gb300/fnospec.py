"""Thin ctypes binding of libfnospec (include/fnospec.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the
library is missing or fails to load, every entry point raises; there is no
fallback computation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# FNO_DEBUG_BOUNDS=1 selects the range-checked build (python -m
# fourier_neural_spectral_gb300.build --debug): every global store of the main
# kernels is checked against its launch's output ranges.
LIB_PATH = os.path.join(_PKG, "libfnospec_debug.so" if os.environ.get("FNO_DEBUG_BOUNDS") == "1"
                        else "libfnospec.so")

FNO_OK = 0
FNO_ERR_INVALID_ARG = 1
FNO_ERR_UNSUPPORTED = 2
FNO_ERR_CUDA = 3
FNO_ERR_WORKSPACE = 4
FNO_ERR_TIMEOUT = 5
FNO_ERR_DEVICE = 6

FNO_PREC_FP32 = 0
FNO_PREC_TF32 = 1
FNO_PREC_3XTF32 = 2
FNO_ACT_NONE = 0
FNO_ACT_GELU = 1
ACTIVATIONS = {"none": FNO_ACT_NONE, "gelu": FNO_ACT_GELU}
PRECISIONS = {"fp32": FNO_PREC_FP32, "tf32": FNO_PREC_TF32, "3xtf32": FNO_PREC_3XTF32}

# Every symbol include/fnospec.h declares.
EXPORTS = (
    "fno_status_string", "fno_plan_create", "fno_plan_workspace_size", "fno_plan_launch_count",
    "fno_plan_describe", "fno_plan_kernel_info", "fno_plan_record_events", "fno_plan_execute", "fno_plan_destroy", "fno_spectral_conv2d",
    "fno_release_cache", "fno_forward_modes", "fno_mix_modes", "fno_inverse_modes",
    "fno_get_device_status", "fno_spectral_conv2d_noalloc", "fno_plan_backward",
    "fno_block_epilogue", "fno_block_execute", "fno_plan_create_1d",
    "fno_plan_debug_force_timeout", "fno_plan_set_single_launch", "fno_plan_debug_bounds_margin",
)


class FnoError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libfnospec and declare the C signatures.  Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libfnospec not built ({path} missing): run "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        st = ctypes.c_int
        sig = {
            "fno_status_string": (ctypes.c_char_p, [st]),
            "fno_plan_create": (st, [ctypes.POINTER(vp), i, i, i, i, i, i, i, i]),
            "fno_plan_create_1d": (st, [ctypes.POINTER(vp), i, i, i, i, i, i]),
            "fno_plan_debug_force_timeout": (st, [vp, i]),
            "fno_plan_set_single_launch": (st, [vp, i]),
            "fno_plan_debug_bounds_margin": (st, [vp, sz]),
            "fno_plan_workspace_size": (st, [vp, ctypes.POINTER(sz)]),
            "fno_plan_launch_count": (st, [vp, ctypes.POINTER(i)]),
            "fno_plan_describe": (st, [vp, ctypes.c_char_p, sz]),
            "fno_plan_kernel_info": (st, [vp, i, ctypes.c_char_p, sz, ctypes.POINTER(sz),
                                          ctypes.POINTER(sz)]),
            "fno_plan_record_events": (st, [vp, ctypes.POINTER(vp), i]),
            "fno_plan_execute": (st, [vp, vp, vp, vp, vp, sz, vp]),
            "fno_plan_destroy": (st, [vp]),
            "fno_spectral_conv2d": (st, [vp, vp, vp, i, i, i, i, i, i, i, vp]),
            "fno_release_cache": (st, []),
            "fno_forward_modes": (st, [vp, vp, vp, vp, sz, vp]),
            "fno_mix_modes": (st, [vp, vp, vp, vp, vp]),
            "fno_inverse_modes": (st, [vp, vp, vp, vp, sz, vp]),
            "fno_get_device_status": (st, [vp, vp]),
            "fno_spectral_conv2d_noalloc": (st, [vp, vp, vp, i, i, i, i, i, i, i, vp]),
            "fno_plan_backward": (st, [vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "fno_block_epilogue": (st, [vp, vp, vp, vp, i, vp, vp]),
            "fno_block_execute": (st, [vp, vp, vp, vp, vp, i, vp, vp, sz, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library().fno_status_string(status).decode()
    except Exception:
        return f"status {status}"


def _check(status: int, where: str):
    if status != FNO_OK:
        raise FnoError(status, where)


def _ptr(t) -> int | None:
    """Device address of a tensor, or an int/None passed through unchanged."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor or an address, got {type(t)}")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libfnospec must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _weight_ptr(w) -> int:
    if isinstance(w, torch.Tensor) and w.dtype == torch.complex64:
        return _ptr(w)
    if isinstance(w, torch.Tensor) and w.dtype != torch.float32:
        raise TypeError("w must be complex64 or float32 (re, im) pairs")
    return _ptr(w)


def _precision(precision) -> int:
    return PRECISIONS[precision] if isinstance(precision, str) else int(precision)


class Plan:
    """fno_plan_t owner.  Holds its workspace as a torch tensor on the device."""

    def __init__(self, B, Cin, Cout, H, W, m1, m2, precision="fp32", allocate_workspace=True):
        h = ctypes.c_void_p()
        _check(load_library().fno_plan_create(ctypes.byref(h), B, Cin, Cout, H, W, m1, m2,
                                              _precision(precision)), "fno_plan_create")
        self._setup(h, (B, Cin, Cout, H, W, m1, m2), precision, allocate_workspace)

    def _setup(self, h, shape, precision, allocate_workspace):
        lib = load_library()
        self._h = h
        self.shape = shape
        self.precision = precision
        n = ctypes.c_size_t()
        _check(lib.fno_plan_workspace_size(h, ctypes.byref(n)), "fno_plan_workspace_size")
        self.workspace_bytes = int(n.value)
        self._describe()
        self._event_array = None
        self.workspace = None
        if allocate_workspace and self.workspace_bytes:
            self.workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8, device="cuda")

    def _describe(self):
        """Launch count, description and kernel list of the plan as it stands."""
        lib = load_library()
        h = self._h
        k = ctypes.c_int()
        _check(lib.fno_plan_launch_count(h, ctypes.byref(k)), "fno_plan_launch_count")
        self.launches = int(k.value)
        buf = ctypes.create_string_buffer(256)
        _check(lib.fno_plan_describe(h, buf, 256), "fno_plan_describe")
        self.description = buf.value.decode()
        self.kernels = []
        for k in range(self.launches):
            nm = ctypes.create_string_buffer(64)
            nb, nf = ctypes.c_size_t(), ctypes.c_size_t()
            _check(lib.fno_plan_kernel_info(h, k, nm, 64, ctypes.byref(nb), ctypes.byref(nf)),
                   "fno_plan_kernel_info")
            self.kernels.append({"name": nm.value.decode(), "bytes": int(nb.value),
                                 "flops": int(nf.value)})

    @property
    def handle(self):
        return self._h

    def _ws(self, workspace):
        ws = self.workspace if workspace is None else workspace
        nbytes = 0 if ws is None else ws.numel() * ws.element_size()
        return _ptr(ws), nbytes

    def fno_plan_execute(self, x, w, y, workspace=None, stream=None):
        wp, wn = self._ws(workspace)
        _check(load_library().fno_plan_execute(self._h, _ptr(x), _weight_ptr(w), _ptr(y), wp, wn,
                                               _stream(stream)), "fno_plan_execute")
        return y

    def fno_forward_modes(self, x, X, workspace=None, stream=None):
        wp, wn = self._ws(workspace)
        _check(load_library().fno_forward_modes(self._h, _ptr(x), _ptr(X), wp, wn,
                                                _stream(stream)), "fno_forward_modes")
        return X

    def fno_mix_modes(self, X, w, Z, stream=None):
        _check(load_library().fno_mix_modes(self._h, _ptr(X), _weight_ptr(w), _ptr(Z),
                                            _stream(stream)), "fno_mix_modes")
        return Z

    def fno_inverse_modes(self, Z, y, workspace=None, stream=None):
        wp, wn = self._ws(workspace)
        _check(load_library().fno_inverse_modes(self._h, _ptr(Z), _ptr(y), wp, wn,
                                                _stream(stream)), "fno_inverse_modes")
        return y

    def fno_block_epilogue(self, x, w_pw, bias, y, activation="gelu", stream=None):
        """y <- act(y + w_pw x + bias) in place (y: the spectral layer's output)."""
        act = ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)
        _check(load_library().fno_block_epilogue(self._h, _ptr(x), _ptr(w_pw), _ptr(bias), act,
                                                 _ptr(y), _stream(stream)), "fno_block_epilogue")
        return y

    def fno_block_execute(self, x, w, w_pw, bias, y, activation="gelu", workspace=None,
                          stream=None):
        """One FNO block: y = act(layer(x, w) + w_pw x + bias)."""
        act = ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)
        wp, wn = self._ws(workspace)
        _check(load_library().fno_block_execute(self._h, _ptr(x), _weight_ptr(w), _ptr(w_pw),
                                                _ptr(bias), act, _ptr(y), wp, wn,
                                                _stream(stream)), "fno_block_execute")
        return y

    def fno_plan_backward(self, x, w, gy, gx=None, gw=None, workspace=None, stream=None):
        """dL/dx into gx and dL/dRe(w) + i dL/dIm(w) into gw (either may be None)
        from gy = dL/dy; see include/fnospec.h."""
        wp, wn = self._ws(workspace)
        _check(load_library().fno_plan_backward(
            self._h, _ptr(x), None if w is None else _weight_ptr(w), _ptr(gy), _ptr(gx),
            None if gw is None else _weight_ptr(gw), wp, wn, _stream(stream)),
            "fno_plan_backward")
        return gx, gw

    def fno_plan_record_events(self, events):
        """Arm per-kernel timing with a list of launches + 1 torch.cuda.Event
        (created with enable_timing=True and already recorded once so that the
        underlying CUDA event exists), or disarm with None."""
        lib = load_library()
        if events is None:
            self._event_array = None
            _check(lib.fno_plan_record_events(self._h, None, 0), "fno_plan_record_events")
            return
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        self._event_array = arr  # keep alive while armed
        _check(lib.fno_plan_record_events(self._h, arr, len(events)), "fno_plan_record_events")

    def fno_plan_debug_force_timeout(self, enable: bool):
        """Test hook: make this plan's bounded device waits give up at once
        (see include/fnospec.h)."""
        _check(load_library().fno_plan_debug_force_timeout(self._h, 1 if enable else 0),
               "fno_plan_debug_force_timeout")

    def fno_plan_set_single_launch(self, enable: bool):
        """Run execute as one cooperative launch (True) or three (False); the
        launch count, kernel list and description follow."""
        lib = load_library()
        _check(lib.fno_plan_set_single_launch(self._h, 1 if enable else 0),
               "fno_plan_set_single_launch")
        self._describe()

    def fno_get_device_status(self, stream=None) -> int:
        return int(load_library().fno_get_device_status(self._h, _stream(stream)))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load_library().fno_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Plan1d(Plan):
    """fno_plan_create_1d owner: the 1D layer over x float32 [B, Cin, L] with
    w complex64 [Cin, Cout, m] and y float32 [B, Cout, L]; every Plan method
    applies (execute, stages, backward, block epilogue)."""

    def __init__(self, B, Cin, Cout, L, m, precision="fp32", allocate_workspace=True):
        h = ctypes.c_void_p()
        _check(load_library().fno_plan_create_1d(ctypes.byref(h), B, Cin, Cout, L, m,
                                                 _precision(precision)), "fno_plan_create_1d")
        self._setup(h, (B, Cin, Cout, L, m), precision, allocate_workspace)


def fno_spectral_conv2d(x, w, y, B, Cin, Cout, H, W, m1, m2, stream=None):
    """One-shot call with the exact C signature (fp32 path, cached plan)."""
    _check(load_library().fno_spectral_conv2d(_ptr(x), _weight_ptr(w), _ptr(y), B, Cin, Cout, H,
                                              W, m1, m2, _stream(stream)), "fno_spectral_conv2d")
    return y


def fno_spectral_conv2d_noalloc(x, w, y, B, Cin, Cout, H, W, m1, m2, stream=None):
    """The layer without any device allocation (static scratch inside the
    library, small shapes only); see include/fnospec.h."""
    _check(load_library().fno_spectral_conv2d_noalloc(_ptr(x), _weight_ptr(w), _ptr(y), B, Cin,
                                                      Cout, H, W, m1, m2, _stream(stream)),
           "fno_spectral_conv2d_noalloc")
    return y


def spectral_conv2d(x: torch.Tensor, w: torch.Tensor, m1: int, m2: int, out=None, stream=None):
    """Convenience wrapper: shapes from the tensors, allocates y if needed."""
    B, Cin, H, W = x.shape
    Cout = w.shape[1]
    if out is None:
        out = torch.empty((B, Cout, H, W), dtype=torch.float32, device=x.device)
    return fno_spectral_conv2d(x, w, out, B, Cin, Cout, H, W, m1, m2, stream)


_autograd_plans = {}


def _autograd_plan(B, Cin, Cout, H, W, m1, m2, device):
    key = (B, Cin, Cout, H, W, m1, m2, device)
    plan = _autograd_plans.get(key)
    if plan is None:
        with torch.cuda.device(device):
            plan = Plan(B, Cin, Cout, H, W, m1, m2)
        _autograd_plans[key] = plan
    return plan


def _autograd_plan_1d(B, Cin, Cout, L, m, device):
    key = ("1d", B, Cin, Cout, L, m, device)
    plan = _autograd_plans.get(key)
    if plan is None:
        with torch.cuda.device(device):
            plan = Plan1d(B, Cin, Cout, L, m)
        _autograd_plans[key] = plan
    return plan


class SpectralConv2dFunction(torch.autograd.Function):
    """y = layer(x, w) with gradients for x (float32 [B, Cin, H, W]) and w
    (complex64 [Cin, Cout, 2*m1, m2]) through fno_plan_execute and
    fno_plan_backward.  Plans are cached per (shape, device); calls with the
    same shape share the plan's workspace and run on the current stream."""

    @staticmethod
    def forward(ctx, x, w, m1, m2):
        B, Cin, H, W = x.shape
        Cout = w.shape[1]
        plan = _autograd_plan(B, Cin, Cout, H, W, m1, m2, x.device.index)
        y = torch.empty((B, Cout, H, W), dtype=torch.float32, device=x.device)
        plan.fno_plan_execute(x, w, y)
        ctx.save_for_backward(x, w)
        ctx.plan = plan
        return y

    @staticmethod
    def backward(ctx, gy):
        x, w = ctx.saved_tensors
        gy = gy.contiguous()
        gx = torch.empty_like(x) if ctx.needs_input_grad[0] else None
        gw = torch.empty_like(w) if ctx.needs_input_grad[1] else None
        if gx is None and gw is None:
            return None, None, None, None
        ctx.plan.fno_plan_backward(x, w, gy, gx, gw)
        return gx, gw, None, None


def spectral_conv2d_autograd(x: torch.Tensor, w: torch.Tensor, m1: int, m2: int):
    """Differentiable layer (see SpectralConv2dFunction)."""
    return SpectralConv2dFunction.apply(x, w, m1, m2)


class SpectralConv1dFunction(torch.autograd.Function):
    """The 1D layer with gradients for x (float32 [B, Cin, L]) and w
    (complex64 [Cin, Cout, m]); plans cached per (shape, device) as for
    SpectralConv2dFunction."""

    @staticmethod
    def forward(ctx, x, w, m):
        B, Cin, L = x.shape
        Cout = w.shape[1]
        plan = _autograd_plan_1d(B, Cin, Cout, L, m, x.device.index)
        y = torch.empty((B, Cout, L), dtype=torch.float32, device=x.device)
        plan.fno_plan_execute(x, w, y)
        ctx.save_for_backward(x, w)
        ctx.plan = plan
        return y

    @staticmethod
    def backward(ctx, gy):
        x, w = ctx.saved_tensors
        gy = gy.contiguous()
        gx = torch.empty_like(x) if ctx.needs_input_grad[0] else None
        gw = torch.empty_like(w) if ctx.needs_input_grad[1] else None
        if gx is None and gw is None:
            return None, None, None
        ctx.plan.fno_plan_backward(x, w, gy, gx, gw)
        return gx, gw, None


def spectral_conv1d_autograd(x: torch.Tensor, w: torch.Tensor, m: int):
    """Differentiable 1D layer (see SpectralConv1dFunction)."""
    return SpectralConv1dFunction.apply(x, w, m)


def fno_release_cache():
    _check(load_library().fno_release_cache(), "fno_release_cache")
