"""CPU oracle for conv2d backward-data (dgrad).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
CUDA library never loads it and shares no code with it.

The arithmetic lives in ``dgrad_oracle.c`` (plain C, fp64 accumulation), built
with gcc into ``oracle/_build/liboracle.so`` and called through ctypes.  This
module only marshals numpy arrays.

Functions (all return float64 numpy arrays):

* ``dgrad(go, w, H, W, stride, pad_h, pad_w)`` -> ``(acc, mag)``: the
  definition as a direct scatter over grad_out (O1).  ``mag`` is the per-element
  sum of |terms|.
* ``conv2d_fwd(x, w, stride, pad_h, pad_w)``: the forward convolution (O-fwd).
* ``dgrad_gather(...)``: doppler's per-input-element gather (O2).
* ``dgrad_gemm_p1(...)``: meganeura's implicit-GEMM index map (O3).
* ``dgrad_phase(...)``: the sub-pixel phase split (O-phase).
* ``dgrad_at(go, w, H, W, stride, pad_h, pad_w, idx)``: the definition at
  sampled elements.
* ``dgrad_fused(..., relu_in=None, grad_in=None)``: O1 followed by a ReLU
  backward mask and gradient accumulation, composed elementwise in numpy.
* ``wgrad(go, x, stride, pad_h, pad_w)`` -> ``(acc, mag)``: the weight
  gradient dW[co,ci,kh,kw] (O-w), as a direct sum over the batch and grad_out
  positions; ``mag`` the per-element sum of |terms|.

Pins: every function is checked in ``tests/test_oracle.py`` against hand-worked
fixtures, brute-force adjoints, finite differences, the transposed-padding
identity, closed forms and torch's CPU fp64 convolution routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dgrad_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_LOCK = threading.Lock()
_LIB = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, no fast-math) and return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
             "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            lib = ctypes.CDLL(build())
            i, p = ctypes.c_int, ctypes.c_void_p
            shape = [i] * 10
            lib.oracle_dgrad_scatter.argtypes = shape + [p, p, p, p, i]
            lib.oracle_conv2d_fwd.argtypes = shape + [p, p, p]
            lib.oracle_dgrad_gather.argtypes = shape + [p, p, p]
            lib.oracle_dgrad_gemm_p1.argtypes = shape + [p, p, p]
            lib.oracle_dgrad_phase.argtypes = shape + [p, p, p]
            lib.oracle_dgrad_at.argtypes = shape + [p, p, p, ctypes.c_long, p, p]
            lib.oracle_out_extent.argtypes = [i, i, i, i]
            lib.oracle_wgrad.argtypes = shape + [p, p, p, p, i]
            for f in (lib.oracle_dgrad_scatter, lib.oracle_conv2d_fwd, lib.oracle_dgrad_gather,
                      lib.oracle_dgrad_gemm_p1, lib.oracle_dgrad_phase, lib.oracle_dgrad_at,
                      lib.oracle_out_extent, lib.oracle_wgrad):
                f.restype = ctypes.c_int
            _LIB = lib
    return _LIB


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch CPU tensor
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def out_extent(n_in: int, k: int, stride: int, pad: int) -> int:
    """floor((n_in + 2*pad - k)/stride) + 1, or 0 when the window does not fit."""
    return int(_lib().oracle_out_extent(n_in, k, stride, pad))


def _dims(go, w, H, W, stride, pad_h, pad_w):
    N, Co, oH, oW = go.shape
    Co2, Ci, kH, kW = w.shape
    if Co2 != Co:
        raise ValueError(f"grad_out has {Co} channels, weight has {Co2} output channels")
    if (oH, oW) != (out_extent(H, kH, stride, pad_h), out_extent(W, kW, stride, pad_w)):
        raise ValueError("grad_out spatial shape does not match H, W, kernel, stride, padding")
    return N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w


def _check(rc: int):
    if rc != 0:
        raise ValueError("oracle rejected the shape")


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def dgrad(go, w, H: int, W: int, stride: int, pad_h: int, pad_w: int,
          nthreads: int | None = None, with_mag: bool = True):
    """O1 (direct scatter).  Returns (acc, mag) as float64 [N, Ci, H, W]."""
    go, w = _f32(go), _f32(w)
    d = _dims(go, w, H, W, stride, pad_h, pad_w)
    acc = np.empty((d[0], d[1], H, W), np.float64)
    mag = np.empty_like(acc) if with_mag else None
    nt = default_threads() if nthreads is None else nthreads
    _check(_lib().oracle_dgrad_scatter(*d, _ptr(go), _ptr(w), _ptr(acc),
                                       _ptr(mag) if with_mag else None, nt))
    return acc, mag


def conv2d_fwd(x, w, stride: int, pad_h: int, pad_w: int) -> np.ndarray:
    """O-fwd.  x [N, Ci, H, W], w [Co, Ci, kH, kW], both taken as float64."""
    x, w = _f64(x), _f64(w)
    N, Ci, H, W = x.shape
    Co, Ci2, kH, kW = w.shape
    if Ci2 != Ci:
        raise ValueError("channel mismatch")
    oH, oW = out_extent(H, kH, stride, pad_h), out_extent(W, kW, stride, pad_w)
    if oH < 1 or oW < 1:
        raise ValueError("window does not fit")
    y = np.empty((N, Co, oH, oW), np.float64)
    _check(_lib().oracle_conv2d_fwd(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w,
                                    _ptr(x), _ptr(w), _ptr(y)))
    return y


def _single(fn, go, w, H, W, stride, pad_h, pad_w):
    go, w = _f32(go), _f32(w)
    d = _dims(go, w, H, W, stride, pad_h, pad_w)
    acc = np.empty((d[0], d[1], H, W), np.float64)
    _check(fn(*d, _ptr(go), _ptr(w), _ptr(acc)))
    return acc


def dgrad_gather(go, w, H, W, stride, pad_h, pad_w) -> np.ndarray:
    """O2: doppler's per-input-element gather."""
    return _single(_lib().oracle_dgrad_gather, go, w, H, W, stride, pad_h, pad_w)


def dgrad_gemm_p1(go, w, H, W, stride, pad_h, pad_w) -> np.ndarray:
    """O3: meganeura's implicit-GEMM index map (its stride-1 path assumes 'same' padding)."""
    return _single(_lib().oracle_dgrad_gemm_p1, go, w, H, W, stride, pad_h, pad_w)


def dgrad_phase(go, w, H, W, stride, pad_h, pad_w) -> np.ndarray:
    """O-phase: the sub-pixel phase split."""
    return _single(_lib().oracle_dgrad_phase, go, w, H, W, stride, pad_h, pad_w)


def dgrad_at(go, w, H, W, stride, pad_h, pad_w, idx):
    """The definition at sampled elements; idx is an int array [S, 4] of (n, ci, ih, iw)."""
    go, w = _f32(go), _f32(w)
    d = _dims(go, w, H, W, stride, pad_h, pad_w)
    idx = np.ascontiguousarray(idx, dtype=np.int32).reshape(-1, 4)
    acc = np.empty(len(idx), np.float64)
    mag = np.empty(len(idx), np.float64)
    _check(_lib().oracle_dgrad_at(*d, _ptr(go), _ptr(w), _ptr(idx), len(idx), _ptr(acc), _ptr(mag)))
    return acc, mag


def dgrad_fused(go, w, H, W, stride, pad_h, pad_w, relu_in=None, grad_in=None, nthreads=None):
    """O1, then the two elementwise steps of ferrotensor's kernels.wgsl that an
    autograd chain applies to it: section 12 "Relu", relu_backward (the
    gradient passes where the ReLU input is > 0, else 0), and section 20
    "Gradient Accumulation" (grad = grad + new_grad).  Returns (acc, mag):
    acc float64; mag the per-element sum of |terms| of the dgrad part (0 where
    masked), the basis of the TF32 bound."""
    acc, mag = dgrad(go, w, H, W, stride, pad_h, pad_w, nthreads=nthreads)
    if relu_in is not None:
        keep = _f32(relu_in) > np.float32(0.0)
        acc = np.where(keep, acc, 0.0)
        mag = np.where(keep, mag, 0.0)
    if grad_in is not None:
        acc = _f32(grad_in).astype(np.float64) + acc
    return acc, mag


def wgrad(go, x, kH: int, kW: int, stride: int, pad_h: int, pad_w: int, nthreads: int | None = None):
    """O-w: the weight gradient of the convolution whose grad_out is ``go``
    [N, Co, oH, oW] and whose forward input is ``x`` [N, Ci, H, W].  Returns
    (acc, mag) as float64 [Co, Ci, kH, kW]."""
    go, x = _f32(go), _f32(x)
    N, Co, oH, oW = go.shape
    N2, Ci, H, W = x.shape
    if N2 != N:
        raise ValueError("batch mismatch")
    if (oH, oW) != (out_extent(H, kH, stride, pad_h), out_extent(W, kW, stride, pad_w)):
        raise ValueError("grad_out spatial shape does not match H, W, kernel, stride, padding")
    acc = np.empty((Co, Ci, kH, kW), np.float64)
    mag = np.empty_like(acc)
    nt = default_threads() if nthreads is None else nthreads
    _check(_lib().oracle_wgrad(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, _ptr(go), _ptr(x),
                               _ptr(acc), _ptr(mag), nt))
    return acc, mag
