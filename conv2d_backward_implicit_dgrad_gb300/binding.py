"""ctypes binding over libdgrad_gb300.so (the C ABI in include/dgrad.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  If the library is missing or cannot be loaded, every call raises:
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_LOCK = threading.Lock()
_LIB = None

# dgrad_status_t
STATUS = {
    0: "DGRAD_OK", 1: "DGRAD_ERR_INVALID_ARG", 2: "DGRAD_ERR_UNSUPPORTED", 3: "DGRAD_ERR_MISALIGNED",
    4: "DGRAD_ERR_ALIAS", 5: "DGRAD_ERR_OOM", 6: "DGRAD_ERR_CUDA", 7: "DGRAD_ERR_DEVICE_TIMEOUT",
    8: "DGRAD_ERR_NO_DEVICE", 9: "DGRAD_ERR_WRONG_DEVICE",
}
PREC = {"fp32": 0, "tf32": 1, "tf32x3": 2}
PATH = {"auto": 0, "simt": 1, "tcgen05": 2, "col2im": 3}
PATH_NAME = {v: k for k, v in PATH.items()}

# Every function declared in include/dgrad.h (checked by the CPU tests).
EXPORTS = ("dgrad_plan", "dgrad_plan_ex", "dgrad_describe", "dgrad_describe_taps", "dgrad_plan_info", "dgrad_run",
           "dgrad_run_fused", "dgrad_prepack", "dgrad_run_packed", "dgrad_pack_grad_out", "dgrad_run_main", "dgrad_run_host", "dgrad_run_noalloc", "dgrad_plan_check",
           "dgrad_plan_destroy", "dgrad_status_string", "dgrad_cuda_error_string",
           "wgrad_describe", "wgrad_describe_taps", "wgrad_describe_run", "wgrad_plan", "wgrad_plan_ex", "wgrad_plan_info",
           "wgrad_run", "wgrad_plan_check", "wgrad_plan_destroy", "dgrad_probe_ffma")


class Options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("tile_blocks", ctypes.c_int), ("slice_n", ctypes.c_int),
                ("chunk_k", ctypes.c_int), ("grid", ctypes.c_int), ("sm_count", ctypes.c_int),
                ("a_source", ctypes.c_int), ("group_taps", ctypes.c_int), ("b_stages", ctypes.c_int),
                ("timeout_us", ctypes.c_int), ("wait_test", ctypes.c_int)]


class WgradPlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("N", "Ci", "H", "W", "Co", "kH", "kW", "stride", "pad_h", "pad_w",
                                            "oH", "oW", "precision", "interleave", "mode", "Wf", "Kimg", "Lx",
                                            "n_copies",
                                            "seg_rows",
                                            "n_mt", "n_nt", "n_ks", "slice_n", "n_units", "grid", "stages",
                                            "smem_bytes", "tmem_cols")] + [
        ("workspace_bytes", ctypes.c_size_t), ("useful_flops", ctypes.c_double),
        ("algorithmic_bytes", ctypes.c_double)]

    def as_dict(self):
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["precision"] = {0: "fp32", 1: "tf32", 2: "tf32x3"}.get(d["precision"], d["precision"])
        return d


class WgradOptions(ctypes.Structure):
    _fields_ = [("timeout_us", ctypes.c_int), ("wait_test", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("N", "Ci", "H", "W", "Co", "kH", "kW", "stride", "pad_h", "pad_w",
                                            "oH", "oW", "precision", "path", "n_phases", "n_taps",
                                            "Ph", "Pw", "Hv", "Wp")] + [
        ("positions", ctypes.c_longlong), ("max_shift", ctypes.c_int),
        ("tile_blocks", ctypes.c_int), ("slice_n", ctypes.c_int), ("n_slices", ctypes.c_int),
        ("chunk_k", ctypes.c_int), ("n_chunks", ctypes.c_int), ("n_work", ctypes.c_longlong),
        ("grid", ctypes.c_int), ("b_resident", ctypes.c_int), ("a_source", ctypes.c_int),
        ("smem_bytes", ctypes.c_int),
        ("tmem_cols", ctypes.c_int), ("group_taps", ctypes.c_int), ("tile_step", ctypes.c_int),
        ("a_stages", ctypes.c_int), ("b_stages", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
        ("packed_weight_bytes", ctypes.c_size_t), ("useful_flops", ctypes.c_double),
        ("algorithmic_bytes", ctypes.c_double), ("band_rows", ctypes.c_int), ("stg_box", ctypes.c_int),
        ("img_tiles", ctypes.c_int), ("a_rows", ctypes.c_int)]

    def as_dict(self):
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["path"] = PATH_NAME.get(d["path"], d["path"])
        d["a_source"] = A_SOURCE_NAME.get(d["a_source"], d["a_source"])
        d["precision"] = {0: "fp32", 1: "tf32", 2: "tf32x3"}.get(d["precision"], d["precision"])
        return d


class DgradError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        name = STATUS.get(status, str(status))
        msg = f"{where}: {name}" if where else name
        if _LIB is not None:
            msg += f" ({_LIB.dgrad_status_string(status).decode()})"
            if status == 6:
                msg += f": {_LIB.dgrad_cuda_error_string().decode()}"
        super().__init__(msg)


def load_library(path: str | None = None):
    """Load (building if needed and possible) libdgrad_gb300.so."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        if path is None:
            path = _build.LIB
            if not _build.up_to_date():
                try:
                    _build.build()
                except Exception as e:  # no toolchain: fail loudly, never fall back
                    if not os.path.exists(path):
                        raise RuntimeError(f"libdgrad_gb300.so is missing and could not be built: {e}") from e
        lib = ctypes.CDLL(path)
        i, p, vp = ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        shape = [i] * 10
        lib.dgrad_plan.argtypes = shape + [i, ctypes.POINTER(vp)]
        lib.dgrad_plan_ex.argtypes = shape + [i, ctypes.POINTER(Options), ctypes.POINTER(vp)]
        lib.dgrad_describe.argtypes = shape + [i, ctypes.POINTER(Options), ctypes.POINTER(PlanInfo)]
        lib.dgrad_describe_taps.argtypes = shape + [i, p, ctypes.POINTER(i), p, ctypes.POINTER(i)]
        lib.dgrad_plan_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        lib.dgrad_run.argtypes = [vp, p, p, p, vp]
        lib.dgrad_run_fused.argtypes = [vp, p, p, p, p, i, vp]
        lib.dgrad_prepack.argtypes = [vp, p, vp]
        lib.dgrad_run_packed.argtypes = [vp, p, p, vp]
        lib.dgrad_pack_grad_out.argtypes = [vp, p, vp]
        lib.dgrad_run_main.argtypes = [vp, p, p, vp]
        lib.dgrad_run_host.argtypes = [vp, p, p, p, vp]
        lib.dgrad_plan_check.argtypes = [vp]
        lib.dgrad_plan_destroy.argtypes = [vp]
        lib.dgrad_plan_destroy.restype = None
        lib.dgrad_status_string.argtypes = [i]
        lib.dgrad_status_string.restype = ctypes.c_char_p
        lib.dgrad_cuda_error_string.argtypes = []
        lib.dgrad_cuda_error_string.restype = ctypes.c_char_p
        lib.wgrad_describe.argtypes = shape + [i, i, ctypes.POINTER(WgradPlanInfo)]
        lib.wgrad_describe_taps.argtypes = shape + [i, p, p, p, p, ctypes.POINTER(i), ctypes.POINTER(i)]
        lib.wgrad_plan.argtypes = shape + [i, ctypes.POINTER(vp)]
        lib.wgrad_plan_ex.argtypes = shape + [i, ctypes.POINTER(WgradOptions), ctypes.POINTER(vp)]
        lib.wgrad_plan_info.argtypes = [vp, ctypes.POINTER(WgradPlanInfo)]
        lib.wgrad_run.argtypes = [vp, p, p, p, vp]
        lib.wgrad_plan_check.argtypes = [vp]
        lib.wgrad_plan_destroy.argtypes = [vp]
        lib.wgrad_plan_destroy.restype = None
        lib.dgrad_probe_ffma.argtypes = [i, i, p, vp]
        lib.dgrad_probe_ffma.restype = i
        for f in ("wgrad_describe", "wgrad_describe_taps", "wgrad_plan", "wgrad_plan_ex", "wgrad_plan_info",
                  "wgrad_run", "wgrad_plan_check"):
            getattr(lib, f).restype = i
        for f in ("dgrad_plan", "dgrad_plan_ex", "dgrad_describe", "dgrad_describe_taps", "dgrad_plan_info",
                  "dgrad_run", "dgrad_run_fused", "dgrad_prepack", "dgrad_run_packed", "dgrad_pack_grad_out", "dgrad_run_main",
                  "dgrad_run_host", "dgrad_plan_check"):
            getattr(lib, f).restype = i
        _LIB = lib
        return lib


A_SOURCE = {"auto": 0, "frame": 1, "producers": 2, "staged": 3, "tmem": 4}
A_SOURCE_NAME = {v: k for k, v in A_SOURCE.items()}


GROUP_TAPS = {"auto": 0, "on": 1, "rows": 1, "off": 2, "phases": 3}


def _options(path="auto", tile_blocks=0, slice_n=0, chunk_k=0, grid=0, sm_count=0, a_source="auto",
             group_taps="auto", b_stages=0, timeout_us=0, wait_test=0):
    return Options(PATH[path] if isinstance(path, str) else int(path), tile_blocks, slice_n, chunk_k, grid,
                   sm_count, A_SOURCE[a_source] if isinstance(a_source, str) else int(a_source),
                   GROUP_TAPS[group_taps] if isinstance(group_taps, str) else int(group_taps), int(b_stages),
                   int(timeout_us), int(wait_test))


def describe(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision="tf32", **opts) -> dict:
    """Host-only planning decisions (no GPU needed)."""
    lib = load_library()
    info = PlanInfo()
    o = _options(**opts)
    st = lib.dgrad_describe(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, PREC[precision], ctypes.byref(o),
                            ctypes.byref(info))
    if st != 0:
        raise DgradError(st, "dgrad_describe")
    return info.as_dict()


def describe_taps(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w):
    """Host-only phase and tap tables: (phases, taps) as lists of dicts."""
    lib = load_library()
    cap = 256
    ph = (ctypes.c_int * (7 * cap))()
    tp = (ctypes.c_int * (3 * cap))()
    nph, ntp = ctypes.c_int(), ctypes.c_int()
    st = lib.dgrad_describe_taps(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, cap, ph, ctypes.byref(nph), tp,
                                 ctypes.byref(ntp))
    if st != 0:
        raise DgradError(st, "dgrad_describe_taps")
    phases = [dict(zip(("a", "b", "Hq", "Wq", "tap_begin", "tap_count", "row_len"), ph[7 * i:7 * i + 7]))
              for i in range(nph.value)]
    taps = [dict(zip(("kh", "kw", "shift"), tp[3 * i:3 * i + 3])) for i in range(ntp.value)]
    return phases, taps


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


class Plan:
    """A dgrad plan bound to the current CUDA device.

    Plan(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision="tf32" | "tf32x3" | "fp32", path=..., ...)
    plan.run(grad_out, weight, grad_input=None, stream=None) -> grad_input (device tensors)
    plan.prepack(weight); plan.run_packed(grad_out, grad_input=None) -> the two halves of run
    plan.run_host(grad_out, weight, grad_input) -> grad_input (host tensors; synchronous)
    """

    def __init__(self, N, Ci, H, W, Co, kH, kW, stride=1, pad_h=0, pad_w=0, precision="tf32", **opts):
        self._lib = load_library()
        self._h = ctypes.c_void_p()
        self.args = (N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w)
        self.precision = precision
        o = _options(**opts)
        st = self._lib.dgrad_plan_ex(*self.args, PREC[precision], ctypes.byref(o), ctypes.byref(self._h))
        if st != 0:
            raise DgradError(st, "dgrad_plan")
        info = PlanInfo()
        self._lib.dgrad_plan_info(self._h, ctypes.byref(info))
        self.info = info.as_dict()
        self.oH, self.oW = self.info["oH"], self.info["oW"]

    @property
    def go_shape(self):
        N, Ci, H, W, Co = self.args[:5]
        return (N, Co, self.oH, self.oW)

    @property
    def gi_shape(self):
        N, Ci, H, W = self.args[:4]
        return (N, Ci, H, W)

    @property
    def w_shape(self):
        N, Ci, H, W, Co, kH, kW = self.args[:7]
        return (Co, Ci, kH, kW)

    def _check_tensor(self, t, shape, name, device):
        import torch
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32, got {t.dtype}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if device == "cuda" and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if device == "cpu" and t.is_cuda:
            raise ValueError(f"{name} must be a CPU tensor")

    def run(self, grad_out, weight, grad_input=None, stream=None, relu_in=None, accumulate=False):
        """grad_input = (accumulate ? grad_input : 0) + (relu_in > 0 if given) * dgrad."""
        import torch
        self._check_tensor(grad_out, self.go_shape, "grad_out", "cuda")
        self._check_tensor(weight, self.w_shape, "weight", "cuda")
        if grad_input is None:
            if accumulate:
                raise ValueError("accumulate needs grad_input")
            grad_input = torch.empty(self.gi_shape, dtype=torch.float32, device=grad_out.device)
        self._check_tensor(grad_input, self.gi_shape, "grad_input", "cuda")
        if relu_in is None and not accumulate:
            st = self._lib.dgrad_run(self._h, ctypes.c_void_p(grad_out.data_ptr()),
                                     ctypes.c_void_p(weight.data_ptr()), ctypes.c_void_p(grad_input.data_ptr()),
                                     _stream_handle(stream))
            where = "dgrad_run"
        else:
            if relu_in is not None:
                self._check_tensor(relu_in, self.gi_shape, "relu_in", "cuda")
            st = self._lib.dgrad_run_fused(
                self._h, ctypes.c_void_p(grad_out.data_ptr()), ctypes.c_void_p(weight.data_ptr()),
                ctypes.c_void_p(grad_input.data_ptr()),
                ctypes.c_void_p(relu_in.data_ptr() if relu_in is not None else 0), 1 if accumulate else 0,
                _stream_handle(stream))
            where = "dgrad_run_fused"
        if st != 0:
            raise DgradError(st, where)
        return grad_input

    def prepack(self, weight, stream=None):
        """Pack `weight` into the plan's workspace (first half of run)."""
        self._check_tensor(weight, self.w_shape, "weight", "cuda")
        st = self._lib.dgrad_prepack(self._h, ctypes.c_void_p(weight.data_ptr()), _stream_handle(stream))
        if st != 0:
            raise DgradError(st, "dgrad_prepack")

    def run_packed(self, grad_out, grad_input=None, stream=None):
        """Main kernel on the weights packed last (second half of run)."""
        import torch
        self._check_tensor(grad_out, self.go_shape, "grad_out", "cuda")
        if grad_input is None:
            grad_input = torch.empty(self.gi_shape, dtype=torch.float32, device=grad_out.device)
        self._check_tensor(grad_input, self.gi_shape, "grad_input", "cuda")
        st = self._lib.dgrad_run_packed(self._h, ctypes.c_void_p(grad_out.data_ptr()),
                                        ctypes.c_void_p(grad_input.data_ptr()), _stream_handle(stream))
        if st != 0:
            raise DgradError(st, "dgrad_run_packed")
        return grad_input

    def pack_grad_out(self, grad_out, stream=None):
        """Pack grad_out into the plan's frame (frame path; no-op otherwise)."""
        self._check_tensor(grad_out, self.go_shape, "grad_out", "cuda")
        st = self._lib.dgrad_pack_grad_out(self._h, ctypes.c_void_p(grad_out.data_ptr()), _stream_handle(stream))
        if st != 0:
            raise DgradError(st, "dgrad_pack_grad_out")

    def run_main(self, grad_out, grad_input=None, stream=None):
        """The main kernel alone, on the weights and frame packed last."""
        import torch
        self._check_tensor(grad_out, self.go_shape, "grad_out", "cuda")
        if grad_input is None:
            grad_input = torch.empty(self.gi_shape, dtype=torch.float32, device=grad_out.device)
        self._check_tensor(grad_input, self.gi_shape, "grad_input", "cuda")
        st = self._lib.dgrad_run_main(self._h, ctypes.c_void_p(grad_out.data_ptr()),
                                      ctypes.c_void_p(grad_input.data_ptr()), _stream_handle(stream))
        if st != 0:
            raise DgradError(st, "dgrad_run_main")
        return grad_input

    def run_host(self, grad_out, weight, grad_input=None, stream=None):
        import torch
        self._check_tensor(grad_out, self.go_shape, "grad_out", "cpu")
        self._check_tensor(weight, self.w_shape, "weight", "cpu")
        if grad_input is None:
            grad_input = torch.empty(self.gi_shape, dtype=torch.float32, pin_memory=True)
        self._check_tensor(grad_input, self.gi_shape, "grad_input", "cpu")
        st = self._lib.dgrad_run_host(self._h, ctypes.c_void_p(grad_out.data_ptr()),
                                      ctypes.c_void_p(weight.data_ptr()), ctypes.c_void_p(grad_input.data_ptr()),
                                      _stream_handle(stream))
        if st != 0:
            raise DgradError(st, "dgrad_run_host")
        return grad_input

    def check(self):
        """Raise if a kernel of this plan recorded an error (call after synchronising)."""
        st = self._lib.dgrad_plan_check(self._h)
        if st != 0:
            raise DgradError(st, "dgrad_plan_check")

    def close(self):
        if self._h:
            self._lib.dgrad_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def dgrad(grad_out, weight, H, W, stride=1, pad_h=0, pad_w=0, precision="tf32", **opts):
    """One-shot convenience: plan, run on the current stream, return grad_input."""
    import torch
    N, Co, oH, oW = grad_out.shape
    _, Ci, kH, kW = weight.shape
    with Plan(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision, **opts) as p:
        out = p.run(grad_out, weight)
        torch.cuda.current_stream().synchronize()
        return out


# ---------------------------------------------------------------- weight gradient
def wgrad_describe(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision="tf32", sm_count=0) -> dict:
    """Host-only planning decisions of the weight gradient (no GPU needed)."""
    lib = load_library()
    info = WgradPlanInfo()
    st = lib.wgrad_describe(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, PREC[precision], sm_count,
                            ctypes.byref(info))
    if st != 0:
        raise DgradError(st, "wgrad_describe")
    return info.as_dict()


def wgrad_describe_taps(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w) -> dict:
    """Host-only tap table of the weight gradient: per tap (kh*kW + kw) the input
    copy and K offset it reads; per input copy its row phase, column phase and
    column shift; the copies' leading zero rows and columns; the number of
    images interleaved along K."""
    lib = load_library()
    cap = 1024
    cp, off = (ctypes.c_int * cap)(), (ctypes.c_int * cap)()
    crh, crw, csh = (ctypes.c_int * cap)(), (ctypes.c_int * cap)(), (ctypes.c_int * cap)()
    nc, ty, tu, f = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    st = lib.wgrad_describe_taps(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, cap, cp, off, crh, crw, csh,
                                 ctypes.byref(nc), ctypes.byref(ty), ctypes.byref(tu), ctypes.byref(f))
    if st != 0:
        raise DgradError(st, "wgrad_describe_taps")
    taps, n = kH * kW, nc.value
    return {"copy": list(cp[:taps]), "offset": list(off[:taps]), "copy_rh": list(crh[:n]),
            "copy_rw": list(crw[:n]), "copy_shift": list(csh[:n]), "Ty": ty.value, "Tu": tu.value,
            "interleave": f.value}


def wgrad_describe_run(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, sm_count=0):
    """Host-only run-mode table of the weight gradient (None when the shape
    runs the segment mode): tap groups, tiles, stage length and tiles per unit."""
    lib = load_library()
    cap = 1024
    hdr = (ctypes.c_int * 15)()
    grp, taps, tiles = (ctypes.c_int * (6 * cap))(), (ctypes.c_int * cap)(), (ctypes.c_int * (2 * cap))()
    st = lib.wgrad_describe_run(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, sm_count, cap, hdr, grp, taps,
                                   tiles)
    if st == 2:
        return None
    if st != 0:
        raise DgradError(st, "wgrad_describe_run")
    keys = ("n_groups", "n_tiles", "spt", "seg_rows", "stages", "Pg", "Px", "cps", "nksq", "cpt", "n_nt", "Q", "L",
            "tpu", "n_sets")
    d = dict(zip(keys, hdr[:15]))
    d["groups"] = [dict(zip(("copy", "base", "n_taps", "n_mt", "unused", "tap0"), grp[6 * i:6 * i + 6]))
                   for i in range(d["n_groups"])]
    d["taps"] = list(taps[:kH * kW])
    d["tiles"] = [(tiles[2 * t], tiles[2 * t + 1]) for t in range(d["n_tiles"])]
    return d


class WgradPlan:
    """A weight-gradient plan bound to the current CUDA device.

    WgradPlan(N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w, precision="tf32", timeout_us=0, wait_test=0)
    plan.run(grad_out, input, grad_weight=None, stream=None) -> grad_weight [Co, Ci, kH, kW]
    (timeout_us, wait_test: the in-kernel wait limit and the failure-detection test hook, see wgrad.h)
    """

    def __init__(self, N, Ci, H, W, Co, kH, kW, stride=1, pad_h=0, pad_w=0, precision="tf32", timeout_us=0,
                 wait_test=0):
        self._lib = load_library()
        self._h = ctypes.c_void_p()
        self.args = (N, Ci, H, W, Co, kH, kW, stride, pad_h, pad_w)
        opts = WgradOptions(timeout_us, wait_test)
        st = self._lib.wgrad_plan_ex(*self.args, PREC[precision], ctypes.byref(opts), ctypes.byref(self._h))
        if st != 0:
            raise DgradError(st, "wgrad_plan")
        info = WgradPlanInfo()
        self._lib.wgrad_plan_info(self._h, ctypes.byref(info))
        self.info = info.as_dict()
        oH, oW = self.info["oH"], self.info["oW"]
        self.go_shape = (N, Co, oH, oW)
        self.x_shape = (N, Ci, H, W)
        self.w_shape = (Co, Ci, kH, kW)

    def run(self, grad_out, input, grad_weight=None, stream=None):
        import torch
        for t, shape, name in ((grad_out, self.go_shape, "grad_out"), (input, self.x_shape, "input")):
            if tuple(t.shape) != shape or t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
                raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape {shape}")
        if grad_weight is None:
            grad_weight = torch.empty(self.w_shape, dtype=torch.float32, device=grad_out.device)
        if (tuple(grad_weight.shape) != self.w_shape or grad_weight.dtype != torch.float32
                or not grad_weight.is_contiguous() or not grad_weight.is_cuda):
            raise ValueError(f"grad_weight must be a contiguous float32 CUDA tensor of shape {self.w_shape}")
        st = self._lib.wgrad_run(self._h, ctypes.c_void_p(grad_out.data_ptr()), ctypes.c_void_p(input.data_ptr()),
                                 ctypes.c_void_p(grad_weight.data_ptr()), _stream_handle(stream))
        if st != 0:
            raise DgradError(st, "wgrad_run")
        return grad_weight

    def check(self):
        st = self._lib.wgrad_plan_check(self._h)
        if st != 0:
            raise DgradError(st, "wgrad_plan_check")

    def close(self):
        if self._h:
            self._lib.wgrad_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
