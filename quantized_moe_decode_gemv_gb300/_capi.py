"""ctypes binding of the C ABI in include/moe_layer.h.

Argument marshalling only: every step of the layer runs in the CUDA library.
PyTorch is used for device memory and streams.  If the shared library has not
been built this module raises on import -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Any, Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_CHECKS=1: the debug build (kernel index checks, NVTX ranges)
LIB_NAME = "libmoe_gb300_checks.so" if os.environ.get("MOE_CHECKS") == "1" else "libmoe_gb300.so"
LIB_PATH = os.path.join(_HERE, LIB_NAME)

# enums (include/moe_layer.h)
MOE_OK = 0
STATUS_NAMES = ["MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_TOPK_GT_E",
                "MOE_ERR_LATENT_PROJ", "MOE_ERR_SHAPE", "MOE_ERR_DEVICE", "MOE_ERR_OOM",
                "MOE_ERR_CUDA", "MOE_ERR_TIMEOUT", "MOE_ERR_NONFINITE", "MOE_ERR_INDEX"]
ACT = {"swiglu": 0, "relu2": 1}
ROUTER = {"softmax": 0, "sigmoid": 1}
DTYPE = {"bf16": 0, "fp16": 1, "fp32": 2}
WFMT = {"affine": 0, "nvfp4": 1, "mxfp4": 2}
PATH = {"auto": 0, "gemv": 1, "grouped": 2}
NUM_STAGES = 5
STAGE_NAMES = ["dense_in", "route", "expert_up", "expert_down", "dense_out"]


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{name}: {message}")


class moe_layer_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("expert_ffn", ctypes.c_int32),
                ("latent", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("shared_ffn", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("act", ctypes.c_int32), ("router", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("routed_scale", ctypes.c_float),
                ("has_router_bias", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("scale_dtype", ctypes.c_int32), ("router_dtype", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("weight_format", ctypes.c_int32)]


_WEIGHT_FIELDS = ["router_w", "router_bias", "fc1_latent", "fc2_latent", "gate_q", "up_q",
                  "down_q", "gate_s", "gate_b", "up_s", "up_b", "down_s", "down_b", "sh_gate",
                  "sh_up", "sh_down"]


class moe_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _WEIGHT_FIELDS]


# symbol -> (restype, argtypes)
SIGNATURES = {
    "moe_abi_version": (ctypes.c_int32, []),
    "moe_build_flags": (ctypes.c_int32, []),
    "moe_layer_validate": (ctypes.c_int, [ctypes.POINTER(moe_layer_config),
                                          ctypes.POINTER(moe_layer_weights)]),
    "moe_layer_create": (ctypes.c_int, [ctypes.POINTER(moe_layer_config),
                                        ctypes.POINTER(moe_layer_weights), ctypes.c_void_p,
                                        ctypes.POINTER(ctypes.c_void_p)]),
    "moe_layer_forward": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_forward_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_forward_host": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                              ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_set_path": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "moe_layer_device_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_profile": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "moe_layer_stage_times": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_float),
                                             ctypes.c_int32]),
    "moe_layer_path_for": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_int32]),
    "moe_layer_last_launch_count": (ctypes.c_int32, [ctypes.c_void_p]),
    "moe_layer_device_bytes": (ctypes.c_int64, [ctypes.c_void_p]),
    "moe_layer_destroy": (ctypes.c_int, [ctypes.c_void_p]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_layer_last_error": (ctypes.c_char_p, [ctypes.c_void_p]),
    "moe_router_topk_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                               ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_void_p]),
    "moe_debug_live_allocations": (ctypes.c_int64, []),
    "moe_debug_fail_allocation": (None, [ctypes.c_int32]),
}

_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (built by ``build.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{LIB_NAME} is not built (expected at {path}); run "
                           "quantized_moe_decode_gemv_gb300.build.build() first -- the layer "
                           "has no CPU implementation")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _last_error(handle=None) -> str:
    msg = load_library().moe_layer_last_error(handle)
    return msg.decode() if msg else ""


def _check(status: int, handle=None):
    if status != MOE_OK:
        raise MoEError(status, _last_error(handle))


@dataclasses.dataclass
class MoEConfig:
    """Python mirror of ``moe_layer_config``."""
    hidden: int
    n_experts: int
    top_k: int
    expert_ffn: int
    latent: int = 0
    group_size: int = 64
    shared_ffn: int = 0
    max_tokens: int = 16
    act: str = "swiglu"
    router: str = "softmax"
    renormalize: bool = True
    routed_scale: float = 1.0
    router_bias: bool = False
    act_dtype: str = "bf16"
    scale_dtype: str = "bf16"
    router_dtype: str = "bf16"
    bits: int = 4
    fmt: str = "affine"          # expert weight format: "affine", "nvfp4" or "mxfp4"

    @classmethod
    def from_spec(cls, spec: Any, max_tokens: int) -> "MoEConfig":
        """Build from any object carrying the same attribute names."""
        kw = {f.name: getattr(spec, f.name) for f in dataclasses.fields(cls)
              if f.name != "max_tokens" and hasattr(spec, f.name)}
        return cls(max_tokens=max_tokens, **kw)

    def to_c(self) -> moe_layer_config:
        return moe_layer_config(
            hidden=self.hidden, n_experts=self.n_experts, top_k=self.top_k,
            expert_ffn=self.expert_ffn, latent=self.latent, group_size=self.group_size,
            shared_ffn=self.shared_ffn, max_tokens=self.max_tokens, act=ACT[self.act],
            router=ROUTER[self.router], renormalize=int(bool(self.renormalize)),
            routed_scale=float(self.routed_scale), has_router_bias=int(bool(self.router_bias)),
            act_dtype=DTYPE[self.act_dtype], scale_dtype=DTYPE[self.scale_dtype],
            router_dtype=DTYPE[self.router_dtype], bits=int(self.bits),
            weight_format=WFMT[self.fmt])


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return int(t.data_ptr())


def weights_struct(weights: Dict[str, Any]) -> moe_layer_weights:
    """``moe_layer_weights`` from a dict of device tensors (missing -> NULL)."""
    return moe_layer_weights(**{n: _ptr(weights.get(n)) for n in _WEIGHT_FIELDS})


# storage-array names of the input generator -> C field names
_ARRAY_TO_FIELD = {"router_w": "router_w", "router_bias": "router_bias", "fc1": "fc1_latent",
                   "fc2": "fc2_latent", "gate_q": "gate_q", "up_q": "up_q", "down_q": "down_q",
                   "gate_s": "gate_s", "gate_b": "gate_b", "up_s": "up_s", "up_b": "up_b",
                   "down_s": "down_s", "down_b": "down_b", "sh_gate": "sh_gate",
                   "sh_up": "sh_up", "sh_down": "sh_down"}


def upload_arrays(arrays: Dict[str, np.ndarray], device="cuda") -> Dict[str, Any]:
    """Copy host arrays (numpy) to device tensors keyed by C field name.  Bit
    patterns are kept as is (uint16 bf16 -> int16 storage, uint32 -> int32)."""
    import torch
    out = {}
    for name, arr in arrays.items():
        field = _ARRAY_TO_FIELD.get(name)
        if field is None or arr is None:
            continue
        a = np.ascontiguousarray(arr)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        elif a.dtype == np.uint32:
            a = a.view(np.int32)
        out[field] = torch.from_numpy(a).to(device)
    return out


def torch_act_dtype(name: str):
    import torch
    return {"bf16": torch.bfloat16, "fp16": torch.float16}[name]


# ---------------------------------------------------------------------------
# thin wrappers with the C names
# ---------------------------------------------------------------------------

def moe_layer_validate(config: MoEConfig, weights: Optional[Dict[str, Any]] = None) -> int:
    lib = load_library()
    c = config.to_c()
    w = ctypes.byref(weights_struct(weights)) if weights is not None else None
    return lib.moe_layer_validate(ctypes.byref(c), w)


def moe_layer_create(config: MoEConfig, weights: Dict[str, Any], stream: int = 0) -> int:
    lib = load_library()
    c = config.to_c()
    w = weights_struct(weights)
    h = ctypes.c_void_p()
    _check(lib.moe_layer_create(ctypes.byref(c), ctypes.byref(w), ctypes.c_void_p(stream),
                                ctypes.byref(h)))
    return h.value


def moe_layer_forward(handle: int, x, T: int, out, stream: int = 0) -> None:
    lib = load_library()
    _check(lib.moe_layer_forward(handle, _ptr(x), T, _ptr(out), ctypes.c_void_p(stream)), handle)


def moe_layer_forward_ex(handle: int, x, T: int, out, stream: int = 0, topk_ids=None,
                         topk_w=None, delta=None) -> None:
    lib = load_library()
    _check(lib.moe_layer_forward_ex(handle, _ptr(x), T, _ptr(out), ctypes.c_void_p(stream),
                                    _ptr(topk_ids), _ptr(topk_w), _ptr(delta)), handle)


def moe_layer_forward_host(handle: int, x_host_ptr: int, T: int, out_host_ptr: int,
                           stream: int = 0) -> None:
    lib = load_library()
    _check(lib.moe_layer_forward_host(handle, ctypes.c_void_p(x_host_ptr), T,
                                      ctypes.c_void_p(out_host_ptr), ctypes.c_void_p(stream)),
           handle)


def moe_layer_set_path(handle: int, path: str) -> None:
    _check(load_library().moe_layer_set_path(handle, PATH[path]), handle)


def moe_layer_device_status(handle: int, stream: int = 0) -> int:
    return load_library().moe_layer_device_status(handle, ctypes.c_void_p(stream))


def moe_router_topk_noalloc(x, T: int, hidden: int, x_dtype: str, router_w, router_dtype: str,
                            router_bias, n_experts: int, top_k: int, router: str,
                            renormalize: bool, routed_scale: float, topk_ids, topk_w,
                            stream: int = 0, key_status=None) -> None:
    """Router gemv + top-k with no device allocation (see include/moe_layer.h).
    ``key_status``: optional device int32 tensor of one element that receives 1
    when a selection key was NaN or infinite, else 0."""
    lib = load_library()
    _check(lib.moe_router_topk_noalloc(_ptr(x), T, hidden, DTYPE[x_dtype], _ptr(router_w),
                                       DTYPE[router_dtype], _ptr(router_bias), n_experts, top_k,
                                       ROUTER[router], int(bool(renormalize)), float(routed_scale),
                                       _ptr(topk_ids), _ptr(topk_w), _ptr(key_status),
                                       ctypes.c_void_p(stream)))


def moe_layer_destroy(handle: int) -> None:
    if handle:
        _check(load_library().moe_layer_destroy(handle))


class MoELayer:
    """One layer handle.  ``weights`` are device tensors keyed by C field name
    (see ``upload_arrays``); they may be freed after construction."""

    def __init__(self, config: MoEConfig, weights: Dict[str, Any], stream: int = 0):
        import torch
        self.config = config
        self.handle = moe_layer_create(config, weights, stream)
        self._torch = torch

    def _stream(self, stream):
        if stream is None:
            return self._torch.cuda.current_stream().cuda_stream
        if hasattr(stream, "cuda_stream"):
            return int(stream.cuda_stream)
        return int(stream)

    def forward(self, x, out=None, stream=None):
        torch = self._torch
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        moe_layer_forward(self.handle, x, T, out, self._stream(stream))
        return out

    __call__ = forward

    def forward_ex(self, x, stream=None):
        """Returns (out, ids [T,k] int32, weights [T,k] fp32, delta [T,H] fp32)."""
        torch = self._torch
        T, k = x.shape[0], self.config.top_k
        out = torch.empty_like(x)
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, k), dtype=torch.float32, device=x.device)
        delta = torch.empty((T, self.config.hidden), dtype=torch.float32, device=x.device)
        moe_layer_forward_ex(self.handle, x, T, out, self._stream(stream), ids, w, delta)
        return out, ids, w, delta

    def forward_host(self, x_host, out_host, stream=None):
        """x_host/out_host: (pinned) host tensors [T, H] of the activation dtype."""
        moe_layer_forward_host(self.handle, x_host.data_ptr(), x_host.shape[0],
                               out_host.data_ptr(), self._stream(stream))
        return out_host

    def set_path(self, path: str):
        moe_layer_set_path(self.handle, path)

    def device_status(self, stream=None) -> int:
        return moe_layer_device_status(self.handle, self._stream(stream))

    def profile(self, enable: bool = True):
        _check(load_library().moe_layer_profile(self.handle, int(enable)), self.handle)

    def stage_times(self):
        """Durations (ms) of the kernel stages of the last profiled forward."""
        buf = (ctypes.c_float * NUM_STAGES)()
        _check(load_library().moe_layer_stage_times(self.handle, buf, NUM_STAGES), self.handle)
        return list(buf)

    def device_bytes(self) -> int:
        return load_library().moe_layer_device_bytes(self.handle)

    def path_for(self, T: int) -> str:
        """The path ("gemv" or "grouped") a forward of T rows takes."""
        v = load_library().moe_layer_path_for(self.handle, int(T))
        if v < 0:
            raise MoEError(f"no path for T={T}")
        return {p: n for n, p in PATH.items()}[v]

    def last_launch_count(self) -> int:
        """Kernel launches of the last forward."""
        return int(load_library().moe_layer_last_launch_count(self.handle))

    def close(self):
        if getattr(self, "handle", None):
            moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
