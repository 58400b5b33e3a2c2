"""GB300-native MoE token dispatch + expert GEMM in one persistent kernel.

Thin ctypes binding over the C ABI in ``include/mk.h``: the functions below
carry the C names and only marshal arguments (tensor -> device pointer,
current torch stream -> cudaStream_t).  Every step of the path runs in the
CUDA library ``_build/libmk.so``; there is no CPU fallback.  When the library
is missing every call raises ``MkLibraryMissing`` (build it with
``moe_token_dispatch_persistent_gb300.build.build()``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmk.so")

MK_OK = 0
MK_ERR_INVALID_ARG = 1
MK_ERR_UNSUPPORTED = 2
MK_ERR_CUDA = 3
MK_ERR_TIMEOUT = 4
MK_ERR_DEVICE_FAULT = 5
MK_ERR_NOT_IMPLEMENTED = 6
MK_ERR_WORKSPACE = 7

MK_MODE_FUSED = 0
MK_MODE_UNFUSED = 1
MK_MODE_DISPATCH_ONLY = 2
MK_OUT_BF16 = 0
MK_OUT_F32 = 1
MK_FAULT_NONE = 0
MK_FAULT_DROP_TILE_FLAG = 1
MK_MMA_AUTO = 0
MK_MMA_SINGLE = 1
MK_MMA_PAIR = 2
MK_MMA_WIDE = 3
MK_GATHER_AUTO = 0
MK_GATHER_STAGED = 1
MK_GATHER_DIRECT = 2
MK_GATHER_GATHER4 = 3

# Entry points declared in include/mk.h (checked by the tests).
ABI_FUNCTIONS = (
    "mk_config_default",
    "mk_moe_dispatch_gemm",
    "mk_moe_dispatch_gemm_ex",
    "mk_moe_dispatch_gemm_combine",
    "mk_moe_dispatch_gated",
    "mk_moe_dispatch_gemm_host",
    "mk_moe_dispatch_gemm_noalloc",
    "mk_moe_ep_sim",
    "mk_moe_ep_sim_gated",
    "mk_ep_workspace_size",
    "mk_workspace_size",
    "mk_get_status",
    "mk_last_error_detail",
    "mk_last_launch_info",
    "mk_read_trace",
    "mk_release_workspace",
    "mk_status_string",
    "mk_version",
)


class MkLibraryMissing(RuntimeError):
    pass


class MkError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_name(status)} ({status})")


class mk_config_t(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("dispatch_ctas", ctypes.c_int32),
        ("grid_ctas", ctypes.c_int32),
        ("n_group", ctypes.c_int32),
        ("debug_fault", ctypes.c_int32),
        ("spin_limit_ns", ctypes.c_int64),
        ("trace", ctypes.c_int32),
        ("l2_prefetch", ctypes.c_int32),
        ("mma_pair", ctypes.c_int32),
        ("gather", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 4),
    ]


class mk_launch_info_t(ctypes.Structure):
    _fields_ = [
        ("grid_ctas", ctypes.c_int32),
        ("dispatch_ctas", ctypes.c_int32),
        ("launches", ctypes.c_int32),
        ("n_group", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64),
        ("mma_pair", ctypes.c_int32),
        ("gather", ctypes.c_int32),
        ("route_lanes", ctypes.c_int32),
        ("route_chunks", ctypes.c_int32),
    ]


_lib_handle = None
_p = ctypes.c_void_p
_i = ctypes.c_int


def lib(path: str | None = None) -> ctypes.CDLL:
    """The loaded CUDA library (raises MkLibraryMissing if it was not built)."""
    global _lib_handle
    if _lib_handle is not None and path is None:
        return _lib_handle
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise MkLibraryMissing(f"CUDA library not found at {p}; build it first")
    h = ctypes.CDLL(p)
    h.mk_config_default.argtypes = [ctypes.POINTER(mk_config_t)]
    h.mk_config_default.restype = None
    sig = [_p, _p, _i, _i, _i, _i, _p, _i, _p, _p, _p, _p, _p]
    h.mk_moe_dispatch_gemm.argtypes = sig
    h.mk_moe_dispatch_gemm.restype = _i
    h.mk_moe_dispatch_gemm_ex.argtypes = sig + [ctypes.POINTER(mk_config_t), _p, ctypes.c_size_t]
    h.mk_moe_dispatch_gemm_ex.restype = _i
    h.mk_moe_dispatch_gemm_combine.argtypes = sig[:-1] + [_p, _p, ctypes.POINTER(mk_config_t), _p,
                                                           ctypes.c_size_t]
    h.mk_moe_dispatch_gemm_combine.restype = _i
    h.mk_moe_dispatch_gated.argtypes = [_p, _p, _i, _i, _i, _i, _p, _p, _i, _p, _p, _p, _p, _p,
                                        ctypes.POINTER(mk_config_t), _p, ctypes.c_size_t]
    h.mk_moe_dispatch_gated.restype = _i
    h.mk_moe_dispatch_gemm_host.argtypes = sig + [ctypes.POINTER(mk_config_t)]
    h.mk_moe_dispatch_gemm_host.restype = _i
    h.mk_moe_dispatch_gemm_noalloc.argtypes = sig + [ctypes.POINTER(mk_config_t)]
    h.mk_moe_dispatch_gemm_noalloc.restype = _i
    h.mk_moe_ep_sim.argtypes = [_p, _p, _i, _i, _i, _i, _p, _i, _i, _p, _p, _p, _p, _p, _p,
                                ctypes.POINTER(mk_config_t), _p, ctypes.c_size_t]
    h.mk_moe_ep_sim.restype = _i
    h.mk_moe_ep_sim_gated.argtypes = [_p, _p, _i, _i, _i, _i, _p, _p, _i, _i, _p, _p, _p, _p, _p, _p,
                                      ctypes.POINTER(mk_config_t), _p, ctypes.c_size_t]
    h.mk_moe_ep_sim_gated.restype = _i
    h.mk_ep_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
    h.mk_ep_workspace_size.restype = ctypes.c_size_t
    h.mk_workspace_size.argtypes = [_i, _i, _i, _i, _i, ctypes.POINTER(mk_config_t)]
    h.mk_workspace_size.restype = ctypes.c_size_t
    h.mk_get_status.argtypes = [_p]
    h.mk_get_status.restype = _i
    h.mk_last_error_detail.argtypes = [ctypes.POINTER(ctypes.c_int32)] * 3
    h.mk_last_error_detail.restype = None
    h.mk_last_launch_info.argtypes = [ctypes.POINTER(mk_launch_info_t)]
    h.mk_last_launch_info.restype = None
    h.mk_read_trace.argtypes = [_p, _p, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_uint64), ctypes.c_size_t]
    h.mk_read_trace.restype = _i
    h.mk_release_workspace.argtypes = []
    h.mk_release_workspace.restype = None
    h.mk_status_string.argtypes = [_i]
    h.mk_status_string.restype = ctypes.c_char_p
    h.mk_version.argtypes = []
    h.mk_version.restype = _i
    if path is None:
        _lib_handle = h
    return h


def status_name(s: int) -> str:
    try:
        return lib().mk_status_string(int(s)).decode()
    except MkLibraryMissing:
        return str(s)


# ------------------------------------------------------------ marshalling --

def _ptr(v):
    if v is None:
        return None
    if hasattr(v, "data_ptr"):
        return v.data_ptr() or None
    return int(v) or None


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def _check(status: int, what: str):
    if status != MK_OK:
        raise MkError(status, what)


# ----------------------------------------------------------- C-named calls --

def mk_config_default() -> mk_config_t:
    c = mk_config_t()
    lib().mk_config_default(ctypes.byref(c))
    return c


def mk_version() -> int:
    return int(lib().mk_version())


def mk_status_string(s: int) -> str:
    return lib().mk_status_string(int(s)).decode()


def mk_workspace_size(T, H, F, E, k, cfg: mk_config_t | None = None) -> int:
    return int(lib().mk_workspace_size(T, H, F, E, k, ctypes.byref(cfg) if cfg is not None else None))


def mk_moe_dispatch_gemm(x, logits, T, H, E, k, W, F, y_sorted, src_index, expert_offsets, gate_w, stream=None) -> int:
    return int(lib().mk_moe_dispatch_gemm(_ptr(x), _ptr(logits), T, H, E, k, _ptr(W), F, _ptr(y_sorted),
                                          _ptr(src_index), _ptr(expert_offsets), _ptr(gate_w), _stream(stream)))


def mk_moe_dispatch_gemm_ex(x, logits, T, H, E, k, W, F, y_sorted, src_index, expert_offsets, gate_w, stream=None,
                            cfg: mk_config_t | None = None, workspace=None, ws_bytes: int = 0) -> int:
    return int(lib().mk_moe_dispatch_gemm_ex(_ptr(x), _ptr(logits), T, H, E, k, _ptr(W), F, _ptr(y_sorted),
                                             _ptr(src_index), _ptr(expert_offsets), _ptr(gate_w), _stream(stream),
                                             ctypes.byref(cfg) if cfg is not None else None, _ptr(workspace),
                                             int(ws_bytes)))


def mk_moe_dispatch_gemm_combine(x, logits, T, H, E, k, W, F, y_sorted, src_index, expert_offsets, gate_w, out,
                                 stream=None, cfg: mk_config_t | None = None, workspace=None, ws_bytes: int = 0) -> int:
    return int(lib().mk_moe_dispatch_gemm_combine(_ptr(x), _ptr(logits), T, H, E, k, _ptr(W), F, _ptr(y_sorted),
                                                  _ptr(src_index), _ptr(expert_offsets), _ptr(gate_w), _ptr(out),
                                                  _stream(stream), ctypes.byref(cfg) if cfg is not None else None,
                                                  _ptr(workspace), int(ws_bytes)))


def mk_moe_dispatch_gated(x, logits, T, H, E, k, W1, W3, F, h_sorted, src_index, expert_offsets, gate_w,
                          stream=None, cfg: mk_config_t | None = None, workspace=None, ws_bytes: int = 0) -> int:
    return int(lib().mk_moe_dispatch_gated(_ptr(x), _ptr(logits), T, H, E, k, _ptr(W1), _ptr(W3), F, _ptr(h_sorted),
                                           _ptr(src_index), _ptr(expert_offsets), _ptr(gate_w), _stream(stream),
                                           ctypes.byref(cfg) if cfg is not None else None, _ptr(workspace),
                                           int(ws_bytes)))


def moe_gated(x, logits, W1, W3, k, cfg: mk_config_t | None = None, stream=None, check=True):
    """Dispatch + gated expert FFN on torch tensors; ``y_sorted`` holds h."""
    T, H = x.shape
    E, _, F = W1.shape
    o = alloc_outputs(T, F, E, k, cfg.out_dtype if cfg is not None else MK_OUT_BF16, x.device)
    st = mk_moe_dispatch_gated(x, logits, T, H, E, k, W1, W3, F, o["y_sorted"], o["src_index"],
                               o["expert_offsets"], o["gate_w"], stream, cfg)
    _check(st, "mk_moe_dispatch_gated")
    if check:
        _check(mk_get_status(stream), "device status")
    return o


def moe_layer(x, logits, W, k, cfg: mk_config_t | None = None, stream=None, check=True):
    """Dispatch + expert GEMM + combine on torch tensors; returns the outputs
    of moe_dispatch_gemm plus ``out[T,F]``."""
    import torch

    T, H = x.shape
    E, _, F = W.shape
    o = alloc_outputs(T, F, E, k, cfg.out_dtype if cfg is not None else MK_OUT_BF16, x.device)
    o["out"] = torch.empty((T, F), dtype=o["y_sorted"].dtype, device=x.device)
    st = mk_moe_dispatch_gemm_combine(x, logits, T, H, E, k, W, F, o["y_sorted"], o["src_index"],
                                      o["expert_offsets"], o["gate_w"], o["out"], stream, cfg)
    _check(st, "mk_moe_dispatch_gemm_combine")
    if check:
        _check(mk_get_status(stream), "device status")
    return o


def mk_moe_ep_sim(x, logits, T, H, E, k, W, F, ranks, y_tok, src_index, expert_offsets, gate_w, out=None,
                  stream=None, cfg: mk_config_t | None = None, workspace=None, ws_bytes: int = 0) -> int:
    return int(lib().mk_moe_ep_sim(_ptr(x), _ptr(logits), T, H, E, k, _ptr(W), F, ranks, _ptr(y_tok),
                                   _ptr(src_index), _ptr(expert_offsets), _ptr(gate_w), _ptr(out), _stream(stream),
                                   ctypes.byref(cfg) if cfg is not None else None, _ptr(workspace), int(ws_bytes)))


def mk_moe_ep_sim_gated(x, logits, T, H, E, k, W1, W3, F, ranks, h_tok, src_index, expert_offsets, gate_w,
                        out=None, stream=None, cfg: mk_config_t | None = None, workspace=None, ws_bytes: int = 0) -> int:
    return int(lib().mk_moe_ep_sim_gated(_ptr(x), _ptr(logits), T, H, E, k, _ptr(W1), _ptr(W3), F, ranks,
                                         _ptr(h_tok), _ptr(src_index), _ptr(expert_offsets), _ptr(gate_w), _ptr(out),
                                         _stream(stream), ctypes.byref(cfg) if cfg is not None else None,
                                         _ptr(workspace), int(ws_bytes)))


def mk_ep_workspace_size(T, H, F, E, k, ranks) -> int:
    return int(lib().mk_ep_workspace_size(T, H, F, E, k, ranks))


def moe_ep_sim(x, logits, W, k, ranks, cfg: mk_config_t | None = None, stream=None, combine=True, check=True,
               W3=None):
    """Expert parallelism over ``ranks`` logical ranks simulated on one GPU;
    returns ``y_tok[T*k,F]`` (token-major), the receive metadata
    (``src_index``, ``gate_w``, ``expert_offsets``) and, with ``combine``,
    ``out[T,F]``.  With ``W3`` the experts are the gated (SwiGLU) FFN with
    ``W`` as W1, and ``y_tok`` holds h."""
    import torch

    T, H = x.shape
    E, _, F = W.shape
    o = alloc_outputs(T, F, E, k, cfg.out_dtype if cfg is not None else MK_OUT_BF16, x.device)
    o["y_tok"] = o.pop("y_sorted")
    o["out"] = torch.empty((T, F), dtype=o["y_tok"].dtype, device=x.device) if combine else None
    if W3 is None:
        st = mk_moe_ep_sim(x, logits, T, H, E, k, W, F, ranks, o["y_tok"], o["src_index"], o["expert_offsets"],
                           o["gate_w"], o["out"], stream, cfg)
    else:
        st = mk_moe_ep_sim_gated(x, logits, T, H, E, k, W, W3, F, ranks, o["y_tok"], o["src_index"],
                                 o["expert_offsets"], o["gate_w"], o["out"], stream, cfg)
    _check(st, "mk_moe_ep_sim")
    if check:
        _check(mk_get_status(stream), "device status")
    return o


def mk_moe_dispatch_gemm_host(x_host, logits_host, T, H, E, k, W, F, y_host, src_host, offsets_host, gate_host,
                              stream=None, cfg: mk_config_t | None = None) -> int:
    return int(lib().mk_moe_dispatch_gemm_host(_ptr(x_host), _ptr(logits_host), T, H, E, k, _ptr(W), F,
                                               _ptr(y_host), _ptr(src_host), _ptr(offsets_host), _ptr(gate_host),
                                               _stream(stream), ctypes.byref(cfg) if cfg is not None else None))


MK_NOALLOC_SCRATCH_BYTES = 64 << 20


def mk_moe_dispatch_gemm_noalloc(x, logits, T, H, E, k, W, F, y_sorted, src_index, expert_offsets, gate_w,
                                 stream=None, cfg: mk_config_t | None = None) -> int:
    """Allocation-free call: the library's fixed 64 MiB device array is the
    workspace (for callers that may not allocate device memory while they
    run this, e.g. inside a framework that owns the device-memory budget).
    Calls that overlap on the GPU share that array and race."""
    return int(lib().mk_moe_dispatch_gemm_noalloc(_ptr(x), _ptr(logits), T, H, E, k, _ptr(W), F, _ptr(y_sorted),
                                                  _ptr(src_index), _ptr(expert_offsets), _ptr(gate_w),
                                                  _stream(stream), ctypes.byref(cfg) if cfg is not None else None))


def mk_get_status(stream=None) -> int:
    return int(lib().mk_get_status(_stream(stream)))


def mk_last_error_detail():
    a, b, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    lib().mk_last_error_detail(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    return dict(site=a.value, cta=b.value, info=c.value)


def mk_last_launch_info() -> dict:
    i = mk_launch_info_t()
    lib().mk_last_launch_info(ctypes.byref(i))
    return {f: getattr(i, f) for f, _ in mk_launch_info_t._fields_}


def mk_read_trace(T, H, E, k, n_ctas, stream=None, workspace=None):
    import numpy as np

    buf = (ctypes.c_uint64 * (n_ctas * 16))()
    _check(int(lib().mk_read_trace(_stream(stream), _ptr(workspace), T, H, E, k, buf, n_ctas * 16)), "mk_read_trace")
    return np.frombuffer(buf, dtype=np.uint64).reshape(n_ctas, 16).copy()


def mk_release_workspace() -> None:
    lib().mk_release_workspace()


# ------------------------------------------------------------- convenience --

def make_config(mode=MK_MODE_FUSED, out_dtype=MK_OUT_BF16, dispatch_ctas=0, grid_ctas=0, n_group=0,
                debug_fault=MK_FAULT_NONE, spin_limit_ns=0, trace=0, l2_prefetch=0,
                mma_pair=0, gather=0) -> mk_config_t:
    c = mk_config_default()
    c.mode, c.out_dtype, c.dispatch_ctas, c.grid_ctas = mode, out_dtype, dispatch_ctas, grid_ctas
    c.n_group, c.debug_fault, c.spin_limit_ns, c.trace = n_group, debug_fault, spin_limit_ns, trace
    c.l2_prefetch, c.mma_pair, c.gather = l2_prefetch, mma_pair, gather
    return c


def alloc_outputs(T, F, E, k, out_dtype=MK_OUT_BF16, device="cuda"):
    """Output tensors of the right shapes (torch, on ``device``)."""
    import torch

    ydt = torch.float32 if out_dtype == MK_OUT_F32 else torch.bfloat16
    return dict(
        y_sorted=torch.empty((T * k, F), dtype=ydt, device=device),
        src_index=torch.empty(T * k, dtype=torch.int32, device=device),
        expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=device),
        gate_w=torch.empty(T * k, dtype=torch.float32, device=device),
    )


def moe_dispatch_gemm(x, logits, W, k, cfg: mk_config_t | None = None, out=None, stream=None, workspace=None,
                      ws_bytes=0, check=True):
    """Run the path on torch tensors x[T,H] bf16, logits[T,E] f32, W[E,H,F] bf16 (device).

    Returns the dict of outputs (allocated when ``out`` is None).  With
    ``check`` the stream is synchronised and device errors are raised.
    """
    T, H = x.shape
    E, H2, F = W.shape
    if H2 != H or tuple(logits.shape) != (T, E):
        raise ValueError("shape mismatch between x, logits and W")
    if out is None:
        out = alloc_outputs(T, F, E, k, cfg.out_dtype if cfg is not None else MK_OUT_BF16, x.device)
    st = mk_moe_dispatch_gemm_ex(x, logits, T, H, E, k, W, F, out["y_sorted"], out["src_index"],
                                 out["expert_offsets"], out["gate_w"], stream, cfg, workspace, ws_bytes)
    _check(st, "mk_moe_dispatch_gemm_ex")
    if check:
        _check(mk_get_status(stream), "device status")
    return out
