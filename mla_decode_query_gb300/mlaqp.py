"""ctypes binding of ``libmlaqp.so`` (declared in ``include/mlaqp.h``).

Argument marshalling only: every function here forwards to the C entry point
of the same name and returns its status code unchanged; all of the operation
runs in the library's CUDA kernels.  Tensor arguments may be ``torch.Tensor``
objects on the GPU (their ``data_ptr()`` is passed) or raw integer device
addresses; ``None`` passes NULL.  ``stream=None`` means PyTorch's current
CUDA stream.

If the library has not been built the first call raises ``RuntimeError``:
there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import re
import threading
from pathlib import Path

from .build import INCLUDE, LIB_PATH

MLAQP_WEIGHT_BF16 = 0
MLAQP_WEIGHT_MXFP8 = 1
MLAQP_OUT_BF16 = 0
MLAQP_OUT_E4M3 = 1

MLAQP_OK = 0
MLAQP_ERR_UNSUPPORTED = 1
MLAQP_ERR_INVALID_ARG = 2
MLAQP_ERR_CUDA = 3

MLAQP_DEVSTATUS_WAIT_TIMEOUT = 1

NOPE_DIM = 128
LATENT_DIM = 512
ROPE_DIM = 64
OUT_DIM = 576
MAX_M = 256
MAX_M_DECODE = 32
V_HEAD_DIM = 128

WEIGHT_FORMATS = {"bf16": MLAQP_WEIGHT_BF16, "mxfp8": MLAQP_WEIGHT_MXFP8}
OUT_DTYPES = {"bf16": MLAQP_OUT_BF16, "e4m3": MLAQP_OUT_E4M3}

_lock = threading.Lock()
_lib = None

_c_void_p = ctypes.c_void_p
_c_int = ctypes.c_int
_SIGNATURES = {
    "mlaqp_can_implement": (_c_int, [_c_int] * 8),
    "mlaqp_prewarm": (_c_int, [_c_int] * 5),
    "mlaqp_run": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, ctypes.c_int64,
                           _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p]),
    "mlaqp_run_pdl": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p, ctypes.c_int64,
                               _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p]),
    "mlaqp_run_strided": (_c_int, [_c_void_p, ctypes.c_int64, ctypes.c_int64, _c_void_p, ctypes.c_int64,
                                   ctypes.c_int64, _c_void_p, _c_void_p, _c_void_p, ctypes.c_int64, _c_void_p,
                                   _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_void_p]),
    "mlaqp_debug_run_arm": (_c_int, [_c_void_p, ctypes.c_int64, ctypes.c_int64, _c_void_p, ctypes.c_int64,
                                     ctypes.c_int64, _c_void_p, _c_void_p, _c_void_p, ctypes.c_int64, _c_void_p,
                                     _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_void_p]),
    "mlaqp_debug_set_policy": (_c_int, [_c_int, _c_int]),
    "mlaqp_prefetch_weights": (_c_int, [_c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_void_p]),
    "mlaqp_launch_shape": (_c_int, [_c_int, _c_int, _c_int, _c_int, ctypes.POINTER(_c_int),
                                    ctypes.POINTER(_c_int)]),
    "mlaqp_debug_plan": (_c_int, [_c_int] * 8 + [ctypes.POINTER(_c_int)] * 6),
    "mlaqp_debug_v_plan": (_c_int, [_c_int] * 5 + [ctypes.POINTER(_c_int)] * 7),
    "mlaqp_device_status": (_c_int, [ctypes.POINTER(ctypes.c_uint), _c_int]),
    "mlaqp_debug_run_bounded_wait": (_c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                              ctypes.c_int64, _c_void_p, _c_int, _c_int, _c_int, _c_int,
                                              ctypes.c_ulonglong, ctypes.c_uint, _c_void_p]),
    "mlaqp_debug_launch_null": (_c_int, [_c_int, _c_int, _c_int, _c_void_p]),
    "mlaqp_v_up_run": (_c_int, [_c_void_p, ctypes.c_int64, ctypes.c_int64, _c_void_p, _c_void_p, _c_void_p,
                                ctypes.c_int64, _c_int, _c_int, _c_int, _c_int, _c_void_p]),
    "mlaqp_v_up_can_implement": (_c_int, [_c_int] * 4),
    "mlaqp_v_up_prewarm": (_c_int, [_c_int] * 4),
    "mlaqp_debug_v_up_bounded_wait": (_c_int, [_c_void_p, ctypes.c_int64, ctypes.c_int64, _c_void_p, _c_void_p,
                                               _c_void_p, ctypes.c_int64, _c_int, _c_int, _c_int,
                                               ctypes.c_ulonglong, ctypes.c_uint, _c_void_p]),
    "mlaqp_last_error": (ctypes.c_char_p, []),
    "mlaqp_version": (_c_int, []),
}


def header_functions(header: Path | None = None) -> list[str]:
    """Names of the functions ``include/*.h`` declares (parsed from text)."""
    names = []
    for h in ([header] if header else sorted(INCLUDE.glob("*.h"))):
        text = re.sub(r"/\*.*?\*/", "", Path(h).read_text(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(mlaqp_\w+)\s*\(", text, flags=re.M)
    return names


def load_library(path: Path | str | None = None) -> ctypes.CDLL:
    """Load ``libmlaqp.so`` once and attach the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = Path(path) if path else LIB_PATH
        if not p.exists():
            raise RuntimeError(
                f"{p} is missing: build the CUDA library first "
                "(python -m mla_decode_query_gb300.build, or __graft_entry__.build())")
        lib = ctypes.CDLL(str(p))
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a tensor, an int address or None, got {type(x)!r}")


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    raise TypeError(f"expected a torch.cuda.Stream, an int handle or None, got {type(stream)!r}")


def _fmt(v, table) -> int:
    return table[v] if isinstance(v, str) else int(v)


def mlaqp_can_implement(num_heads, max_m, nope_dim=NOPE_DIM, latent_dim=LATENT_DIM, rope_dim=ROPE_DIM,
                        weight_format="bf16", out_dtype="bf16", device=-1) -> int:
    return load_library().mlaqp_can_implement(num_heads, max_m, nope_dim, latent_dim, rope_dim,
                                              _fmt(weight_format, WEIGHT_FORMATS),
                                              _fmt(out_dtype, OUT_DTYPES), device)


def mlaqp_prewarm(num_heads, max_m, weight_format="bf16", out_dtype="bf16", device=-1) -> int:
    return load_library().mlaqp_prewarm(num_heads, max_m, _fmt(weight_format, WEIGHT_FORMATS),
                                        _fmt(out_dtype, OUT_DTYPES), device)


def _run_args(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H, weight_format,
              out_dtype):
    return (_ptr(q_nope), _ptr(q_pe), _ptr(weight), _ptr(weight_scale), _ptr(out), int(out_row_stride),
            _ptr(q_scale), int(M), int(H), _fmt(weight_format, WEIGHT_FORMATS), _fmt(out_dtype, OUT_DTYPES))


def mlaqp_run(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H, weight_format,
              out_dtype, stream=None) -> int:
    a = _run_args(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H, weight_format,
                  out_dtype)
    return load_library().mlaqp_run(*a, _stream(stream))


def mlaqp_run_pdl(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H, weight_format,
                  out_dtype, stream=None) -> int:
    a = _run_args(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H, weight_format,
                  out_dtype)
    return load_library().mlaqp_run_pdl(*a, _stream(stream))


def mlaqp_run_strided(q_nope, q_nope_token_stride, q_nope_head_stride, q_pe, q_pe_token_stride, q_pe_head_stride,
                      weight, weight_scale, out, out_row_stride, q_scale, M, H, nope_dim, weight_format, out_dtype,
                      pdl=False, stream=None) -> int:
    return load_library().mlaqp_run_strided(
        _ptr(q_nope), int(q_nope_token_stride), int(q_nope_head_stride), _ptr(q_pe), int(q_pe_token_stride),
        int(q_pe_head_stride), _ptr(weight), _ptr(weight_scale), _ptr(out), int(out_row_stride), _ptr(q_scale),
        int(M), int(H), int(nope_dim), _fmt(weight_format, WEIGHT_FORMATS), _fmt(out_dtype, OUT_DTYPES),
        int(pdl), _stream(stream))


def mlaqp_prefetch_weights(weight, weight_scale, H, nope_dim, weight_format, pdl=False, stream=None) -> int:
    return load_library().mlaqp_prefetch_weights(_ptr(weight), _ptr(weight_scale), int(H), int(nope_dim),
                                                 _fmt(weight_format, WEIGHT_FORMATS), int(pdl),
                                                 _stream(stream))


ARMS = {"auto": 0, "warp_mma": 1, "warp_fma": 2, "cta_mma": 3, "tcgen05": 4}


def mlaqp_debug_run_arm(q_nope, q_nope_token_stride, q_nope_head_stride, q_pe, q_pe_token_stride, q_pe_head_stride,
                        weight, weight_scale, out, out_row_stride, q_scale, M, H, nope_dim, weight_format, out_dtype,
                        pdl=False, arm="auto", stream=None) -> int:
    return load_library().mlaqp_debug_run_arm(
        _ptr(q_nope), int(q_nope_token_stride), int(q_nope_head_stride), _ptr(q_pe), int(q_pe_token_stride),
        int(q_pe_head_stride), _ptr(weight), _ptr(weight_scale), _ptr(out), int(out_row_stride), _ptr(q_scale),
        int(M), int(H), int(nope_dim), _fmt(weight_format, WEIGHT_FORMATS), _fmt(out_dtype, OUT_DTYPES),
        int(pdl), _fmt(arm, ARMS), _stream(stream))


def mlaqp_debug_set_policy(trig, cta_cap) -> int:
    return load_library().mlaqp_debug_set_policy(int(trig), int(cta_cap))


def mlaqp_debug_run_bounded_wait(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H,
                                 weight_format, out_dtype, wait_limit_ns, extra_tx_bytes, stream=None) -> int:
    a = _run_args(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H, weight_format,
                  out_dtype)
    return load_library().mlaqp_debug_run_bounded_wait(*a, int(wait_limit_ns), int(extra_tx_bytes),
                                                       _stream(stream))


def mlaqp_debug_launch_null(ctas, threads, pdl, stream=None) -> int:
    return load_library().mlaqp_debug_launch_null(int(ctas), int(threads), int(pdl), _stream(stream))


def mlaqp_v_up_run(x, x_token_stride, x_head_stride, weight, weight_scale, out, out_row_stride, M, H,
                   weight_format, pdl=False, stream=None) -> int:
    return load_library().mlaqp_v_up_run(_ptr(x), int(x_token_stride), int(x_head_stride), _ptr(weight),
                                         _ptr(weight_scale), _ptr(out), int(out_row_stride), int(M), int(H),
                                         _fmt(weight_format, WEIGHT_FORMATS), int(pdl), _stream(stream))


def mlaqp_v_up_can_implement(num_heads, max_m, weight_format="bf16", device=-1) -> int:
    return load_library().mlaqp_v_up_can_implement(num_heads, max_m, _fmt(weight_format, WEIGHT_FORMATS), device)


def mlaqp_v_up_prewarm(num_heads, max_m, weight_format="bf16", device=-1) -> int:
    return load_library().mlaqp_v_up_prewarm(num_heads, max_m, _fmt(weight_format, WEIGHT_FORMATS), device)


def mlaqp_debug_v_up_bounded_wait(x, x_token_stride, x_head_stride, weight, weight_scale, out, out_row_stride, M,
                                  H, weight_format, wait_limit_ns, extra_tx_bytes, stream=None) -> int:
    return load_library().mlaqp_debug_v_up_bounded_wait(
        _ptr(x), int(x_token_stride), int(x_head_stride), _ptr(weight), _ptr(weight_scale), _ptr(out),
        int(out_row_stride), int(M), int(H), _fmt(weight_format, WEIGHT_FORMATS), int(wait_limit_ns),
        int(extra_tx_bytes), _stream(stream))


def mlaqp_launch_shape(M, H, weight_format="bf16", out_dtype="bf16"):
    """Returns ``(status, grid_ctas, threads_per_cta)``."""
    g, t = _c_int(0), _c_int(0)
    st = load_library().mlaqp_launch_shape(int(M), int(H), _fmt(weight_format, WEIGHT_FORMATS),
                                           _fmt(out_dtype, OUT_DTYPES), ctypes.byref(g), ctypes.byref(t))
    return st, g.value, t.value


ARM_NAMES = {v: k for k, v in ARMS.items()}


def mlaqp_debug_plan(M, H, weight_format="bf16", out_dtype="bf16", nope_dim=128, pdl=1, arm="auto", sm_count=152):
    """The launch a query call would make on a device with ``sm_count`` SMs
    (host-side, no device).  Returns ``(status, plan)`` with plan a dict:
    arm (name), chunk_tokens, trig, cta_cap, grid_ctas, threads_per_cta."""
    out = [_c_int(0) for _ in range(6)]
    st = load_library().mlaqp_debug_plan(int(M), int(H), int(nope_dim), _fmt(weight_format, WEIGHT_FORMATS),
                                         _fmt(out_dtype, OUT_DTYPES), int(pdl), _fmt(arm, ARMS), int(sm_count),
                                         *[ctypes.byref(o) for o in out])
    keys = ("arm", "chunk_tokens", "trig", "cta_cap", "grid_ctas", "threads_per_cta")
    plan = {k: o.value for k, o in zip(keys, out)}
    plan["arm"] = ARM_NAMES.get(plan["arm"], plan["arm"])
    return st, plan


V_FORMS = {0: "plain", 1: "multicast", 2: "cluster"}


def mlaqp_debug_v_plan(M, H, weight_format="bf16", pdl=1, sm_count=152):
    """As mlaqp_debug_plan for a V call with contiguous x.  Returns
    ``(status, plan)``: form (plain / multicast / cluster), chunk_tokens,
    trig, cta_cap, grid_ctas, threads_per_cta, cluster."""
    out = [_c_int(0) for _ in range(7)]
    st = load_library().mlaqp_debug_v_plan(int(M), int(H), _fmt(weight_format, WEIGHT_FORMATS), int(pdl),
                                           int(sm_count), *[ctypes.byref(o) for o in out])
    keys = ("form", "chunk_tokens", "trig", "cta_cap", "grid_ctas", "threads_per_cta", "cluster")
    plan = {k: o.value for k, o in zip(keys, out)}
    plan["form"] = V_FORMS.get(plan["form"], plan["form"])
    return st, plan


def mlaqp_device_status(reset=False):
    """Returns ``(status, word)``."""
    v = ctypes.c_uint(0)
    st = load_library().mlaqp_device_status(ctypes.byref(v), 1 if reset else 0)
    return st, v.value


def mlaqp_last_error() -> str:
    return load_library().mlaqp_last_error().decode()


def mlaqp_version() -> int:
    return load_library().mlaqp_version()


class MlaqpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"mlaqp status {status}: {message}")
        self.status = status


def check(status: int) -> None:
    """Raise ``MlaqpError`` with the library's message for a non-OK status."""
    if status != MLAQP_OK:
        raise MlaqpError(status, mlaqp_last_error())
