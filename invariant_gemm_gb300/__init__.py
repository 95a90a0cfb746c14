"""Python binding of the invariant_gemm C ABI (ctypes).

Argument marshalling only: every step of the path runs in the CUDA kernels of
`libinvariant_gemm.so`, built in-tree by `invariant_gemm_gb300.build`. There is
no fallback: if the library is missing, every call raises.

Tensors are torch CUDA tensors (device memory and streams come from torch);
their data pointers are handed to the library unchanged. Layouts:
  x        bf16  [M][K]
  A_stack  bf16  [L][slices][r][K]
  B_stack  bf16  [L][slices][N][r]
  z        f32   [slices][M][r]
  y        bf16  [M][slices*N]   (updated in place)
  idx      int32 [M]             (-1 = no adapter)
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "MODE_DET", "MODE_ATOMIC", "MODE_UNSPLIT", "MODE_DET_TREE", "PATH_AUTO", "PATH_WARP", "PATH_MMA", "PATH_FMA",
    "FLAG_STATIC_WEIGHTS", "FLAG_UNFUSED", "FLAG_Z_FP32", "FLAG_TEST_COPY_TIMEOUT",
    "FLAG_INPUT_READY",
    "IGError", "Shape", "PlanInfo", "lib", "lib_path", "make_shape", "workspace_bytes",
    "plan_query", "workspace", "workspace_init", "map_tokens", "lora_shrink",
    "lora_expand", "lora_apply", "lora_shrink_noalloc", "check_status", "status_string",
    "EXPORTS",
]

MODE_DET, MODE_ATOMIC, MODE_UNSPLIT, MODE_DET_TREE = 0, 1, 2, 3
FLAG_STATIC_WEIGHTS = 1
FLAG_UNFUSED = 2
FLAG_Z_FP32 = 4
FLAG_TEST_COPY_TIMEOUT = 8   # testing only: the first A-copy wait of each block expires
FLAG_INPUT_READY = 16        # x not written by work still running on the stream
PATH_AUTO, PATH_WARP, PATH_MMA, PATH_FMA = 0, 1, 2, 3

STATUS = {
    0: "IG_OK", -1: "IG_ERR_ARG", -2: "IG_ERR_SHAPE", -3: "IG_ERR_ALIGN",
    -4: "IG_ERR_WS_SMALL", -5: "IG_ERR_CUDA", -6: "IG_ERR_WS_CORRUPT",
    -7: "IG_ERR_ADAPTER_RANGE", -8: "IG_ERR_TIMEOUT", -9: "IG_ERR_UNSUPPORTED",
}

# every function declared in include/invariant_gemm.h
EXPORTS = [
    "ig_version", "ig_status_string", "ig_workspace_bytes", "ig_plan_query",
    "ig_workspace_init", "ig_map_tokens", "lora_shrink", "lora_expand", "lora_apply",
    "ig_check_status", "lora_shrink_noalloc",
]

_HERE = os.path.dirname(os.path.abspath(__file__))


def lib_path() -> str:
    return os.path.join(_HERE, "libinvariant_gemm.so")


class IGError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)} ({status_string(code)})")


class Shape(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("N", ctypes.c_int64),
        ("r", ctypes.c_int64), ("slices", ctypes.c_int32), ("num_adapters", ctypes.c_int32),
        ("split_k", ctypes.c_int32), ("mode", ctypes.c_int32), ("path", ctypes.c_int32),
        ("flags", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int32), ("split_k", ctypes.c_int32), ("k_split", ctypes.c_int64),
        ("shrink_bm", ctypes.c_int32), ("shrink_bn", ctypes.c_int32),
        ("expand_bm", ctypes.c_int32), ("expand_bn", ctypes.c_int32),
        ("shrink_tiles_max", ctypes.c_int64), ("shrink_ctas_max", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64), ("determinism_key", ctypes.c_uint64),
        ("apply_kernels", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]


_LIB = None
_P = ctypes.c_void_p
_SP = ctypes.POINTER(Shape)


def lib() -> ctypes.CDLL:
    """The loaded library. Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise ImportError(
                f"{path} is missing: build it with `python -m invariant_gemm_gb300.build`")
        L = ctypes.CDLL(path, mode=ctypes.RTLD_LOCAL)
        L.ig_version.restype = ctypes.c_char_p
        L.ig_version.argtypes = []
        L.ig_status_string.restype = ctypes.c_char_p
        L.ig_status_string.argtypes = [ctypes.c_int]
        L.ig_workspace_bytes.restype = ctypes.c_size_t
        L.ig_workspace_bytes.argtypes = [_SP]
        L.ig_plan_query.restype = ctypes.c_int
        L.ig_plan_query.argtypes = [_SP, ctypes.POINTER(PlanInfo)]
        L.ig_workspace_init.restype = ctypes.c_int
        L.ig_workspace_init.argtypes = [_P, ctypes.c_size_t, _SP, _P]
        L.ig_map_tokens.restype = ctypes.c_int
        L.ig_map_tokens.argtypes = [_SP, _P, _P, ctypes.c_size_t, _P]
        L.lora_shrink.restype = ctypes.c_int
        L.lora_shrink.argtypes = [_SP, _P, _P, _P, ctypes.c_float, _P, _P, ctypes.c_size_t, _P]
        L.lora_expand.restype = ctypes.c_int
        L.lora_expand.argtypes = [_SP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
        L.lora_apply.restype = ctypes.c_int
        L.lora_apply.argtypes = [_SP, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                 ctypes.c_size_t, _P]
        L.lora_shrink_noalloc.restype = ctypes.c_int
        L.lora_shrink_noalloc.argtypes = [_SP, _P, _P, _P, ctypes.c_float, _P, _P]
        L.ig_check_status.restype = ctypes.c_int
        L.ig_check_status.argtypes = [_P, ctypes.c_size_t, _P]
        _LIB = L
    return _LIB


def status_string(code: int) -> str:
    try:
        return lib().ig_status_string(int(code)).decode()
    except ImportError:
        return STATUS.get(code, "unknown")


def make_shape(M, K, N, r, *, slices=1, num_adapters=1, split_k=8, mode=MODE_DET,
               path=PATH_AUTO, flags=0) -> Shape:
    return Shape(int(M), int(K), int(N), int(r), int(slices), int(num_adapters),
                 int(split_k), int(mode), int(path), int(flags))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(ws):
    return ws.numel() * ws.element_size()


def _check(rc: int, what: str):
    if rc != 0:
        raise IGError(rc, what)


def workspace_bytes(shape: Shape) -> int:
    return int(lib().ig_workspace_bytes(ctypes.byref(shape)))


def plan_query(shape: Shape) -> dict:
    info = PlanInfo()
    _check(lib().ig_plan_query(ctypes.byref(shape), ctypes.byref(info)), "ig_plan_query")
    return {f: getattr(info, f) for f, _ in PlanInfo._fields_}


def workspace_init(shape: Shape, ws, stream=None):
    _check(lib().ig_workspace_init(_ptr(ws), _nbytes(ws), ctypes.byref(shape), _stream(stream)),
           "ig_workspace_init")


def workspace(shape: Shape, device="cuda", stream=None, min_bytes: int = 0):
    """Allocate (with torch) and initialise a workspace large enough for shape."""
    import torch
    n = workspace_bytes(shape)
    if n == 0:
        plan_query(shape)  # raises with the reason
        raise IGError(-2, "ig_workspace_bytes")
    ws = torch.empty(max(n, int(min_bytes)), dtype=torch.uint8, device=device)
    workspace_init(shape, ws, stream)
    return ws


def map_tokens(shape: Shape, adapter_idx, ws, stream=None):
    _check(lib().ig_map_tokens(ctypes.byref(shape), _ptr(adapter_idx), _ptr(ws), _nbytes(ws),
                               _stream(stream)), "ig_map_tokens")


def lora_shrink(shape: Shape, x, A_stack, adapter_idx, scale, z, ws, stream=None):
    _check(lib().lora_shrink(ctypes.byref(shape), _ptr(x), _ptr(A_stack), _ptr(adapter_idx),
                             float(scale), _ptr(z), _ptr(ws), _nbytes(ws), _stream(stream)),
           "lora_shrink")


def lora_expand(shape: Shape, z, B_stack, adapter_idx, y, ws, stream=None):
    _check(lib().lora_expand(ctypes.byref(shape), _ptr(z), _ptr(B_stack), _ptr(adapter_idx),
                             _ptr(y), _ptr(ws), _nbytes(ws), _stream(stream)), "lora_expand")


def lora_apply(shape: Shape, x, y, adapter_idx, A_stack, B_stack, scale, z, ws, stream=None):
    _check(lib().lora_apply(ctypes.byref(shape), _ptr(x), _ptr(y), _ptr(adapter_idx),
                            _ptr(A_stack), _ptr(B_stack), float(scale), _ptr(z), _ptr(ws),
                            _nbytes(ws), _stream(stream)), "lora_apply")


def lora_shrink_noalloc(shape: Shape, x, A_stack, adapter_idx, scale, z, stream=None):
    """lora_shrink with the library's built-in 4 MiB scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    _check(lib().lora_shrink_noalloc(ctypes.byref(shape), _ptr(x), _ptr(A_stack),
                                     _ptr(adapter_idx), float(scale), _ptr(z), _stream(stream)),
           "lora_shrink_noalloc")


def check_status(ws, stream=None) -> int:
    """Synchronise and return the device status (0 or a negative code)."""
    return int(lib().ig_check_status(_ptr(ws), _nbytes(ws), _stream(stream)))
