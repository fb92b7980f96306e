"""Python binding of libpoetx.so, the C ABI of the POET-X orthogonal-equivalence
linear layer on one B300 (declared in include/poetx.h).

The functions below carry the C names and only marshal arguments: torch
tensors become device pointers, the stream defaults to torch's current
stream, and a non-OK status raises PoetxError.  Every step of the layer runs
in the library's CUDA kernels; there is no other implementation behind these
calls, and importing this package fails if the library cannot be loaded.

``Layer`` is a small convenience that owns the device buffers a layer needs
(params, pre-merged weight, workspace), allocated with torch.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

__all__ = [
    "PoetxError", "poetx_layer_desc", "LIB", "lib_path", "POETX_OK", "POETX_ERR_INVALID_ARG",
    "POETX_ERR_UNSUPPORTED", "POETX_ERR_MISALIGNED", "POETX_ERR_CUDA", "POETX_ERR_TIMEOUT",
    "MODE_CAYLEY", "MODE_NEUMANN", "DTYPE_FP32", "DTYPE_BF16", "WEIGHT_DENSE", "WEIGHT_INT8",
    "make_desc", "poetx_weight_size", "poetx_blocks_build", "poetx_generator_adamw",
    "poetx_status_string", "poetx_version", "poetx_perm_generate", "poetx_gen_length",
    "poetx_params_size", "poetx_params_build", "poetx_weight_premerge", "poetx_workspace_size",
    "poetx_linear_fwd", "poetx_linear_bwd", "poetx_merge_workspace_size", "poetx_merge",
    "poetx_linear_step_host", "poetx_linear_step_host_async", "poetx_device_status",
    "poetx_selftest_bounded_wait",
    "poetx_set_wait_timeout_ns", "poetx_set_dependent_launch",
    "poetx_set_fused_gather_max_features", "poetx_profile_enable",
    "poetx_profile_reset", "poetx_profile_read", "poetx_profile_kind_name", "poetx_launch_count",
    "KIND_NAMES", "Layer",
    "EXPORTED_SYMBOLS", "poetx_linear_fwd_noalloc", "NOALLOC_SCRATCH_BYTES",
]

POETX_OK, POETX_ERR_INVALID_ARG, POETX_ERR_UNSUPPORTED = 0, 1, 2
POETX_ERR_MISALIGNED, POETX_ERR_CUDA, POETX_ERR_TIMEOUT = 3, 4, 5
MODE_CAYLEY, MODE_NEUMANN = 0, 1
DTYPE_FP32, DTYPE_BF16 = 0, 1
WEIGHT_DENSE, WEIGHT_INT8 = 0, 1

EXPORTED_SYMBOLS = [
    "poetx_status_string", "poetx_version", "poetx_perm_generate", "poetx_gen_length",
    "poetx_params_size", "poetx_params_build", "poetx_weight_premerge", "poetx_workspace_size",
    "poetx_linear_fwd", "poetx_linear_bwd", "poetx_merge_workspace_size", "poetx_merge",
    "poetx_linear_step_host", "poetx_linear_step_host_async", "poetx_device_status",
    "poetx_selftest_bounded_wait",
    "poetx_set_wait_timeout_ns", "poetx_set_dependent_launch",
    "poetx_set_fused_gather_max_features", "poetx_profile_enable",
    "poetx_profile_reset", "poetx_profile_read", "poetx_profile_kind_name", "poetx_launch_count",
    "poetx_linear_fwd_noalloc",
    "poetx_weight_size", "poetx_blocks_build", "poetx_generator_adamw",
]

# Size of the library's fixed forward scratch (POETX_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 32 << 20

KIND_NAMES = ["gemm_fwd", "gemm_dgrad", "blockdiag", "gradred", "gather", "build", "genbwd",
              "merge", "simt", "dequant"]


class PoetxError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {poetx_status_string(status)} ({status})")


class poetx_layer_desc(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("n", ctypes.c_int32), ("b_R", ctypes.c_int32),
                ("b_P", ctypes.c_int32), ("seed_R", ctypes.c_uint64), ("seed_P", ctypes.c_uint64),
                ("mode", ctypes.c_int32), ("neumann_k", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("weight_format", ctypes.c_int32)]

    def __repr__(self):
        return (f"poetx_layer_desc(m={self.m}, n={self.n}, b_R={self.b_R}, b_P={self.b_P}, "
                f"seed_R={self.seed_R}, seed_P={self.seed_P}, mode={self.mode}, "
                f"neumann_k={self.neumann_k}, dtype={self.dtype}, "
                f"weight_format={self.weight_format})")


def make_desc(m, n, b_R, b_P, seed_R, seed_P, dtype="bf16", mode="cayley", neumann_k=3,
              weight="dense"):
    """weight: "dense" (W0' in the layer dtype) or "int8" (POET-XQ storage)."""
    return poetx_layer_desc(
        m, n, b_R, b_P, seed_R, seed_P,
        MODE_NEUMANN if mode in ("neumann", MODE_NEUMANN) else MODE_CAYLEY, neumann_k,
        DTYPE_BF16 if dtype in ("bf16", DTYPE_BF16) else DTYPE_FP32,
        WEIGHT_INT8 if weight in ("int8", WEIGHT_INT8) else WEIGHT_DENSE)


def _load():
    path = _build.build()   # compiles in-tree if missing or stale; raises on failure
    lib = ctypes.CDLL(path, mode=ctypes.RTLD_GLOBAL)
    P, V, I32, I64, U64, SZ = (ctypes.c_void_p, None, ctypes.c_int32, ctypes.c_int64,
                               ctypes.c_uint64, ctypes.c_size_t)
    D = ctypes.POINTER(poetx_layer_desc)
    F = ctypes.POINTER(ctypes.c_float)
    sig = {
        "poetx_status_string": (ctypes.c_char_p, [I32]),
        "poetx_version": (I32, []),
        "poetx_perm_generate": (I32, [U64, I32, ctypes.POINTER(ctypes.c_int32)]),
        "poetx_gen_length": (I64, [I32, I32]),
        "poetx_params_size": (SZ, [D]),
        "poetx_params_build": (I32, [D, P, P, P, P]),
        "poetx_blocks_build": (I32, [D, P, P, P, P]),
        "poetx_weight_premerge": (I32, [D, P, P, P, P]),
        "poetx_workspace_size": (SZ, [D, I64]),
        "poetx_weight_size": (SZ, [D]),
        "poetx_linear_fwd": (I32, [D, P, P, P, I64, P, P, P, P, P]),
        "poetx_linear_bwd": (I32, [D, P, P, P, P, P, P, I64, P, P, P, I32, P, P]),
        "poetx_merge_workspace_size": (SZ, [D]),
        "poetx_merge": (I32, [D, P, P, U64, U64, P, P]),
        "poetx_linear_step_host": (I32, [D, P, P, P, P, I64, P, P, P, P, P, P, P, P, P, P, P, P]),
        "poetx_linear_step_host_async": (I32, [D, P, P, P, P, I64, P, P, P, P, P, P, P, P, P, P, P, P]),
        "poetx_device_status": (I32, [I32]),
        "poetx_generator_adamw": (I32, [P, P, P, P, I64, I64, ctypes.c_float, ctypes.c_float,
                                        ctypes.c_float, ctypes.c_float, ctypes.c_float, P]),
        "poetx_selftest_bounded_wait": (I32, [U64, P]),
        "poetx_set_wait_timeout_ns": (V, [U64]),
        "poetx_set_dependent_launch": (V, [I32]),
        "poetx_set_fused_gather_max_features": (V, [I32]),
        "poetx_profile_enable": (V, [I32]),
        "poetx_profile_reset": (V, []),
        "poetx_profile_read": (I32, [I32, ctypes.POINTER(ctypes.c_int64),
                                     ctypes.POINTER(ctypes.c_double)]),
        "poetx_profile_kind_name": (ctypes.c_char_p, [I32]),
        "poetx_launch_count": (I64, []),
        "poetx_linear_fwd_noalloc": (I32, [D, P, P, P, I64, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib, path


LIB, lib_path = _load()


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != POETX_OK:
        raise PoetxError(status, where)


def poetx_status_string(status: int) -> str:
    return LIB.poetx_status_string(status).decode()


def poetx_version() -> int:
    return LIB.poetx_version()


def poetx_perm_generate(seed: int, d: int):
    """Host permutation of 0..d-1 from `seed` (numpy int32 array)."""
    import numpy as np
    out = np.empty(d, dtype=np.int32)
    _check(LIB.poetx_perm_generate(seed, d, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "poetx_perm_generate")
    return out


def poetx_gen_length(d: int, b: int) -> int:
    return LIB.poetx_gen_length(d, b)


def poetx_params_size(desc) -> int:
    return LIB.poetx_params_size(ctypes.byref(desc))


def poetx_params_build(desc, genR, genP, params, stream=None):
    _check(LIB.poetx_params_build(ctypes.byref(desc), _ptr(genR), _ptr(genP), _ptr(params),
                                  _stream(stream)), "poetx_params_build")


def poetx_blocks_build(desc, genR, genP, params, stream=None):
    """Rebuild only the blocks of params (device work only; capturable in a
    CUDA graph).  params must already hold the permutations of desc's seeds."""
    _check(LIB.poetx_blocks_build(ctypes.byref(desc), _ptr(genR), _ptr(genP), _ptr(params),
                                  _stream(stream)), "poetx_blocks_build")


def poetx_weight_premerge(desc, params, W0, W0p, stream=None):
    _check(LIB.poetx_weight_premerge(ctypes.byref(desc), _ptr(params), _ptr(W0), _ptr(W0p),
                                     _stream(stream)), "poetx_weight_premerge")


def poetx_workspace_size(desc, T: int) -> int:
    return LIB.poetx_workspace_size(ctypes.byref(desc), T)


def poetx_weight_size(desc) -> int:
    return LIB.poetx_weight_size(ctypes.byref(desc))


def poetx_linear_fwd(desc, params, W0p, X, T, Y, saved_h, saved_u, workspace, stream=None):
    _check(LIB.poetx_linear_fwd(ctypes.byref(desc), _ptr(params), _ptr(W0p), _ptr(X), T, _ptr(Y),
                                _ptr(saved_h), _ptr(saved_u), _ptr(workspace), _stream(stream)),
           "poetx_linear_fwd")


def poetx_linear_bwd(desc, params, W0p, X, dY, saved_h, saved_u, T, dX, dGenR, dGenP, accumulate,
                     workspace, stream=None):
    _check(LIB.poetx_linear_bwd(ctypes.byref(desc), _ptr(params), _ptr(W0p), _ptr(X), _ptr(dY),
                                _ptr(saved_h), _ptr(saved_u), T, _ptr(dX), _ptr(dGenR),
                                _ptr(dGenP), int(accumulate), _ptr(workspace), _stream(stream)),
           "poetx_linear_bwd")


def poetx_linear_fwd_noalloc(desc, params, W0p, X, T, Y, saved_h, saved_u, stream=None):
    """Forward without a workspace argument: the library's fixed device scratch
    of NOALLOC_SCRATCH_BYTES serves as workspace, so the call allocates
    nothing (for callers that cannot allocate device memory).  Calls that
    overlap on the GPU share that scratch and race."""
    _check(LIB.poetx_linear_fwd_noalloc(ctypes.byref(desc), _ptr(params), _ptr(W0p), _ptr(X), T,
                                        _ptr(Y), _ptr(saved_h), _ptr(saved_u), _stream(stream)),
           "poetx_linear_fwd_noalloc")


def poetx_merge_workspace_size(desc) -> int:
    return LIB.poetx_merge_workspace_size(ctypes.byref(desc))


def poetx_merge(desc, params, W0p, new_seed_R, new_seed_P, workspace, stream=None):
    _check(LIB.poetx_merge(ctypes.byref(desc), _ptr(params), _ptr(W0p), new_seed_R, new_seed_P,
                           _ptr(workspace), _stream(stream)), "poetx_merge")


def poetx_linear_step_host(desc, params, W0p, X_host, dY_host, T, X_dev, dY_dev, Y_dev,
                           saved_h_dev, saved_u_dev, dX_dev, dGenR_dev, dGenP_dev, dGenR_host,
                           dGenP_host, workspace, stream=None):
    _check(LIB.poetx_linear_step_host(
        ctypes.byref(desc), _ptr(params), _ptr(W0p), _ptr(X_host), _ptr(dY_host), T, _ptr(X_dev),
        _ptr(dY_dev), _ptr(Y_dev), _ptr(saved_h_dev), _ptr(saved_u_dev), _ptr(dX_dev), _ptr(dGenR_dev),
        _ptr(dGenP_dev), _ptr(dGenR_host), _ptr(dGenP_host), _ptr(workspace), _stream(stream)),
        "poetx_linear_step_host")


def poetx_linear_step_host_async(desc, params, W0p, X_host, dY_host, T, X_dev, dY_dev, Y_dev,
                                 saved_h_dev, saved_u_dev, dX_dev, dGenR_dev, dGenP_dev, dGenR_host,
                                 dGenP_host, workspace, stream=None):
    _check(LIB.poetx_linear_step_host_async(
        ctypes.byref(desc), _ptr(params), _ptr(W0p), _ptr(X_host), _ptr(dY_host), T, _ptr(X_dev),
        _ptr(dY_dev), _ptr(Y_dev), _ptr(saved_h_dev), _ptr(saved_u_dev), _ptr(dX_dev), _ptr(dGenR_dev),
        _ptr(dGenP_dev), _ptr(dGenR_host), _ptr(dGenP_host), _ptr(workspace), _stream(stream)),
        "poetx_linear_step_host_async")


def poetx_generator_adamw(gen, grad, m1, m2, length, step, lr, beta1=0.9, beta2=0.999, eps=1e-8,
                          weight_decay=0.0, stream=None):
    _check(LIB.poetx_generator_adamw(_ptr(gen), _ptr(grad), _ptr(m1), _ptr(m2), length, step, lr,
                                     beta1, beta2, eps, weight_decay, _stream(stream)),
           "poetx_generator_adamw")


def poetx_device_status(reset: bool = False) -> int:
    return LIB.poetx_device_status(1 if reset else 0)


def poetx_selftest_bounded_wait(timeout_ns: int, stream=None) -> int:
    return LIB.poetx_selftest_bounded_wait(timeout_ns, _stream(stream))


def poetx_set_wait_timeout_ns(timeout_ns: int):
    LIB.poetx_set_wait_timeout_ns(timeout_ns)


def poetx_set_dependent_launch(on: bool = True):
    """Programmatic dependent launch of the pass kernels (on by default)."""
    LIB.poetx_set_dependent_launch(1 if on else 0)


def poetx_set_fused_gather_max_features(max_features: int = -1):
    """Column permutation inside the block transform for bf16 sides of 256
    to `max_features` features (0: off, the default; negative: the default)."""
    LIB.poetx_set_fused_gather_max_features(int(max_features))


def poetx_profile_enable(on: bool = True):
    LIB.poetx_profile_enable(1 if on else 0)


def poetx_profile_reset():
    LIB.poetx_profile_reset()


def poetx_profile_read(kind: int):
    """(groups, total_ms) of the timed launch groups of one kernel class."""
    g, ms = ctypes.c_int64(), ctypes.c_double()
    _check(LIB.poetx_profile_read(kind, ctypes.byref(g), ctypes.byref(ms)), "poetx_profile_read")
    return g.value, ms.value


def poetx_profile_kind_name(kind: int) -> str:
    return LIB.poetx_profile_kind_name(kind).decode()


def poetx_launch_count() -> int:
    return LIB.poetx_launch_count()


class Layer:
    """Device buffers of one POET-X layer plus calls into the library.

    Holds params (poetx_params_size bytes), the pre-merged weight W0'
    (m x n, layer dtype) and a workspace sized for ``max_tokens``.  All memory
    comes from torch's caching allocator; the library allocates none.
    """

    def __init__(self, desc, max_tokens: int, device="cuda"):
        import torch
        self.desc = desc
        self.device = torch.device(device)
        self.dtype = torch.bfloat16 if desc.dtype == DTYPE_BF16 else torch.float32
        self.params = torch.empty(poetx_params_size(desc), dtype=torch.uint8, device=self.device)
        if desc.weight_format == WEIGHT_INT8:   # codes, then row scales (poetx_weight_size bytes)
            self.W0p = torch.empty(poetx_weight_size(desc), dtype=torch.uint8, device=self.device)
        else:
            self.W0p = torch.empty(desc.m, desc.n, dtype=self.dtype, device=self.device)
        self.max_tokens = max_tokens
        ws = max(poetx_workspace_size(desc, max_tokens), poetx_merge_workspace_size(desc))
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.device)
        self.len_R = poetx_gen_length(desc.m, desc.b_R)
        self.len_P = poetx_gen_length(desc.n, desc.b_P)

    def build(self, genR, genP, stream=None):
        poetx_params_build(self.desc, genR, genP, self.params, stream)

    def rebuild(self, genR, genP, stream=None):
        """New generators, same seeds: blocks only (capturable in a CUDA graph)."""
        poetx_blocks_build(self.desc, genR, genP, self.params, stream)

    def premerge(self, W0, stream=None):
        poetx_weight_premerge(self.desc, self.params, W0, self.W0p, stream)

    def forward(self, X, Y, saved_h=None, saved_u=None, stream=None):
        T = X.shape[0]
        assert T <= self.max_tokens
        poetx_linear_fwd(self.desc, self.params, self.W0p, X, T, Y, saved_h, saved_u,
                         self.workspace, stream)

    def backward(self, X, dY, dX, dGenR, dGenP, saved_h=None, saved_u=None, accumulate=False,
                 stream=None):
        T = dY.shape[0]
        assert T <= self.max_tokens
        poetx_linear_bwd(self.desc, self.params, self.W0p, X, dY, saved_h, saved_u, T, dX, dGenR,
                         dGenP, accumulate, self.workspace, stream)

    def merge(self, new_seed_R, new_seed_P, stream=None):
        poetx_merge(self.desc, self.params, self.W0p, new_seed_R, new_seed_P, self.workspace,
                    stream)
