"""Thin ctypes binding of libklt.so, with the same names as the C ABI in include/klt.h.

Argument marshalling only: every step of the tail runs in the library's CUDA kernels.
PyTorch supplies device memory and the stream.  There is no fallback path: if the
library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

from .build import LIB_PATH

KLT_OK = 0
KLT_ERR_INVALID_ARG = 1
KLT_ERR_UNSUPPORTED = 2
KLT_ERR_ALIGN = 3
KLT_ERR_CUDA = 4
KLT_ERR_DEVICE_TIMEOUT = 5
KLT_ERR_OOM = 6
KLT_ERR_TOO_LARGE = 7
KLT_NOALLOC_MAX_PAIRS = 65536
KLT_FMT_FP8_B128 = 0
KLT_FMT_NVFP4 = 1
KLT_FMT_MXFP8 = 2
KLT_FMT_NVFP4_W4A4 = 3
KLT_FLAG_NO_PDL = 1
KLT_FLAG_PHASED = 2
KLT_FLAG_DETERMINISTIC = 4

EXPORTS = ("klt_create", "klt_forward", "klt_forward_hidden", "klt_status", "klt_destroy",
           "klt_strerror", "klt_launch_count", "klt_gemm_tile", "klt_route_noalloc")


class KltDims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("L", ctypes.c_int32), ("E", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("I", ctypes.c_int32), ("Is", ctypes.c_int32),
                ("routed_fmt", ctypes.c_int32), ("eps", ctypes.c_float),
                ("max_tokens", ctypes.c_int32)]


class KltWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w13", "w13_scale", "w13_global", "w2", "w2_scale", "w2_global", "ws13", "ws2",
        "w_up", "gamma", "w_lat", "w_gate")]


class KltRouting(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "ids", "weights", "cnt", "off", "gidx", "slot", "pos")]


class KltDebug(ctypes.Structure):
    _fields_ = [("zq", ctypes.c_void_p), ("zs", ctypes.c_void_p), ("aq", ctypes.c_void_p),
                ("as_", ctypes.c_void_p), ("r", ctypes.c_void_p), ("n", ctypes.c_void_p),
                ("a_s", ctypes.c_void_p), ("events", ctypes.c_void_p * 8),
                ("stall_after_kblocks", ctypes.c_int32), ("timeout_ms", ctypes.c_int32),
                ("trace", ctypes.c_void_p), ("trace_entries", ctypes.c_int32),
                ("force_bn", ctypes.c_int32), ("z", ctypes.c_void_p),
                ("logits", ctypes.c_void_p), ("zsx", ctypes.c_void_p)]


_LIB: Optional[ctypes.CDLL] = None


class KltError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libklt.so (built by ``build.build()``); raises if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libklt.so not built at {path}; run "
                           "latent_moe_layer_route_gb300.build.build() first")
    lib = ctypes.CDLL(path)
    lib.klt_create.argtypes = [ctypes.POINTER(KltDims), ctypes.POINTER(KltWeights),
                               ctypes.c_uint32, ctypes.POINTER(ctypes.c_void_p)]
    lib.klt_create.restype = ctypes.c_int
    lib.klt_forward.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                ctypes.POINTER(KltRouting), ctypes.POINTER(KltDebug),
                                ctypes.c_void_p]
    lib.klt_forward.restype = ctypes.c_int
    lib.klt_forward_hidden.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                       ctypes.c_void_p, ctypes.POINTER(KltRouting),
                                       ctypes.POINTER(KltDebug), ctypes.c_void_p]
    lib.klt_forward_hidden.restype = ctypes.c_int
    lib.klt_status.argtypes = [ctypes.c_void_p]
    lib.klt_status.restype = ctypes.c_int
    lib.klt_destroy.argtypes = [ctypes.c_void_p]
    lib.klt_destroy.restype = ctypes.c_int
    lib.klt_strerror.argtypes = [ctypes.c_int]
    lib.klt_strerror.restype = ctypes.c_char_p
    lib.klt_launch_count.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    lib.klt_launch_count.restype = ctypes.c_int
    lib.klt_gemm_tile.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32]
    lib.klt_gemm_tile.restype = ctypes.c_int
    lib.klt_route_noalloc.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32] + [ctypes.c_void_p] * 8
    lib.klt_route_noalloc.restype = ctypes.c_int
    _LIB = lib
    return lib


def strerror(code: int) -> str:
    return load_library().klt_strerror(code).decode()


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def dims_of(cfg, max_tokens: Optional[int] = None) -> KltDims:
    fmt = {"nvfp4": KLT_FMT_NVFP4, "mxfp8": KLT_FMT_MXFP8,
           "nvfp4_w4a4": KLT_FMT_NVFP4_W4A4}.get(cfg.routed_fmt, KLT_FMT_FP8_B128)
    return KltDims(cfg.H, cfg.L, cfg.E, cfg.topk, cfg.I, cfg.Is, fmt, cfg.eps,
                   cfg.M if max_tokens is None else max_tokens)


def weights_of(w: Dict) -> KltWeights:
    """Weight dict (CUDA tensors, names as produced by ``inputs.make_weights``, plus the
    optional ``w_lat``/``w_gate`` of ``inputs.make_projection_weights``)."""
    proj = (_ptr(w.get("w_lat")), _ptr(w.get("w_gate")))
    if "w13_sx" in w:  # MXFP8: UE8M0 scale bytes per 32 K-elements
        return KltWeights(_ptr(w["w13_q"]), _ptr(w["w13_sx"]), None, _ptr(w["w2_q"]),
                          _ptr(w["w2_sx"]), None, _ptr(w["ws13"]), _ptr(w["ws2"]),
                          _ptr(w["w_up"]), _ptr(w["gamma"]), *proj)
    if "w13_s" in w:
        return KltWeights(_ptr(w["w13_q"]), _ptr(w["w13_s"]), None, _ptr(w["w2_q"]),
                          _ptr(w["w2_s"]), None, _ptr(w["ws13"]), _ptr(w["ws2"]),
                          _ptr(w["w_up"]), _ptr(w["gamma"]), *proj)
    return KltWeights(_ptr(w["w13_q"]), _ptr(w["w13_sb"]), _ptr(w["w13_g"]), _ptr(w["w2_q"]),
                      _ptr(w["w2_sb"]), _ptr(w["w2_g"]), _ptr(w["ws13"]), _ptr(w["ws2"]),
                      _ptr(w["w_up"]), _ptr(w["gamma"]), *proj)


def klt_create(dims: KltDims, weights: KltWeights, flags: int = 0) -> ctypes.c_void_p:
    lib = load_library()
    h = ctypes.c_void_p()
    rc = lib.klt_create(ctypes.byref(dims), ctypes.byref(weights), flags, ctypes.byref(h))
    if rc != KLT_OK:
        raise KltError(rc, "klt_create")
    return h


def klt_forward(h, x, z, logits, M: int, out, routing: Optional[KltRouting] = None,
                debug: Optional[KltDebug] = None, stream: Optional[int] = None) -> int:
    lib = load_library()
    return lib.klt_forward(h, _ptr(x), _ptr(z), _ptr(logits), M, _ptr(out),
                           ctypes.byref(routing) if routing is not None else None,
                           ctypes.byref(debug) if debug is not None else None,
                           stream)


def klt_forward_hidden(h, x, M: int, out, routing: Optional[KltRouting] = None,
                       debug: Optional[KltDebug] = None, stream: Optional[int] = None) -> int:
    lib = load_library()
    return lib.klt_forward_hidden(h, _ptr(x), M, _ptr(out),
                                  ctypes.byref(routing) if routing is not None else None,
                                  ctypes.byref(debug) if debug is not None else None, stream)


def klt_status(h) -> int:
    return load_library().klt_status(h)


def klt_destroy(h) -> int:
    return load_library().klt_destroy(h)


def klt_launch_count(h, M: int) -> int:
    return load_library().klt_launch_count(h, M)


def klt_gemm_tile(h, M: int, force_bn: int = 0) -> int:
    return load_library().klt_gemm_tile(h, M, force_bn)


def klt_route_noalloc(logits, topk: int, ids, weights, cnt, off, gidx, slot, pos,
                      stream: Optional[int] = None) -> int:
    """Routing + permutation with no device allocation (fixed internal scratch); tensors
    are caller-owned CUDA tensors with the klt_routing layouts."""
    M, E = logits.shape
    return load_library().klt_route_noalloc(
        _ptr(logits), M, E, topk, _ptr(ids), _ptr(weights), _ptr(cnt), _ptr(off), _ptr(gidx),
        _ptr(slot), _ptr(pos), stream)


class LatentMoETail:
    """One tail layer on the current CUDA device (owns a klt handle)."""

    def __init__(self, cfg, weights: Dict, max_tokens: Optional[int] = None, flags: int = 0):
        self.cfg = cfg
        self.max_tokens = cfg.M if max_tokens is None else max_tokens
        self.handle = klt_create(dims_of(cfg, self.max_tokens), weights_of(weights), flags)

    def forward(self, x, z, logits, out=None, routing: Optional[KltRouting] = None,
                debug: Optional[KltDebug] = None, stream=None):
        import torch
        M = x.shape[0]
        if out is None:
            out = torch.empty((M, self.cfg.H), dtype=torch.bfloat16, device=x.device)
        if stream is None:
            stream = torch.cuda.current_stream(x.device).cuda_stream
        rc = klt_forward(self.handle, x, z, logits, M, out, routing, debug, stream)
        if rc != KLT_OK:
            raise KltError(rc, "klt_forward")
        return out

    __call__ = forward

    def forward_hidden(self, x, out=None, routing: Optional[KltRouting] = None,
                       debug: Optional[KltDebug] = None, stream=None):
        """The step before the tail (latent input and router logits from x), then the
        tail; the handle must have been created with ``w_lat`` and ``w_gate``."""
        import torch
        M = x.shape[0]
        if out is None:
            out = torch.empty((M, self.cfg.H), dtype=torch.bfloat16, device=x.device)
        if stream is None:
            stream = torch.cuda.current_stream(x.device).cuda_stream
        rc = klt_forward_hidden(self.handle, x, M, out, routing, debug, stream)
        if rc != KLT_OK:
            raise KltError(rc, "klt_forward_hidden")
        return out

    def status(self) -> int:
        return klt_status(self.handle)

    def launch_count(self, M: int) -> int:
        return klt_launch_count(self.handle, M)

    def gemm_tile(self, M: int, force_bn: int = 0) -> int:
        """256 for the token-major engine, else the feature-major engine's token tile."""
        return klt_gemm_tile(self.handle, M, force_bn)

    def close(self):
        if self.handle is not None and self.handle.value:
            klt_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
