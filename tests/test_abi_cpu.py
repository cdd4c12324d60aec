"""The C-ABI library loads, exports every entry point declared in include/klt.h and rejects
bad arguments on the host before touching a device.  No compute call runs here."""
import ctypes
import os
import re

import pytest

from latent_moe_layer_route_gb300 import binding as B
from latent_moe_layer_route_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "klt.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(klt_\w+)\s*\(", text, re.M)))


def test_header_declares_binding_exports():
    assert declared_functions() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror(lib):
    assert B.strerror(B.KLT_OK) == "ok"
    assert "timeout" in B.strerror(B.KLT_ERR_DEVICE_TIMEOUT) or "expired" in B.strerror(
        B.KLT_ERR_DEVICE_TIMEOUT)
    assert B.strerror(12345) == "unknown status"


def _dims(**kw):
    base = dict(H=256, L=256, E=4, topk=2, I=128, Is=128, routed_fmt=B.KLT_FMT_FP8_B128,
                eps=1e-6, max_tokens=8)
    base.update(kw)
    return B.KltDims(**base)


def _create(lib, dims, weights):
    h = ctypes.c_void_p()
    rc = lib.klt_create(ctypes.byref(dims) if dims is not None else None,
                        ctypes.byref(weights) if weights is not None else None, 0,
                        ctypes.byref(h))
    return rc, h


def test_create_rejects_null_and_bad_shapes(lib):
    w = B.KltWeights(*([0x1000] * 10))
    assert _create(lib, None, w)[0] == B.KLT_ERR_INVALID_ARG
    assert _create(lib, _dims(), None)[0] == B.KLT_ERR_INVALID_ARG
    assert lib.klt_create(ctypes.byref(_dims()), ctypes.byref(w), 0, None) == \
        B.KLT_ERR_INVALID_ARG
    assert _create(lib, _dims(H=200), w)[0] == B.KLT_ERR_UNSUPPORTED
    assert _create(lib, _dims(I=100), w)[0] == B.KLT_ERR_UNSUPPORTED
    assert _create(lib, _dims(topk=5), w)[0] == B.KLT_ERR_UNSUPPORTED
    assert _create(lib, _dims(E=300, topk=2), w)[0] == B.KLT_ERR_UNSUPPORTED
    assert _create(lib, _dims(routed_fmt=7), w)[0] == B.KLT_ERR_UNSUPPORTED
    assert _create(lib, _dims(eps=0.0), w)[0] == B.KLT_ERR_INVALID_ARG
    assert _create(lib, _dims(max_tokens=0), w)[0] == B.KLT_ERR_INVALID_ARG
    assert _create(lib, _dims(max_tokens=1 << 20, topk=2), w)[0] == B.KLT_ERR_UNSUPPORTED
    # one past the largest supported sizes: 32 k-blocks of L and I, 32 choices per token
    assert _create(lib, _dims(L=4224), w)[0] == B.KLT_ERR_UNSUPPORTED
    assert _create(lib, _dims(I=4224), w)[0] == B.KLT_ERR_UNSUPPORTED
    assert _create(lib, _dims(E=64, topk=33), w)[0] == B.KLT_ERR_UNSUPPORTED


def test_create_rejects_the_deterministic_combine_with_phased_launches(lib):
    w = B.KltWeights(*([0x1000] * 10))
    h = ctypes.c_void_p()
    flags = B.KLT_FLAG_DETERMINISTIC | B.KLT_FLAG_PHASED
    assert lib.klt_create(ctypes.byref(_dims()), ctypes.byref(w), flags, ctypes.byref(h)) == \
        B.KLT_ERR_UNSUPPORTED
    assert not h.value


def test_create_rejects_null_and_misaligned_weight_pointers(lib):
    ptrs = [0x1000] * 10
    ptrs[2] = ptrs[5] = 0  # fp8 layers do not use the global scales
    for i in (0, 1, 3, 4, 6, 7, 8, 9):
        p = list(ptrs)
        p[i] = 0
        assert _create(lib, _dims(), B.KltWeights(*p))[0] == B.KLT_ERR_INVALID_ARG, i
        p[i] = 0x1008
        assert _create(lib, _dims(), B.KltWeights(*p))[0] == B.KLT_ERR_ALIGN, i


def test_forward_and_status_reject_null_handle(lib):
    assert lib.klt_forward(None, None, None, None, 4, None, None, None, None) == \
        B.KLT_ERR_INVALID_ARG
    assert lib.klt_status(None) == B.KLT_ERR_INVALID_ARG
    assert lib.klt_destroy(None) == B.KLT_OK
    assert lib.klt_launch_count(None, 16) == 0
    assert lib.klt_gemm_tile(None, 16, 0) == -B.KLT_ERR_INVALID_ARG


def test_forward_hidden_rejects_null_handle(lib):
    assert lib.klt_forward_hidden(None, None, 4, None, None, None, None) == \
        B.KLT_ERR_INVALID_ARG


def test_create_wants_both_projection_weights_or_neither(lib):
    ptrs = [0x1000] * 12
    ptrs[2] = ptrs[5] = 0
    for i in (10, 11):  # only one of w_lat / w_gate
        p = list(ptrs)
        p[i] = 0
        assert _create(lib, _dims(), B.KltWeights(*p))[0] == B.KLT_ERR_INVALID_ARG, i
    p = list(ptrs)
    p[11] = 0x1008
    assert _create(lib, _dims(), B.KltWeights(*p))[0] == B.KLT_ERR_ALIGN
