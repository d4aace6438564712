"""Host-side argument checks of the C ABI that return before any device work
(no GPU): every configuration rule of moe_reader_prepare, and the null or
malformed arguments of the decode, stack, shared and readout entry points."""

import ctypes

import numpy as np
import pytest

from calibration_free_sparse_gb300 import build as B
from calibration_free_sparse_gb300 import reader as RD


@pytest.fixture(scope="module")
def lib():
    lib = ctypes.CDLL(B.build())
    lib.moe_reader_prepare.restype = ctypes.c_int
    lib.moe_reader_prepare.argtypes = [ctypes.POINTER(RD.Config)] + [ctypes.c_void_p] * 5 + [
        ctypes.POINTER(ctypes.c_void_p)]
    return lib


GOOD = dict(hidden=256, num_experts=8, experts_per_token=2, inter=128, screen_coords=80, rank=8,
            max_batch=4, flags=0)
FAKE = 256 * 1024   # an aligned address that is never dereferenced: the checks reject first


def prepare(lib, **over):
    c = dict(GOOD, **over)
    cfg = RD.Config(c["hidden"], c["num_experts"], c["experts_per_token"], c["inter"],
                    c["screen_coords"], c["rank"], c["max_batch"], c["flags"])
    sigma = np.ones(512, np.int8)
    out = ctypes.c_void_p(123)
    code = lib.moe_reader_prepare(ctypes.byref(cfg), FAKE, FAKE, FAKE, sigma.ctypes.data, None,
                                  ctypes.byref(out))
    assert out.value is None   # *out is cleared whenever prepare fails
    return code


@pytest.mark.parametrize("over", [
    dict(flags=4), dict(flags=RD.FLAG_RHO_RANK),            # an unknown bit; the ranking needs c = 128
    dict(flags=RD.FLAG_RHO_RANK | RD.FLAG_TRIT5),
    dict(hidden=100), dict(hidden=0), dict(num_experts=0),
    dict(experts_per_token=9), dict(experts_per_token=0),
    dict(inter=96), dict(inter=0), dict(inter=16384),
    dict(screen_coords=0), dict(screen_coords=129),
    dict(rank=0), dict(rank=65), dict(max_batch=0), dict(max_batch=1025),
])
def test_configuration_rules(lib, over):
    assert prepare(lib, **over) == RD.EINVAL


def test_sigma_must_be_signs(lib):
    cfg = RD.Config(256, 8, 2, 128, 80, 8, 4, 0)
    out = ctypes.c_void_p()
    sigma = np.ones(256, np.int8)
    sigma[7] = 0
    assert lib.moe_reader_prepare(ctypes.byref(cfg), FAKE, FAKE, FAKE, sigma.ctypes.data, None,
                                  ctypes.byref(out)) == RD.EINVAL
    # misaligned weights
    assert lib.moe_reader_prepare(ctypes.byref(cfg), FAKE + 16, FAKE, FAKE,
                                  np.ones(256, np.int8).ctypes.data, None,
                                  ctypes.byref(out)) == RD.EINVAL


def test_null_handles_and_arguments(lib):
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.moe_reader_decode_shared.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp]
    lib.moe_reader_decode_stack.argtypes = [vp, i32, vp, i32, vp, vp, i32, vp, vp, vp]
    lib.moe_reader_get_kept_shared.argtypes = [vp, vp, i64, ctypes.POINTER(ctypes.c_int32)]
    lib.moe_reader_get_kept.argtypes = [vp, vp, i64]
    lib.moe_reader_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    assert lib.moe_reader_decode_shared(None, None, 1, None, None, 1, None, None) == RD.EINVAL
    assert lib.moe_reader_decode_stack(None, 2, None, 1, None, None, 1, None, None, None) == RD.EINVAL
    layers = (ctypes.c_void_p * 2)(None, None)
    assert lib.moe_reader_decode_stack(layers, 0, None, 1, None, None, 1, None, None, None) == RD.EINVAL
    assert lib.moe_reader_decode_stack(layers, 2, None, 1, None, None, 1, None, None, None) == RD.EINVAL
    K = ctypes.c_int32(0)
    assert lib.moe_reader_get_kept_shared(None, None, 0, ctypes.byref(K)) == RD.EINVAL
    assert lib.moe_reader_get_kept(None, None, 0) == RD.EINVAL
    assert lib.moe_reader_status(None, None) == RD.EINVAL


def test_fault_injection_arguments(lib):
    lib.moe_reader_inject_fault.argtypes = [ctypes.c_void_p, ctypes.c_uint32]
    lib.moe_reader_inject_fault.restype = ctypes.c_int
    lib.moe_reader_set_wait_limit.argtypes = [ctypes.c_void_p, ctypes.c_uint64]
    lib.moe_reader_set_wait_limit.restype = ctypes.c_int
    assert lib.moe_reader_inject_fault(None, 0) == RD.EINVAL              # nothing to inject
    assert lib.moe_reader_inject_fault(None, 0x8) == RD.EINVAL            # unknown bit
    assert lib.moe_reader_inject_fault(None, RD.INJECT_DECODE_STALL) == RD.EINVAL   # needs a handle
    assert lib.moe_reader_set_wait_limit(None, 1000) == RD.EINVAL


def test_injected_allocation_failure_is_enomem(lib):
    """An injected allocation failure makes prepare return ENOMEM before it
    touches a device pointer, on any host; without the injection, a host with
    no GPU fails its first allocation as a CUDA error, not as ENOMEM."""
    lib.moe_reader_inject_fault.argtypes = [ctypes.c_void_p, ctypes.c_uint32]
    lib.moe_reader_inject_fault.restype = ctypes.c_int
    assert lib.moe_reader_inject_fault(None, RD.INJECT_ALLOC_FAIL) == RD.OK
    assert prepare(lib) == RD.ENOMEM
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except ImportError:
        has_gpu = False
    if not has_gpu:   # with a GPU the call would run on the fake weight pointers
        assert prepare(lib) == RD.ECUDA
