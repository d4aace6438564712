"""Failure detection on the GPU without faulting it: every failure is made on
purpose through the library's one-shot injections (a wait on a count that
nothing reaches, a grid barrier that waits for a CTA that was never
launched, an allocation reported as failed), the bounded waits run out after
the limit the test sets, the error surfaces as a status, and the next call on
the same handle is clean and in parity with the oracle."""

import time

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from calibration_free_sparse_gb300 import reader as RD
from oracle import reader as R
from tests import gpu_common as C

pytestmark = pytest.mark.gpu

H, E, TOPK, I, CC, RANK, K = 256, 16, 2, 128, 80, 8, 32


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def pair():
    _torch()
    return C.Pair(H, E, TOPK, I, CC, RANK, max_batch=4, seed=0)


def test_decode_wait_runs_out_and_the_next_decode_is_clean(pair):
    x, ids, w = pair.tokens(3, 5)
    pair.reader.set_wait_limit(2_000_000)                  # 2 ms
    RD.inject_fault(RD.INJECT_DECODE_STALL, pair.reader)
    t0 = time.perf_counter()
    pair.decode_gpu(x, ids, w, K)
    code, bits = pair.reader.status()
    assert code == RD.ETIMEOUT and bits & RD.ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0                  # bounded, far from the 1 s default
    # the injection fired once: the next decode, normal limit, is clean and in parity
    pair.reader.set_wait_limit(0)
    y = pair.decode_gpu(x, ids, w, K)
    assert pair.reader.status() == (RD.OK, 0)
    C.check_decode(pair, x, ids, w, K, y)


def test_host_decode_reports_the_timeout(pair):
    x, ids, w = pair.tokens(2, 6)
    pair.reader.set_wait_limit(2_000_000)
    RD.inject_fault(RD.INJECT_DECODE_STALL, pair.reader)
    with pytest.raises(RD.ReaderError) as e:
        pair.reader.decode_host(x, ids, w, K)
    assert e.value.code == RD.ETIMEOUT
    pair.reader.set_wait_limit(0)
    y = pair.reader.decode_host(x, ids, w, K)
    C.check_decode(pair, x, ids, w, K, y)


def test_shared_decode_wait_runs_out(pair):
    torch = _torch()
    x, ids, w = pair.tokens(3, 7)
    pair.reader.set_wait_limit(2_000_000)
    RD.inject_fault(RD.INJECT_DECODE_STALL, pair.reader)
    xd = torch.from_numpy(x).cuda()
    y = torch.empty_like(xd)
    pair.reader.decode_shared(xd, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), K, y)
    code, bits = pair.reader.status()
    assert code == RD.ETIMEOUT and bits & RD.ERR_TIMEOUT
    pair.reader.set_wait_limit(0)
    pair.reader.decode_shared(xd, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), K, y)
    torch.cuda.synchronize()
    assert pair.reader.status() == (RD.OK, 0)
    res = R.decode_shared(pair.layer, x, ids, w, K)
    for t in range(3):
        C.assert_y_close(y[t].cpu().numpy(), res.tokens[t].y)


def test_stack_layer_timeout_reaches_later_layers():
    torch = _torch()
    L, B, k = 3, 2, 92
    pairs = [C.Pair(256, 8, 2, 256, 80, 8, max_batch=B, seed=30 + l) for l in range(L)]
    readers = [p.reader for p in pairs]
    h0 = S.activations(31, B, 256)
    ids = np.ascontiguousarray(np.stack([S.routing(40 + l, B, 8, 2)[0] for l in range(L)]))
    w = np.ascontiguousarray(np.stack([S.routing(40 + l, B, 8, 2)[1] for l in range(L)]))
    hd, idd, wd = (torch.from_numpy(a).cuda() for a in (h0, ids, w))
    hout = torch.empty_like(hd)
    ys = torch.empty((L, B, 256), device="cuda")
    readers[1].set_wait_limit(2_000_000)
    RD.inject_fault(RD.INJECT_DECODE_STALL, readers[1])
    RD.decode_stack(readers, hd, idd, wd, k, hout, ys)
    torch.cuda.synchronize()
    assert readers[0].status() == (RD.OK, 0)
    for rd in readers[1:]:                  # the stalled layer and the one it feeds
        code, bits = rd.status()
        assert code == RD.ETIMEOUT and bits & RD.ERR_TIMEOUT
    # the next step on the same handles is clean: exact residual chain, layers in parity
    readers[1].set_wait_limit(0)
    RD.decode_stack(readers, hd, idd, wd, k, hout, ys)
    torch.cuda.synchronize()
    for rd in readers:
        assert rd.status() == (RD.OK, 0)
    y = ys.cpu().numpy()
    h = h0.astype(np.float32)
    for l, p in enumerate(pairs):
        ss = np.sum(h.astype(np.float64) ** 2, axis=-1, keepdims=True)
        x = (h * (1.0 / np.sqrt(ss / 256 + 1e-6)).astype(np.float32)).astype(np.float32)
        C.check_decode(p, x, ids[l], w[l], k, y[l])
        h = (h + y[l]).astype(np.float32)
    assert np.array_equal(hout.cpu().numpy(), h)


def test_prepare_barrier_timeout_then_prepare_works():
    _torch()
    RD.inject_fault(RD.INJECT_PREPARE_STALL)
    with pytest.raises(RD.ReaderError) as e:
        C.Pair(H, E, TOPK, I, CC, RANK, max_batch=2, seed=3)
    assert e.value.code == RD.ETIMEOUT
    p = C.Pair(H, E, TOPK, I, CC, RANK, max_batch=2, seed=3)     # the injection fired once
    x, ids, w = p.tokens(2, 8)
    y = p.decode_gpu(x, ids, w, K)
    assert p.reader.status() == (RD.OK, 0)
    C.check_decode(p, x, ids, w, K, y)


def test_allocation_failure_is_enomem_and_leaks_nothing():
    torch = _torch()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    RD.inject_fault(RD.INJECT_ALLOC_FAIL)
    with pytest.raises(RD.ReaderError) as e:
        C.Pair(H, E, TOPK, I, CC, RANK, max_batch=2, seed=4)
    assert e.value.code == RD.ENOMEM
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free1 - free0) < (64 << 20)        # the weights the test itself uploaded
    p = C.Pair(H, E, TOPK, I, CC, RANK, max_batch=2, seed=4)
    x, ids, w = p.tokens(2, 9)
    p.decode_gpu(x, ids, w, K)
    RD.inject_fault(RD.INJECT_ALLOC_FAIL)          # get_kept's staging allocation
    with pytest.raises(RD.ReaderError) as e:
        p.reader.kept(2, K)
    assert e.value.code == RD.ENOMEM
    assert p.reader.kept(2, K).shape == (2, K)
