"""Many decode launches on one handle, of every kind, with batches that grow
and shrink, and a launch that aborts in between.  The decode leaves nothing
to reset at the end of a launch: each launch takes a generation from a
counter of CTAs, releases token flags with it, and counters are zeroed by
their last reader.  A word that a launch left behind would make a later
launch read stale counts or kept lists, so every repeated decode here must
reproduce its first result: the same kept lists, the same y up to the order
of fp32 atomic additions."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import reader as RD
from tests import gpu_common as C

pytestmark = pytest.mark.gpu

H, E, TOPK, I, CC, RANK, K = 256, 16, 2, 128, 80, 8, 32
BATCHES = (5, 1, 8, 2, 8, 3)


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def pair():
    _torch()
    return C.Pair(H, E, TOPK, I, CC, RANK, max_batch=8, seed=21)


def _per_token(pair, B, host):
    x, ids, w = pair.tokens(B, 100 + B)
    y = pair.reader.decode_host(x, ids, w, K) if host else pair.decode_gpu(x, ids, w, K)
    assert pair.reader.status() == (RD.OK, 0)
    return y, pair.reader.kept(B, K)


def _shared(pair, torch, seed):
    x, ids, w = pair.tokens(3, seed)
    xd = torch.from_numpy(x).cuda()
    y = torch.empty_like(xd)
    pair.reader.decode_shared(xd, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), K, y)
    torch.cuda.synchronize()
    assert pair.reader.status() == (RD.OK, 0)
    return y.cpu().numpy(), pair.reader.kept_shared()


def _stack(pair, torch, seed):
    B = 4
    x, ids, w = pair.tokens(B, seed)
    h_in = torch.from_numpy(x).cuda()
    h_out = torch.empty_like(h_in)
    y_layers = torch.empty((1, B, H), device="cuda")
    RD.decode_stack([pair.reader], h_in, torch.from_numpy(ids[None]).cuda(),
                    torch.from_numpy(w[None]).cuda(), K, h_out, y_layers)
    torch.cuda.synchronize()
    assert pair.reader.status() == (RD.OK, 0)
    return y_layers[0].cpu().numpy()


def _same_y(a, b):
    scale = np.abs(a).max(axis=1, keepdims=True) + 1e-30
    return (np.abs(b - a) / scale).max() <= 1e-5


def test_repeated_launches_of_every_kind(pair):
    torch = _torch()
    # the first decode of each batch size on this handle, against the oracle
    refs = {}
    for B in sorted(set(BATCHES)):
        y, kept = _per_token(pair, B, host=False)
        x, ids, w = pair.tokens(B, 100 + B)
        C.check_decode(pair, x, ids, w, K, y)
        refs[B] = (y, kept)
    y_sh0, k_sh0 = _shared(pair, torch, 300)
    y_st0 = _stack(pair, torch, 400)
    for rep in range(4):
        for i, B in enumerate(BATCHES):
            y, kept = _per_token(pair, B, host=(rep + i) % 3 == 0)
            assert np.array_equal(kept, refs[B][1]), (rep, i, B)
            assert _same_y(refs[B][0], y), (rep, i, B)
            if i % 2 == 1:   # a batch-shared decode in between
                y_sh, k_sh = _shared(pair, torch, 300)
                assert np.array_equal(k_sh, k_sh0) and _same_y(y_sh0, y_sh), (rep, i)
            if i == 2:       # a one-layer stack in between
                assert _same_y(y_st0, _stack(pair, torch, 400)), (rep, i)
            if rep == 1 and i == 3:
                # a launch that gives up on a wait; the status call clears the
                # handle's words and the next launches carry on
                pair.reader.set_wait_limit(2_000_000)
                RD.inject_fault(RD.INJECT_DECODE_STALL, pair.reader)
                x, ids, w = pair.tokens(B, 100 + B)
                pair.decode_gpu(x, ids, w, K)
                code, bits = pair.reader.status()
                assert code == RD.ETIMEOUT and bits & RD.ERR_TIMEOUT
                pair.reader.set_wait_limit(0)
