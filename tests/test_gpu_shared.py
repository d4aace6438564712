"""GPU parity of the batch-shared selection (moe_reader_decode_shared) against
the oracle's decode_shared: the batch's kept set bit-exact except channels
whose batch score lies within the band of the K-th, every token's output
within the tolerances, read accounting exact; at batch 1 it is the per-token
decode.  Shapes: a small layer, a GPT-OSS-like layer with up to 32 tokens per
expert, and the full Qwen3-30B-A3B-shaped layer at batch 16."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from calibration_free_sparse_gb300 import reader as RD
from oracle import reader as R
from tests import gpu_common as C

pytestmark = pytest.mark.gpu


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def decode_shared_gpu(pair, x, ids, w, k):
    torch = _torch()
    xd = torch.from_numpy(x).cuda()
    y = torch.empty_like(xd)
    pair.reader.decode_shared(xd, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), k, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check_against_oracle(pair, x, ids, w, k, band=C.KEPT_BAND, tokens=None):
    y = decode_shared_gpu(pair, x, ids, w, k)
    assert pair.reader.status() == (0, 0)
    kept = pair.reader.kept_shared()
    B, I = x.shape[0], pair.shape.I
    gm = C.gpu_masks(pair, B)
    res = R.decode_shared(pair.layer, x, ids, w, k)
    if any(not np.array_equal(gm[t], res.tokens[t].mask) for t in range(B)):
        for t in range(B):
            if not np.array_equal(gm[t], res.tokens[t].mask):
                C.check_near_tie(pair, x[t], res.tokens[t], gm[t])
        res = R.decode_shared(pair.layer, x, ids, w, k, masks=gm)
    assert kept.size == res.K
    got, ref = set(int(v) for v in kept), set(int(v) for v in res.kept)
    diff = got ^ ref
    if diff:
        rank = {int(e): r for r, e in enumerate(res.experts)}
        for g in diff:
            sc = res.batch_score[rank[g // I], g % I]
            assert abs(sc - res.kth_score) <= band * res.kth_score, (g, sc, res.kth_score)
    for t in (range(B) if tokens is None else tokens):
        C.assert_y_close(y[t], res.tokens[t].y)
    # read accounting of the kernel's own screened sets and kept set, always
    mine = [np.array([g for g in kept if int(g) // I in set(int(e) for e in ids[t])], np.int64)
            for t in range(B)]
    st = C.assert_read_accounting(pair, ids, gm, mine)
    if not diff:
        refs = C.oracle_sectors(pair, ids, res.tokens)
        for name in refs:
            assert st[name] == refs[name], name
    return y, kept, res, len(diff)


@pytest.fixture(scope="module")
def small():
    _torch()
    return C.Pair(256, 8, 2, 256, 80, 8, max_batch=8, seed=41)


@pytest.mark.parametrize("B", [1, 3, 8])
def test_small_against_oracle(small, B):
    x, ids, w = small.tokens(B, 500 + B)
    check_against_oracle(small, x, ids, w, 92)


@pytest.mark.parametrize("k", [0, 1, 511, 512])
def test_small_edge_budgets(small, k):
    x, ids, w = small.tokens(5, 600 + k)
    y, kept, res, _ = check_against_oracle(small, x, ids, w, k)
    if k == small.shape.N:
        assert kept.size == res.experts.size * small.shape.I


def test_batch_of_one_is_the_per_token_decode(small):
    x, ids, w = small.tokens(1, 650)
    ys = decode_shared_gpu(small, x, ids, w, 92)
    kept_s = small.reader.kept_shared()
    yp = small.decode_gpu(x, ids, w, 92)
    kept_p = small.reader.kept(1, 92)[0]
    assert np.array_equal(kept_s, kept_p)
    assert np.abs(ys - yp).max() <= 1e-5 * np.abs(yp).max()


def test_identical_tokens_keep_the_per_token_set(small):
    x, ids, w = small.tokens(1, 660)
    B = 6
    xb, idb, wb = (np.ascontiguousarray(np.repeat(a, B, 0)) for a in (x, ids, w))
    ys = decode_shared_gpu(small, xb, idb, wb, 92)
    kept_s = small.reader.kept_shared()
    yp = small.decode_gpu(x, ids, w, 92)
    assert np.array_equal(kept_s, small.reader.kept(1, 92)[0])
    for t in range(B):
        assert np.abs(ys[t] - yp[0]).max() <= 1e-5 * np.abs(yp).max()


def test_kept_readout_states(small):
    x, ids, w = small.tokens(2, 670)
    small.decode_gpu(x, ids, w, 92)
    with pytest.raises(RD.ReaderError) as e:
        small.reader.kept_shared()
    assert e.value.code == RD.ESTATE
    decode_shared_gpu(small, x, ids, w, 92)
    with pytest.raises(RD.ReaderError) as e:
        small.reader.kept(2, 92)
    assert e.value.code == RD.ESTATE


@pytest.fixture(scope="module")
def gptoss_like():
    _torch()
    return C.Pair(2880, 8, 4, 2880, 80, 32, max_batch=64, seed=43)


@pytest.mark.parametrize("B", [16, 64])
def test_many_tokens_per_expert(gptoss_like, B):
    """B 64 routes 32 tokens to an expert on average: each kept row serves
    them all.  The oracle checks sampled tokens."""
    k = S.budget_to_k(0.178, 4 * 2880)
    x, ids, w = gptoss_like.tokens(B, 700 + B)
    check_against_oracle(gptoss_like, x, ids, w, k, tokens=sorted({0, B // 2, B - 1}))


@pytest.fixture(scope="module")
def qwen3():
    _torch()
    WL = S.QWEN3_30B
    return C.Pair(WL.H, WL.E, WL.topk, WL.I, WL.c, WL.r, max_batch=16, seed=47,
                  device_weights=True)


def test_qwen3_30b_batch16(qwen3):
    WL = S.QWEN3_30B
    x, ids, w = qwen3.tokens(16, 810)
    y, kept, res, nd = check_against_oracle(qwen3, x, ids, w, WL.k, tokens=(0, 7, 15))
    # the shared set reads fewer kept rows than the union of per-token sets
    st_shared = qwen3.reader.stats()
    qwen3.decode_gpu(x, ids, w, WL.k)
    st_tok = qwen3.reader.stats()
    assert st_shared["G"] < st_tok["G"]
