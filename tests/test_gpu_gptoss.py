"""GPU parity on the full GPT-OSS-120B-shaped layer (H 2880 zero-padded to
2944, E 32, top-4, I 2880, c 80, r 32, k 1417 = the 17.8% read budget) from
batch 1 up to the large-batch stress of batch 128: the oracle on batch 1 and
on sampled tokens of batch 128 (it computes tokens one by one), and, for every
token of batch 128, the per-token identity that holds at any size: a token's
kept set and output do not depend on the batch it is decoded in."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from oracle import reader as R
from tests import gpu_common as C

pytestmark = pytest.mark.gpu

WL = S.GPT_OSS_120B
BMAX = 128


@pytest.fixture(scope="module")
def pair():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return C.Pair(WL.H, WL.E, WL.topk, WL.I, WL.c, WL.r, max_batch=BMAX, seed=5,
                  device_weights=True)


def test_batch1_against_oracle(pair):
    x, ids, w = pair.tokens(1, 600)
    y = pair.decode_gpu(x, ids, w, WL.k)
    assert pair.reader.status() == (0, 0)
    res = R.decode(pair.layer, x, ids, w, WL.k)
    kept = pair.reader.kept(1, WL.k)
    nd = C.assert_kept_match(kept[0], res[0], ids[0], WL.k)
    C.assert_y_close(y[0], res[0].y)
    if nd == 0:
        st = pair.reader.stats()
        ref = C.oracle_sectors(pair, ids, res)
        for name in ref:
            assert st[name] == ref[name], name


@pytest.mark.parametrize("B", [16, BMAX])
def test_large_batch(pair, B):
    x, ids, w = pair.tokens(B, 700 + B)
    y = pair.decode_gpu(x, ids, w, WL.k)
    assert pair.reader.status() == (0, 0)
    kept = pair.reader.kept(B, WL.k)
    # sampled tokens against the oracle
    for t in sorted({0, 1, B // 2, B - 1}):
        res = R.decode_token(pair.layer, x[t], ids[t], w[t], WL.k)
        C.assert_kept_match(kept[t], res, ids[t], WL.k)
        C.assert_y_close(y[t], res.y)
    # every token: the same result when decoded in batches of 8
    for t0 in range(0, B, 8):
        sl = slice(t0, min(B, t0 + 8))
        ys = pair.decode_gpu(x[sl], ids[sl], w[sl], WL.k)
        assert pair.reader.status() == (0, 0)
        ks = pair.reader.kept(ys.shape[0], WL.k)
        assert np.array_equal(ks, kept[sl]), t0
        scale = np.abs(y[sl]).max(axis=1, keepdims=True)
        assert np.all(np.abs(ys - y[sl]) <= 1e-5 * scale), t0
