"""GPU parity on the full GPT-OSS-120B-shaped layer (H 2880 zero-padded to
2944, E 32, top-4, I 2880, c 80, r 32, k 1417 = the 17.8% read budget) from
batch 1 up to the large-batch stress of batch 128: the oracle on batch 1 and
on sampled tokens of batch 128 (it computes tokens one by one), and, for every
token of batch 128, the per-token identity that holds at any size: a token's
kept set and output do not depend on the batch it is decoded in."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
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
    C.check_decode(pair, x, ids, w, WL.k, y)


@pytest.mark.parametrize("B", [16, BMAX])
def test_large_batch(pair, B):
    x, ids, w = pair.tokens(B, 700 + B)
    y = pair.decode_gpu(x, ids, w, WL.k)
    assert pair.reader.status() == (0, 0)
    kept = pair.reader.kept(B, WL.k)
    # sampled tokens against the oracle; read accounting of the whole batch
    C.check_decode(pair, x, ids, w, WL.k, y, tokens=sorted({0, 1, B // 2, B - 1}))
    # every token: the same result when decoded in batches of 8
    for t0 in range(0, B, 8):
        sl = slice(t0, min(B, t0 + 8))
        ys = pair.decode_gpu(x[sl], ids[sl], w[sl], WL.k)
        assert pair.reader.status() == (0, 0)
        ks = pair.reader.kept(ys.shape[0], WL.k)
        assert np.array_equal(ks, kept[sl]), t0
        scale = np.abs(y[sl]).max(axis=1, keepdims=True)
        assert np.all(np.abs(ys - y[sl]) <= 1e-5 * scale), t0
