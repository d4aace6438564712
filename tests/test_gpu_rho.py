"""GPU parity of the full-screen ranking by the expected squared output error
(MOE_READER_FLAG_RHO_RANK) against the oracle's decode_token_rho: kept sets
bit-exact except channels whose key lies within the band of the k-th, y
within the tolerances, the ranking keys (exported scores) close to the
oracle's; configuration errors."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from calibration_free_sparse_gb300 import reader as RD
from oracle import reader as R
from tests import gpu_common as C

pytestmark = pytest.mark.gpu

SHAPES = {
    "small": dict(H=256, E=8, topk=2, I=256, r=8, budget=0.287, batches=(1, 3)),
    "qwen3_like": dict(H=2048, E=16, topk=8, I=768, r=32, budget=0.35, batches=(1, 2)),
}


@pytest.fixture(scope="module", params=sorted(SHAPES))
def case(request):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sh = SHAPES[request.param]
    pair = C.Pair(sh["H"], sh["E"], sh["topk"], sh["I"], 128, sh["r"],
                  max_batch=max(sh["batches"]), seed=23, flags=RD.FLAG_RHO_RANK)
    k = S.budget_to_k(sh["budget"], sh["topk"] * sh["I"])
    return request.param, sh, pair, k


def test_against_oracle(case):
    name, sh, pair, k = case
    for B in sh["batches"]:
        x, ids, w = pair.tokens(B, 900 + B)
        y = pair.decode_gpu(x, ids, w, k)
        assert pair.reader.status() == (0, 0), name
        kept = pair.reader.kept(B, k)
        keys = pair.reader.export("score")
        gm = C.gpu_masks(pair, B)
        assert gm.all()                      # the full screen reads every coordinate
        for t in range(B):
            res = R.decode_token_rho(pair.layer, x[t], ids[t], w[t], k)
            ref = res.score.reshape(-1)
            assert np.abs(keys[t] - ref).max() <= 1e-4 * np.abs(ref).max(), name
            C.assert_kept_match(kept[t], res, ids[t], k)
            C.assert_y_close(y[t], res.y)
        C.assert_read_accounting(pair, ids, gm, [kept[t] for t in range(B)])


def test_flag_needs_the_full_screen():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    with pytest.raises(RD.ReaderError) as e:
        C.Pair(256, 4, 2, 64, 80, 8, max_batch=2, seed=1, flags=RD.FLAG_RHO_RANK)
    assert e.value.code == RD.EINVAL
