"""GPU parity on layer shapes that take the other paths of the decode kernel:
an odd screened-coordinate count, padded coordinate runs and a padded hidden
size, several code words per thread, multi-chunk staging and the largest
routed width the configuration allows.  Expert counts are cut down so the
fp64 oracle (whose recovery basis needs the whole layer's Gram matrix)
finishes in seconds; every other dimension is the named model's.

  odd_c_wide       H 512,  E 8, top-2, I 1536, c 81, r 16
  gpt_oss_like     H 2880 (Hp 2944), E 8, top-4, I 2880 (run 720 -> 736 bytes), c 80, r 32
  qwen3_235b_like  H 4096, E 8, top-8, I 1536, c 80, r 32, 12.8% read budget
  wide_inter       H 256,  E 4, top-2, I 4160 (run 1040 -> 1056 bytes), c 80, r 8
  max_inter        H 128,  E 4, top-4, I 8192 (N = 32768), c 128, r 4
"""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from tests import gpu_common as C

pytestmark = pytest.mark.gpu

SHAPES = {
    "odd_c_wide": dict(H=512, E=8, topk=2, I=1536, c=81, r=16, budget=0.178, batches=(1, 5)),
    "gpt_oss_like": dict(H=2880, E=8, topk=4, I=2880, c=80, r=32, budget=0.178, batches=(1, 3)),
    "qwen3_235b_like": dict(H=4096, E=8, topk=8, I=1536, c=80, r=32, budget=0.128, batches=(1, 2)),
    "wide_inter": dict(H=256, E=4, topk=2, I=4160, c=80, r=8, budget=0.178, batches=(2,)),
    "max_inter": dict(H=128, E=4, topk=4, I=8192, c=128, r=4, budget=0.178, batches=(1, 2)),
}


@pytest.fixture(scope="module", params=sorted(SHAPES))
def case(request):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sh = SHAPES[request.param]
    pair = C.Pair(sh["H"], sh["E"], sh["topk"], sh["I"], sh["c"], sh["r"],
                  max_batch=max(sh["batches"]), seed=11)
    k = S.budget_to_k(sh["budget"], sh["topk"] * sh["I"])
    return request.param, sh, pair, k


def test_decode_parity(case):
    name, sh, pair, k = case
    for B in sh["batches"]:
        x, ids, w = pair.tokens(B, 40 + B)
        y = pair.decode_gpu(x, ids, w, k)
        assert pair.reader.status() == (0, 0), name
        C.check_decode(pair, x, ids, w, k, y)


def test_screen_estimates(case):
    """ghat and vhat of every routed channel against the oracle's sketch sums."""
    name, sh, pair, k = case
    B = sh["batches"][-1]
    x, ids, w = pair.tokens(B, 70 + B)
    y = pair.decode_gpu(x, ids, w, k)
    res, _, _ = C.check_decode(pair, x, ids, w, k, y)
    ghat = pair.reader.export("ghat")
    vhat = pair.reader.export("vhat")
    for t in range(B):
        rg = res[t].ghat.reshape(-1)
        rv = res[t].vhat.reshape(-1)
        assert np.abs(ghat[t] - rg).max() <= 1e-5 * np.abs(rg).max(), name
        assert np.abs(vhat[t] - rv).max() <= 1e-5 * np.abs(rv).max(), name
