"""GPU parity of the five-trits-per-byte sketch (MOE_READER_FLAG_TRIT5, the
pages' ~1.6-bit codes): the stored runs bit-exact against the oracle's
pack_codes5 (TWN threshold ties excused), every decode in parity with the
oracle with its read accounting in the five-trit sector model, and the same
estimates and kept sets as the 2-bit layout of the same layer."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from calibration_free_sparse_gb300 import reader as RD
from oracle import reader as R
from oracle import sectors as SC
from tests import gpu_common as C

pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny": dict(H=256, E=16, topk=2, I=128, c=80, r=8, k=32, batches=(1, 3)),
    "qwen3_like": dict(H=2048, E=16, topk=8, I=768, c=80, r=32, k=756, batches=(1, 4)),
    "odd_c": dict(H=512, E=8, topk=2, I=1536, c=81, r=16, k=None, batches=(2,)),
}


@pytest.fixture(scope="module", params=sorted(SHAPES))
def pairs(request):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sh = SHAPES[request.param]
    p5 = C.Pair(sh["H"], sh["E"], sh["topk"], sh["I"], sh["c"], sh["r"],
                max_batch=max(sh["batches"]), seed=61, flags=RD.FLAG_TRIT5)
    p2 = C.Pair(sh["H"], sh["E"], sh["topk"], sh["I"], sh["c"], sh["r"],
                max_batch=max(sh["batches"]), seed=61)
    k = sh["k"] if sh["k"] is not None else S.budget_to_k(0.178, sh["topk"] * sh["I"])
    return request.param, sh, p5, p2, k


def _tie_margin(pair, e):
    sh = pair.shape
    out = []
    for W in (pair.layer.g(e), pair.layer.v(e)):
        wt = R.rotate(R.pad_hidden(W, sh.Hp), pair.sigma).reshape(sh.I, sh.nb, 128)
        delta = R.TWN_DELTA * np.abs(wt).mean(-1, keepdims=True)
        out.append(np.abs(np.abs(wt) - delta) / np.maximum(delta, 1e-300))
    return np.stack(out)     # [2][I][nb][128]


def test_runs_match_pack_codes5(pairs):
    name, sh, p5, _, _ = pairs
    codes = p5.reader.export("codes")                 # [E][nb][128][2][S5]
    assert codes.shape[-1] == R.run_stride5(sh["I"]), name
    for e in range(sh["E"]):
        tt = np.transpose(p5.layer.sketch(e).t, (2, 3, 0, 1))   # [nb][128][2][I]
        ref = R.pack_codes5(tt)
        if np.array_equal(codes[e], ref):
            continue
        got_t = R.unpack_codes5(codes[e], sh["I"])
        bad = np.argwhere(got_t != tt)
        margin = _tie_margin(p5, e)
        for b, c, gv, i in bad:
            assert margin[gv, i, b, c] < 1e-9, (name, e, b, c, gv, i)


def test_decode_parity_and_read_accounting(pairs):
    name, sh, p5, _, k = pairs
    for B in sh["batches"]:
        x, ids, w = p5.tokens(B, 30 + B)
        y = p5.decode_gpu(x, ids, w, k)
        assert p5.reader.status() == (0, 0), name
        C.check_decode(p5, x, ids, w, k, y)


def test_same_estimates_and_kept_sets_as_two_bit(pairs):
    """The trits are the same; only their packing differs: the screen's sums
    run in the same order, so the estimates are bit-identical."""
    name, sh, p5, p2, k = pairs
    B = sh["batches"][-1]
    x, ids, w = p5.tokens(B, 50 + B)
    y5 = p5.decode_gpu(x, ids, w, k)
    g5, v5, kept5, st5 = (p5.reader.export("ghat"), p5.reader.export("vhat"),
                          p5.reader.kept(B, k), p5.reader.stats())
    y2 = p2.decode_gpu(x, ids, w, k)
    g2, v2, kept2, st2 = (p2.reader.export("ghat"), p2.reader.export("vhat"),
                          p2.reader.kept(B, k), p2.reader.stats())
    assert np.array_equal(g5, g2) and np.array_equal(v5, v2), name
    assert np.array_equal(kept5, kept2), name
    assert np.abs(y5 - y2).max() <= 1e-6 * np.abs(y2).max(), name
    # the screen reads ceil(I/5) instead of ceil(I/4) bytes a run; all else equal
    run5, run2 = (sh["I"] + 4) // 5, (sh["I"] + 3) // 4
    assert st5["codes"] * -(-run2 // 32) == st2["codes"] * -(-run5 // 32), name
    for a in ("scales", "dnorm", "G", "V", "Dt", "b", "U", "dense"):
        assert st5[a] == st2[a], (name, a)


def test_qwen3_30b_read_fraction_is_the_pages_17_8_percent():
    """The full Qwen3-30B-A3B-shaped layer at k = 756: five-trit codes bring
    the reads to the pages' 17.8% (the 2-bit layout reads 18.7%)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    WL = S.QWEN3_30B
    p5 = C.Pair(WL.H, WL.E, WL.topk, WL.I, WL.c, WL.r, max_batch=1, seed=3, device_weights=True,
                flags=RD.FLAG_TRIT5)
    x, ids, w = p5.tokens(1, 101)
    y = p5.decode_gpu(x, ids, w, WL.k)
    assert p5.reader.status() == (0, 0)
    C.check_decode(p5, x, ids, w, WL.k, y)
    st = p5.reader.stats()
    frac = sum(st[a] for a in SC.ARRAYS) / st["dense"]
    assert abs(frac - 0.178) < 1.5e-3, frac
