"""moe_reader_topk_noalloc: the selection step for callers that cannot call
cudaMalloc (graph capture, engine plugins, locked allocators).  Checked
against the kept sets of the regular decode entry point on the same scores,
on two calls in a row, and against a numpy brute force (lexicographic sort)
on rows full of exact ties, repeated ids, signed zeros and NaNs of both
signs.  This file is collected last on purpose."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _gids(ids, I):
    return np.stack([np.concatenate([int(e) * I + np.arange(I) for e in row]) for row in ids])


def test_noalloc_topk_matches_decode_kept_sets():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from calibration_free_sparse_gb300 import reader as rd
    from tests import gpu_common as C

    H, E, topk, I = 512, 32, 8, 256
    pair = C.Pair(H, E, topk, I, 80, 16, max_batch=8, seed=5)
    for call, (B, k, seed) in enumerate([(8, 300, 51), (5, 77, 52)]):
        x, ids, w = pair.tokens(B, seed)
        pair.decode_gpu(x, ids, w, k)
        assert pair.reader.status() == (0, 0)
        ref = pair.reader.kept(B, k)                       # global ids, ascending
        scores = torch.from_numpy(pair.reader.export("score").copy()).cuda()
        gid = _gids(ids, I).astype(np.int32)
        kept = torch.full((B, k), -1, dtype=torch.int32, device="cuda")
        rd.topk_noalloc(scores, k, kept, ids=torch.from_numpy(gid).cuda())
        torch.cuda.synchronize()
        cols = kept.cpu().numpy()
        for t in range(B):
            assert np.all(np.diff(cols[t]) > 0)
            got = np.sort(gid[t][cols[t]])
            assert np.array_equal(got, ref[t]), (call, t)


def test_noalloc_rejects_oversize_and_bad_k():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from calibration_free_sparse_gb300 import reader as rd

    big = torch.zeros((2, (1 << 17) + 1), device="cuda")
    out = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(rd.ReaderError) as ei:
        rd.topk_noalloc(big, 4, out)
    assert ei.value.code == rd.ETOOBIG
    small = torch.rand((3, 100), device="cuda")
    with pytest.raises(rd.ReaderError) as ei:
        rd.topk_noalloc(small, 101, torch.zeros((3, 101), dtype=torch.int32, device="cuda"))
    assert ei.value.code == rd.EINVAL


def brute_topk(scores, ids, k):
    """Columns of the k largest entries per row, ascending: larger float first
    (-0 ties with +0, any NaN above +inf, NaNs tie), then the smaller id, then
    the smaller column."""
    out = []
    for r in range(scores.shape[0]):
        s = scores[r].astype(np.float64)
        nan = np.isnan(s)
        val = np.where(nan, 0.0, s)
        val = np.where(val == 0.0, 0.0, val)          # -0 -> +0
        idr = np.arange(s.size) if ids is None else ids[r].astype(np.int64)
        cols = np.arange(s.size)
        order = np.lexsort((cols, idr, -val, -nan.astype(np.int64)))
        out.append(np.sort(order[:k]))
    return np.stack(out)


def test_noalloc_matches_brute_force_with_ties_nans_and_repeated_ids():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from calibration_free_sparse_gb300 import reader as rd

    rng = np.random.default_rng(9)
    rows, cols = 6, 3000
    for call in range(2):
        # few distinct values: the k-th score sits inside a large tied group
        sc = rng.integers(-3, 4, (rows, cols)).astype(np.float32) * 0.5
        sc[0, :50] = np.nan                                          # +NaN above everything
        sc[1, 10:40] = -np.nan                                       # sign bit set: still above
        sc[1, 40:45] = np.float32(np.inf)
        sc[2] = np.where(rng.random(cols) < 0.5, np.float32(-0.0), np.float32(0.0))   # +-0 tie
        sc[3, ::7] = np.float32(-np.inf)
        # ids with repeats (a row of 30 distinct values) and one row of equal ids
        ids = rng.integers(0, 30, (rows, cols)).astype(np.int32)
        ids[4] = 7
        for k in (1, 37, 1500, cols - 1, cols):
            for use_ids in (True, False):
                ref = brute_topk(sc, ids if use_ids else None, k)
                kept = torch.full((rows, k), -1, dtype=torch.int32, device="cuda")
                rd.topk_noalloc(torch.from_numpy(sc).cuda(), k, kept,
                                ids=torch.from_numpy(ids).cuda() if use_ids else None)
                torch.cuda.synchronize()
                got = kept.cpu().numpy()
                assert np.array_equal(got, ref), (call, k, use_ids)


def test_noalloc_wrapper_checks_types_and_shapes():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from calibration_free_sparse_gb300 import reader as rd

    sc = torch.rand((2, 64), device="cuda")
    ok = torch.zeros((2, 5), dtype=torch.int32, device="cuda")
    with pytest.raises(TypeError):
        rd.topk_noalloc(sc.double(), 5, ok)
    with pytest.raises(TypeError):
        rd.topk_noalloc(sc, 5, ok.long())
    with pytest.raises(ValueError):
        rd.topk_noalloc(sc, 5, torch.zeros((2, 4), dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        rd.topk_noalloc(sc, 5, ok, ids=torch.zeros((2, 63), dtype=torch.int32, device="cuda"))
    with pytest.raises(TypeError):
        rd.topk_noalloc(sc.cpu(), 5, ok)
