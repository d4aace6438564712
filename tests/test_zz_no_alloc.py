"""moe_reader_topk_noalloc: the selection step for callers that cannot call
cudaMalloc (graph capture, engine plugins, locked allocators).  Checked
against the kept sets of the regular decode entry point on the same scores,
on two calls in a row.  This file is collected last on purpose."""

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
