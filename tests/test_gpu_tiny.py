"""GPU parity of the whole path on the tiny layer (H 256, E 16, top-2, I 128,
k 32, c 80, r 8), element by element against the fp64 oracle."""

import numpy as np
import pytest

from oracle import reader as R
from tests import gpu_common as C

pytestmark = pytest.mark.gpu

H, E, TOPK, I, CC, RANK, K = 256, 16, 2, 128, 80, 8, 32


@pytest.fixture(scope="module")
def pair():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return C.Pair(H, E, TOPK, I, CC, RANK, max_batch=8, seed=0)


def _tie_margin(pair, e):
    """Relative distance of every rotated weight magnitude from its block's TWN threshold."""
    sh = pair.shape
    out = []
    for W in (pair.layer.g(e), pair.layer.v(e)):
        wt = R.rotate(R.pad_hidden(W, sh.Hp), pair.sigma).reshape(sh.I, sh.nb, 128)
        delta = R.TWN_DELTA * np.abs(wt).mean(-1, keepdims=True)
        out.append(np.abs(np.abs(wt) - delta) / np.maximum(delta, 1e-300))
    return np.stack(out)     # [2][I][nb][128]


def test_codes_bit_exact(pair):
    codes = pair.reader.export("codes")            # [E][nb][128][2][S]
    for e in range(E):
        sk = pair.layer.sketch(e)
        ref = sk.packed()
        if np.array_equal(codes[e], ref):
            continue
        got_t = R.unpack_codes(codes[e], I)        # [nb][128][2][I]
        ref_t = R.unpack_codes(ref, I)
        bad = np.argwhere(got_t != ref_t)
        margin = _tie_margin(pair, e)
        for b, c, gv, i in bad:
            assert margin[gv, i, b, c] < 1e-9, (e, b, c, gv, i)


def test_scales_and_rho(pair):
    sc = pair.reader.export("scales")
    rho = pair.reader.export("rho")
    for e in range(E):
        sk = pair.layer.sketch(e)
        assert np.array_equal(sc[e], sk.alpha)
        d = np.abs(rho[e].astype(np.float64) - sk.rho.astype(np.float64))
        ulp = np.spacing(sk.rho.astype(np.float16)).astype(np.float64)
        assert np.all(d <= ulp)


def test_dnorm_and_transpose(pair):
    dn = pair.reader.export("dnorm")
    Dt = pair.reader.export("Dt")
    for e in range(E):
        ref = pair.layer.dnorm(e)
        assert np.allclose(dn[e], ref, rtol=2.5e-7, atol=0)
        assert np.array_equal(Dt[e], pair.D[e].T)


def test_recovery_basis(pair):
    U = pair.reader.export("U").astype(np.float64)
    Uo = pair.layer.U.astype(np.float64)
    P, Po = U @ U.T, Uo @ Uo.T
    assert np.linalg.norm(P - Po, 2) < 1e-2
    ev = pair.reader.export("eigvals")
    assert np.allclose(ev, pair.layer.eigenvalues, rtol=1e-5)
    # columns agree after the shared sign convention, up to fp16 rounding
    assert np.all(np.abs(np.sum(U * Uo, axis=0)) > 0.99)
    b = pair.reader.export("b").astype(np.float64)
    for e in range(E):
        bo = pair.layer.b(e).astype(np.float64)
        assert np.abs(b[e] - bo).max() <= 1e-2 * np.abs(bo).max()


@pytest.mark.parametrize("B,k,seed", [(1, K, 1), (3, K, 2), (8, K, 3), (2, 0, 4), (2, 256, 5),
                                      (1, 1, 6), (4, 255, 7)])
def test_decode_parity(pair, B, k, seed):
    x, ids, w = pair.tokens(B, seed)
    y = pair.decode_gpu(x, ids, w, k)
    code, bits = pair.reader.status()
    assert code == 0 and bits == 0
    res, _, _ = C.check_decode(pair, x, ids, w, k, y)
    ghat = pair.reader.export("ghat")
    vhat = pair.reader.export("vhat")
    score = pair.reader.export("score")
    for t in range(B):
        ref_g = res[t].ghat.reshape(-1)
        ref_v = res[t].vhat.reshape(-1)
        assert np.abs(ghat[t] - ref_g).max() <= 1e-5 * np.abs(ref_g).max()
        assert np.abs(vhat[t] - ref_v).max() <= 1e-5 * np.abs(ref_v).max()
        ref_s = res[t].score.reshape(-1)
        assert np.abs(score[t] - ref_s).max() <= 1e-5 * ref_s.max()


@pytest.mark.parametrize("B,k", [(1, K), (3, K), (2, 0), (2, 256)])
def test_read_accounting_exact(pair, B, k):
    x, ids, w = pair.tokens(B, 10 + B + k)
    y = pair.decode_gpu(x, ids, w, k)
    _, ndiff, _ = C.check_decode(pair, x, ids, w, k, y)
    assert ndiff == 0


def test_host_abi_matches_device(pair):
    x, ids, w = pair.tokens(3, 21)
    y_dev = pair.decode_gpu(x, ids, w, K)
    y_host = pair.reader.decode_host(x, ids, w, K)
    # the recovery vector is summed with fp32 atomics: equal up to summation order
    assert np.abs(y_dev - y_host).max() <= 1e-6 * np.abs(y_dev).max()


def test_empty_batch_and_argument_errors(pair):
    import torch

    from calibration_free_sparse_gb300 import reader as rd

    x = torch.zeros((0, H), device="cuda")
    ids = torch.zeros((0, TOPK), dtype=torch.int32, device="cuda")
    w = torch.zeros((0, TOPK), device="cuda")
    y = torch.zeros((0, H), device="cuda")
    pair.reader.decode(x, ids, w, K, y)          # B = 0 is a no-op
    x1 = torch.zeros((1, H), device="cuda")
    i1 = torch.zeros((1, TOPK), dtype=torch.int32, device="cuda")
    w1 = torch.zeros((1, TOPK), device="cuda")
    y1 = torch.zeros((1, H), device="cuda")
    for bad_k in (-1, E * 0 + TOPK * I + 1):
        with pytest.raises(rd.ReaderError) as ei:
            pair.reader.decode(x1, i1, w1, bad_k, y1)
        assert ei.value.code == rd.EINVAL
    x9 = torch.zeros((9, H), device="cuda")
    with pytest.raises(rd.ReaderError):
        pair.reader.decode(x9, i1, w1, K, y1)     # B > max_batch


def test_device_input_checks(pair):
    from calibration_free_sparse_gb300 import reader as rd

    x, ids, w = pair.tokens(2, 31)
    bad = ids.copy()
    bad[0, 0] = E + 5
    pair.decode_gpu(x, bad, w, K)
    code, bits = pair.reader.status()
    assert code == rd.EDEVICE and bits & rd.ERR_EXPERT_RANGE
    dup = ids.copy()
    dup[1, 1] = dup[1, 0]
    pair.decode_gpu(x, dup, w, K)
    code, bits = pair.reader.status()
    assert code == rd.EDEVICE and bits & rd.ERR_EXPERT_DUP
    wn = w.copy()
    wn[0, 1] = -0.5
    pair.decode_gpu(x, ids, wn, K)
    code, bits = pair.reader.status()
    assert code == rd.EDEVICE and bits & rd.ERR_WEIGHT
    xn = x.copy()
    xn[1, 7] = np.nan
    pair.decode_gpu(xn, ids, w, K)
    code, bits = pair.reader.status()
    assert code == rd.EDEVICE and bits & rd.ERR_X_NONFINITE
    # the error word is cleared by status(): a clean decode reports OK again
    pair.decode_gpu(x, ids, w, K)
    assert pair.reader.status() == (0, 0)


def test_prepare_rejects_bad_config():
    import torch

    from calibration_free_sparse_gb300 import reader as rd

    g = torch.zeros((2, 64, 256), dtype=torch.bfloat16, device="cuda")
    d = torch.zeros((2, 256, 64), dtype=torch.bfloat16, device="cuda")
    sig = np.ones(256, np.int8)
    for kw in (dict(inter=60), dict(screen_coords=0), dict(screen_coords=129), dict(rank=0),
               dict(max_batch=0)):
        args = dict(hidden=256, num_experts=2, experts_per_token=1, inter=64, screen_coords=80,
                    rank=8, max_batch=4)
        args.update(kw)
        with pytest.raises(rd.ReaderError) as ei:
            rd.MoeReader(args["hidden"], args["num_experts"], args["experts_per_token"],
                         args["inter"], g, g, d, sig, screen_coords=args["screen_coords"],
                         rank=args["rank"], max_batch=args["max_batch"])
        assert ei.value.code == rd.EINVAL
    bad_sig = sig.copy()
    bad_sig[3] = 0
    with pytest.raises(rd.ReaderError):
        rd.MoeReader(256, 2, 1, 64, g, g, d, bad_sig, rank=8)
