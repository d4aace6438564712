"""GPU parity of the layer stack: L prepared layers decoded by one call with
the residual stream carried on the device (layer l reads h_l / RMS(h_l),
h_{l+1} = h_l + y_l), against the oracle's stack and against properties that
hold at any size: the fp32 residual chain is exact, and every layer of the
stack gives what a lone decode of that layer gives on the same input."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from calibration_free_sparse_gb300 import reader as RD
from oracle import reader as R
from tests import gpu_common as C

pytestmark = pytest.mark.gpu

SMALL = dict(H=256, E=8, topk=2, I=256, c=80, r=8)
L_SMALL = 4
K_SMALL = 92            # 17.8% of N = 512
WL = S.QWEN3_30B


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def small():
    _torch()
    return [C.Pair(SMALL["H"], SMALL["E"], SMALL["topk"], SMALL["I"], SMALL["c"], SMALL["r"],
                   max_batch=5, seed=70 + l) for l in range(L_SMALL)]


def routing_stack(L, B, E, topk, seed):
    ids, w = zip(*(S.routing(seed + l, B, E, topk) for l in range(L)))
    return np.ascontiguousarray(np.stack(ids)), np.ascontiguousarray(np.stack(w))


def run_stack(readers, h0, ids, w, k, with_y=True):
    torch = _torch()
    L, (B, H) = len(readers), h0.shape
    hd = torch.from_numpy(np.ascontiguousarray(h0)).cuda()
    idd = torch.from_numpy(ids).cuda()
    wd = torch.from_numpy(w).cuda()
    hout = torch.empty_like(hd)
    y = torch.empty((L, B, H), dtype=torch.float32, device="cuda") if with_y else None
    RD.decode_stack(readers, hd, idd, wd, k, hout, y)
    torch.cuda.synchronize()
    return hout.cpu().numpy(), (y.cpu().numpy() if with_y else None)


def fp32_chain(h0, y):
    """h_0 .. h_L with h_{l+1} = h_l + y_l rounded to fp32 at every step."""
    hs = [h0.astype(np.float32)]
    for yl in y:
        hs.append((hs[-1] + yl).astype(np.float32))
    return hs


def kernel_input(h):
    """x = h * (1 / sqrt(mean(h^2) + 1e-6)) with the mean and root in fp64 and
    the factor and product in fp32: the stack's stated input arithmetic."""
    ss = np.sum(h.astype(np.float64) ** 2, axis=-1, keepdims=True)
    f = (1.0 / np.sqrt(ss / h.shape[-1] + 1e-6)).astype(np.float32)
    return (h * f).astype(np.float32)


def oracle_layers_on_gpu_inputs(pairs, h0, ids, w, k, y, tokens=None):
    """Every layer of the last stack call against the oracle on the layer's
    own input as the kernel formed it (the exact fp32 residual chain and the
    stated normalisation), at the 1e-4 kept-set band, with read accounting of
    each layer's screened and kept sets."""
    hs = fp32_chain(h0, y)
    for l, p in enumerate(pairs):
        x = kernel_input(hs[l])
        C.check_decode(p, x, ids[l], w[l], k, y[l], tokens=tokens)
    return hs


@pytest.mark.parametrize("B", [1, 5])
def test_stack_against_oracle(small, B):
    sh = small[0].shape
    h0 = S.activations(80 + B, B, sh.H)
    ids, w = routing_stack(L_SMALL, B, sh.E, sh.topk, seed=90 + B)
    h_out, y = run_stack([p.reader for p in small], h0, ids, w, K_SMALL)
    for p in small:
        assert p.reader.status() == (0, 0)
    hs = oracle_layers_on_gpu_inputs(small, h0, ids, w, K_SMALL, y)
    assert np.array_equal(h_out, hs[-1])
    # the oracle's own stack (float64 residual) stays within the summed bounds
    res, h_ref = R.decode_stack([p.layer for p in small], h0, ids, w, K_SMALL)
    bound = np.zeros(B)
    for l in range(L_SMALL):
        for t in range(B):
            C.assert_y_close(y[l, t], res[l][t].y)
            bound[t] += C.Y_MAX_REL * np.abs(res[l][t].y).max()
    for t in range(B):
        assert np.abs(h_out[t] - h_ref[t]).max() <= bound[t]


def test_residual_chain_is_exact_fp32(small):
    B = 4
    sh = small[0].shape
    h0 = S.activations(120, B, sh.H)
    ids, w = routing_stack(L_SMALL, B, sh.E, sh.topk, seed=130)
    h_out, y = run_stack([p.reader for p in small], h0, ids, w, K_SMALL)
    assert np.array_equal(h_out, fp32_chain(h0, y)[-1])


def test_each_layer_equals_a_lone_decode_of_its_input(small):
    torch = _torch()
    B = 3
    sh = small[0].shape
    h0 = 2.5 * S.activations(140, B, sh.H)
    ids, w = routing_stack(L_SMALL, B, sh.E, sh.topk, seed=150)
    h_out, y = run_stack([p.reader for p in small], h0, ids, w, K_SMALL)
    kept = [p.reader.kept(B, K_SMALL) for p in small]
    hs = fp32_chain(h0, y)
    for l, p in enumerate(small):
        x = kernel_input(hs[l])
        yl = p.decode_gpu(x, ids[l], w[l], K_SMALL)
        assert p.reader.status() == (0, 0)
        assert np.array_equal(p.reader.kept(B, K_SMALL), kept[l]), l
        # the same arithmetic up to the order of the fp32 output atomics
        assert np.abs(yl - y[l]).max() <= 1e-5 * np.abs(y[l]).max(), l
    del torch


def test_repeated_steps_and_scratch_outputs(small):
    """Back-to-back steps reuse every counter; without y_layers the layers'
    outputs stay in the handles' scratch and only h_out comes back."""
    sh = small[0].shape
    B = 5
    outs = []
    for step in range(3):
        h0 = S.activations(160 + step, B, sh.H)
        ids, w = routing_stack(L_SMALL, B, sh.E, sh.topk, seed=170 + 10 * step)
        h_out, y = run_stack([p.reader for p in small], h0, ids, w, K_SMALL)
        h_bare, _ = run_stack([p.reader for p in small], h0, ids, w, K_SMALL, with_y=False)
        assert np.abs(h_bare - h_out).max() <= 1e-5 * np.abs(h_out).max()
        outs.append((h0, ids, w, h_out))
    for p in small:
        assert p.reader.status() == (0, 0)
    h0, ids, w, h_out = outs[-1]
    res, h_ref = R.decode_stack([p.layer for p in small], h0, ids, w, K_SMALL)
    for t in range(B):
        assert np.abs(h_out[t] - h_ref[t]).max() <= 5e-3 * np.abs(h_ref[t]).max()


def test_argument_errors(small):
    torch = _torch()
    sh = small[0].shape
    B = 2
    h0 = torch.from_numpy(S.activations(1, B, sh.H)).cuda()
    ids, w = routing_stack(2, B, sh.E, sh.topk, seed=3)
    idd, wd = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    hout = torch.empty_like(h0)
    r = [p.reader for p in small]

    def code(readers, h_in, h_out, Bv=None, y=None):
        try:
            RD.decode_stack(readers, h_in if Bv is None else h_in[:Bv], idd, wd, K_SMALL, h_out,
                            y)
        except RD.ReaderError as e:
            return e.code
        return RD.OK

    assert code([r[0], r[0]], h0, hout) == RD.EINVAL          # one handle twice
    assert code(r[:2], h0, h0) == RD.EINVAL                    # h_out is h_in
    y_all = torch.empty((2, B, sh.H), device="cuda")
    assert code(r[:2], h0, hout, y=y_all) == RD.OK
    assert code(r[:2], h0, hout, y=h0) == RD.EINVAL            # y_layers over h_in
    big = torch.zeros((6, sh.H), device="cuda")
    assert code(r[:2], big, torch.empty_like(big)) == RD.EINVAL   # B above max_batch
    assert code(r[:2], h0, hout, Bv=0) == RD.OK                   # B = 0: nothing to do
    other = C.Pair(sh.H, sh.E, sh.topk, 128, sh.c, sh.r, max_batch=5, seed=1)
    assert code([r[0], other.reader], h0, hout) == RD.EINVAL      # shapes differ
    torch.cuda.synchronize()
    for p in small[:2]:
        assert p.reader.status() == (0, 0)


def _hp(wl):
    return R.Shape(H=wl.H, E=wl.E, topk=wl.topk, I=wl.I).Hp


class _HostPair:
    """A prepared reader and the oracle's view of the same layer (the shape of
    gpu_common.Pair, for layers prepared outside it)."""

    def __init__(self, reader, wl, G, V, D, sigma):
        self.reader = reader
        self.shape = R.Shape(H=wl.H, E=wl.E, topk=wl.topk, I=wl.I, c=wl.c, r=wl.r)
        self.sigma = sigma
        self.layer = R.Layer(self.shape, G, V, D, sigma)


@pytest.fixture(scope="module")
def qwen3_stack():
    torch = _torch()
    from calibration_free_sparse_gb300.reader import MoeReader

    readers, keep = [], []
    for l in range(3):
        g, v, d = S.weights_device(200 + l, WL.E, WL.I, WL.H, "cuda")
        sigma = S.signs(200 + l, R.Shape(H=WL.H, E=WL.E, topk=WL.topk, I=WL.I).Hp)
        readers.append(MoeReader(WL.H, WL.E, WL.topk, WL.I, g, v, d, sigma, screen_coords=WL.c,
                                 rank=WL.r, max_batch=16))
        keep.append((g, v))
        del d
    torch.cuda.synchronize()
    return readers, keep


def test_qwen3_30b_stack_properties(qwen3_stack):
    """Three Qwen3-30B-A3B-shaped layers at batch 16, k 756, the benchmark's
    launch configuration: exact fp32 residual chain, and each layer's kept set
    and y equal to a lone decode of the same input."""
    torch = _torch()
    readers, _ = qwen3_stack
    B = 16
    h0 = S.activations(210, B, WL.H)
    ids, w = routing_stack(len(readers), B, WL.E, WL.topk, seed=220)
    h_out, y = run_stack(readers, h0, ids, w, WL.k)
    for rd in readers:
        assert rd.status() == (0, 0)
    kept = [rd.kept(B, WL.k) for rd in readers]
    hs = fp32_chain(h0, y)
    assert np.array_equal(h_out, hs[-1])
    for l, rd in enumerate(readers):
        x = torch.from_numpy(kernel_input(hs[l])).cuda()
        yl = torch.empty_like(x)
        rd.decode(x, torch.from_numpy(ids[l]).cuda(), torch.from_numpy(w[l]).cuda(), WL.k, yl)
        torch.cuda.synchronize()
        assert rd.status() == (0, 0)
        assert np.array_equal(rd.kept(B, WL.k), kept[l]), l
        yl = yl.cpu().numpy()
        assert np.abs(yl - y[l]).max() <= 1e-5 * np.abs(y[l]).max(), l


def test_qwen3_30b_48_layer_stack():
    """The 48-layer stack of Qwen3-30B-A3B-shaped layers (independent weights
    per layer, residual carried) at batch 1 and 8 and at the 17.8% and 12.8%
    budgets: every layer's status clean, the fp32 residual chain exact, the
    first and last layers against the oracle on their own inputs (sampled
    tokens, 1e-4 kept-set band, read accounting of the whole batch), and
    sampled layers equal to a lone decode of their input."""
    torch = _torch()
    from calibration_free_sparse_gb300.reader import MoeReader

    L = 48
    readers, keep = [], []
    for l in range(L):
        g, v, d = S.weights_device(400 + l, WL.E, WL.I, WL.H, "cuda")
        sigma = S.signs(400 + l, R.Shape(H=WL.H, E=WL.E, topk=WL.topk, I=WL.I).Hp)
        readers.append(MoeReader(WL.H, WL.E, WL.topk, WL.I, g, v, d, sigma, screen_coords=WL.c,
                                 rank=WL.r, max_batch=8))
        keep.append((g, v))
        del d
    torch.cuda.synchronize()
    host = {}
    try:
        for B, k in ((1, WL.k), (8, WL.k), (8, S.QWEN3_30B_LOW.k)):
            h0 = S.activations(500 + B + k, B, WL.H)
            ids, w = routing_stack(L, B, WL.E, WL.topk, seed=600 + B)
            h_out, y = run_stack(readers, h0, ids, w, k)
            for rd in readers:
                assert rd.status() == (0, 0)
            hs = fp32_chain(h0, y)
            assert np.array_equal(h_out, hs[-1])
            assert np.isfinite(h_out).all()
            for l in (0, 47):
                # the oracle on the layer's own input as the kernel formed it
                if l not in host:
                    g, v, d = S.weights_device(400 + l, WL.E, WL.I, WL.H, "cuda")
                    G, V, D = (S.bf16_tensor_to_bits(a) for a in (g, v, d))
                    del g, v, d
                    host[l] = _HostPair(readers[l], WL, G, V, D, S.signs(400 + l, _hp(WL)))
                C.check_decode(host[l], kernel_input(hs[l]), ids[l], w[l], k, y[l],
                               tokens=sorted({0, B - 1}))
            for l in (0, 23, 47):
                kept = readers[l].kept(B, k)
                x = torch.from_numpy(kernel_input(hs[l])).cuda()
                yl = torch.empty_like(x)
                readers[l].decode(x, torch.from_numpy(ids[l]).cuda(), torch.from_numpy(w[l]).cuda(),
                                  k, yl)
                torch.cuda.synchronize()
                assert readers[l].status() == (0, 0)
                assert np.array_equal(readers[l].kept(B, k), kept), (B, k, l)
                assert np.abs(yl.cpu().numpy() - y[l]).max() <= 1e-5 * np.abs(y[l]).max(), (B, k, l)
    finally:
        for rd in readers:
            rd.close()
