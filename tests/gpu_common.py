"""Shared pieces of the GPU parity tests: build seeded layers on both sides
and compare the CUDA library against the fp64 oracle."""

import numpy as np

from calibration_free_sparse_gb300 import synthetic as S
from oracle import reader as R
from oracle import sectors as SC

# Acceptance (floating point): max |y - y*| / ||y*||_inf and ||y - y*||_2 / ||y*||_2
Y_MAX_REL = 2e-2
Y_L2_REL = 5e-3
# Kept sets: bit-exact except channels whose oracle score lies within this
# relative distance of the oracle's k-th score.
KEPT_BAND = 1e-4


def to_device_bf16(bits, torch):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


class Pair:
    """The same layer prepared by the CUDA library and described to the oracle."""

    def __init__(self, H, E, topk, I, c, r, max_batch, seed=0, device_weights=False, flags=0):
        import torch

        from calibration_free_sparse_gb300.reader import MoeReader

        self.shape = R.Shape(H=H, E=E, topk=topk, I=I, c=c, r=r)
        if device_weights:
            g, v, d = S.weights_device(seed, E, I, H, "cuda")
            self.G, self.V, self.D = (S.bf16_tensor_to_bits(t) for t in (g, v, d))
        else:
            self.G, self.V, self.D = S.weights(seed, E, I, H)
            g, v, d = (to_device_bf16(a, torch) for a in (self.G, self.V, self.D))
        self.sigma = S.signs(seed, self.shape.Hp)
        self.dev = (g, v, d)
        self.reader = MoeReader(H, E, topk, I, g, v, d, self.sigma, screen_coords=c, rank=r,
                                max_batch=max_batch, flags=flags)
        self.layer = R.Layer(self.shape, self.G, self.V, self.D, self.sigma)

    def tokens(self, B, seed):
        x = S.activations(seed, B, self.shape.H)
        ids, w = S.routing(seed, B, self.shape.E, self.shape.topk)
        return x, ids, w

    def decode_gpu(self, x, ids, w, k):
        import torch

        xd = torch.from_numpy(x).cuda()
        idd = torch.from_numpy(ids).cuda()
        wd = torch.from_numpy(w).cuda()
        y = torch.empty_like(xd)
        self.reader.decode(xd, idd, wd, k, y)
        torch.cuda.synchronize()
        return y.cpu().numpy()


def oracle_scores_by_id(res, ids):
    """Map global channel id -> oracle score for one token."""
    I = res.score.shape[1]
    out = {}
    for s, e in enumerate(ids):
        for i in range(I):
            out[int(e) * I + i] = float(res.score[s, i])
    return out


def assert_kept_match(gpu_kept, res, ids, k, band=KEPT_BAND):
    got = set(int(v) for v in gpu_kept)
    ref = set(int(v) for v in res.kept)
    assert len(got) == k, (len(got), k)
    diff = got ^ ref
    if diff:
        sc = oracle_scores_by_id(res, ids)
        kth = res.kth_score
        for g in diff:
            assert abs(sc[g] - kth) <= band * kth, (g, sc[g], kth)
    return len(diff)


def assert_y_close(y, ref):
    ref = np.asarray(ref, np.float64)
    err = np.asarray(y, np.float64) - ref
    scale_inf = np.abs(ref).max()
    scale_2 = np.linalg.norm(ref)
    assert np.abs(err).max() <= Y_MAX_REL * scale_inf, (np.abs(err).max() / scale_inf)
    assert np.linalg.norm(err) <= Y_L2_REL * scale_2, (np.linalg.norm(err) / scale_2)
    return np.abs(err).max() / scale_inf, np.linalg.norm(err) / scale_2


def oracle_sectors(pair, ids, results):
    masks = np.stack([r.mask for r in results])
    kept = [r.kept for r in results]
    return SC.decode_sectors(pair.shape, ids, masks, kept)


def mask_bits_to_bool(words, nb):
    """u32 [nb][4] -> bool [nb][128]."""
    out = np.zeros((nb, 128), bool)
    for b in range(nb):
        for w in range(4):
            for j in range(32):
                out[b, 32 * w + j] = (int(words[b, w]) >> j) & 1
    return out
