"""fp64 oracle of the weight-only channel reader (prepare + per-token decode).

TEST INFRASTRUCTURE ONLY -- see the package docstring for who may import it.

Every step follows the two summaries of "Channel Selection for
Mixture-of-Experts Decoding Needs No Calibration Data":
[CN] the Chinese summary page (sections 前置知识 / 核心方法 / 方法步骤详情) and
[KR] the Korean summary page (section 어떻게 쓰나).  Where the pages leave a
step open, the reading taken is stated in the function's docstring.

Inputs are the stored values: BF16 weights as uint16 bit patterns, fp32 x,
int32 expert ids, fp32 routing weights and an int8 sign vector.  All method
arithmetic runs in float64.  Numpy library primitives (matmul, eigh, sort) are
used as single steps; nothing is blocked, fused or reordered beyond the
definitions written here.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 128          # rotation block: [CN] §方法步骤详情, load-time (1)
TWN_DELTA = 0.7      # Ternary Weight Networks threshold factor ([CN] §技术新颖性 credits TWN)


# --------------------------------------------------------------------------
# shapes
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Shape:
    """Layer shape: hidden H, experts E, experts per token topk, expert width I,
    screened coordinates per block c, recovery rank r."""
    H: int
    E: int
    topk: int
    I: int
    c: int = 80
    r: int = 32

    @property
    def Hp(self) -> int:
        """Hidden size zero-padded to whole 128-coordinate blocks."""
        return BLOCK * math.ceil(self.H / BLOCK)

    @property
    def nb(self) -> int:
        return self.Hp // BLOCK

    @property
    def N(self) -> int:
        """Routed channels per token: every channel of the token's topk experts
        ([CN] §核心方法: 8 experts x 768 = 6144 channels for Qwen3-Thinking)."""
        return self.topk * self.I


# --------------------------------------------------------------------------
# stored-value decoding (exact)
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of BF16 bit patterns (upper half of an fp32)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pad_hidden(a: np.ndarray, Hp: int) -> np.ndarray:
    """Zero-pad the last axis to Hp (a block that runs past H holds zeros)."""
    pad = Hp - a.shape[-1]
    if pad == 0:
        return a
    width = [(0, 0)] * (a.ndim - 1) + [(0, pad)]
    return np.pad(a, width)


# --------------------------------------------------------------------------
# randomized block Hadamard rotation
# --------------------------------------------------------------------------
def sylvester_hadamard(n: int = BLOCK) -> np.ndarray:
    """Sylvester Hadamard matrix, entry (i, j) = (-1)^popcount(i & j)."""
    i = np.arange(n)
    anded = np.bitwise_and.outer(i, i)
    parity = np.zeros_like(anded)
    v = anded.copy()
    while v.any():
        parity ^= v & 1
        v >>= 1
    return np.where(parity == 0, 1.0, -1.0)


def rotate(a: np.ndarray, sigma: np.ndarray) -> np.ndarray:
    """R a, applied on the last axis (length Hp = 128 * nb).

    R is block diagonal; block b is R_b = H_128 diag(sigma_b) / sqrt(128), an
    orthogonal matrix, so g^T x = (R g)^T (R x)  ([CN] §前置知识 "Hadamard旋转与
    三元Sketch"; [KR] §어떻게 쓰나).  Reading: the randomization is one
    independent +-1 sign per coordinate (sigma), applied before the Sylvester
    Hadamard of each block.
    """
    Hm = sylvester_hadamard()
    a = np.asarray(a, dtype=np.float64)
    nb = a.shape[-1] // BLOCK
    s = np.asarray(sigma, dtype=np.float64)
    u = (a * s).reshape(a.shape[:-1] + (nb, BLOCK))
    out = (u @ Hm.T) / math.sqrt(BLOCK)
    return out.reshape(a.shape)


def select_coordinates(mag: np.ndarray, c: int) -> np.ndarray:
    """Partial-screen coordinate set T_b: the c coordinates with the largest
    |Rx| in each 128-block ([CN] §方法步骤详情, decode (1); [KR] §어떻게 쓰나:
    80 of 128).  Ties go to the lower coordinate index.  Returns bool [nb, 128].
    """
    nb = mag.shape[0]
    mask = np.zeros((nb, BLOCK), dtype=bool)
    for b in range(nb):
        order = np.argsort(-mag[b].astype(np.float64), kind="stable")
        mask[b, order[:c]] = True
    return mask


def selection_gaps(mag: np.ndarray, c: int) -> np.ndarray:
    """Per block, the relative gap (m_c - m_{c+1}) / m_c between the c-th and
    the (c+1)-th largest |Rx| (m sorted descending, float64); +inf when every
    coordinate is screened (c = 128) or the block is zero.  A block whose gap
    is tiny is a near-tie: an implementation that rounds Rx differently (an
    fp32 butterfly, say) may legitimately screen the other coordinate, so
    parity checks of the screened set excuse such blocks.  Returns float64 [nb].
    """
    srt = -np.sort(-np.asarray(mag, dtype=np.float64), axis=1)
    out = np.full(srt.shape[0], np.inf)
    if c >= BLOCK:
        return out
    top, nxt = srt[:, c - 1], srt[:, c]
    pos = top > 0
    out[pos] = (top[pos] - nxt[pos]) / top[pos]
    return out


# --------------------------------------------------------------------------
# ternary sketch (load time)
# --------------------------------------------------------------------------
def ternarize(wt: np.ndarray):
    """Ternary code, FP16 scale and FP16 block mean-squared error of rotated blocks.

    wt: float64 [..., 128], one rotated 128-block per leading index.
    Ternary Weight Networks rule (reading of [CN] §前置知识 / load-time (1): codes
    in {-1, 0, 1}, an FP16 scale and the block's quantisation MSE rho_b):
        Delta = 0.7 * mean|w|,  t_i = sign(w_i) if |w_i| > Delta else 0,
        alpha = mean of |w_i| over {t_i != 0}  (0 if empty), stored FP16,
        rho   = mean_i (w_i - alpha_fp16 * t_i)^2, stored FP16.
    Returns (t int8 [..., 128], alpha float16 [...], rho float16 [...]).
    """
    absw = np.abs(wt)
    delta = TWN_DELTA * absw.mean(axis=-1, keepdims=True)
    support = absw > delta
    t = np.where(support, np.sign(wt), 0.0)
    nnz = support.sum(axis=-1)
    total = np.where(support, absw, 0.0).sum(axis=-1)
    alpha = np.where(nnz > 0, total / np.maximum(nnz, 1), 0.0)
    alpha16 = alpha.astype(np.float16)
    resid = wt - alpha16.astype(np.float64)[..., None] * t
    rho16 = (resid * resid).mean(axis=-1).astype(np.float16)
    return t.astype(np.int8), alpha16, rho16


def run_bytes(I: int) -> int:
    """Bytes of one coordinate run of 2-bit codes (I channels, 4 per byte)."""
    return (I + 3) // 4


def run_stride(I: int) -> int:
    """Run length padded to whole 32-byte sectors."""
    return 32 * math.ceil(run_bytes(I) / 32)


def pack_codes(t: np.ndarray) -> np.ndarray:
    """2-bit packing of ternary codes along the last axis (channels).

    Code values: 0 -> 0b00, +1 -> 0b01, -1 -> 0b11 (two's complement of the
    trit).  Channel i sits in byte i // 4 at bits 2 * (i % 4).  The run is
    zero-padded to a whole number of 32-byte sectors.
    """
    I = t.shape[-1]
    q = np.where(t == 1, 1, np.where(t == -1, 3, 0)).astype(np.uint8)
    padI = 4 * run_bytes(I)
    if padI != I:
        q = np.concatenate([q, np.zeros(q.shape[:-1] + (padI - I,), np.uint8)], axis=-1)
    q = q.reshape(q.shape[:-1] + (padI // 4, 4))
    packed = (q[..., 0] | (q[..., 1] << 2) | (q[..., 2] << 4) | (q[..., 3] << 6)).astype(np.uint8)
    stride = run_stride(I)
    if stride != packed.shape[-1]:
        packed = np.concatenate(
            [packed, np.zeros(packed.shape[:-1] + (stride - packed.shape[-1],), np.uint8)], axis=-1)
    return packed


def unpack_codes(packed: np.ndarray, I: int) -> np.ndarray:
    """Inverse of pack_codes: int8 trits [..., I]."""
    b = packed[..., : run_bytes(I)].astype(np.uint8)
    fields = np.stack([(b >> (2 * k)) & 3 for k in range(4)], axis=-1)
    fields = fields.reshape(b.shape[:-1] + (4 * b.shape[-1],))[..., :I]
    out = np.zeros(fields.shape, np.int8)
    out[fields == 1] = 1
    out[fields == 3] = -1
    if np.any(fields == 2):
        raise ValueError("invalid 2-bit code 0b10")
    return out


# 1.6 bit per trit: five trits per byte ([CN] §方法步骤详情 load-time (1): a
# 128-coordinate block of 256 BF16 bytes shrinks to about 30 bytes; 128 trits
# at 8/5 bits are 26 bytes, plus the FP16 scale and the FP16 rho)
TRIT5_DIGIT = {0: 0, 1: 1, -1: 2}   # the base-3 digit of a trit (the 2-bit code order)


def run_bytes5(I: int) -> int:
    """Bytes of one coordinate run of five-trit bytes (I channels, 5 per byte)."""
    return (I + 4) // 5


def run_stride5(I: int) -> int:
    """Five-trit run length padded to whole 32-byte sectors."""
    return 32 * math.ceil(run_bytes5(I) / 32)


def pack_codes5(t: np.ndarray) -> np.ndarray:
    """Five trits per byte along the last axis (channels): byte j holds
    channels 5j .. 5j+4 as sum_m digit(t[5j+m]) * 3^m, digit 0 -> 0, +1 -> 1,
    -1 -> 2 (at most 242).  Zero-padded to a whole number of 32-byte sectors."""
    I = t.shape[-1]
    q = np.where(t == 1, 1, np.where(t == -1, 2, 0)).astype(np.int64)
    padI = 5 * run_bytes5(I)
    if padI != I:
        q = np.concatenate([q, np.zeros(q.shape[:-1] + (padI - I,), np.int64)], axis=-1)
    q = q.reshape(q.shape[:-1] + (padI // 5, 5))
    packed = (q * (3 ** np.arange(5))).sum(axis=-1).astype(np.uint8)
    stride = run_stride5(I)
    if stride != packed.shape[-1]:
        packed = np.concatenate(
            [packed, np.zeros(packed.shape[:-1] + (stride - packed.shape[-1],), np.uint8)], axis=-1)
    return packed


def unpack_codes5(packed: np.ndarray, I: int) -> np.ndarray:
    """Inverse of pack_codes5: int8 trits [..., I]."""
    b = packed[..., : run_bytes5(I)].astype(np.int64)
    if np.any(b > 242):
        raise ValueError("invalid five-trit byte (> 242)")
    digits = np.stack([(b // 3 ** m) % 3 for m in range(5)], axis=-1)
    digits = digits.reshape(b.shape[:-1] + (5 * b.shape[-1],))[..., :I]
    out = np.zeros(digits.shape, np.int8)
    out[digits == 1] = 1
    out[digits == 2] = -1
    return out


@dataclass
class ExpertSketch:
    """Sketch of one expert: trits t[gv][I][nb][128] (gv 0 = gate, 1 = up),
    alpha and rho float16 [nb][2][I]."""
    t: np.ndarray
    alpha: np.ndarray
    rho: np.ndarray

    def packed(self) -> np.ndarray:
        """Documented layout of one expert: u8 [nb][128][2][run_stride(I)]."""
        tt = np.transpose(self.t, (2, 3, 0, 1))  # [nb][128][2][I]
        return pack_codes(tt)


def sketch_expert(G_e: np.ndarray, V_e: np.ndarray, sigma: np.ndarray, Hp: int) -> ExpertSketch:
    """Rotate every gate row g_j and up row v_j in 128-blocks, then ternarise
    each block ([CN] §方法步骤详情, load-time (1); [KR] §어떻게 쓰나).
    G_e, V_e: float64 [I][H] (exact BF16 values)."""
    I = G_e.shape[0]
    nb = Hp // BLOCK
    ts, alphas, rhos = [], [], []
    for W in (G_e, V_e):
        Wr = rotate(pad_hidden(W, Hp), sigma).reshape(I, nb, BLOCK)
        t, a, r = ternarize(Wr)
        ts.append(t)
        alphas.append(a.T)  # [nb][I]
        rhos.append(r.T)
    return ExpertSketch(
        t=np.stack(ts),                                  # [2][I][nb][128]
        alpha=np.stack(alphas, axis=1),                  # [nb][2][I]
        rho=np.stack(rhos, axis=1),
    )


# --------------------------------------------------------------------------
# down norms and per-layer recovery basis (load time)
# --------------------------------------------------------------------------
def down_norms(D_e: np.ndarray) -> np.ndarray:
    """||d_j|| for every channel j of one expert; D_e float64 [H][I] (column j
    is d_j).  Stored fp32 ([CN] §方法步骤详情, load-time (2))."""
    return np.sqrt((D_e * D_e).sum(axis=0)).astype(np.float32)


def canonical_signs(U: np.ndarray) -> np.ndarray:
    """Flip each column so its largest-magnitude entry (first on ties) is positive.
    The recovery term U U^T v does not depend on this choice."""
    U = U.copy()
    for j in range(U.shape[1]):
        i = int(np.argmax(np.abs(U[:, j])))
        if U[i, j] < 0:
            U[:, j] = -U[:, j]
    return U


def recovery_basis(down_blocks, r: int):
    """Top-r left singular vectors of the layer's stacked down columns.

    [CN] §前置知识 "低秩恢复" and §方法步骤详情 load-time (3): stack the down
    columns d_j of all experts of one layer and keep the top-32 left singular
    vectors U.  Computed as the top-r eigenvectors of M = sum_j d_j d_j^T
    (the same vectors), accumulated expert by expert.
    down_blocks: iterable of float64 [H][I] arrays (one per expert).
    Returns (U float16 [H][r], eigenvalues float64 [r] in descending order).
    """
    M = None
    for D_e in down_blocks:
        part = D_e @ D_e.T
        M = part if M is None else M + part
    evals, evecs = np.linalg.eigh(M)
    order = np.argsort(-evals, kind="stable")[:r]
    U = canonical_signs(evecs[:, order])
    return U.astype(np.float16), evals[order]


def recovery_coeffs(U16: np.ndarray, D_e: np.ndarray) -> np.ndarray:
    """b_j = U^T d_j for every channel of one expert, with the stored FP16 U;
    stored FP16, shape [I][r] ([CN] §前置知识 "低秩恢复")."""
    return (U16.astype(np.float64).T @ D_e).T.astype(np.float16)


# --------------------------------------------------------------------------
# prepared layer
# --------------------------------------------------------------------------
@dataclass
class Layer:
    """One MoE layer's stored weights (BF16 bit patterns) and the oracle's
    prepared arrays, computed lazily per expert."""
    shape: Shape
    G: np.ndarray        # uint16 [E][I][H]
    V: np.ndarray        # uint16 [E][I][H]
    D: np.ndarray        # uint16 [E][H][I]
    sigma: np.ndarray    # int8 [Hp]
    _sketch: dict = field(default_factory=dict)
    _dnorm: dict = field(default_factory=dict)
    _b: dict = field(default_factory=dict)
    _U: np.ndarray | None = None
    eigenvalues: np.ndarray | None = None

    def g(self, e):
        return bf16_bits_to_f64(self.G[e])

    def v(self, e):
        return bf16_bits_to_f64(self.V[e])

    def d(self, e):
        return bf16_bits_to_f64(self.D[e])

    def sketch(self, e) -> ExpertSketch:
        if e not in self._sketch:
            self._sketch[e] = sketch_expert(self.g(e), self.v(e), self.sigma, self.shape.Hp)
        return self._sketch[e]

    def dnorm(self, e) -> np.ndarray:
        if e not in self._dnorm:
            self._dnorm[e] = down_norms(self.d(e))
        return self._dnorm[e]

    @property
    def U(self) -> np.ndarray:
        if self._U is None:
            self._U, self.eigenvalues = recovery_basis(
                (self.d(e) for e in range(self.shape.E)), self.shape.r)
        return self._U

    def b(self, e) -> np.ndarray:
        if e not in self._b:
            self._b[e] = recovery_coeffs(self.U, self.d(e))
        return self._b[e]


# --------------------------------------------------------------------------
# decode (per token)
# --------------------------------------------------------------------------
def silu(z):
    """phi(z) = z / (1 + e^{-z}), the experts' gate activation (SiLU)."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


@dataclass
class TokenResult:
    y: np.ndarray            # float64 [H]: y_exact + y_recovery
    y_exact: np.ndarray      # sum over kept channels
    y_recovery: np.ndarray   # U sum over skipped channels
    kept: np.ndarray         # int64 sorted global channel ids e*I + i of K
    kept_order: np.ndarray   # K in selection order (-s, id)
    score: np.ndarray        # float64 [topk][I]
    p: np.ndarray            # float64 [topk][I]: phi(ghat) vhat
    ghat: np.ndarray
    vhat: np.ndarray
    mask: np.ndarray         # bool [nb][128] screened coordinates
    kth_score: float         # score of the k-th kept channel (nan if k == 0)
    next_score: float        # best skipped score (nan if k == N)
    gap: np.ndarray = None   # float64 [nb]: relative gap at the screen's c-th |Rx| per block


def screen_estimates(layer: Layer, e: int, Rx: np.ndarray, mask: np.ndarray):
    """Sketch activation estimates for every channel of expert e.

    ghat_j = sum_b alpha^g_{j,b} sum_{c in T_b} t^g_{j,b,c} (Rx)_{b,c}; vhat
    likewise with the up sketch ([CN] §核心方法 step 1; [KR] §어떻게 쓰나).  The
    omitted coordinates are not rescaled (the pages are silent; plain reading).
    Rx: float64 [nb][128]; mask: bool [nb][128].
    """
    sk = layer.sketch(e)
    rx = np.where(mask, Rx, 0.0)                              # [nb][128]
    partial = np.einsum("gibc,bc->gib", sk.t.astype(np.float64), rx)  # [2][I][nb]
    alpha = np.transpose(sk.alpha.astype(np.float64), (1, 2, 0))     # [2][I][nb]
    est = (alpha * partial).sum(axis=-1)
    return est[0], est[1]


@dataclass
class TokenScreen:
    """Steps 1-2 of one token up to its scores (before any selection)."""
    mask: np.ndarray         # bool [nb][128]
    ghat: np.ndarray         # float64 [topk][I]
    vhat: np.ndarray
    p: np.ndarray            # phi(ghat) vhat
    score: np.ndarray        # w ||d|| |p|
    gap: np.ndarray          # float64 [nb]: selection_gaps of the token's blocks


def screen_token(layer: Layer, x: np.ndarray, ids, w, mask=None) -> TokenScreen:
    """Rotate x once, partial screen of the c largest-|Rx| coordinates per
    block, and the output-unit score s_j = w_j ||d_j|| |phi(ghat_j) vhat_j| of
    every routed channel ([CN] §方法步骤详情, decode (1)-(2); the placement of
    |.| follows [KR] §어떻게 쓰나, [CN] writes phi(ghat)|vhat|).

    mask (bool [nb][128], optional) replaces the screened set: a parity check
    passes the other side's set where a block's c-th and (c+1)-th |Rx| are a
    near-tie (selection_gaps), so that both sides then screen the same
    coordinates.  Every other step is unchanged."""
    sh = layer.shape
    x64 = np.asarray(x, dtype=np.float64)
    xpad = pad_hidden(x64, sh.Hp)
    Rx = rotate(xpad, layer.sigma).reshape(sh.nb, BLOCK)
    gap = selection_gaps(np.abs(Rx), sh.c)
    if mask is None:
        mask = select_coordinates(np.abs(Rx), sh.c)
    else:
        mask = np.asarray(mask, dtype=bool).reshape(sh.nb, BLOCK)
    ids = [int(e) for e in ids]
    topk = len(ids)
    ghat = np.zeros((topk, sh.I))
    vhat = np.zeros((topk, sh.I))
    dn = np.zeros((topk, sh.I))
    for s, e in enumerate(ids):
        ghat[s], vhat[s] = screen_estimates(layer, e, Rx, mask)
        dn[s] = layer.dnorm(e).astype(np.float64)
    p = silu(ghat) * vhat
    wv = np.asarray(w, dtype=np.float64)
    score = wv[:, None] * dn * np.abs(p)
    return TokenScreen(mask=mask, ghat=ghat, vhat=vhat, p=p, score=score, gap=gap)


def exact_and_recovery(layer: Layer, x: np.ndarray, ids, w, p: np.ndarray, keep: np.ndarray):
    """Steps 3-4 for one token given its kept channels (keep: bool [topk][I]):
    kept channels from the native BF16 g_j, v_j with the original fp32 x,
    a_j = phi(g_j^T x)(v_j^T x), y_exact = sum_K w_j a_j d_j; skipped ones
    recovered as y_recovery = U sum_S w_j b_j p_j."""
    sh = layer.shape
    x64 = np.asarray(x, dtype=np.float64)
    wv = np.asarray(w, dtype=np.float64)
    y_exact = np.zeros(sh.H)
    coef = np.zeros(sh.r)
    any_skip = False
    for s, e in enumerate(int(v) for v in ids):
        rows = np.nonzero(keep[s])[0]
        if rows.size:
            g_rows = bf16_bits_to_f64(layer.G[e][rows])          # [n][H]
            v_rows = bf16_bits_to_f64(layer.V[e][rows])
            d_cols = bf16_bits_to_f64(layer.D[e][:, rows])        # [H][n]
            a = silu(g_rows @ x64) * (v_rows @ x64)
            y_exact += d_cols @ (wv[s] * a)
        skip = np.nonzero(~keep[s])[0]
        if skip.size:
            any_skip = True
            coef += (wv[s] * p[s, skip]) @ layer.b(e)[skip].astype(np.float64)
    y_rec = layer.U.astype(np.float64) @ coef if any_skip else np.zeros(sh.H)
    return y_exact, y_rec


def decode_token(layer: Layer, x: np.ndarray, ids: np.ndarray, w: np.ndarray, k: int,
                 mask=None) -> TokenResult:
    """One token through the reader ([CN] §方法步骤详情, decode (1)-(4)).
    `mask` optionally fixes the screened coordinates (see screen_token).

    1. Rotate x once; partial screen of the c largest-|Rx| coordinates per block.
    2. s_j = w_j ||d_j|| |phi(ghat_j) vhat_j| for every routed channel, then the
       exact top-k over all routed experts' channels together; ties go to the
       lower global channel id e*I + i.
    3. Kept channels: native BF16 g_j, v_j with the original fp32 x,
       a_j = phi(g_j^T x)(v_j^T x); y_exact = sum_K w_j a_j d_j.
    4. Skipped channels: y_recovery = U sum_S w_j b_j p_j, p_j = phi(ghat_j) vhat_j.
    """
    sh = layer.shape
    sc = screen_token(layer, x, ids, w, mask=mask)
    ids = [int(e) for e in ids]
    gid = np.array([[e * sh.I + i for i in range(sh.I)] for e in ids], dtype=np.int64)
    flat_s = sc.score.reshape(-1)
    flat_id = gid.reshape(-1)
    order = np.lexsort((flat_id, -flat_s))       # primary -s, secondary id
    kept_idx = order[:k]
    kth = float(flat_s[order[k - 1]]) if k > 0 else float("nan")
    nxt = float(flat_s[order[k]]) if k < flat_s.size else float("nan")
    keep = np.zeros(flat_s.size, bool)
    keep[kept_idx] = True
    y_exact, y_rec = exact_and_recovery(layer, x, ids, w, sc.p, keep.reshape(len(ids), sh.I))
    return TokenResult(
        y=y_exact + y_rec, y_exact=y_exact, y_recovery=y_rec,
        kept=np.sort(flat_id[kept_idx]), kept_order=flat_id[kept_idx],
        score=sc.score, p=sc.p, ghat=sc.ghat, vhat=sc.vhat, mask=sc.mask,
        kth_score=kth, next_score=nxt, gap=sc.gap)


def decode(layer: Layer, x: np.ndarray, ids: np.ndarray, w: np.ndarray, k: int):
    """Batch decode: every token independently (selection is per token; the
    batch-shared selection of [CN] §未来方向 is future work)."""
    return [decode_token(layer, x[t], ids[t], w[t], k) for t in range(x.shape[0])]


# --------------------------------------------------------------------------
# full screen ranked by the expected squared output error (budgets >= 28.7%)
# --------------------------------------------------------------------------
def silu_grad(z):
    """d/dz z sigmoid(z)."""
    sg = 1.0 / (1.0 + np.exp(-z))
    return sg * (1.0 + z * (1.0 - sg))


def expected_skip_error(layer: Layer, x: np.ndarray, ids, w):
    """[topk][I] expected squared output error of skipping each routed channel
    under the full screen ([CN] §方法步骤详情 decode (2): from the 28.7% budget
    the whole sketch is read and rho_b ranks channels by the expected squared
    output error after skipping; the pages give no formula, the reading here):

    - skipping j leaves w_j (a_j d_j - p_j U b_j) in the output (the exact
      term missing, its recovery present); with U orthonormal and a_j = p_j +
      err, its expected squared norm is
      w_j^2 (p_j^2 (||d_j||^2 - ||b_j||^2) + var(a_j) ||d_j||^2), the first
      term clamped at 0 (FP16 b can exceed the FP32 ||d_j|| by rounding);
    - var(a_j) = (phi'(ghat_j) vhat_j)^2 var(g_j) + phi(ghat_j)^2 var(v_j)
      (first order in the sketch errors, which are taken as independent);
    - var(g_j) = sum_b rho^g_{j,b} ||(Rx)_b||^2: the block's ternary error has
      mean square rho_b per coordinate and meets Rx_b in every coordinate;
      var(v_j) likewise.
    Uses the stored FP16 rho and b and the FP32 ||d_j||."""
    sh = layer.shape
    if sh.c != BLOCK:
        raise ValueError("the expected-error ranking uses the full screen (c = 128)")
    sc = screen_token(layer, x, ids, w)
    Rx = rotate(pad_hidden(np.asarray(x, dtype=np.float64), sh.Hp), layer.sigma).reshape(sh.nb, BLOCK)
    rn2 = (Rx * Rx).sum(axis=1)                                  # [nb]
    wv = np.asarray(w, dtype=np.float64)
    out = np.zeros((len(ids), sh.I))
    for s_, e in enumerate(int(v) for v in ids):
        rho = layer.sketch(e).rho.astype(np.float64)             # [nb][2][I]
        var_g = rn2 @ rho[:, 0, :]
        var_v = rn2 @ rho[:, 1, :]
        g, v = sc.ghat[s_], sc.vhat[s_]
        var_a = (silu_grad(g) * v) ** 2 * var_g + silu(g) ** 2 * var_v
        dn2 = layer.dnorm(e).astype(np.float64) ** 2
        bn2 = (layer.b(e).astype(np.float64) ** 2).sum(axis=1)
        out[s_] = wv[s_] ** 2 * (sc.p[s_] ** 2 * np.maximum(dn2 - bn2, 0.0) + var_a * dn2)
    return sc, out


def decode_token_rho(layer: Layer, x: np.ndarray, ids, w, k: int) -> TokenResult:
    """One token with the full screen and the top-k by expected_skip_error
    (ties to the lower global id); kept channels exact, the rest recovered."""
    sh = layer.shape
    sc, err = expected_skip_error(layer, x, ids, w)
    gid = np.array([[int(e) * sh.I + i for i in range(sh.I)] for e in ids], dtype=np.int64)
    flat, flat_id = err.reshape(-1), gid.reshape(-1)
    order = np.lexsort((flat_id, -flat))
    kth = float(flat[order[k - 1]]) if k > 0 else float("nan")
    nxt = float(flat[order[k]]) if k < flat.size else float("nan")
    keep = np.zeros(flat.size, bool)
    keep[order[:k]] = True
    y_exact, y_rec = exact_and_recovery(layer, x, ids, w, sc.p, keep.reshape(len(ids), sh.I))
    return TokenResult(
        y=y_exact + y_rec, y_exact=y_exact, y_recovery=y_rec,
        kept=np.sort(flat_id[order[:k]]), kept_order=flat_id[order[:k]],
        score=err, p=sc.p, ghat=sc.ghat, vhat=sc.vhat, mask=sc.mask,
        kth_score=kth, next_score=nxt, gap=sc.gap)


# --------------------------------------------------------------------------
# batch-shared selection
# --------------------------------------------------------------------------
@dataclass
class SharedResult:
    """One batch through the reader with one kept set for the whole batch."""
    tokens: list             # per token: TokenResult (kept = its share of K; kth/next: the batch's)
    experts: np.ndarray      # ascending distinct routed experts of the batch
    batch_score: np.ndarray  # float64 [len(experts)][I]
    K: int                   # kept channels of the batch
    kept: np.ndarray         # int64 sorted global ids e*I + i of K
    kth_score: float
    next_score: float


def shared_kept_count(k: int, n_experts: int, topk: int) -> int:
    """K_B = k * n_e / topk rounded half up: the per-token kept fraction k / N
    applied to the batch's union of n_e * I routed channels."""
    return (2 * k * n_experts + topk) // (2 * topk)


def decode_shared(layer: Layer, x: np.ndarray, ids: np.ndarray, w: np.ndarray, k: int,
                  masks=None) -> SharedResult:
    """Batch-shared selection: one kept set for the whole batch ([CN] §未来方向
    (1) names it as the way to keep the gains at larger batches and gives no
    formula; the reading taken here):

    - every token is screened and scored as in decode_token (steps 1-2);
    - the union U of the batch's routed channels: all I channels of every
      expert some token routes to;
    - batch score S(e, i) = sum of s_{t,(e,i)} over the tokens t routed to e,
      in token order (the output-unit scores add up the tokens' output error);
    - K = the top-K_B of S over U, K_B = shared_kept_count(k, |experts|, topk),
      ties to the lower global id e*I + i;
    - token t computes its channels in K exactly and recovers its routed
      channels outside K with its own p (steps 3-4).

    At batch 1, U is the token's N routed channels, K_B = k and S = s: the
    per-token reader.  `masks` (bool [B][nb][128], optional) fixes the
    tokens' screened coordinates (see screen_token)."""
    sh = layer.shape
    B = x.shape[0]
    ids = np.asarray(ids)
    screens = [screen_token(layer, x[t], ids[t], w[t], mask=None if masks is None else masks[t])
               for t in range(B)]
    experts = np.array(sorted({int(e) for e in ids.reshape(-1)}), dtype=np.int64)
    rank = {int(e): r for r, e in enumerate(experts)}
    S = np.zeros((experts.size, sh.I))
    for t in range(B):
        for s_, e in enumerate(ids[t]):
            S[rank[int(e)]] += screens[t].score[s_]
    K = shared_kept_count(k, experts.size, sh.topk)
    gid = (experts[:, None] * sh.I + np.arange(sh.I)[None, :]).reshape(-1)
    flat = S.reshape(-1)
    order = np.lexsort((gid, -flat))
    kept = np.sort(gid[order[:K]])
    kth = float(flat[order[K - 1]]) if K > 0 else float("nan")
    nxt = float(flat[order[K]]) if K < flat.size else float("nan")
    kept_set = set(int(g) for g in kept)
    tokens = []
    for t in range(B):
        sc = screens[t]
        tid = np.array([[int(e) * sh.I + i for i in range(sh.I)] for e in ids[t]], dtype=np.int64)
        keep = np.vectorize(lambda g: int(g) in kept_set)(tid) if tid.size else np.zeros_like(tid, bool)
        y_exact, y_rec = exact_and_recovery(layer, x[t], ids[t], w[t], sc.p, keep)
        mine = np.sort(tid[keep])
        tokens.append(TokenResult(
            y=y_exact + y_rec, y_exact=y_exact, y_recovery=y_rec, kept=mine, kept_order=mine,
            score=sc.score, p=sc.p, ghat=sc.ghat, vhat=sc.vhat, mask=sc.mask,
            kth_score=kth, next_score=nxt, gap=sc.gap))
    return SharedResult(tokens=tokens, experts=experts, batch_score=S, K=K, kept=kept,
                        kth_score=kth, next_score=nxt)


# --------------------------------------------------------------------------
# stacked layers
# --------------------------------------------------------------------------
RMS_EPS = 1e-6   # keeps a zero residual finite, as RMS normalisation layers do


def rms_normalise(h: np.ndarray) -> np.ndarray:
    """x = h / sqrt(mean(h^2) + eps) per token, in float64.  The stack's layer
    input: the pages state only that the residual stream is carried from layer
    to layer ([CN] §局限与改进 and §独立分析的弱点 (1) on per-layer fixed costs);
    each layer reading the normalised residual is the plain reading of a
    pre-normalised decoder block."""
    h = np.asarray(h, dtype=np.float64)
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + RMS_EPS)


def decode_stack(layers, h_in: np.ndarray, ids, w, k: int):
    """L stacked layers: x_l = rms_normalise(h_l) handed to the layer as fp32
    (the layer input precision), y_l = decode(layer_l, x_l), h_{l+1} = h_l + y_l
    in float64.  ids, w: [L][B][topk].  Returns (per-layer decode results,
    h_L)."""
    h = np.asarray(h_in, dtype=np.float64)
    results = []
    for l, layer in enumerate(layers):
        x = rms_normalise(h).astype(np.float32)
        res = decode(layer, x, ids[l], w[l], k)
        results.append(res)
        h = h + np.stack([r.y for r in res])
    return results, h
