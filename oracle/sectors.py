"""32-byte-sector read accounting for one decode call.

TEST INFRASTRUCTURE ONLY -- see the package docstring for who may import it.

[CN] §前置知识 "显存带宽受限的解码": the GPU reads memory in 32-byte sectors,
so a read of 80 bytes that touches 4 sectors costs 128 bytes; reads are
counted as a share of the full model's routed-expert reads.  [KR] §전제와 한계:
every weight/parameter read is billed in 32-byte hardware sectors.

Every parameter array below starts on a 256-byte boundary and is laid out
as documented for the library:

  codes   u8   [E][nb][128][2][S]   S = ceil(ceil(I/4)/32)*32; a screened
                                    coordinate reads its gate run and its up run,
                                    ceil(I/4) bytes each (five-trit layout:
                                    ceil(I/5) bytes, S = ceil(ceil(I/5)/32)*32)
  scales  f16  [E][nb][2][I]        a routed expert reads all of them
  dnorm   f32  [E][I]               a routed expert reads all of them
  G, V    bf16 [E][I][H]            a kept channel reads its row
  Dt      bf16 [E][I][H]            a kept channel reads its row
  b       f16  [E][I][r]            a skipped channel reads its row
  U       f16  [H][r]               read whole when any token skips a channel

Counts are sets of distinct sectors, a union over the tokens of the batch.
The denominator is the union of the routed experts' full G, V and D arrays.
"""

from __future__ import annotations

import numpy as np

SECTOR = 32
ARRAYS = ("codes", "scales", "dnorm", "G", "V", "Dt", "b", "U")


def sectors_touched(start: int, length: int) -> set:
    """Set of sector indices touched by the byte range [start, start + length)."""
    if length <= 0:
        return set()
    return set(range(start // SECTOR, (start + length - 1) // SECTOR + 1))


def _ranges_to_sectors(starts: np.ndarray, length: int) -> np.ndarray:
    """Distinct sector ids covered by equal-length byte ranges at `starts`."""
    if starts.size == 0 or length <= 0:
        return np.zeros(0, np.int64)
    starts = np.asarray(starts, dtype=np.int64)
    first = starts // SECTOR
    last = (starts + length - 1) // SECTOR
    span = int((last - first).max()) + 1
    ids = first[:, None] + np.arange(span)[None, :]
    ids = ids[ids <= last[:, None]]
    return np.unique(ids)


def decode_sectors(shape, ids, masks, kept, codes="2bit"):
    """Distinct 32-byte sectors read per parameter array for one decode call.

    shape: oracle.reader.Shape; ids: int [B][topk] routed experts;
    masks: bool [B][nb][128] screened coordinates per token;
    kept: list of B arrays of kept global channel ids (e*I + i);
    codes: "2bit" (4 trits a byte) or "trit5" (5 trits a byte: runs of
    ceil(I/5) bytes, the 1.6-bit layout).
    Returns dict array-name -> sector count, plus "dense" (the denominator).
    """
    E, I, H, r, nb = shape.E, shape.I, shape.H, shape.r, shape.nb
    if codes not in ("2bit", "trit5"):
        raise ValueError(codes)
    run = (I + 3) // 4 if codes == "2bit" else (I + 4) // 5
    stride = SECTOR * ((run + SECTOR - 1) // SECTOR)
    B = len(ids)

    code_starts, scale_starts, dn_starts = [], [], []
    kept_ids, skip_ids = [], []
    routed = set()
    any_skip = False
    for t in range(B):
        experts = [int(e) for e in ids[t]]
        routed.update(experts)
        kb, kc = np.nonzero(masks[t])
        for e in experts:
            base = ((e * nb + kb) * 128 + kc) * 2
            code_starts.append(base * stride)          # gate run
            code_starts.append((base + 1) * stride)    # up run
        kset = set(int(g) for g in kept[t])
        for e in experts:
            for i in range(I):
                g = e * I + i
                (kept_ids if g in kset else skip_ids).append(g)
                if g not in kset:
                    any_skip = True
    for e in sorted(routed):
        for b in range(nb):
            scale_starts.append(((e * nb + b) * 2) * I * 2)
        dn_starts.append(e * I * 4)

    counts = {}
    counts["codes"] = _ranges_to_sectors(np.concatenate(code_starts) if code_starts else np.zeros(0),
                                         run).size
    counts["scales"] = _ranges_to_sectors(np.array(scale_starts), 2 * I * 2).size
    counts["dnorm"] = _ranges_to_sectors(np.array(dn_starts), I * 4).size
    kept_arr = np.unique(np.array(kept_ids, dtype=np.int64))
    row = H * 2
    for name in ("G", "V", "Dt"):
        counts[name] = _ranges_to_sectors(kept_arr * row, row).size
    skip_arr = np.unique(np.array(skip_ids, dtype=np.int64))
    counts["b"] = _ranges_to_sectors(skip_arr * r * 2, r * 2).size
    counts["U"] = _ranges_to_sectors(np.array([0]), H * r * 2).size if any_skip else 0

    expert_bytes = I * H * 2
    dense = 0
    for _ in range(3):  # G, V, D of every routed expert
        dense += _ranges_to_sectors(np.array(sorted(routed), dtype=np.int64) * expert_bytes,
                                    expert_bytes).size
    counts["dense"] = dense
    return counts


def analytic_sectors_b1(shape, k: int) -> dict:
    """Closed-form sector counts for ONE token with distinct experts, k kept
    channels (0 < k < N) and c screened coordinates per block; used to pin the
    set-based count."""
    I, H, r, nb, topk, c = shape.I, shape.H, shape.r, shape.nb, shape.topk, shape.c
    up = lambda nbytes: -(-nbytes // SECTOR)  # noqa: E731  sectors of an aligned range
    N = topk * I
    out = {
        "codes": topk * nb * c * 2 * up((I + 3) // 4),
        "scales": topk * nb * up(2 * I * 2),
        "dnorm": topk * up(I * 4),
        "G": k * up(2 * H), "V": k * up(2 * H), "Dt": k * up(2 * H),
        "U": up(2 * H * r),
        "dense": 3 * topk * up(I * H * 2),
    }
    # b rows: r*2 bytes each; when a row is shorter than a sector, adjacent
    # skipped channels share sectors, so the closed form holds only when
    # r*2 is a multiple of 32.
    if (2 * r) % SECTOR == 0:
        out["b"] = (N - k) * (2 * r // SECTOR)
    return out
