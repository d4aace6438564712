"""Pins of the oracle's 1.6-bit (five trits per byte) code layout (no GPU):
the packing's worked values and round trips, the pages' ~30 bytes per
128-coordinate block, and the read shares of the Qwen3-30B-shaped layer at the
17.8% budget, where five-trit codes bring the sketch to the pages' 4.9% and
the total to their 17.8%."""

import numpy as np
import pytest

from oracle import reader as R
from oracle import sectors as SC


def test_worked_byte_values():
    # digits (0, +1, -1) -> (0, 1, 2), little-endian base 3
    t = np.array([[1, 0, -1, 1, 1]], np.int8)
    assert R.pack_codes5(t)[0, 0] == 1 + 0 * 3 + 2 * 9 + 1 * 27 + 1 * 81 == 127
    assert R.pack_codes5(np.array([[-1] * 5], np.int8))[0, 0] == 242
    assert R.pack_codes5(np.array([[0] * 5], np.int8))[0, 0] == 0
    assert R.pack_codes5(np.array([[1] * 5], np.int8))[0, 0] == 121


def test_every_byte_round_trips():
    digits = np.array([[(b // 3 ** m) % 3 for m in range(5)] for b in range(243)])
    t = np.where(digits == 1, 1, np.where(digits == 2, -1, 0)).astype(np.int8)
    packed = R.pack_codes5(t)
    assert np.array_equal(packed[:, 0], np.arange(243, dtype=np.uint8))
    assert np.array_equal(R.unpack_codes5(packed, 5), t)
    with pytest.raises(ValueError):
        R.unpack_codes5(np.array([[243]], np.uint8), 5)


@pytest.mark.parametrize("I", [128, 768, 1536, 2880, 4160])
def test_random_runs_round_trip(I):
    rng = np.random.default_rng(I)
    t = rng.integers(-1, 2, size=(3, 7, I)).astype(np.int8)
    packed = R.pack_codes5(t)
    assert packed.shape[-1] == R.run_stride5(I) and R.run_stride5(I) % 32 == 0
    assert packed.shape[-1] >= (I + 4) // 5
    assert np.array_equal(R.unpack_codes5(packed, I), t)
    assert not packed[..., R.run_bytes5(I):].any()   # zero padding


def test_block_of_128_trits_is_about_30_bytes():
    # 256 BF16 bytes -> ternary codes at 8/5 bits + FP16 scale + FP16 rho
    assert R.run_bytes5(128) + 2 + 2 == 30
    assert R.run_bytes(128) + 2 + 2 == 36       # the 2-bit layout


def _one_token_reads(codes):
    sh = R.Shape(H=2048, E=128, topk=8, I=768, c=80, r=32)
    ids = np.array([[3, 17, 29, 40, 66, 80, 101, 127]])
    masks = np.zeros((1, sh.nb, 128), bool)
    masks[0, :, :80] = True                      # 80 screened coordinates a block
    # 756 kept rows (any 756 distinct channels read the same number of sectors)
    kept = [np.array([e * sh.I + i for e in ids[0] for i in range(95)][:756])]
    assert kept[0].size == 756
    st = SC.decode_sectors(sh, ids, masks, kept, codes=codes)
    return {k: v / st["dense"] for k, v in st.items() if k != "dense"}


def test_read_shares_match_the_pages_budget():
    two = _one_token_reads("2bit")
    five = _one_token_reads("trit5")
    assert abs(two["codes"] - 0.0521) < 5e-4
    assert abs(five["codes"] - 0.0434) < 5e-4
    # sketch = codes + scales: 4.9% on the pages at the 17.8% budget
    assert abs(five["codes"] + five["scales"] - 0.049) < 5e-4
    assert abs(sum(five.values()) - 0.178) < 1e-3
    assert abs(sum(two.values()) - 0.187) < 1e-3
    for a in ("scales", "dnorm", "G", "V", "Dt", "b", "U"):
        assert two[a] == five[a]
