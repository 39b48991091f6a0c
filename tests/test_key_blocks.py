"""The key-block count of the backward with different query and key lengths
(dash_key_blocks, host only): the largest divisor of the key tile count that
leaves at least as many key tiles per block as query tiles, for as many
key/value heads as query heads and whole key tiles, within the index range."""
import pytest

from tile_scheduling_persistent_gb300 import dash


def brute(B, Hq, Hkv, Sq, Skv):
    if Skv == Sq or Hq != Hkv or Skv % 128:
        return 1
    nq, nkv = (Sq + 127) // 128, Skv // 128
    ok = [g for g in range(1, nkv + 1) if nkv % g == 0 and nkv // g >= nq and B * Hq * g * Sq < 2 ** 31]
    return max(ok)


@pytest.mark.parametrize("shape", [
    (4, 16, 16, 1024, 8192),      # the 1K x 8K workload: 8 blocks of 8 key tiles
    (1, 1, 1, 130, 1024),         # 2 query tiles (ragged), 8 key tiles: 4 blocks
    (1, 2, 2, 256, 640),          # 5 key tiles: no divisor leaves 2 per block
    (1, 4, 2, 640, 256),          # grouped-query heads: no split
    (1, 2, 2, 200, 333),          # ragged keys: no split
    (1, 2, 2, 1024, 1024),        # equal lengths: no split
    (2, 8, 8, 128, 128 * 64),     # one query tile: a block per key tile
    (1, 16, 16, 1_000_000, 1024 * 128 * 16),   # the index range caps G
])
def test_key_blocks_rule(shape):
    assert dash.key_blocks(*shape) == brute(*shape)


def test_key_blocks_examples():
    assert dash.key_blocks(4, 16, 16, 1024, 8192) == 8
    assert dash.key_blocks(2, 8, 8, 128, 128 * 64) == 64
    assert dash.key_blocks(1, 16, 16, 1_000_000, 1024 * 128 * 16) == 2


def test_key_blocks_rejects_bad_sizes():
    with pytest.raises(dash.DashError):
        dash.key_blocks(0, 1, 1, 128, 256)
