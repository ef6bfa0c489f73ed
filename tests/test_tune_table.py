"""The dispatch table's text form, without a GPU: the tuner reads back every
row of the committed table, writes the same rows again, covers every (N, K)
pair of the trace grid with M ranges that tile 1 .. 2^40 without gaps, and a
merge replaces only the re-measured shapes.  (The table is the measured
counterpart of the page's per-shape meta-parameters: "feat: optimize w8a8
block fp8 matmul for Hopper", FlagGems-vllm PR #693, Description.)"""
import re

import pytest

pytest.importorskip("torch")
from block_scaled_fp8_w8a8_gb300 import tune  # noqa: E402

ROW = re.compile(r"^\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+), (\d+)\},")


def committed_rows():
    return [line.rstrip("\n") for line in open(tune.TABLE) if ROW.match(line)]


def test_table_round_trips():
    best = tune.read_table(tune.TABLE)
    assert len(best) == len(committed_rows()) == len(tune.grid_shapes())
    assert tune.table_lines(best, ranges=True) == committed_rows()


def test_ranges_tile_the_m_axis_for_every_grid_pair():
    by_nk = {}
    for line in committed_rows():
        lo, hi, n, k = (int(v) for v in ROW.match(line).groups()[:4])
        by_nk.setdefault((n, k), []).append((lo, hi))
    assert set(by_nk) == {(n, k) for n in tune.GRID_N for k in tune.GRID_K}
    for ranges in by_nk.values():
        ranges.sort()
        assert ranges[0][0] == 1 and ranges[-1][1] == tune.M_OPEN_END
        for (lo0, hi0), (lo1, hi1) in zip(ranges, ranges[1:]):
            assert lo0 <= hi0 and hi0 + 1 == lo1


def test_merge_replaces_only_the_measured_shapes():
    best = tune.read_table(tune.TABLE)
    key = (4096, 4096, 4096)
    new = dict(best)
    new[key] = dict(variant=1, split_k=3, m_tile=0, block_n_tile=256, stages=3, us=1.0)
    lines = tune.table_lines(new, ranges=True)
    changed = [(a, b) for a, b in zip(committed_rows(), lines) if a != b]
    assert len(changed) == 1 and ", 4096, 4096, 1, 3, 0, 256, 3}," in changed[0][1]


def test_half_tail_candidates_only_where_a_last_wave_fits_twice():
    # 4096 x 4096: 512 tiles of 128 x 256 on 152 SMs leave 56 -> halves fit
    assert any(c.get("split_k") == 3 for c in tune.candidates(4096, 4096, 4096, sms=152))
    # 2048 x 4096: 256 tiles leave 104 > 152 / 2 -> no half tail
    assert not any(c.get("split_k") == 3 for c in tune.candidates(2048, 4096, 4096, sms=152))
