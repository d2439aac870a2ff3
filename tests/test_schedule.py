"""Host-side checks of the attention kernel's work schedule (no GPU needed).

attn_flash_schedule returns the plan attn_fwd / attn_fwd_ws would launch: the
mode, the persistent grid, the whole items [0, dp_end) dealt round-robin and,
when the last waves are cut along the key axis, each CTA's run of key tiles
[cut[g], cut[g+1]) and the CTA range its merge waits for (g_last).  The
kernel relies on these invariants: the runs tile the cut units exactly, a run
starts inside an item at most once (its first segment, the only one that
writes a piece), and g_last names the CTA holding the item's last key tile.
"""

import math

import pytest

import head_attention_fwd_gb300 as attn

def n_items(B, h, S):
    return B * h * math.ceil(S / 256)


def run_segments(cut_lo, cut_hi, n_kv):
    """Segments (start, end, starts_mid, ends_at_item_end) of one run."""
    segs, pos = [], cut_lo
    while pos < cut_hi:
        item_end = (pos // n_kv + 1) * n_kv
        end = min(item_end, cut_hi)
        segs.append((pos, end, pos % n_kv != 0, end == item_end))
        pos = end
    return segs


CUT_CASES = [
    (1, 16, 4096, 64, 152),   # the bench workload: 256 items of 32 key tiles
    (2, 16, 8192, 64, 152),   # long sequence: 1024 items of 64 key tiles
    (1, 4, 8192, 64, 152),    # one partial wave: every item cut
    (1, 20, 4096, 64, 148),
    (3, 7, 5000, 64, 132),    # ragged key tail (40 tiles, the last one partial)
    (1, 25, 4096, 64, 300),   # more SMs than a cut plan may use: grid capped at 256
]


@pytest.mark.parametrize("B,h,S,d,sms", CUT_CASES, ids=lambda x: str(x))
def test_cut_runs_tile_the_units_and_merge_ranges_are_right(B, h, S, d, sms, monkeypatch):
    monkeypatch.delenv("ATTN_SPLIT", raising=False)
    plan = attn.attn_flash_schedule(B, h, S, d, sms, True)
    n_kv = math.ceil(S / 128)
    items = n_items(B, h, S)
    assert plan["mode"] == 2
    grid = plan["grid"]
    assert grid == min(sms, 256, items * n_kv)
    # whole items fill complete waves; the rest is cut
    assert plan["dp_end"] % grid == 0
    assert plan["dp_end"] + plan["sk_units"] // n_kv == items
    assert plan["sk_units"] % n_kv == 0
    cut, g_last = plan["cut"], plan["g_last"]
    assert cut[0] == 0 and cut[grid] == plan["sk_units"]
    assert all(cut[g] <= cut[g + 1] for g in range(grid))
    for g in range(grid):
        segs = run_segments(cut[g], cut[g + 1], n_kv)
        # only the first segment of a run may start inside an item (one piece per CTA)
        assert all(not mid for (_, _, mid, _) in segs[1:])
        if not segs:
            continue
        last_unit = ((cut[g + 1] - 1) // n_kv + 1) * n_kv - 1
        holder = next(x for x in range(grid) if cut[x] <= last_unit < cut[x + 1])
        assert g_last[g] == holder
        assert g_last[g] >= g


@pytest.mark.parametrize("B,h,S,d,sms", CUT_CASES, ids=lambda x: str(x))
def test_cut_runs_are_equal(B, h, S, d, sms, monkeypatch):
    """Every CTA's run has floor(U/grid) or ceil(U/grid) key tiles, and the
    whole items before the cut fill complete waves, so every SM does the
    same number of key tiles up to one."""
    monkeypatch.delenv("ATTN_SPLIT", raising=False)
    plan = attn.attn_flash_schedule(B, h, S, d, sms, True)
    grid, U, cut = plan["grid"], plan["sk_units"], plan["cut"]
    lens = {cut[g + 1] - cut[g] for g in range(grid)}
    assert lens <= {U // grid, -(-U // grid)}


def test_modes_without_a_cut(monkeypatch):
    monkeypatch.delenv("ATTN_SPLIT", raising=False)
    # d = 128: one item per CTA
    p = attn.attn_flash_schedule(1, 32, 16384, 128, 152, True)
    assert p["mode"] == 0 and p["grid"] == n_items(1, 32, 16384) and p["sk_units"] == 0
    # whole items requested
    p = attn.attn_flash_schedule(1, 16, 4096, 64, 152, False)
    assert p["mode"] == 1 and p["grid"] == 152 and p["dp_end"] == 256 and p["sk_units"] == 0
    # short items (4 key tiles) never pay for a cut
    p = attn.attn_flash_schedule(8, 12, 512, 64, 152, True)
    assert p["mode"] == 1 and p["sk_units"] == 0
    # an item count that fills whole waves has nothing to balance
    p = attn.attn_flash_schedule(1, 19, 4096, 64, 152, True)
    assert n_items(1, 19, 4096) % 152 == 0 and p["mode"] == 1
    # fewer items than SMs: one item per CTA on a grid of the item count
    p = attn.attn_flash_schedule(1, 2, 1024, 64, 152, True)
    assert p["mode"] == 1 and p["grid"] == n_items(1, 2, 1024)


def test_split_environment_override(monkeypatch):
    monkeypatch.setenv("ATTN_SPLIT", "never")
    assert attn.attn_flash_schedule(1, 16, 4096, 64, 152, True)["mode"] == 1
    monkeypatch.setenv("ATTN_SPLIT", "force")
    p = attn.attn_flash_schedule(8, 12, 512, 64, 152, True)  # short items, cut anyway
    assert p["mode"] == 2 and p["cut"][-1] == p["sk_units"]


def test_schedule_rejects_bad_sizes():
    for args in [(0, 1, 128, 64, 152), (1, 1, 128, 96, 152), (1, 1, 128, 64, 0)]:
        with pytest.raises(ValueError):
            attn.attn_flash_schedule(*args)
