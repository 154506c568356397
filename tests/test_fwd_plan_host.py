"""Host-side launch plan of the forward (no GPU): which grid a shape gets, and
the balanced per-CTA work lists of causal shapes (FlashAttention-4 summary,
section 3.3: work tiles taken longest first, heads of an L2 section innermost).

The lists are checked against the work-order definition, restated here in
plain Python: every work tile appears exactly once, each CTA takes its tiles
in work-list order, and the estimated work per CTA is balanced to within one
tile, the bound that greedy list scheduling guarantees."""

import pytest

from exact_attention_15_gb300 import binding as b

ONE_CTA, STRIDING, BALANCED = b.FWD_ONE_CTA_PER_TILE, b.FWD_STRIDING, b.FWD_BALANCED_LIST
FIXED_COST = 6  # the plan's per-tile start-up estimate, in key tiles


def work_tile_units(v, B, H_q, N, sec_heads, causal, pair=0):
    """Key tiles the two 128-row query tiles of work tile v visit: tiles are
    numbered batch outermost, then sections of sec_heads query heads, then
    m-blocks (reversed under a causal mask), then the heads of the section. A
    work tile is 256 rows of one head, or (pair) the same 128 rows of two
    heads, so m-blocks are 128 rows and heads count in pairs."""
    rows = 256 // (1 + pair)
    heads = H_q // (1 + pair)
    sec_units = sec_heads // (1 + pair)
    nm = (N + rows - 1) // rows
    local = v % (nm * heads)
    sec, rest = divmod(local, nm * sec_units)
    hs = min(sec_units, heads - sec * sec_units)
    mi = rest // hs
    m = nm - 1 - mi if causal else mi
    units = 0
    for i in range(2):
        r0 = rows * m + (0 if pair else 128 * i)
        if r0 >= N:
            continue
        kv_end = min(N, r0 + 128) if causal else N
        units += (kv_end + 127) // 128
    return units


@pytest.mark.parametrize("B,H,N,d", [(4, 16, 8192, 128), (64, 16, 1024, 64), (1, 8, 300, 128)])
def test_equal_tiles_use_striding_or_one_cta_per_tile(B, H, N, d):
    p = b.attn_debug_fwd_plan(B, H, H, N, N, d, d, False, False, 152)
    assert p["tiles"] == B * H * ((N + 255) // 256)
    if p["tiles"] > 152:
        assert (p["mode"], p["grid"]) == (STRIDING, 152)
    else:
        assert (p["mode"], p["grid"]) == (ONE_CTA, p["tiles"])


def test_mode_choice_for_causal_and_packed_shapes():
    # long causal tiles: balanced lists; short ones: striding (saving start-ups wins)
    assert b.attn_debug_fwd_plan(4, 16, 16, 8192, 8192, 128, 128, True, False, 152)["mode"] == BALANCED
    assert b.attn_debug_fwd_plan(64, 16, 16, 1024, 1024, 64, 64, True, False, 152)["mode"] == STRIDING
    # packed inputs never use host lists (their lengths live on the device):
    # with more tiles than SMs, a persistent grid claims them from a counter
    for N in (4096, 40000, 300000):
        p = b.attn_debug_fwd_plan(16, 32, 8, N, N, 128, 128, True, True, 152)
        if p["tiles"] > 152:
            assert (p["mode"], p["grid"]) == (b.FWD_CLAIMED, 152)
        else:
            assert (p["mode"], p["grid"]) == (ONE_CTA, p["tiles"])
    # L2 sections: K + V of 8 heads (4 MiB each at N = 8192, d = 128) fit the 48 MiB share
    assert b.attn_debug_fwd_plan(4, 16, 16, 8192, 8192, 128, 128, True, False, 152)["sec_heads"] == 8


def test_argument_errors():
    with pytest.raises(ValueError):
        b.attn_debug_fwd_plan(1, 16, 16, 1024, 1024, 96, 96, True, False, 152)
    with pytest.raises(ValueError):
        b.attn_debug_fwd_plan(1, 16, 5, 1024, 1024, 128, 128, True, False, 152)
    with pytest.raises(ValueError):
        b.attn_debug_fwd_plan(1, 16, 16, 1024, 1000, 128, 128, True, False, 152)


@pytest.mark.parametrize("B,H_q,H_kv,N,d_qk,d_v,n_sm", [
    (4, 16, 16, 8192, 128, 128, 152),   # the causal benchmark shape
    (1, 16, 16, 32768, 128, 128, 152),  # one long sequence: several L2 sections
    (2, 16, 16, 8192, 64, 64, 148),
    (1, 16, 16, 4096, 192, 128, 152),   # separate head dimensions
    (3, 12, 4, 6000, 128, 128, 152),    # GQA, ragged length, partial last section
    (2, 8, 8, 5000, 128, 128, 20),      # few SMs
    (2, 32, 8, 8192, 128, 128, 152),    # even GQA group: head-pair work tiles
    (1, 16, 4, 3000, 64, 64, 152),      # head pairs, ragged length
])
def test_balanced_lists(B, H_q, H_kv, N, d_qk, d_v, n_sm):
    p = b.attn_debug_fwd_plan(B, H_q, H_kv, N, N, d_qk, d_v, True, False, n_sm)
    assert p["mode"] == BALANCED and p["grid"] == n_sm
    tiles, start, lists = p["tiles"], p["start"], p["tiles_of"]
    assert start[0] == 0 and start[-1] == tiles and len(lists) == tiles
    assert sorted(lists) == list(range(tiles)), "every work tile exactly once"
    pair = p["pair_heads"]
    assert pair == (1 if (H_q // H_kv) % 2 == 0 else 0)
    assert tiles == B * ((N + 255 // (1 + pair)) // (256 // (1 + pair))) * (H_q // (1 + pair))
    cost = {v: FIXED_COST + work_tile_units(v, B, H_q, N, p["sec_heads"], True, pair)
            for v in range(tiles)}
    loads = []
    for c in range(n_sm):
        mine = lists[start[c]:start[c + 1]]
        assert mine, "every CTA has work"
        assert mine == sorted(mine), "a CTA takes its tiles in work-list order"
        loads.append(sum(cost[v] for v in mine))
    assert max(loads) - min(loads) <= max(cost.values())
    # and well below what striding would leave on the long shapes
    stride = [sum(cost[v] for v in range(c, tiles, n_sm)) for c in range(n_sm)]
    assert max(loads) <= max(stride)
