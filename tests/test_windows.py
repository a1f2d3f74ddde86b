"""The window plan of the full-size parity tests (host logic, no GPU)."""
from _windows import TILE, windows
from zero_sharded_mixed_shard_gb300 import synth


def test_windows_cover_every_cta_last_tile():
    """On the 1.3e9 vector at 152 CTAs: the first tile of every CTA's last
    tile lies inside a window, and the random windows add up to ~64 Mi."""
    wl = synth.WORKLOADS["tf1p3b"]
    w = windows(wl, 0, ctas=152)
    ntiles = -(-wl.N // TILE)
    for c in range(152):
        last = c + ((ntiles - 1 - c) // 152) * 152
        assert last + 152 >= ntiles
        b = last * TILE
        assert any(lo <= b and min(wl.N, b + TILE) <= hi for lo, hi in w), c
    assert sum(e - b for b, e in w) >= 64 * (1 << 20) * 0.9


def test_windows_are_sorted_disjoint_and_inside_the_vector():
    for name in ("tf1p3b", "shard7p5b", "folded", "gpt2s"):
        wl = synth.WORKLOADS[name]
        w = windows(wl, wl.seed, ctas=152)
        assert all(0 <= b < e <= wl.elems for b, e in w), name
        assert all(w[i][1] < w[i + 1][0] for i in range(len(w) - 1)), name
