"""Element windows of a full-size workload that the parity tests compare
with the oracle: every shard's first and last 4,096 elements, +-256 around
every tensor boundary, the last tile of every CTA of the bulk-copy pipeline
and random windows.  Host logic only."""
import numpy as np

TILE = 2048          # elements per tile of the bulk-copy pipeline


def windows(wl, seed=0, ctas=None, n_random=64, random_len=1 << 20):
    E = wl.elems
    r = []
    if wl.shard is None:
        for k in range(wl.P):
            b, e = min(k * wl.M, wl.N), min((k + 1) * wl.M, wl.N)
            if b < e:
                r += [(b, min(b + 4096, e)), (max(b, e - 4096), e)]
    else:
        r += [(0, min(4096, E)), (max(0, E - 4096), E)]
    if wl.tensors:
        pos = 0
        for n in wl.tensors[:-1]:
            pos += n
            r.append((max(0, pos - 256), min(E, pos + 256)))
    if ctas:
        # CTA c takes tiles c, c + ctas, ...: its last one is the largest such
        # index below the tile count (buffers start 16-byte aligned: no head)
        ntiles = -(-(E // 8 * 8) // TILE)
        for c in range(min(ctas, ntiles)):
            last = c + ((ntiles - 1 - c) // ctas) * ctas
            r.append((last * TILE, min(E, (last + 1) * TILE)))
    rng = np.random.default_rng(seed)
    for s in rng.integers(0, max(1, E - random_len), size=n_random):
        r.append((int(s), int(min(E, s + random_len))))
    r.sort()
    merged = []
    for b, e in r:
        if merged and b <= merged[-1][1]:
            merged[-1] = (merged[-1][0], max(merged[-1][1], e))
        else:
            merged.append((b, e))
    return merged
