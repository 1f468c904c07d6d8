"""Index arithmetic of the split-over-pages work partition (CPU only).

The decode kernels lay all tiles of all (request, head) lanes end to end and
give worker w the range [floor(w T / W), floor((w + 1) T / W)).  A lane's tiles
[A, A + n) belong to workers floor(((x + 1) W - 1) / T); partial results of a
split lane go to slot lane + w.  These properties must hold for the merge to
read exactly what the split kernel wrote, whatever the mix of lengths.
"""
import numpy as np
import pytest


def begin(w, T, W):
    return (w * T) // W


def worker_of(x, T, W):
    return ((x + 1) * W - 1) // T


def check(tiles_per_req, H, W):
    prefix = np.concatenate([[0], np.cumsum(tiles_per_req)]).astype(np.int64)
    T = H * int(prefix[-1])
    if T == 0:
        return
    # every tile has exactly one worker, and worker_of inverts begin
    owner = np.empty(T, dtype=np.int64)
    for w in range(W):
        b0, b1 = begin(w, T, W), begin(w + 1, T, W)
        owner[b0:b1] = w
    assert all(worker_of(x, T, W) == owner[x] for x in range(T))
    written = {}
    for b, n in enumerate(tiles_per_req):
        for h in range(H):
            if n == 0:
                continue
            lane = b * H + h
            A = H * int(prefix[b]) + h * int(n)
            lo, hi = worker_of(A, T, W), worker_of(A + n - 1, T, W)
            if lo == hi:
                continue                           # finished by one worker
            owners = set(owner[A:A + n].tolist())
            nonempty = {w for w in range(lo, hi + 1) if begin(w, T, W) != begin(w + 1, T, W)}
            assert owners == nonempty              # merge reads exactly the writers
            for w in owners:
                slot = lane + w
                assert slot not in written, "partial slots collide"
                assert slot < (len(tiles_per_req) * H) + W
                written[slot] = lane
    # the first request of each non-empty worker (the plan kernel's search)
    for w in range(W):
        x = begin(w, T, W)
        if x >= T:
            continue
        b = max(i for i in range(len(tiles_per_req)) if H * prefix[i] <= x)
        assert H * prefix[b] <= x < H * prefix[b + 1]


@pytest.mark.parametrize("seed", range(40))
def test_random_mixes(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 12))
    tiles = rng.integers(0, 30, size=B)
    if seed % 3 == 0:
        tiles[rng.integers(0, B)] = 0
    H = int(rng.integers(1, 5))
    W = int(rng.integers(1, 400))
    check(tiles.tolist(), H, W)


def test_more_workers_than_tiles():
    check([3, 0, 1], 1, 64)
    check([1], 1, 1000)
    check([2, 2], 2, 7)
