"""Index arithmetic of the split-over-pages work partition (CPU only).

The decode kernels lay all tiles of all (request, head) lanes end to end and
give worker w the range [floor(w T / W), floor((w + 1) T / W)).  A lane's tiles
[A, A + n) belong to workers floor(((x + 1) W - 1) / T); partial results of a
split lane go to slot lane + w.  These properties must hold for the merge to
read exactly what the split kernel wrote, whatever the mix of lengths.

With more than 8 query heads per KV head, a KV head's lanes are 2^s sub-lanes:
the ranges then partition the KV lanes' tiles (R = W / 2^s ranges), worker w
takes range w >> s for sub-lane w & (2^s - 1), and the partial of KV lane K from
range r goes to slot ((K + r) << s) | sub.  With s = 0 this is the scheme above.
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


def check_sub_lanes(tiles_per_req, Hk, s, W):
    """Sub-lane partition: every (lane, worker) partial has its own slot below
    B * H + W (H = Hk << s lane heads), and the merge of a lane reads exactly the
    ranges that hold its tiles, at the slots their sub-lane worker wrote."""
    NS = 1 << s
    assert W % NS == 0
    R = W // NS
    prefix = np.concatenate([[0], np.cumsum(tiles_per_req)]).astype(np.int64)
    T = Hk * int(prefix[-1])
    if T == 0:
        return
    owner = np.empty(T, dtype=np.int64)                  # range of each KV-lane tile
    for r in range(R):
        owner[begin(r, T, R):begin(r + 1, T, R)] = r
    assert all(worker_of(x, T, R) == owner[x] for x in range(T))
    H = Hk << s
    written = {}
    for b, n in enumerate(tiles_per_req):
        if n == 0:
            continue
        for hk in range(Hk):
            K = b * Hk + hk
            A = Hk * int(prefix[b]) + hk * int(n)
            r_lo, r_hi = worker_of(A, T, R), worker_of(A + n - 1, T, R)
            ranges = set(owner[A:A + n].tolist())
            nonempty = {r for r in range(r_lo, r_hi + 1) if begin(r, T, R) != begin(r + 1, T, R)}
            assert ranges == nonempty
            for sub in range(NS):
                lane = b * H + (hk << s | sub)
                for r in ranges:
                    w = (r << s) | sub                   # the worker that wrote it
                    assert w < W
                    slot = ((K + r) << s) | sub
                    assert slot not in written, "partial slots collide"
                    assert slot < len(tiles_per_req) * H + W
                    written[slot] = (lane, w)


@pytest.mark.parametrize("seed", range(40))
def test_sub_lane_mixes(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 10))
    tiles = rng.integers(0, 30, size=B)
    if seed % 3 == 0:
        tiles[rng.integers(0, B)] = 0
    Hk = int(rng.integers(1, 4))
    s = int(rng.integers(0, 5))
    W = (1 << s) * int(rng.integers(1, 200))
    check_sub_lanes(tiles.tolist(), Hk, s, W)


def test_sub_lanes_reduce_to_the_plain_scheme():
    """s = 0: the slot ((K + r) << 0) | 0 = lane + w of the plain partition."""
    check_sub_lanes([3, 0, 7, 1], 2, 0, 5)
    check_sub_lanes([1], 1, 3, 1000 - 1000 % 8)
