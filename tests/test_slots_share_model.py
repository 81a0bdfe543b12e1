"""Model check, on the CPU, of how the valid-slot kernel shares its pages
out among warps: each warp's fixed contiguous range of the first
``fixed`` pages, then ranges of the rest taken from one counter, of about
(pages left) / (2 warps) and at least a minimum (guided self-scheduling).
Warps are replayed in random order with random speeds; every page must be
walked exactly once, the counter's overshoot must stay within one range per
warp, and taking a range ahead (before the warp is free) is shown to hand
out more of the pool up front, the reason the kernel does not."""

import random

import pytest

FIXED_SHARE = 4
MIN_RANGE = 16


def share_out(items, warps, dynamic, rnd, ahead=False):
    """Pages walked per warp (list of (lo, hi) ranges per warp) and the
    pages handed out before any warp finished its fixed share."""
    fixed = items // FIXED_SHARE if dynamic else items
    counter = 0
    walked = [[] for _ in range(warps)]
    for w in range(warps):
        i0, i1 = fixed * w // warps, fixed * (w + 1) // warps
        if i0 < i1:
            walked[w].append((i0, i1))
    if not dynamic:
        return walked, 0
    # each warp's state: pages left as it last saw them; a pending range
    # when it takes one ahead
    left = [items - fixed] * warps
    pending = [None] * warps
    up_front = 0
    if ahead:
        for w in range(warps):
            n = max(MIN_RANGE, left[w] // (2 * warps))
            pending[w] = (counter, n)
            counter += n
        up_front = min(counter, items - fixed)
    active = list(range(warps))
    while active:
        w = rnd.choice(active)
        if ahead:
            lo0, n = pending[w]
        else:
            n = max(MIN_RANGE, left[w] // (2 * warps))
            lo0 = counter
            counter += n
        lo = fixed + lo0
        if lo >= items:
            active.remove(w)
            continue
        hi = min(lo + n, items)
        left[w] = items - hi
        if ahead:
            n2 = max(MIN_RANGE, left[w] // (2 * warps))
            pending[w] = (counter, n2)
            counter += n2
        walked[w].append((lo, hi))
    assert counter <= items - fixed + warps * max(MIN_RANGE, (items - fixed) // (2 * warps)) * 2
    return walked, up_front


@pytest.mark.parametrize("seed", range(40))
def test_every_page_once(seed):
    rnd = random.Random(seed)
    items = rnd.choice([1, 7, 64, 1000, 4096, 65536, 166400, 300001])
    warps = rnd.choice([1, 8, 64, 640, 2432])
    for dynamic in (False, True):
        walked, _ = share_out(items, warps, dynamic, rnd)
        seen = bytearray(items)
        for ranges in walked:
            for lo, hi in ranges:
                assert 0 <= lo < hi <= items
                for i in range(lo, hi):
                    seen[i] += 1
        assert all(c == 1 for c in seen), (seed, items, warps, dynamic)


def test_ranges_shrink_toward_the_end():
    """Guided ranges start near (pages left) / (2 warps) and end at the
    minimum: the last ranges are short, so warps end close together."""
    rnd = random.Random(1)
    items, warps = 1 << 20, 2432
    walked, _ = share_out(items, warps, True, rnd)
    dyn = sorted((r for ranges in walked for r in ranges[1:]), key=lambda r: r[0])
    first, last = dyn[0], dyn[-1]
    assert first[1] - first[0] == (items - items // FIXED_SHARE) // (2 * warps)
    assert last[1] - last[0] <= MIN_RANGE


def test_taking_ranges_ahead_hands_the_pool_out_early():
    rnd = random.Random(2)
    items, warps = 1 << 20, 2432
    _, up_front = share_out(items, warps, True, rnd, ahead=True)
    # about half the dynamic pool is spoken for before any warp is free
    assert up_front >= 0.45 * (items - items // FIXED_SHARE)
