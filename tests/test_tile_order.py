"""The fused wgrad + SGD kernel's tile schedule (csrc/gemm.cu, decode_tile, contraction-grouped
branch): slot t = c + G*i of a persistent grid of G CTAs maps to a position of the size-sorted
tile list.  Every position must be visited exactly once, whatever the number of tiles (the
kernel runs slots t < ntiles), or a master-weight tile would be updated twice or not at all.
The two rules are written out here as the kernel evaluates them (unsigned 32-bit arithmetic)."""
import random

import pytest


def every_third(t, G, n):
    # front when t % 3 == 0 (position t / 3), else back (position n - 1 - (t - ceil(t / 3)))
    return t // 3 if t % 3 == 0 else n - 1 - (t - (t + 2) // 3)


def alternate(t, G, n):
    # front when c + i is even; position i * G/2 + c/2 from that end
    i, c = t // G, t % G
    fi = i * (G // 2) + c // 2
    return fi if (c + i) % 2 == 0 else n - 1 - fi


def schedule(G):
    if G % 3 != 0:
        return every_third
    if G % 2 == 0:
        return alternate
    return lambda t, G, n: t


@pytest.mark.parametrize("G", [148, 132, 2, 3, 6, 7, 12, 296])
def test_slots_cover_each_tile_once(G):
    rng = random.Random(G)
    f = schedule(G)
    counts = [1, 2, G - 1, G, G + 1, 3 * G + 2] + [rng.randrange(1, 40 * G) for _ in range(20)]
    if G == 148:
        counts += [336 * 1024, 336 * 512]  # the layer step's gate/up and down tile lists
    for n in counts:
        pos = [f(t, G, n) for t in range(n)]
        assert sorted(pos) == list(range(n)), (G, n)


def test_every_third_rotates_each_cta():
    # G = 148: each CTA takes the front every third tile, a third of the CTAs at any one time
    G, n = 148, 336 * 1024
    for c in (0, 1, 2, 77, 147):
        front = [every_third(c + G * i, G, n) < n // 3 for i in range(30)]
        assert sum(front) == 10
        assert all(front[i] == front[i + 3] for i in range(27))
    for i in range(6):
        assert sum(every_third(c + G * i, G, n) < n // 3 for c in range(G)) in (49, 50)
