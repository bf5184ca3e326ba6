"""The decode work-item plan (host logic, no GPU): how each (layer, KV head)
stream of a call is cut into large chunks followed by short ones, checked
through the library's test hook against the rule the hook documents and
against the properties the decode kernels rely on."""
import numpy as np
import pytest

import paged_kv_cache_flash_gb300 as K
from paged_kv_cache_flash_gb300 import build as B

SIZES = (128, 64, 32, 16)     # large chunk sizes, largest first
MIN_SMALL = 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    B.build()


def chunks(m, big, small, tail):
    """Chunk sizes of one stream of m blocks, in claim order."""
    nbig = (m - tail) // big if m > tail else 0
    rest = m - nbig * big
    out = [big] * nbig
    while rest > 0:
        out.append(min(small, rest))
        rest -= small
    return out


def rule(nres, L, H, workers, cap, extra):
    """The documented choice, by enumeration: for each large size (largest
    first) the smallest short size whose partials fit; stop at the first
    large size whose large items give every warp one; else the last that
    fit.  Returns (big, small, tail) or (0, 0, 0)."""
    streams = len(nres) * L * H
    best = (0, 0, 0)
    for c in SIZES:
        fit = None
        for sm in (16, 32, 64, 128):
            if sm > c:
                break
            t = -(-(workers * c // 2) // streams)
            tail = -(-t // sm) * sm
            parts = extra + sum(L * H * len(chunks(m, c, sm, tail)) for m in nres)
            if parts <= cap:
                fit = (c, sm, tail)
                break
        if fit is None:
            break
        best = fit
        big_items = sum(L * H * ((m - fit[2]) // c if m > fit[2] else 0) for m in nres)
        if big_items >= workers:
            break
    return best


def _cases():
    rng = np.random.default_rng(0x6B76 + 7)
    out = []
    for _ in range(300):
        n = int(rng.integers(1, 40))
        hi = int(rng.choice([20, 600, 9000]))
        nres = [int(x) for x in rng.integers(0, hi, size=n)]
        nres[0] = max(nres[0], 1)
        L, H = (int(rng.choice([2, 80])), int(rng.choice([1, 2, 8])))
        workers = int(rng.choice([152, 608, 1216, 1824]))
        full = sum(L * H * (-(-m // 16)) for m in nres)
        cap = int(rng.choice([full + 10, full // 2 + 1, full * 4, 10 ** 9]))
        extra = int(rng.choice([0, 0, 100]))
        out.append((nres, L, H, workers, cap, extra))
    return out


@pytest.mark.parametrize("case", _cases())
def test_plan_follows_rule_and_covers_every_stream(case):
    nres, L, H, workers, cap, extra = case
    big, small, tail = K.debug_chunk_plan(nres, L, H, workers, cap, extra)
    assert (big, small, tail) == rule(nres, L, H, workers, cap, extra)
    if big == 0:
        return
    assert big in SIZES and small >= MIN_SMALL and small <= big and small & (small - 1) == 0
    assert tail % small == 0
    # the short chunks of every stream cover at least its share of half a
    # large chunk per warp
    streams = len(nres) * L * H
    assert 2 * tail * streams >= workers * big - 1
    parts = extra
    for m in nres:
        c = chunks(m, big, small, tail)
        assert sum(c) == m                               # every block, once
        nbig = (m - tail) // big if m > tail else 0
        assert all(x == big for x in c[:nbig]) and all(x <= small for x in c[nbig:])
        assert m - nbig * big >= min(m, tail)            # the short region
        assert all(x <= 128 for x in c)                  # a decode item holds at most 128 blocks
        parts += L * H * len(c)
    assert parts <= cap


def test_bench_workloads():
    # 70B shape (80 layers x 8 KV heads): 1,216 bf16 decode warps, 1,824 FP8 / 2-bit
    assert K.debug_chunk_plan([513], 80, 8, 1216, 10 ** 9) == (128, 16, 128)
    assert K.debug_chunk_plan([8193], 80, 8, 1216, 10 ** 9) == (128, 16, 128)
    assert K.debug_chunk_plan([513], 80, 8, 1824, 10 ** 9) == (64, 16, 96)
    # a small call gets short chunks only
    big, small, tail = K.debug_chunk_plan([17], 2, 2, 1216, 10 ** 9)
    assert chunks(17, big, small, tail) == [16, 1]


def test_short_chunks_grow_when_partials_are_scarce():
    # 8K: 8 x 640 partials with 32-block short chunks (3 x 128 + 4 x 32 + 1),
    # 12 x 640 with 16 (3 x 128 + 8 x 16 + 1)
    assert K.debug_chunk_plan([513], 80, 8, 1216, 640 * 12) == (128, 16, 128)
    assert K.debug_chunk_plan([513], 80, 8, 1216, 640 * 11) == (128, 32, 128)
    assert K.debug_chunk_plan([513], 80, 8, 1216, 640 * 8) == (128, 32, 128)
    assert K.debug_chunk_plan([513], 80, 8, 1216, 100) == (0, 0, 0)


def test_invalid_arguments():
    with pytest.raises(K.KvsError):
        K.debug_chunk_plan([], 80, 8, 1216, 10 ** 9)
    with pytest.raises(K.KvsError):
        K.debug_chunk_plan([10], 80, 8, 0, 10 ** 9)
