"""The MMA issuer-count rule of the swap-AB and tiled kernels, checked by
simulation on the CPU.

The kernels deal a CTA's K groups round robin to n issuer threads (group i to
issuer i mod n).  Group i reads operand stage i mod stages and TMEM buffer
i mod bufs, waiting on that stage's "full" barrier and, from the buffer's
second use on, on its "empty" barrier.  An mbarrier wait names the phase only
by its parity, so a thread that waits for phase k of a barrier while the
barrier is still in phase k - 2 passes at once: every barrier that is waited
for more than once must be waited for by one thread, which then waits for its
phases in order.  The swap-AB kernel's rule (stated next to its issuer loop):
the largest n <= 3 with (groups <= stages or n | stages) and (groups <= bufs
or n | bufs).  It is safe and slightly conservative: the exact condition on
the buffers is groups <= 2 bufs (an empty barrier is first waited for at the
buffer's second use), which would give 3 instead of 2 issuers to 64-column
tiles at K = 1024; that build measured the same times (the activation loads'
issue, not the MMA loop, bounds those shapes), so the kernel keeps the
simpler rule.
"""
import itertools

import pytest


def swapab_issuers(ng, stages, bufs, max_issuers=3):
    """The kernel's rule."""
    for n in range(max_issuers, 1, -1):
        if (ng <= stages or stages % n == 0) and (ng <= bufs or bufs % n == 0):
            return n
    return 1


def exact_issuers(ng, stages, bufs, max_issuers=3):
    for n in range(max_issuers, 1, -1):
        if (ng <= stages or stages % n == 0) and (ng <= 2 * bufs or bufs % n == 0):
            return n
    return 1


def tiled_issuers(bn, stages):
    return 2 if bn == 128 and stages % 2 == 0 and (512 // bn) % 2 == 0 else 1


def safe(ng, stages, bufs, n):
    """True when every barrier waited for more than once is waited for by one
    issuer only (the stage's full barrier: every use; the buffer's empty
    barrier: every use after the first)."""
    full_waiters, empty_waiters = {}, {}
    for i in range(ng):
        issuer = i % n
        full_waiters.setdefault(i % stages, []).append(issuer)
        if i >= bufs:
            empty_waiters.setdefault(i % bufs, []).append(issuer)
    for waiters in list(full_waiters.values()) + list(empty_waiters.values()):
        if len(waiters) > 1 and len(set(waiters)) > 1:
            return False
    return True


GRID = list(itertools.product(range(1, 65), range(1, 9), (2, 4, 8)))


@pytest.mark.parametrize("bufs", [2, 4, 8])
def test_swapab_rule_is_safe(bufs):
    for ng, stages, b in GRID:
        if b != bufs:
            continue
        n = swapab_issuers(ng, stages, bufs)
        assert safe(ng, stages, bufs, n), (ng, stages, bufs, n)
        assert n <= exact_issuers(ng, stages, bufs)


@pytest.mark.parametrize("bufs", [2, 4, 8])
def test_exact_rule_is_safe_and_maximal(bufs):
    for ng, stages, b in GRID:
        if b != bufs:
            continue
        n = exact_issuers(ng, stages, bufs)
        assert safe(ng, stages, bufs, n), (ng, stages, bufs, n)
        for bigger in range(n + 1, 4):
            assert not safe(ng, stages, bufs, bigger), (ng, stages, bufs, n, bigger)


def test_unsafe_counts_exist():
    """The hazard the rule avoids: 3 issuers on 2 buffers over 8 groups (the
    case that passed a parity wait two phases early), and 2 issuers on 5
    reused stages."""
    assert not safe(8, 6, 2, 3)
    assert not safe(8, 5, 8, 2)
    assert swapab_issuers(8, 6, 2) == 2
    assert swapab_issuers(8, 5, 8) == 1
    assert swapab_issuers(8, 8, 4) == 2          # 64-column tiles, K = 1024
    assert exact_issuers(8, 8, 4) == 3
    assert swapab_issuers(8, 8, 8) == 3
    assert swapab_issuers(2, 2, 8) == 3          # no reuse at all: any count


@pytest.mark.parametrize("bn,stages", [(256, 4), (256, 3), (192, 4), (128, 6), (128, 5), (128, 4)])
def test_tiled_rule_is_safe(bn, stages):
    """The tiled kernel walks many tiles: every stage and buffer is reused, so
    two issuers need even stage and buffer counts; the kernel uses them only at
    BN = 128, where the MMAs are short."""
    n = tiled_issuers(bn, stages)
    for ng in (1, 2, 7, 32, 257):
        assert safe(ng, stages, 512 // bn, n), (bn, stages, ng, n)
    assert n == (2 if (bn, stages) in ((128, 6), (128, 4)) else 1)
