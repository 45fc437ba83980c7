"""Host model of the one-launch prefill's scheduling: the quantising CTA pairs
hold their quantisation at most `lead` units ahead of their own GEMM, and
every pair's GEMM needs the jobs (K groups) of its token block from all the
pairs that share the block.  The rule in the kernel takes
lead = max(1, ceil((y_tiles - 1) / pairs)); this model checks, on the unit
order and the job split the kernel uses, that with that lead the pairs can
never wait on each other in a cycle (no reliance on the takeover path), for
every pair count from 1 to 80 and several tile shapes -- and that a smaller
lead does deadlock for a single pair, so the check has teeth.

Model: units u = 0 .. G * x_tiles * y_tiles - 1 with the weight tile fastest
(yt = u % y_tiles, xt = (u // y_tiles) % x_tiles, g = u // (y_tiles *
x_tiles)); pair p walks units p, p + P, ... (ordinal n = its n-th unit); the
jobs of unit (g, xt, yt) are the K groups kg = (yt + xt) % y_tiles + j *
y_tiles < KG, which the pair quantises in order; a job of ordinal n may
start once the pair has finished n - lead units; a pair finishes its current
unit once every K group of that unit's token block (g, xt) is quantised."""

import math

import pytest


def simulate(P, x_tiles, y_tiles, G, KG, lead):
    """True when every pair finishes all its units; False on a deadlock."""
    units = G * x_tiles * y_tiles

    def decode(u):
        return (u // (y_tiles * x_tiles), (u // y_tiles) % x_tiles, u % y_tiles)

    # per pair: its units, its job list [(ordinal, block, kg)], cursors
    pairs = []
    for p in range(P):
        mine = list(range(p, units, P))
        jobs = []
        for n, u in enumerate(mine):
            g, xt, yt = decode(u)
            kg = (yt + xt) % y_tiles
            while kg < KG:
                jobs.append((n, (g, xt), kg))
                kg += y_tiles
        pairs.append({"units": mine, "jobs": jobs, "next_job": 0, "done_units": 0})
    quantised = set()
    remaining = units
    while remaining:
        progress = False
        for pr in pairs:
            # quantise every allowed job in order
            while pr["next_job"] < len(pr["jobs"]):
                n, blk, kg = pr["jobs"][pr["next_job"]]
                if n > pr["done_units"] + lead:
                    break
                quantised.add((blk, kg))
                pr["next_job"] += 1
                progress = True
            # finish the current unit once its block's K groups are all there
            if pr["done_units"] < len(pr["units"]):
                g, xt, _ = decode(pr["units"][pr["done_units"]])
                if all(((g, xt), kg) in quantised for kg in range(KG)):
                    pr["done_units"] += 1
                    remaining -= 1
                    progress = True
        if not progress:
            return False
    return True


def kernel_lead(y_tiles, pairs):
    return max(1, math.ceil((y_tiles - 1) / pairs))


@pytest.mark.parametrize("x_tiles,y_tiles,G,KG", [
    (32, 4, 8, 32),   # the 8K chunk: 1024 units, N = 1024, K = 4096
    (5, 4, 8, 32),    # 1100 tokens (ragged), as in the pair-count tests
    (2, 5, 3, 5),     # five weight tiles, K = 640
    (4, 1, 2, 8),     # one weight tile: each pair quantises every K group
    (3, 8, 2, 18),    # many weight tiles, unaligned K (18 groups)
])
def test_kernel_lead_never_deadlocks(x_tiles, y_tiles, G, KG):
    for P in range(1, 81):
        assert simulate(P, x_tiles, y_tiles, G, KG, kernel_lead(y_tiles, P)), (P, x_tiles, y_tiles)


def test_smaller_lead_deadlocks_for_one_pair():
    # One pair holds all four units of a block at ordinals n .. n + 3: with a
    # lead below 3 the first unit's last K groups are never allowed.
    assert kernel_lead(4, 1) == 3
    assert simulate(1, 2, 4, 1, 32, 3)
    assert not simulate(1, 2, 4, 1, 32, 2)
    assert not simulate(1, 2, 4, 1, 32, 1)
