"""Model check of the decode kernel's per-warp stage protocol (host only).

The decode kernel streams a consumer warp's K/V blocks through P shared-memory
stages: the producer fills stage j % P for tile j ("full" barrier phase), the
consumer waits for that phase by parity and releases the stage ("empty"
barrier), and the producer refills it after the release.  In split launches
tile 0 may first be filled speculatively: kept (verdict 1) or discarded
(verdict 2, stage 0's phases then run one ahead of its tiles, and the verdict
is published only once the discarded fill has landed).

An mbarrier parity wait passes when the barrier's current phase parity
differs from the one asked for, so a waiter two phases behind would pass at
once.  This model replays the protocol's index arithmetic under that rule
with random latencies and checks that no wait passes before the fill it
stands for has landed, that no stage is refilled before its release, and that
every schedule finishes.
"""
import random

import pytest


class _Bar:
    def __init__(self):
        self.done = 0                      # completed phases (current phase index)

    def passes(self, parity):
        return (self.done & 1) != parity


def _run(P, tiles, verdict, lat, seed, publish_after_landing=True):
    rnd = random.Random(seed)
    full = [_Bar() for _ in range(P)]
    empty = [_Bar() for _ in range(P)]
    fills = [[] for _ in range(P)]        # per stage: what each phase holds
    pending = []                          # (landing time, stage)

    def issue(st, what, now):
        fills[st].append(what)
        pending.append((now + rnd.uniform(*lat), st))

    def advance(now):
        for ev in sorted(pending):
            if ev[0] <= now:
                pending.remove(ev)
                full[ev[1]].done += 1

    shift0 = 1 if verdict == 2 else 0
    if verdict in (1, 2):
        issue(0, "spec" if verdict == 2 else 0, 0.0)
    t_verdict = rnd.uniform(0.5, 2.0)
    if verdict == 2 and publish_after_landing:
        while full[0].done < 1:
            t_verdict += 0.05
            advance(t_verdict)
    jj = 1 if verdict == 1 else 0
    t_prod = t_verdict
    t_cons = max(t_verdict, rnd.uniform(0.3, 2.5))
    j, released, steps = 0, [0] * P, 0
    while (j < tiles or jj < tiles) and steps < 100000:
        steps += 1
        advance(min(t_prod, t_cons))
        if t_prod <= t_cons:
            if jj < tiles:
                st = jj % P
                ready = jj < P or empty[st].passes(((jj // P) - 1) & 1)
                if ready and jj == 0 and shift0:
                    ready = full[st].passes(0)
                if ready:
                    if jj >= P:
                        assert released[st] > (jj - P) // P, ("refill before release", jj)
                    issue(st, jj, t_prod)
                    jj += 1
            t_prod += rnd.uniform(0.01, 0.2)
        else:
            if j < tiles:
                st = j % P
                ph = (j // P + (shift0 if st == 0 else 0)) & 1
                if full[st].passes(ph):
                    assert j in fills[st] and full[st].done > fills[st].index(j), (
                        "wait passed early", j, full[st].done, fills[st])
                    t_cons += rnd.uniform(0.2, 1.0)
                    advance(t_cons)
                    empty[st].done += 1
                    released[st] += 1
                    j += 1
                    continue
            t_cons += rnd.uniform(0.01, 0.2)
    assert j == tiles and jj == tiles, ("stalled", j, jj, tiles)


def _cases(n):
    rnd = random.Random(1234)
    for seed in range(n):
        # stages per warp: 1-3 in the CUDA-core build, 3 (bf16) and 6 (E4M3 or
        # head_dim 64) in the tensor-core build
        yield (rnd.choice([1, 2, 3, 6]), rnd.randint(1, 14), rnd.choice([0, 1, 2]),
               rnd.choice([(0.05, 0.3), (0.5, 3.0), (0.01, 5.0)]), seed)


def test_stage_protocol_random_schedules():
    for P, tiles, verdict, lat, seed in _cases(4000):
        _run(P, tiles, verdict, lat, seed)


def test_model_catches_early_verdict():
    # publishing "discarded" before that fill lands lets tile 0's parity wait
    # pass against the still-pending speculative phase
    with pytest.raises(AssertionError, match="wait passed early"):
        for P, tiles, _, lat, seed in _cases(4000):
            _run(P, tiles, 2, (1.0, 5.0), seed, publish_after_landing=False)
