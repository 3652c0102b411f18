"""The library's token-wise scheduler (pps_sched_*, C++) against the reference
scheduler in oracle/, step by step on seeded traces (CPU only): identical
batches, including generation requests that do not fit, chunked prefills,
removals and draft-length changes."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import scheduler as so


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("budget,reserved", [(64, 16), (16, 4), (40, 40), (8192, 256)])
def test_scheduler_matches_reference(pps, seed, budget, reserved):
    rng = np.random.default_rng(seed)
    o, c = so.SchedulerOracle(budget, reserved), pps.Scheduler(budget, reserved)
    live, nxt = [], 0
    scale = max(1, budget // 32)
    for step in range(300):
        for _ in range(int(rng.integers(0, 4))):
            p = int(rng.integers(0, 120 * scale))
            g = int(rng.choice([1, 1, 1, 4, 7]))
            o.add(nxt, p, g)
            c.add(nxt, p, g)
            live.append(nxt)
            nxt += 1
        if live and rng.random() < 0.1:
            r = live[int(rng.integers(len(live)))]
            g = int(rng.integers(1, 9))
            o.set_gen_tokens(r, g)
            c.set_gen_tokens(r, g)
        want = o.step()
        r, t, p = c.step()
        assert [(int(a), int(b), bool(x)) for a, b, x in zip(r, t, p)] == want, step
        for rid in [x for x in live if rng.random() < 0.04]:
            o.remove(rid)
            c.remove(rid)
            live.remove(rid)


def test_scheduler_rejects_bad_use(pps):
    with pytest.raises(pps.PPSError):
        pps.Scheduler(0)
    with pytest.raises(pps.PPSError):
        pps.Scheduler(8, 9)
    s = pps.Scheduler(8, 2)
    s.add(1, 5, 1)
    with pytest.raises(pps.PPSError):
        s.add(1, 3, 1)                       # already queued
    with pytest.raises(pps.PPSError):
        s.remove(2)
    with pytest.raises(pps.PPSError):
        s.add(3, 1, 0)                       # no generation tokens


def test_scheduler_grows_its_output_buffer(pps):
    s = pps.Scheduler(100000, 0)
    for r in range(5000):
        s.add(r, 0, 1)
    req, tok, pre = s.step()
    assert len(req) == 5000 and tok.sum() == 5000 and not pre.any()
