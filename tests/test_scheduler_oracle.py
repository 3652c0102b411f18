"""Pins for the reference token-wise scheduler (oracle/scheduler.py), checked
against properties stated independently of its code:

* budget: a step never holds more than ``budget`` tokens, nor more than
  ``budget - reserved`` prefill tokens;
* conservation: every prompt token is scheduled exactly once, and a request
  generates only after its whole prompt was scheduled;
* generation first: a generation request left out of a step did not fit in
  what the generation requests before it left over;
* first come first served: at most one prefill request is partial in a step,
  it is the last prefill of the step, and no request is skipped for a later one;
* no idle budget: a step ends with prefill work pending only if the prefill
  room or the step is full;
* a worked example, and planted mistakes that these pins catch.
"""
from __future__ import annotations

import os
import types

import numpy as np
import pytest

from oracle import scheduler as so


def _drive(Sched, seed, steps=200, budget=64, reserved=16):
    rng = np.random.default_rng(seed)
    s = Sched(budget, reserved)
    prompt = {}
    arrival = []
    gen_len = {}
    scheduled = {}
    gen_started = {}
    gen_order = []                    # order in which requests started generating
    nxt = 0
    for t in range(steps):
        for _ in range(int(rng.integers(0, 3))):
            r = nxt
            nxt += 1
            prompt[r] = int(rng.integers(0, 120))
            gen_len[r] = int(rng.choice([1, 1, 1, 4, 7]))
            s.add(r, prompt[r], gen_len[r])
            arrival.append(r)
            scheduled[r] = 0
            if prompt[r] == 0:                # nothing to prefill: generates from now on
                gen_started[r] = True
                gen_order.append(r)
        pending_before = [r for r in arrival if scheduled[r] < prompt[r]]
        gens_before = [r for r in gen_order if r in arrival]
        batch = s.step()
        tot = sum(k for _, k, _ in batch)
        pre = [(r, k) for r, k, p in batch if p]
        gen = [(r, k) for r, k, p in batch if not p]
        assert tot <= budget and sum(k for _, k in pre) <= budget - reserved
        assert len({r for r, _, _ in batch}) == len(batch)
        # generation: whole, only for requests whose prompt was done before the step
        for r, k in gen:
            assert k == gen_len[r] and scheduled[r] == prompt[r] and gen_started.get(r, False)
        used = 0
        for r in gens_before:
            if (r, gen_len[r]) in gen:
                used += gen_len[r]
            else:
                assert used + gen_len[r] > budget, "a generation request was left out with room"
        # prefill: in arrival order, a prefix of the pending list, only the last partial
        assert [r for r, _ in pre] == pending_before[:len(pre)]
        for i, (r, k) in enumerate(pre):
            rem = prompt[r] - scheduled[r]
            assert 0 < k <= rem
            if k < rem:
                assert i == len(pre) - 1
        if len(pre) < len(pending_before) or (pre and pre[-1][1] < prompt[pre[-1][0]] - scheduled[pre[-1][0]]):
            assert sum(k for _, k in pre) == budget - reserved or tot == budget, "idle budget"
        for r, k in pre:
            scheduled[r] += k
        for r, _ in pre:
            if scheduled[r] == prompt[r] and not gen_started.get(r):
                gen_started[r] = True
                gen_order.append(r)
        # retire some generating requests
        for r in [r for r in arrival if gen_started.get(r) and rng.random() < 0.05]:
            s.remove(r)
            arrival.remove(r)
    return prompt, scheduled


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("budget,reserved", [(64, 16), (64, 0), (40, 40), (200, 8), (16, 4)])
def test_scheduler_properties(seed, budget, reserved):
    _drive(so.SchedulerOracle, seed, budget=budget, reserved=reserved)


def test_worked_example():
    s = so.SchedulerOracle(16, 4)
    for r in (0, 1, 2):
        s.add(r, 0, 1)                    # decode requests
    s.add(3, 0, 5)                        # verify of a 5-token draft
    s.add(4, 20, 1)                       # a prompt of 20 tokens
    s.add(5, 3, 1)
    # generation first (1+1+1+5 = 8 tokens), then prefill room min(12, 8) -> 8 of request 4
    assert s.step() == [(0, 1, False), (1, 1, False), (2, 1, False), (3, 5, False), (4, 8, True)]
    s.remove(3)
    # 3 decode tokens; prefill room 12, 13 left -> 12 of request 4 (its last 12)
    assert s.step() == [(0, 1, False), (1, 1, False), (2, 1, False), (4, 12, True)]
    # request 4 now generates; request 5 gets its 3 tokens
    assert s.step() == [(0, 1, False), (1, 1, False), (2, 1, False), (4, 1, False), (5, 3, True)]


MUTATIONS = {
    "prefill_uses_reserved": ("room = self.budget - self.reserved", "room = self.budget"),
    "shortest_first": ("        for e in self.prefill:\n            r, rem, k = e\n",
                       "        for e in sorted(self.prefill, key=lambda e: e[1]):\n            r, rem, k = e\n"),
    "gen_not_whole": ("            if k <= left:\n                batch.append((r, k, False))",
                      "            if left > 0:\n                k = min(k, left)\n                batch.append((r, k, False))"),
    "gen_starts_same_step": ("        for e in done:\n            self.prefill.remove(e)\n            self.gen.append([e[0], e[2]])\n        return batch",
                             "        for e in done:\n            self.prefill.remove(e)\n            self.gen.append([e[0], e[2]])\n            batch.append((e[0], e[2], False))\n        return batch"),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_is_caught(name):
    src_path = os.path.join(os.path.dirname(so.__file__), "scheduler.py")
    src = open(src_path).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, name
    mod = types.ModuleType("sched_mutant_" + name)
    exec(compile(src.replace(old, new), src_path, "exec"), mod.__dict__)
    caught = False
    try:
        for seed in range(4):
            for budget, reserved in [(64, 16), (40, 40), (200, 8), (16, 4)]:
                _drive(mod.SchedulerOracle, seed, budget=budget, reserved=reserved)
    except (AssertionError, KeyError, ValueError):
        caught = True
    assert caught, f"mutation {name} slipped past the pins"
