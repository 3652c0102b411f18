"""Reference token-wise budget scheduler (test infrastructure only).

Forms each step's mixed batch from the prefill, decode and verify queues.
Sources: XY-Serve review, "Tackling the Dynamicity in a Production LLM
Serving System ..." (pith.science/paper/ABCKJ6RF), "Core claim" (a token-wise
scheduler selects a budgeted chunk of tokens from mixed prefill, decode and
verify queues; SplitFuse-style chunking) and Fig. 6 (prefills are split into
smaller parts so each scheduled chunk stays within the budget; some slots are
reserved for decode and speculative tokens so prefill does not disturb the
time between tokens).

Rules (the pages give no more; this is the plain reading, followed by the
library too):
* A step has ``budget`` token slots, ``reserved`` of which prefill may never
  use.
* Generation requests (decode: 1 token per step; verify: its draft length)
  are taken first, in the order they became generation requests, each whole;
  one that does not fit in what is left waits for a later step (the ones
  after it may still fit).
* Then prefill requests, first come first served: each gets
  min(remaining prompt tokens, prefill room left) where the prefill room is
  budget - reserved minus the prefill tokens already taken, and never more
  than what the step has left; once either runs out, later ones wait.
* A request whose prompt is done becomes a generation request at the end of
  the step (its first generation step is the next one).
"""
from __future__ import annotations


class SchedulerOracle:
    def __init__(self, budget, reserved):
        if budget <= 0 or reserved < 0 or reserved > budget:
            raise ValueError("bad budget")
        self.budget, self.reserved = int(budget), int(reserved)
        self.prefill = []          # [request, remaining prompt tokens, tokens per generation step]
        self.gen = []              # [request, tokens per generation step]

    def add(self, request, prompt_tokens, gen_tokens=1):
        """Queue a request with ``prompt_tokens`` still to compute, then
        ``gen_tokens`` tokens per generation step (1 = decode, k = verify of a
        k-token draft)."""
        if prompt_tokens < 0 or gen_tokens <= 0:
            raise ValueError("bad request")
        if prompt_tokens == 0:
            self.gen.append([request, gen_tokens])
        else:
            self.prefill.append([request, prompt_tokens, gen_tokens])

    def remove(self, request):
        self.prefill = [e for e in self.prefill if e[0] != request]
        self.gen = [e for e in self.gen if e[0] != request]

    def set_gen_tokens(self, request, gen_tokens):
        for e in self.gen:
            if e[0] == request:
                e[1] = gen_tokens
        for e in self.prefill:
            if e[0] == request:
                e[2] = gen_tokens

    def step(self):
        """The next batch: list of (request, tokens this step, is_prefill)."""
        left = self.budget
        batch = []
        for r, k in self.gen:
            if k <= left:
                batch.append((r, k, False))
                left -= k
        room = self.budget - self.reserved
        done = []
        for e in self.prefill:
            r, rem, k = e
            take = min(rem, room, left)
            if take <= 0:
                break
            batch.append((r, take, True))
            left -= take
            room -= take
            e[1] -= take
            if e[1] == 0:
                done.append(e)
        for e in done:
            self.prefill.remove(e)
            self.gen.append([e[0], e[2]])
        return batch
