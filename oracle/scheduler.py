"""Plain-Python reference of the continuous-batching scheduler (test infrastructure only).

What the pages give:

* Continuous (iteration-level) batching schedules per iteration, not per request: after
  every generated token, finished requests leave the batch at once and release their
  KV cache, and waiting requests join at once, so the batch changes at every step
  ("Continuous batching and PagedAttention", section 2; "Inference optimization",
  continuous batching: the batch is re-evaluated at every decode step).
* Static batching waits for a batch, runs it until every member has finished, and only
  then takes new requests (same sections) -- the comparison policy.
* A long prefill inserted into a decode batch stalls every decoding request; chunked
  prefill cuts it into pieces spread over several iterations, and a per-step prefill
  token budget bounds it ("Continuous batching and PagedAttention", section 2, the
  three remedies).
* The measure of the policy is the batch-slot fill rate per step (GPU utilisation) on
  requests with Pareto-distributed output lengths; continuous batching should keep it
  above 80% ("Inference optimization", exercise 2).  KV memory waste with paging is
  near zero (about 4%; "Inference optimization", PagedAttention).

Readings where the pages are silent (fixed so that the C++ scheduler can be compared
with this one decision by decision):

* A request has P prompt tokens and wants O >= 1 output tokens.  Its KV holds the
  prompt and every output token but the last: the step that completes the prompt
  samples output 1; each later step writes the K/V of the previous output and samples
  the next.  The request finishes after output O, at the start of the next step.
* Step order: (1) retire finished requests (free their blocks); (2) one decode token
  for every running request whose prompt is complete, in admission order; (3) the next
  prefill chunk of running requests whose prompt is incomplete, in admission order,
  while the step's token budget lasts; (4) admit waiting requests first come first
  served while fewer than max_num_seqs run and budget is left.  Decode tokens count
  against the budget (the budget must be at least max_num_seqs).  Static batching
  admits only in steps that start with no running request.
* When the pool cannot give a block: first evict a cached prefix block no request
  holds (least recently used); else preempt the most recently admitted running
  request (free its blocks, forget its progress, put it back at the head of the queue;
  recompute on readmission); a request that is itself the most recently admitted is
  preempted rather than served.  A prefill chunk whose would-be victim already has
  work in this step's plan waits for a later step.  An admission that does not fit
  after eviction stops admission for this step (no preemption for admissions).  A step
  in which nothing finishes and nothing can be scheduled while requests remain is an
  error (the pool is too small for the request at the head).
* Admission looks up the prefix cache (if any): the matched blocks become the start of
  the request's table and its prefill starts after them.  A prompt's full blocks are
  inserted into the cache in the step that completes the prompt.
* Per step, the plan lists decode entries then prefill entries, each with its sequence,
  number of new tokens, context length after the step, and the slots of the new
  tokens in order.
* Statistics per step: running requests (after admission) / max_num_seqs, also
  summed separately over the steps that end with requests still waiting (the
  saturated phase, where a policy can fill every slot), and, over running requests,
  token slots held in their blocks and token slots unused.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

from .block_manager import BlockManagerError, OutOfBlocks


@dataclass
class Request:
    rid: int
    prompt: list
    output_len: int
    computed: int = 0      # tokens whose K/V are in the cache
    generated: int = 0     # output tokens sampled


@dataclass
class Plan:
    seqs: list = field(default_factory=list)        # request ids, decode first
    query_lens: list = field(default_factory=list)
    context_lens: list = field(default_factory=list)
    slots: list = field(default_factory=list)
    cow_pairs: list = field(default_factory=list)
    num_decode: int = 0
    finished: int = 0
    preempted: int = 0


class Scheduler:
    def __init__(self, manager, max_num_seqs: int, max_batched_tokens: int,
                 static: bool = False, cache=None):
        if max_batched_tokens < max_num_seqs or max_num_seqs <= 0:
            raise ValueError("need max_batched_tokens >= max_num_seqs > 0")
        self.bm = manager
        self.cache = cache
        self.max_num_seqs = max_num_seqs
        self.budget_per_step = max_batched_tokens
        self.static = static
        self.waiting: deque[Request] = deque()
        self.running: list[Request] = []
        self.steps = 0
        self.fill_sum = 0.0
        self.busy_steps = 0
        self.busy_fill_sum = 0.0
        self.slots_held = 0
        self.slots_unused = 0
        self.finished = 0
        self.preemptions = 0
        self.decode_tokens = 0
        self.prefill_tokens = 0

    def add_request(self, rid: int, prompt, output_len: int) -> None:
        if output_len < 1 or len(prompt) < 1:
            raise ValueError("a request needs a prompt and at least one output token")
        self.waiting.append(Request(rid, list(prompt), output_len))

    def done(self) -> bool:
        return not self.waiting and not self.running

    # -- helpers --------------------------------------------------------------------
    def _preempt(self, victim: Request, plan: Plan) -> None:
        self.bm.free_seq(victim.rid)
        victim.computed = victim.generated = 0
        self.running.remove(victim)
        self.waiting.appendleft(victim)
        plan.preempted += 1
        self.preemptions += 1

    def _make_room(self, r: Request, plan: Plan, scheduled) -> str:
        """Free one block for request r: evict a cached block, else preempt the most
        recently admitted request.  Returns "ok", "self" (r itself was preempted) or
        "stuck" (that request already has work in this step's plan; r waits)."""
        if self.cache is not None and self.cache.evict_free_one():
            return "ok"
        victim = self.running[-1]
        if any(victim is e for e in scheduled):
            return "stuck"
        self._preempt(victim, plan)
        return "self" if victim is r else "ok"

    # -- one iteration ----------------------------------------------------------------
    def step(self) -> Plan:
        plan = Plan()
        for r in list(self.running):                              # (1) retire
            if r.generated == r.output_len:
                self.bm.free_seq(r.rid)
                self.running.remove(r)
                plan.finished += 1
                self.finished += 1
        budget = self.budget_per_step
        was_empty = not self.running
        decode, prefill = [], []
        for r in list(self.running):                              # (2) decode
            if r not in self.running or r.computed < len(r.prompt):
                continue
            while True:
                try:
                    slot, cow = self.bm.append_slot(r.rid)
                    break
                except OutOfBlocks:
                    if self._make_room(r, plan, [e[0] for e in decode]) != "ok":
                        slot = None
                        break
            if slot is None:
                continue
            r.computed += 1
            decode.append((r, [slot]))
            if cow is not None:
                plan.cow_pairs.append(cow)
            budget -= 1
        for r in list(self.running):                              # (3) prefill chunks
            if r not in self.running or r.computed >= len(r.prompt) or budget <= 0:
                continue
            chunk = min(len(r.prompt) - r.computed, budget)
            while True:
                try:
                    slots, pairs = self.bm.append_tokens(r.rid, chunk)
                    break
                except OutOfBlocks:
                    if self._make_room(r, plan, [e[0] for e in decode + prefill]) != "ok":
                        slots = None
                        break
            if slots is None:
                continue
            r.computed += chunk
            prefill.append((r, slots))
            plan.cow_pairs += pairs
            budget -= chunk
        admit = not self.static or was_empty
        while admit and self.waiting and len(self.running) < self.max_num_seqs and budget > 0:
            r = self.waiting[0]                                   # (4) admission
            matched = self.cache.lookup(r.prompt) if self.cache is not None else []
            start = len(matched) * self.bm.block_size
            chunk = min(len(r.prompt) - start, budget)
            bs = self.bm.block_size
            need = (start + chunk + bs - 1) // bs - len(matched)
            self.bm.add_seq_shared(r.rid, matched)
            while self.bm.num_free() < need and self.cache is not None \
                    and self.cache.evict_free_one():
                pass
            if self.bm.num_free() < need:
                self.bm.free_seq(r.rid)
                break
            if self.cache is not None:
                self.cache.use(r.prompt, len(matched))
            slots, pairs = self.bm.append_tokens(r.rid, chunk)
            r.computed = start + chunk
            self.waiting.popleft()
            self.running.append(r)
            prefill.append((r, slots))
            plan.cow_pairs += pairs
            budget -= chunk
        for r, slots in decode:                                   # sample
            r.generated += 1
        for r, slots in prefill:
            if r.computed == len(r.prompt):
                r.generated = 1
                if self.cache is not None:
                    self.cache.insert(r.prompt, self.bm.block_table(r.rid))
        for r, slots in decode + prefill:
            plan.seqs.append(r.rid)
            plan.query_lens.append(len(slots))
            plan.context_lens.append(r.computed)
            plan.slots += list(slots)
        plan.num_decode = len(decode)
        if not plan.seqs and not self.done() and plan.finished == 0:
            raise BlockManagerError("no request can make progress: the pool is too small")
        self.steps += 1
        self.fill_sum += len(self.running) / self.max_num_seqs
        if self.waiting:
            self.busy_steps += 1
            self.busy_fill_sum += len(self.running) / self.max_num_seqs
        for r in self.running:
            held = len(self.bm.tables[r.rid]) * self.bm.block_size
            self.slots_held += held
            self.slots_unused += held - self.bm.num_tokens[r.rid]
        self.decode_tokens += len(decode)
        self.prefill_tokens += sum(len(s) for _, s in prefill)
        return plan
