"""Cache capacity under a fixed memory budget: a block pool and an admission /
preemption scheduler, simulated over synthetic request lengths.

The pages attribute the low-bit cache's whole-job gain to capacity, not to
attention speed: BF16 caches grow linearly with context, and under load the
serving system runs out of cache memory, evicts sequences and later
recomputes them, while C4R4 served the same long-context workload with no
preemption ("QuantMLA's INT4/INT2 KV-cache quantization reports 5x
long-context throughput over BF16", sections "Where BF16 caches fall over"
and "What the low-bit cache changes").  There is no serving engine here;
this module replays that mechanism with the library's block sizes:

* ``BlockPool`` hands out the ids of a pool of ``budget // block_bytes``
  64-token blocks (the pool ``PagedCache`` addresses) and takes them back;
* ``simulate`` runs continuous batching, one decode step at a time: every
  running sequence appends one token (a new block every 64 tokens); when the
  pool has no block for a sequence that needs one, the most recently
  admitted sequence is preempted (all its blocks released, its tokens to be
  recomputed on readmission); waiting sequences are admitted first come
  first served while their whole current context plus one token fits.

Reported per format: preemptions, tokens recomputed on readmission, decode
steps to finish the job, the mean number of running sequences, and the
tokens attended over the whole job (the sum over steps of every running
sequence's context: the decode work, which divided by a measured decode rate
in tokens/s gives the job's decode time).
"""
from __future__ import annotations

import dataclasses
from collections import deque
from typing import Dict, List, Optional, Sequence

import torch

BLOCK = 64


class BlockPool:
    """Ids 0 .. num_blocks-1 of a pool of cache blocks, with a free list."""

    def __init__(self, num_blocks: int):
        if num_blocks < 0:
            raise ValueError("num_blocks < 0")
        self.num_blocks = int(num_blocks)
        self._free = list(range(self.num_blocks - 1, -1, -1))  # pop() gives the lowest id
        self._used = bytearray(self.num_blocks)

    @property
    def available(self) -> int:
        return len(self._free)

    def alloc(self, n: int = 1) -> Optional[List[int]]:
        """n block ids, or None (and nothing taken) if fewer are free."""
        if n > len(self._free):
            return None
        ids = [self._free.pop() for _ in range(n)]
        for i in ids:
            self._used[i] = 1
        return ids

    def release(self, ids: Sequence[int]) -> None:
        for i in ids:
            if not (0 <= i < self.num_blocks) or not self._used[i]:
                raise ValueError(f"block {i} is not allocated")
            self._used[i] = 0
            self._free.append(i)


@dataclasses.dataclass
class Request:
    rid: int
    prompt: int   # tokens in the cache when the sequence is admitted
    output: int   # tokens it generates (one per decode step)


def synthetic_requests(n: int, prompt_lo: int, prompt_hi: int, output: int,
                       seed: int = 0) -> List[Request]:
    """n requests with prompt lengths uniform in [prompt_lo, prompt_hi]
    (seeded) and a fixed number of generated tokens."""
    g = torch.Generator()
    g.manual_seed(int(seed) * 1000003 + 71)
    lens = torch.randint(prompt_lo, prompt_hi + 1, (n,), generator=g).tolist()
    return [Request(i, int(p), int(output)) for i, p in enumerate(lens)]


def blocks_for(tokens: int) -> int:
    return (tokens + BLOCK - 1) // BLOCK


def simulate(block_bytes: int, budget_bytes: int, requests: Sequence[Request],
             max_running: int) -> Dict[str, float]:
    """Run the job to completion; see the module docstring for the policy.

    A request whose prompt plus output can never fit in the pool is
    rejected up front (counted, not run)."""
    pool = BlockPool(budget_bytes // block_bytes)
    cap_tokens = pool.num_blocks * BLOCK
    waiting = deque()
    rejected = 0
    for r in requests:
        if r.prompt + r.output > cap_tokens:
            rejected += 1
        else:
            waiting.append([r, 0])  # (request, tokens generated so far)
    running: List[list] = []        # [request, generated, block ids], admission order
    steps = preemptions = recomputed = generated_total = attended = 0
    running_sum = 0
    ever_admitted = set()

    def admit() -> None:
        nonlocal recomputed
        while waiting and len(running) < max_running:
            r, gen = waiting[0]
            ctx = r.prompt + gen
            ids = pool.alloc(blocks_for(ctx + 1))
            if ids is None:
                return
            waiting.popleft()
            if r.rid in ever_admitted:
                recomputed += ctx  # the evicted context is rebuilt
            ever_admitted.add(r.rid)
            running.append([r, gen, ids])

    admit()
    while running:
        # every running sequence needs room for the token of this step
        i = 0
        while i < len(running):
            ent = running[i]
            r, gen, ids = ent
            need = blocks_for(r.prompt + gen + 1) - len(ids)
            evicted_self = False
            while need > 0:
                got = pool.alloc(1)
                if got is not None:
                    ids.extend(got)
                    need -= 1
                    continue
                victim = running.pop()  # the most recently admitted
                pool.release(victim[2])
                preemptions += 1
                waiting.appendleft([victim[0], victim[1]])
                if victim is ent:       # it was the last one admitted itself
                    evicted_self = True
                    break
            if not evicted_self:
                i += 1
        steps += 1
        running_sum += len(running)
        still = []
        for ent in running:
            r = ent[0]
            attended += r.prompt + ent[1] + 1  # the context the new token attends to
            ent[1] += 1
            generated_total += 1
            if ent[1] >= r.output:
                pool.release(ent[2])
            else:
                still.append(ent)
        running[:] = still
        admit()
    if pool.available != pool.num_blocks:
        raise AssertionError("blocks leaked")
    return {"steps": steps, "preemptions": preemptions, "recomputed_tokens": recomputed,
            "generated_tokens": generated_total, "attended_tokens": attended,
            "rejected": rejected,
            "mean_running": (running_sum / steps) if steps else 0.0,
            "pool_blocks": pool.num_blocks}
