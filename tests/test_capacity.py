"""Host logic of the capacity simulation (block pool and admission /
preemption scheduler): hand-traced cases and invariants."""
import random

import pytest

from bit_mla_kv_qmla_gb300 import capacity as C


def test_block_pool_conserves_blocks():
    pool = C.BlockPool(5)
    a = pool.alloc(3)
    assert sorted(a) == [0, 1, 2] and pool.available == 2
    assert pool.alloc(3) is None and pool.available == 2  # nothing taken
    b = pool.alloc(2)
    assert pool.available == 0 and not set(a) & set(b)
    pool.release(a)
    with pytest.raises(ValueError):
        pool.release([a[0]])  # double free
    with pytest.raises(ValueError):
        pool.release([7])     # outside the pool
    pool.release(b)
    assert pool.available == 5


def test_no_pressure_runs_in_waves():
    # 10 equal requests, 4 at a time, 5 tokens each: waves of 4, 4, 2
    reqs = [C.Request(i, 100, 5) for i in range(10)]
    r = C.simulate(1000, 10 ** 9, reqs, 4)
    assert (r["steps"], r["preemptions"], r["recomputed_tokens"]) == (15, 0, 0)
    assert r["generated_tokens"] == 50 and abs(r["mean_running"] - 50 / 15) < 1e-12
    # every token attends to its prompt plus the tokens before it and itself
    assert r["attended_tokens"] == 10 * sum(100 + g + 1 for g in range(5))


def test_preempts_the_most_recent_sequence():
    """Pool of 4 blocks, A and B with 64-token prompts hold two each.  At
    step 65 A needs a third block: B (admitted last) is evicted with 64
    tokens generated; A finishes at step 70 and frees 3 blocks; B comes back
    with its 128-token context rebuilt and generates its last 6 tokens."""
    reqs = [C.Request(0, 64, 70), C.Request(1, 64, 70)]
    r = C.simulate(1000, 4 * 1000, reqs, 2)
    assert (r["steps"], r["preemptions"], r["recomputed_tokens"]) == (76, 1, 128)
    assert r["generated_tokens"] == 140 and abs(r["mean_running"] - 140 / 76) < 1e-12


def test_sequence_that_was_admitted_last_evicts_itself():
    """A (64-token prompt) and B (100) hold two blocks each; B needs a third
    first (step 29) and, being the most recent, is evicted itself with 28
    tokens generated; A runs alone to step 150; B returns with 128 tokens
    rebuilt and finishes its last 22 tokens at step 172."""
    reqs = [C.Request(0, 64, 150), C.Request(1, 100, 50)]
    r = C.simulate(1000, 4 * 1000, reqs, 2)
    assert (r["steps"], r["preemptions"], r["recomputed_tokens"]) == (172, 1, 128)
    assert r["generated_tokens"] == 200 and abs(r["mean_running"] - 200 / 172) < 1e-12


def test_request_larger_than_the_pool_is_rejected():
    reqs = [C.Request(0, 200, 57), C.Request(1, 10, 5)]  # 257 > 4 blocks of 64
    r = C.simulate(1000, 4 * 1000, reqs, 2)
    assert r["rejected"] == 1 and r["generated_tokens"] == 5


def test_random_jobs_finish_and_release_every_block():
    rnd = random.Random(3)
    for _ in range(40):
        n = rnd.randint(1, 12)
        reqs = [C.Request(i, rnd.randint(0, 300), rnd.randint(1, 120)) for i in range(n)]
        blocks = rnd.randint(1, 12)
        r = C.simulate(100, blocks * 100, reqs, rnd.randint(1, 5))
        ok = [q for q in reqs if q.prompt + q.output <= blocks * 64]
        assert r["rejected"] == n - len(ok)
        assert r["generated_tokens"] == sum(q.output for q in ok)
        assert r["steps"] >= max([q.output for q in ok], default=0)


def test_compressed_cache_fits_what_bf16_cannot():
    """Same budget and requests: the low-bit block holds 3.56x the tokens."""
    reqs = C.synthetic_requests(64, 8192, 32768, 256, seed=2)
    budget = 10 ** 9  # BF16: 0.87 M tokens; C4R4: 3.1 M; the 64 prompts need ~1.3 M
    bf16 = C.simulate(73728, budget, reqs, 64)
    c4r4 = C.simulate(20736, budget, reqs, 64)
    assert c4r4["preemptions"] == 0 and bf16["preemptions"] > 0
    assert c4r4["steps"] < bf16["steps"] and c4r4["mean_running"] > bf16["mean_running"]
