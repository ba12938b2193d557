"""Failure path of the bounded device waits, on the GPU without a fault: the
test hook qmla_decode_timeout_test makes a tensor-core kernel withhold one
barrier arrival (16 heads: every worker; 128 heads: the first CTA of every
CTA pair, whose partner then waits in vain for its P rows), the waits give up
after their 1 s limit, every role of both CTAs unwinds and the host reads
QMLA_STATUS_TIMEOUT.  The same process then decodes normally and matches the
oracle: the context stayed usable.  A second check: a query value beyond
binary16's range sets QMLA_STATUS_BAD_QUERY in the tensor-core decodes."""
import numpy as np
import pytest
import torch

from bit_mla_kv_qmla_gb300 import (QMLA_STATUS_BAD_QUERY, QMLA_STATUS_TIMEOUT,
                                   qmla_decode_timeout_test)
from bit_mla_kv_qmla_gb300 import workloads as W
from bit_mla_kv_qmla_gb300.cache import Decoder, build_cache

from helpers import compare_rows, oracle_pool_for_seq
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,heads", [("C4R4", 16), ("C2R4", 128)])
def test_withheld_arrival_times_out_and_context_stays_usable(fmt, heads):
    w = W.Workload(f"timeout_{fmt}_h{heads}", fmt, 3, heads, 700, 0, "lognormal8", 0, 71)
    lens = [700, 130, 64]
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    dec = Decoder(cache, heads, max(lens))
    qc, qr = W.queries(w)
    qc, qr = qc.cuda(), qr.cuda()
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    qmla_decode_timeout_test(cache.fmt, cache.blocks, cache.block_table, cache.seq_lens,
                             max(lens), qc, qr, w.scale, dec.out, dec.lse, dec.workspace,
                             cache.status)
    torch.cuda.synchronize()
    assert cache.status.item() & QMLA_STATUS_TIMEOUT
    # the next decode on the same context is correct
    cache.status.zero_()
    out, lse = dec(qc, qr, w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    table = cache.block_table.cpu().numpy()
    hs = list(range(heads)) if heads <= 16 else [0, 1, 63, 64, 100, 127]
    for b, L in enumerate(lens):
        pool = oracle_pool_for_seq(w, b, L, table[b], cache.num_blocks, "cpu")
        ro, rl = oracle.decode(W.FORMATS[w.fmt], pool, table[b:b + 1], np.array([L]),
                               qc[b:b + 1, hs].cpu(), qr[b:b + 1, hs].cpu(), w.scale)
        compare_rows(out[b, hs], lse[b, hs], ro[0], rl[0], f"after timeout, seq {b}")


@pytest.mark.parametrize("heads", [16, 128])
def test_query_beyond_binary16_sets_status(heads):
    w = W.Workload(f"badq_h{heads}", "C4R4", 2, heads, 200, 0, "lognormal8", 0, 72)
    lens = [200, 64]
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    dec = Decoder(cache, heads, max(lens))
    qc, qr = W.queries(w)
    qc, qr = qc.cuda(), qr.cuda()
    dec(qc, qr, w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    qc[1, 3, 17] = 1.0e5  # beyond 65504: no binary16 operand holds it
    dec(qc, qr, w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() & QMLA_STATUS_BAD_QUERY
