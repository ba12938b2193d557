"""Failure path of the bounded device waits, on the GPU without a fault: the
test hook qmla_decode_timeout_test makes the 16-head tensor-core kernel
withhold one barrier arrival, its waits give up after their 1 s limit, every
role unwinds and the host reads QMLA_STATUS_TIMEOUT.  The same process then
decodes normally and matches the oracle: the context stayed usable."""
import numpy as np
import pytest
import torch

from bit_mla_kv_qmla_gb300 import (QMLA_STATUS_TIMEOUT, qmla_decode_timeout_test)
from bit_mla_kv_qmla_gb300 import workloads as W
from bit_mla_kv_qmla_gb300.cache import Decoder, build_cache

from helpers import compare_rows, oracle_pool_for_seq
import oracle

pytestmark = pytest.mark.gpu


def test_withheld_arrival_times_out_and_context_stays_usable():
    w = W.Workload("timeout_c4r4_h16", "C4R4", 3, 16, 700, 0, "lognormal8", 0, 71)
    lens = [700, 130, 64]
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    dec = Decoder(cache, 16, max(lens))
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
    for b, L in enumerate(lens):
        pool = oracle_pool_for_seq(w, b, L, table[b], cache.num_blocks, "cpu")
        ro, rl = oracle.decode(W.FORMATS[w.fmt], pool, table[b:b + 1], np.array([L]),
                               qc[b:b + 1].cpu(), qr[b:b + 1].cpu(), w.scale)
        compare_rows(out[b], lse[b], ro[0], rl[0], f"after timeout, seq {b}")
