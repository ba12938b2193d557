"""GPU parity of the benchmarked decode step in its own launch configuration:
append one token per sequence (qmla_append_advance) and decode the whole
cache (qmla_decode: the 16-head tensor-core kernel planning its own pieces,
then the merge), both captured once into a CUDA graph and replayed step after
step, at the full size of the default workload (32 sequences x 8192 tokens,
16 heads, C4R4).  Sampled (sequence, head) rows of the last step are checked
against the oracle, which appends the same tokens to its own cache."""
import numpy as np
import pytest
import torch

import oracle
from bit_mla_kv_qmla_gb300 import workloads as W
from bit_mla_kv_qmla_gb300.cache import Decoder, build_cache

from helpers import compare_rows, oracle_pool_for_seq, sample_heads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["C4R4", "C2R4"])
def test_graph_replayed_append_decode_step(fmt):
    w = W.with_format(W.WORKLOADS[1], fmt)
    steps = 3
    lens0 = W.seq_lens(w)
    cache = build_cache(w, "cuda", extra_tokens=steps, gen_device="cuda")
    dec = Decoder(cache, w.heads, max(lens0) + steps)
    qc, qr = W.queries(w, device="cuda")
    g = torch.Generator().manual_seed(99)
    new_lat = torch.randn(w.batch, 1, 512, generator=g).to(torch.bfloat16)
    new_rope = torch.randn(w.batch, 1, 64, generator=g).to(torch.bfloat16)
    d_lat, d_rope = new_lat.cuda(), new_rope.cuda()
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cache.append(d_lat, d_rope)
        dec(qc, qr, w.scale)
    torch.cuda.synchronize()
    # capture records without running: the cache is still at its start
    assert cache.seq_lens.cpu().tolist() == lens0
    for _ in range(steps):
        graph.replay()
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    assert cache.seq_lens.cpu().tolist() == [L + steps for L in lens0]
    out, lse = dec.out.clone(), dec.lse.clone()

    fcode = W.FORMATS[fmt]
    table = cache.block_table.cpu().numpy()
    for b in (0, 13, 31):
        pool = oracle_pool_for_seq(w, b, lens0[b], table[b], cache.num_blocks, "cuda")
        for k in range(steps):
            skipped = oracle.append(fcode, pool, table[b:b + 1], np.array([lens0[b] + k], np.int32),
                                    new_lat[b:b + 1], new_rope[b:b + 1])
            assert skipped == 0
        hs = sample_heads(w.heads, 6, 300 + b)
        ro, rl = oracle.decode(fcode, pool, table[b:b + 1], np.array([lens0[b] + steps]),
                               qc[b:b + 1, hs].cpu(), qr[b:b + 1, hs].cpu(), w.scale)
        compare_rows(out[b, hs], lse[b, hs], ro[0], rl[0], f"{w.name} seq {b}")
