"""qmla_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a serving loop that forbids cudaMalloc once running,
a plugin that may only enqueue work on the stream it is given).  It takes no
workspace; its split partials live in the library's fixed per-device scratch
array.  Checked here through the C ABI against qmla_decode on the same cache,
on two calls in a row with different shapes, so the second call runs on the
scratch contents the first one left behind, and against the oracle; a third
case has so many sequences that the usual split's partials do not fit the
scratch and the call spreads the context over fewer workers.

This file sorts last so that a run stopping at the first failure has already
run every other test."""
import numpy as np
import pytest
import torch

import oracle
import bit_mla_kv_qmla_gb300 as q
from bit_mla_kv_qmla_gb300 import workloads as W
from bit_mla_kv_qmla_gb300.cache import Decoder, build_cache

from helpers import LSE_TOL, O_TOL, compare_rows, oracle_pool_for_seq

pytestmark = pytest.mark.gpu


def _case(fmt, heads, lens, seed):
    w = W.Workload(f"noalloc_{fmt}_{heads}", fmt, len(lens), heads, max(lens), 0,
                   "lognormal8", 0, seed)
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    qc, qr = W.queries(w)
    return w, cache, qc.cuda(), qr.cuda()


def _check_close(o1, l1, o2, l2):
    both_inf = torch.isneginf(l1) & torch.isneginf(l2)
    assert torch.equal(torch.isneginf(l1), torch.isneginf(l2))
    assert (l1[~both_inf] - l2[~both_inf]).abs().max().item() <= LSE_TOL
    ref = o2.float()
    denom = ref.abs().amax(dim=-1).clamp_min(1e-30)
    err = ((o1.float() - ref).abs().amax(dim=-1) / denom)
    err = torch.where(ref.abs().amax(dim=-1) == 0, o1.float().abs().amax(dim=-1), err)
    assert err.max().item() <= O_TOL


def _check_oracle(w, cache, lens, qc, qr, out, lse, seqs):
    table = cache.block_table.cpu().numpy()
    for b in seqs:
        pool = oracle_pool_for_seq(w, b, lens[b], table[b], cache.num_blocks, "cpu")
        ro, rl = oracle.decode(W.FORMATS[w.fmt], pool, table[b:b + 1], np.array([lens[b]]),
                               qc[b:b + 1].cpu(), qr[b:b + 1].cpu(), w.scale)
        compare_rows(out[b:b + 1], lse[b:b + 1], ro, rl, f"noalloc {w.name} seq {b}")


def _scratch_need(batch, heads, slots):
    # the workspace layout of the decode: merge table, partial LSE, partial O,
    # piece table and worker table, each region rounded up to 256 bytes
    def a(x):
        return (x + 255) // 256 * 256
    return (a(batch * 8) + a(slots * heads * 4) + a(slots * heads * 512 * 4) + a(slots * 16)
            + a(slots * 8))


def test_noalloc_matches_decode_two_calls_in_a_row():
    cases = [_case("C4R4", 128, [3000, 1, 700, 0], 21), _case("C2R4", 16, [65, 5000, 64], 22)]
    refs = []
    for w, cache, qc, qr in cases:
        max_len = int(cache.seq_lens.max().item())
        ref_o, ref_l = Decoder(cache, w.heads, max_len)(qc, qr, w.scale)
        refs.append((ref_o.clone(), ref_l.clone(), max_len))
    torch.cuda.synchronize()
    outs = []
    for (w, cache, qc, qr), (_, _, max_len) in zip(cases, refs):  # two calls in a row
        out = torch.full((qc.shape[0], qc.shape[1], 512), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        lse = torch.full((qc.shape[0], qc.shape[1]), float("nan"), device="cuda")
        q.qmla_decode_noalloc(w.fmt, cache.blocks, cache.block_table, cache.seq_lens, max_len,
                              qc, qr, w.scale, out, lse, cache.status)
        outs.append((out, lse))
    torch.cuda.synchronize()
    for (w, cache, qc, qr), (out, lse), (ref_o, ref_l, _) in zip(cases, outs, refs):
        assert cache.status.item() == 0
        _check_close(out, lse, ref_o, ref_l)
        lens = cache.seq_lens.cpu().tolist()
        _check_oracle(w, cache, lens, qc, qr, out, lse, range(len(lens)))


def test_noalloc_fewer_workers_when_partials_do_not_fit():
    """100 short sequences at 128 heads: one partial per sequence plus one per
    CTA pair of the usual split needs more than the scratch holds, so the
    call takes the largest worker count that fits."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    batch, heads = 100, 128
    scratch = 32 << 20
    assert _scratch_need(batch, heads, batch + sms // 2) > scratch
    fit = max(w for w in range(1, sms // 2 + 1) if _scratch_need(batch, heads, batch + w) <= scratch)
    assert 1 < fit < sms // 2
    rng = np.random.default_rng(31)
    lens = [int(x) for x in rng.integers(1, 400, batch)]
    lens[3] = 0
    w, cache, qc, qr = _case("C2R4", heads, lens, 24)
    max_len = max(lens)
    ref_o, ref_l = Decoder(cache, heads, max_len)(qc, qr, w.scale)
    out = torch.full((batch, heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((batch, heads), float("nan"), device="cuda")
    for _ in range(2):  # twice: the second call reuses what the first left in the scratch
        q.qmla_decode_noalloc(w.fmt, cache.blocks, cache.block_table, cache.seq_lens, max_len,
                              qc, qr, w.scale, out, lse, cache.status)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    _check_close(out, lse, ref_o, ref_l)
    _check_oracle(w, cache, lens, qc, qr, out, lse, [0, 3, 50, 99])


def test_noalloc_rejects_batch_beyond_scratch():
    w, cache, qc, qr = _case("C4R4", 128, [64], 23)
    big_b = 200  # 200 sequences x 128 heads of partials exceed the 32 MiB scratch
    qcb = qc.expand(big_b, -1, -1).contiguous()
    qrb = qr.expand(big_b, -1, -1).contiguous()
    table = cache.block_table.expand(big_b, -1).contiguous()
    lens = cache.seq_lens.expand(big_b).contiguous()
    out = torch.empty(big_b, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(big_b, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmlaError) as e:
        q.qmla_decode_noalloc("C4R4", cache.blocks, table, lens, 64, qcb, qrb, w.scale, out, lse,
                              cache.status)
    assert e.value.code == -3
