"""GPU checks of qmla_decode_step, the decode step from host memory to host
memory in one C-ABI call: the step's packed host input (new tokens and
queries) is copied in, the tokens appended, the lengths advanced, the decode
run and out / lse copied into a host buffer.

Each case runs the same steps twice on identical caches: once through
qmla_decode_step with page-locked host buffers, once through the
device-buffer calls (qmla_append_advance, qmla_decode).  The same kernels
see the same inputs, so outputs, pools and lengths must agree bit for bit;
sampled rows of the last step are also checked against the oracle, which
appends the same tokens to its own cache."""
import numpy as np
import pytest
import torch

import oracle
import bit_mla_kv_qmla_gb300 as q
from bit_mla_kv_qmla_gb300 import workloads as W
from bit_mla_kv_qmla_gb300.cache import Decoder, build_cache

from helpers import compare_rows, oracle_pool_for_seq, sample_heads

pytestmark = pytest.mark.gpu


def _workload(fmt, heads, lens, seed):
    return W.Workload(f"step_host_{fmt}_{heads}", fmt, len(lens), heads, max(lens), 0,
                      "lognormal8", 0, seed)


def _pack(o, lat, rope, qc, qr):
    """Step input packed at qmla_decode_step_layout's offsets, page-locked."""
    h = torch.zeros(o[4], dtype=torch.uint8).pin_memory()
    parts = ([(o[0], lat), (o[1], rope)] if lat is not None else []) + [(o[2], qc), (o[3], qr)]
    for off, t in parts:
        raw = t.contiguous().reshape(-1).view(torch.uint8)
        h[off:off + raw.numel()].copy_(raw)
    return h


def _unpack(o, h_out, batch, heads):
    out = h_out[o[5]:o[5] + batch * heads * 512 * 2].view(torch.bfloat16).view(batch, heads, 512)
    lse = h_out[o[6]:o[6] + batch * heads * 4].view(torch.float32).view(batch, heads)
    return out, lse


@pytest.mark.parametrize("fmt,heads,lens,n_new", [
    ("C4R4", 128, [700, 65, 2000, 1], 1),
    ("C2R4", 16, [300, 5000, 64], 2),
    ("BF16", 128, [129, 64], 1),
    ("C4R4", 16, [0, 4000, 63, 64, 65], 3),
])
def test_host_step_matches_device_calls_and_oracle(fmt, heads, lens, n_new):
    steps = 3
    w = _workload(fmt, heads, lens, 41)
    caches = [build_cache(w, "cuda", lens=lens, extra_tokens=steps * n_new, gen_device="cpu")
              for _ in range(2)]
    assert torch.equal(caches[0].blocks, caches[1].blocks)
    max_len = max(lens) + steps * n_new
    B = len(lens)
    o = q.qmla_decode_step_layout(B, heads, n_new)
    ws = torch.empty(q.qmla_decode_step_workspace_bytes(fmt, B, heads, n_new, max_len),
                     dtype=torch.uint8, device="cuda")
    h_out = torch.full((o[7],), 0xff, dtype=torch.uint8).pin_memory()
    dec = Decoder(caches[1], heads, max_len)
    g = torch.Generator().manual_seed(7)
    news = []
    for k in range(steps):
        lat = torch.randn(B, n_new, 512, generator=g).to(torch.bfloat16)
        rope = torch.randn(B, n_new, 64, generator=g).to(torch.bfloat16)
        qc, qr = W.queries(w, step=k + 1)
        news.append((lat, rope))
        # one call from host memory to host memory
        h_in = _pack(o, lat, rope, qc, qr)
        c = caches[0]
        q.qmla_decode_step(fmt, c.blocks, c.block_table, c.seq_lens, max_len, heads, n_new, h_in,
                           w.scale, h_out, ws, c.status)
        out_h, lse_h = _unpack(o, h_out, B, heads)
        # the device-buffer calls
        caches[1].append(lat.cuda(), rope.cuda())
        ref_o, ref_l = dec(qc.cuda(), qr.cuda(), w.scale)
        torch.cuda.synchronize()
        assert torch.equal(out_h.view(torch.int16), ref_o.cpu().view(torch.int16)), f"out step {k}"
        assert torch.equal(lse_h.view(torch.int32), ref_l.cpu().view(torch.int32)), f"lse step {k}"
    for c in caches:
        assert c.status.item() == 0
        assert c.seq_lens.cpu().tolist() == [L + steps * n_new for L in lens]
    assert torch.equal(caches[0].blocks, caches[1].blocks)

    # the oracle: its own cache with the same appended tokens, sampled heads
    fcode = W.FORMATS[fmt]
    table = caches[0].block_table.cpu().numpy()
    qc, qr = W.queries(w, step=steps)
    for b in sorted({0, B - 1, int(np.argmax(lens))}):
        pool = oracle_pool_for_seq(w, b, lens[b], table[b], caches[0].num_blocks, "cpu")
        for k, (lat, rope) in enumerate(news):
            skipped = oracle.append(fcode, pool, table[b:b + 1],
                                    np.array([lens[b] + k * n_new], np.int32),
                                    lat[b:b + 1], rope[b:b + 1])
            assert skipped == 0
        hs = sample_heads(heads, 6, 500 + b)
        ro, rl = oracle.decode(fcode, pool, table[b:b + 1], np.array([lens[b] + steps * n_new]),
                               qc[b:b + 1, hs], qr[b:b + 1, hs], w.scale)
        compare_rows(out_h[b, hs], lse_h[b, hs], ro[0], rl[0], f"{w.name} seq {b}")


def test_host_step_without_new_tokens_is_a_decode():
    lens = [333, 1, 4097]
    w = _workload("C4R4", 128, lens, 43)
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    B, heads, max_len = len(lens), 128, max(lens)
    o = q.qmla_decode_step_layout(B, heads, 0)
    assert o[0] == o[1] == 0 and o[2] == 0
    ws = torch.empty(q.qmla_decode_step_workspace_bytes("C4R4", B, heads, 0, max_len),
                     dtype=torch.uint8, device="cuda")
    qc, qr = W.queries(w)
    h_in = _pack(o, None, None, qc, qr)
    h_out = torch.zeros(o[7], dtype=torch.uint8).pin_memory()
    q.qmla_decode_step("C4R4", cache.blocks, cache.block_table, cache.seq_lens, max_len, heads, 0,
                       h_in, w.scale, h_out, ws, cache.status)
    out_h, lse_h = _unpack(o, h_out, B, heads)
    ref_o, ref_l = Decoder(cache, heads, max_len)(qc.cuda(), qr.cuda(), w.scale)
    torch.cuda.synchronize()
    assert cache.seq_lens.cpu().tolist() == lens
    assert torch.equal(out_h.view(torch.int16), ref_o.cpu().view(torch.int16))
    assert torch.equal(lse_h.view(torch.int32), ref_l.cpu().view(torch.int32))


def test_host_step_small_workspace_enqueues_nothing():
    lens = [100, 200]
    w = _workload("C4R4", 16, lens, 44)
    cache = build_cache(w, "cuda", lens=lens, extra_tokens=1, gen_device="cpu")
    B, heads = len(lens), 16
    o = q.qmla_decode_step_layout(B, heads, 1)
    need = q.qmla_decode_step_workspace_bytes("C4R4", B, heads, 1, 256)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    qc, qr = W.queries(w)
    lat = torch.zeros(B, 1, 512, dtype=torch.bfloat16)
    h_in = _pack(o, lat, lat[:, :, :64], qc, qr)
    h_out = torch.zeros(o[7], dtype=torch.uint8).pin_memory()
    blocks0 = cache.blocks.clone()
    with pytest.raises(q.QmlaError) as e:
        q.qmla_decode_step("C4R4", cache.blocks, cache.block_table, cache.seq_lens, 256, heads, 1,
                           h_in, w.scale, h_out, ws, cache.status)
    assert e.value.code == -4
    torch.cuda.synchronize()
    assert cache.seq_lens.cpu().tolist() == lens
    assert torch.equal(cache.blocks, blocks0)
