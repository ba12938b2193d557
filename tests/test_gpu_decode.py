"""GPU parity of qmla_decode against the oracle.

Small cases are compared in full (several blocks, ragged tails, empty
sequences, every format and the served head counts); the full-size workloads
are built on the GPU and compared on sampled (sequence, head) rows, with the
oracle building its own cache from the same seeded tokens."""
import numpy as np
import pytest
import torch

import oracle
from bit_mla_kv_qmla_gb300 import QMLA_STATUS_BAD_BLOCK, QMLA_STATUS_BAD_LEN
from bit_mla_kv_qmla_gb300 import workloads as W
from bit_mla_kv_qmla_gb300.cache import Decoder, PagedCache, build_cache

from helpers import boundary_sequences, compare_rows, oracle_pool_for_seq, sample_heads

pytestmark = pytest.mark.gpu

# blocks the 128-head kernel's split charges for each sequence a worker
# starts (decode_tc.cu, launch_decode_tc128)
TC128_PIECE_COST = 6
FMTS = ["C4R4", "C2R4", "BF16", "C4R2", "C2R2"]


def _small_workload(fmt, heads, seed):
    return W.Workload(f"small_{fmt}_{heads}", fmt, 5, heads, 1000, 0, "lognormal8", 0, seed)


def _oracle_full(w, cache, lens, qc, qr, gen_device):
    table = cache.block_table.cpu().numpy()
    refs_o, refs_l = [], []
    for b, L in enumerate(lens):
        pool = oracle_pool_for_seq(w, b, L, table[b], cache.num_blocks, gen_device)
        o, l = oracle.decode(W.FORMATS[w.fmt], pool, table[b:b + 1], np.array([L]),
                             qc[b:b + 1].cpu(), qr[b:b + 1].cpu(), w.scale)
        refs_o.append(o[0])
        refs_l.append(l[0])
    return np.stack(refs_o), np.stack(refs_l)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("heads", [16, 32, 128])
def test_decode_small_ragged(fmt, heads):
    w = _small_workload(fmt, heads, 11)
    lens = [1, 63, 65, 1000, 0]  # one token, partial block, block + 1, many blocks, empty
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    qc, qr = W.queries(w)
    dec = Decoder(cache, heads, max(lens))
    out, lse = dec(qc.cuda(), qr.cuda(), w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    ref_o, ref_l = _oracle_full(w, cache, lens, qc, qr, "cpu")
    compare_rows(out, lse, ref_o, ref_l, f"{fmt} H{heads}")
    assert torch.all(out[4] == 0) and torch.all(torch.isneginf(lse[4]))


@pytest.mark.parametrize("fmt,heads", [("C4R4", 16), ("C2R4", 16), ("C4R4", 128)])
def test_decode_large_batch_short_sequences(fmt, heads):
    """More sequences than the 16-head kernel plans for itself (so its pieces
    come from the planner kernel) and than workers, with ragged short lengths
    and empty sequences: many workers see several sequences."""
    w = W.Workload(f"batch_{fmt}_{heads}", fmt, 150, heads, 300, 0, "lognormal8", 0, 23)
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(0, 300, 150)]
    lens[7] = 0
    lens[8] = 1
    lens[9] = 64
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    qc, qr = W.queries(w)
    out, lse = Decoder(cache, heads, max(lens))(qc.cuda(), qr.cuda(), w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    rows = [0, 7, 8, 9, 10, 77, 149]
    table = cache.block_table.cpu().numpy()
    for b in rows:
        L = lens[b]
        pool = oracle_pool_for_seq(w, b, L, table[b], cache.num_blocks, "cpu")
        o, l = oracle.decode(W.FORMATS[w.fmt], pool, table[b:b + 1], np.array([L]),
                             qc[b:b + 1].cpu(), qr[b:b + 1].cpu(), w.scale)
        compare_rows(out[b:b + 1], lse[b:b + 1], o, l, f"{fmt} H{heads} seq {b}")


@pytest.mark.parametrize("fmt,heads", [("C4R4", 16), ("C2R4", 16), ("C4R4", 128)])
def test_decode_many_short_sequences(fmt, heads):
    """Up to 64 sequences (the 16-head kernel plans its own pieces) of a few
    blocks each, with empty and one-token sequences: fewer blocks than
    workers, so with a piece cost many workers own no real block, and every
    worker boundary falls near a sequence start.  Every row is compared."""
    w = W.Workload(f"short_{fmt}_{heads}", fmt, 60, heads, 200, 0, "lognormal8", 0, 29)
    rng = np.random.default_rng(9)
    lens = [int(x) for x in rng.integers(0, 200, 60)]
    lens[0] = 0
    lens[1] = 1
    lens[2] = 64
    lens[59] = 0
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    qc, qr = W.queries(w)
    out, lse = Decoder(cache, heads, max(lens))(qc.cuda(), qr.cuda(), w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    ref_o, ref_l = _oracle_full(w, cache, lens, qc, qr, "cpu")
    compare_rows(out, lse, ref_o, ref_l, f"{fmt} H{heads} short")


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_tiny_workload(fmt):
    w = W.with_format(W.WORKLOADS[0], fmt)
    cache = build_cache(w, "cuda", gen_device="cpu")
    qc, qr = W.queries(w)
    out, lse = Decoder(cache, w.heads, w.seq_len)(qc.cuda(), qr.cuda(), w.scale)
    torch.cuda.synchronize()
    ref_o, ref_l = _oracle_full(w, cache, W.seq_lens(w), qc, qr, "cpu")
    compare_rows(out, lse, ref_o, ref_l, w.name)


# seqs None: the sequences of the 128-head split plan whose context a worker
# boundary cuts into the shortest pieces, and the one split the most
FULL = [(1, "C4R4", [0, 19], 6), (2, "C4R4", [3], 8), (3, "C2R4", None, 6),
        (4, "C4R4", None, 8), (4, "C2R4", None, 6), (4, "BF16", [0], 6), (1, "BF16", [5, 30], 16),
        (1, "C2R2", [4], 8), (2, "C4R2", [11], 6), (2, "C2R4", [7], 6), (3, "C4R4", None, 6)]


@pytest.mark.parametrize("cfg,fmt,seqs,nheads", FULL)
def test_decode_full_size_sampled(cfg, fmt, seqs, nheads):
    w = W.with_format(W.WORKLOADS[cfg], fmt)
    lens = W.seq_lens(w)
    if seqs is None:
        assert w.heads == 128
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        # the 128-head kernel: one worker per CTA pair, six blocks of piece cost
        seqs = boundary_sequences([(L + 63) // 64 for L in lens], sms // 2, TC128_PIECE_COST)
    cache = build_cache(w, "cuda", gen_device="cuda")
    qc, qr = W.queries(w, device="cuda")
    out, lse = Decoder(cache, w.heads, max(lens))(qc, qr, w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    table = cache.block_table.cpu().numpy()
    for b in seqs:
        hs = sample_heads(w.heads, nheads, 100 + b)
        pool = oracle_pool_for_seq(w, b, lens[b], table[b], cache.num_blocks, "cuda")
        ro, rl = oracle.decode(W.FORMATS[fmt], pool, table[b:b + 1], np.array([lens[b]]),
                               qc[b:b + 1, hs].cpu(), qr[b:b + 1, hs].cpu(), w.scale)
        compare_rows(out[b, hs], lse[b, hs], ro[0], rl[0], f"{w.name} seq {b}")


def test_decode_block_permutation_invariance():
    """Same tokens, different physical block placement: bitwise equal output."""
    w = _small_workload("C4R4", 128, 12)
    lens = [700, 64, 130]
    c1 = build_cache(w, "cuda", lens=lens, permute=True, gen_device="cpu")
    c2 = build_cache(w, "cuda", lens=lens, permute=False, gen_device="cpu")
    assert not torch.equal(c1.block_table, c2.block_table)
    qc, qr = W.queries(w)
    qc, qr = qc[:3].cuda(), qr[:3].cuda()
    o1, l1 = Decoder(c1, 128, 700)(qc, qr, w.scale)
    o2, l2 = Decoder(c2, 128, 700)(qc, qr, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("heads", [16, 128])
def test_decode_deterministic(heads):
    w = _small_workload("C2R4", heads, 13)
    lens = [3000, 1, 2000, 640, 64]
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    qc, qr = W.queries(w)
    dec = Decoder(cache, heads, 3000)
    o1, l1 = dec(qc.cuda(), qr.cuda(), w.scale)
    o1, l1 = o1.clone(), l1.clone()
    o2, l2 = dec(qc.cuda(), qr.cuda(), w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_bad_block_and_length_are_flagged():
    w = _small_workload("C4R4", 16, 14)
    cache = build_cache(w, "cuda", lens=[200, 100], gen_device="cpu")
    qc, qr = W.queries(w)
    qc, qr = qc[:2].cuda(), qr[:2].cuda()
    dec = Decoder(cache, 16, 200)
    cache.block_table[1, 0] = 10_000  # outside the pool
    dec(qc, qr, w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() & QMLA_STATUS_BAD_BLOCK
    cache.status.zero_()
    cache.block_table.copy_(build_cache(w, "cuda", lens=[200, 100]).block_table)
    dec2 = Decoder(cache, 16, 150)  # max_seq_len below the first sequence's length
    out, lse = dec2(qc, qr, w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() & QMLA_STATUS_BAD_LEN
    assert torch.isfinite(lse).all()


@pytest.mark.parametrize("fmt,heads,q_len", [("C4R4", 16, 8), ("C2R4", 16, 8), ("BF16", 16, 8),
                                             ("C4R4", 64, 2), ("C4R4", 8, 2), ("C4R4", 16, 2),
                                             ("C2R2", 16, 4)])
def test_decode_multi_query(fmt, heads, q_len):
    """Multi-token query decode (q_len queries per sequence, causal) against the
    oracle, every row: 16 x 8 and 64 x 2 query rows run on the 128-head
    tensor-core kernel, 8 x 2 and 16 x 2 on the CUDA cores.
    Sequences shorter than q_len leave their first queries nothing to attend."""
    w = W.Workload(f"multi_{fmt}_{heads}_{q_len}", fmt, 5, heads, 1000, 0, "lognormal8", 0, 37)
    lens = [1, q_len + 1, 63, 130, 1000]
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    g = torch.Generator().manual_seed(41)
    qc = torch.randn(5, q_len, heads, 512, generator=g).to(torch.bfloat16)
    qr = torch.randn(5, q_len, heads, 64, generator=g).to(torch.bfloat16)
    out, lse = Decoder(cache, heads, max(lens), q_len=q_len)(qc.cuda(), qr.cuda(), w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    table = cache.block_table.cpu().numpy()
    for b, L in enumerate(lens):
        pool = oracle_pool_for_seq(w, b, L, table[b], cache.num_blocks, "cpu")
        ro, rl = oracle.decode_multi(W.FORMATS[fmt], pool, table[b:b + 1], np.array([L]),
                                     qc[b:b + 1], qr[b:b + 1], w.scale)
        compare_rows(out[b], lse[b], ro[0], rl[0], f"{fmt} {heads}x{q_len} seq {b}")


@pytest.mark.parametrize("fmt", ["C4R4", "C2R4"])
def test_decode_folded_rotation(fmt):
    """Latents and content queries rotated by an orthogonal R (a transform
    folded into the weights offline): the GPU decode of the rotated cache
    matches the oracle on the same inputs, and on latents with 10x outlier
    channels its error against the exact decode of the unrotated inputs is
    smaller than without R (the oracle-side pin shows the same)."""
    w = W.Workload(f"fold_{fmt}", fmt, 3, 16, 300, 0, "x10pct1", 0, 5)
    R = W.orthogonal(512, 3)
    lens = [300, 257, 64]
    table, nblocks = W.block_table(w, lens)
    qc, qr = W.queries(w)
    toks = [W.tokens(w, b, L) for b, L in enumerate(lens)]
    results = {}
    for rot in (False, True):
        cache = PagedCache(fmt, table, nblocks)
        pool = np.zeros(nblocks * oracle.block_bytes(W.FORMATS[fmt]), np.uint8)
        tbl = cache.block_table.cpu().numpy()
        for b, (lat, rope) in enumerate(toks):
            lat_b = W.rotate(lat, R) if rot else lat
            cache.append_seq(b, lat_b.cuda(), rope.cuda())
            oracle.append(W.FORMATS[fmt], pool, tbl[b:b + 1], np.array([0], np.int32),
                          lat_b.unsqueeze(0), rope.unsqueeze(0))
        q = W.rotate(qc, R) if rot else qc
        out, lse = Decoder(cache, 16, max(lens))(q.cuda(), qr.cuda(), w.scale)
        torch.cuda.synchronize()
        assert cache.status.item() == 0
        ro, rl = oracle.decode(W.FORMATS[fmt], pool, tbl, np.array(lens), q, qr, w.scale)
        compare_rows(out, lse, ro, rl, f"{fmt} rotated={rot}")
        o = out.double().cpu().numpy()
        results[rot] = (o @ R.numpy().T if rot else o, lse.double().cpu().numpy())
    # exact reference: the unquantized decode of the unrotated inputs
    pool = np.zeros(nblocks * oracle.block_bytes(oracle.BF16), np.uint8)
    tbl = table.numpy().astype(np.int32)
    for b, (lat, rope) in enumerate(toks):
        oracle.append(oracle.BF16, pool, tbl[b:b + 1], np.array([0], np.int32), lat.unsqueeze(0),
                      rope.unsqueeze(0))
    O0, l0 = oracle.decode(oracle.BF16, pool, tbl, np.array(lens), qc, qr, w.scale)
    rms = {k: np.sqrt(((v[0] - O0) ** 2).mean() / (O0 ** 2).mean()) for k, v in results.items()}
    dl = {k: np.abs(v[1] - l0).mean() for k, v in results.items()}
    assert dl[True] < 0.6 * dl[False] and rms[True] < 0.75 * rms[False], (dl, rms)


@pytest.mark.parametrize("batch", [64, 65])
def test_decode_plan_source_boundary(batch):
    """64 sequences: the 16-head kernel plans its own pieces; 65: the planner
    kernel does.  Same tokens, same results within the tolerance."""
    w = W.Workload(f"bound_{batch}", "C4R4", batch, 16, 200, 0, "lognormal8", 0, 43)
    rng = np.random.default_rng(batch)
    lens = [int(x) for x in rng.integers(0, 200, batch)]
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    qc, qr = W.queries(w)
    out, lse = Decoder(cache, 16, max(lens))(qc.cuda(), qr.cuda(), w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    table = cache.block_table.cpu().numpy()
    for b in (0, 31, batch - 1):
        L = lens[b]
        pool = oracle_pool_for_seq(w, b, L, table[b], cache.num_blocks, "cpu")
        o, l = oracle.decode(W.FORMATS[w.fmt], pool, table[b:b + 1], np.array([L]),
                             qc[b:b + 1].cpu(), qr[b:b + 1].cpu(), w.scale)
        compare_rows(out[b:b + 1], lse[b:b + 1], o, l, f"batch {batch} seq {b}")


@pytest.mark.parametrize("fmt,heads", [("C4R4", 16), ("C2R4", 16), ("C4R4", 128)])
def test_decode_one_long_sequence(fmt, heads):
    """One 131072-token sequence: the split gives every worker a piece of it
    (152 pieces at 16 heads, 76 at 128), the most partials the merge ever
    combines for one sequence (in rounds of eight).  Sampled heads against
    the oracle, plus an empty second sequence whose row must be O = 0,
    LSE = -inf."""
    w = W.Workload(f"long_{fmt}_{heads}", fmt, 2, heads, 131072, 0, "x10pct1", 0, 53)
    lens = [131072, 0]
    cache = build_cache(w, "cuda", lens=lens, gen_device="cuda")
    qc, qr = W.queries(w, device="cuda")
    out, lse = Decoder(cache, heads, max(lens))(qc, qr, w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    table = cache.block_table.cpu().numpy()
    hs = sample_heads(heads, 4, 61)
    pool = oracle_pool_for_seq(w, 0, lens[0], table[0], cache.num_blocks, "cuda")
    ro, rl = oracle.decode(W.FORMATS[fmt], pool, table[0:1], np.array([lens[0]]),
                           qc[0:1, hs].cpu(), qr[0:1, hs].cpu(), w.scale)
    compare_rows(out[0, hs], lse[0, hs], ro[0], rl[0], w.name)
    assert torch.count_nonzero(out[1]).item() == 0
    assert torch.isneginf(lse[1]).all()


def test_decode_max_heads():
    """256 query heads, the most any kernel serves (the CUDA-core kernel)."""
    w = W.Workload("heads256", "C4R4", 2, 256, 300, 0, "lognormal8", 0, 47)
    lens = [300, 65]
    cache = build_cache(w, "cuda", lens=lens, gen_device="cpu")
    qc, qr = W.queries(w)
    out, lse = Decoder(cache, 256, max(lens))(qc.cuda(), qr.cuda(), w.scale)
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    ref_o, ref_l = _oracle_full(w, cache, lens, qc, qr, "cpu")
    hs = sample_heads(256, 24, 5)
    compare_rows(out[:, hs], lse[:, hs], ref_o[:, hs], ref_l[:, hs], "H256")


def test_plan_matches_host_restatement():
    """The planner kernel's pieces (read back from the decode's workspace)
    equal the tests' host restatement of the split, on the varied-length
    128-head workload, so the full-size samples drawn from that restatement
    sit at real worker boundaries."""
    from helpers import plan_pieces
    w = W.WORKLOADS[3]
    lens = W.seq_lens(w)
    cache = build_cache(w, "cuda", gen_device="cuda")
    qc, qr = W.queries(w, device="cuda")
    dec = Decoder(cache, w.heads, max(lens))
    dec(qc, qr, w.scale)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H = w.batch, w.heads
    slots = B + 2 * sms  # batch + the larger of the decode kernels' worker counts
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    ws = dec.workspace.cpu()
    seq_table = ws[:B * 8].view(torch.int32).view(B, 2)
    off = a256(B * 8) + a256(slots * H * 4) + a256(slots * H * 512 * 4)
    pieces = ws[off:off + slots * 16].view(torch.int32).view(slots, 4)
    want = plan_pieces([(L + 63) // 64 for L in lens], sms // 2, TC128_PIECE_COST)
    for b in range(B):
        base, n = seq_table[b].tolist()
        assert n == len(want[b]), b
        for i, (_, j0, j1) in enumerate(want[b]):
            assert pieces[base + i].tolist() == [b, j0, j1, 0], (b, i)
