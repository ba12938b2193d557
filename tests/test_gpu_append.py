"""GPU parity of qmla_append: the packed bytes (codes, scales, zeros) must equal
the oracle's bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from bit_mla_kv_qmla_gb300 import (QMLA_STATUS_BAD_BLOCK, QMLA_STATUS_BAD_LEN, qmla_append,
                                   qmla_append_advance, qmla_block_bytes)
from bit_mla_kv_qmla_gb300 import workloads as W
from bit_mla_kv_qmla_gb300.cache import PagedCache, build_cache

from helpers import oracle_pool_for_seq

pytestmark = pytest.mark.gpu
FMTS = ["C4R4", "C2R4", "BF16", "C4R2", "C2R2"]


def _seq_blocks(pool: np.ndarray, row: np.ndarray, n: int, bb: int) -> np.ndarray:
    return np.concatenate([pool[int(k) * bb:(int(k) + 1) * bb] for k in row[:n]])


def _check_seqs(w, cache, seqs, gen_device):
    lens = W.seq_lens(w)
    table = cache.block_table.cpu().numpy()
    gpu_pool = cache.blocks.cpu().numpy()
    bb = qmla_block_bytes(w.fmt)
    for b in seqs:
        L = lens[b]
        n = (L + 63) // 64
        ref = oracle_pool_for_seq(w, b, L, table[b], cache.num_blocks, gen_device)
        assert np.array_equal(_seq_blocks(gpu_pool, table[b], n, bb),
                              _seq_blocks(ref, table[b], n, bb)), f"sequence {b} differs"


@pytest.mark.parametrize("fmt", FMTS)
def test_append_tiny_workload_bitexact(fmt):
    w = W.with_format(W.WORKLOADS[0], fmt)
    cache = build_cache(w, "cuda", gen_device="cpu")
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    _check_seqs(w, cache, [0], "cpu")


@pytest.mark.parametrize("cfg,fmt,seqs", [(1, "C4R4", [0, 31]), (2, "C4R4", [5]),
                                          (3, "C2R4", [0, 17, 63]), (4, "C4R4", [2]),
                                          (4, "C2R4", [1]), (4, "BF16", [3]),
                                          (1, "C2R2", [3, 30]), (3, "C4R2", [9])])
def test_append_full_size_sampled_bitexact(cfg, fmt, seqs):
    w = W.with_format(W.WORKLOADS[cfg], fmt)
    cache = build_cache(w, "cuda", gen_device="cuda")
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    _check_seqs(w, cache, seqs, "cuda")


def _hard_tokens(n, seed):
    """Groups that stress the rounding rules: wide dynamic range, binary16
    subnormal range, values far below binary16, constant groups, single
    outliers, large magnitudes."""
    g = torch.Generator().manual_seed(seed)
    lat = torch.randn(n, 512, generator=g)
    for t in range(n):
        k = t % 8
        if k == 6:
            lat[t] *= 1e-30  # far below binary16: the grid bottoms out at 2^-24
        elif k == 7:
            lat[t] *= 1e-3
            lat[t, 100] = -31000.0  # one huge outlier next to tiny values
        elif k == 1:
            lat[t] *= 4e-6
        elif k == 2:
            lat[t, :64] = 1.25
            lat[t, 64:128] = -7.0
        elif k == 3:
            lat[t] *= torch.exp(torch.randn(512, generator=g) * 3)
        elif k == 4:
            lat[t] = lat[t] * 1000 + 20000
        elif k == 5:
            lat[t, 3] = 300.0
    rope = torch.randn(n, 64, generator=g) * torch.exp(torch.randn(1, generator=g) * 2)
    lat = lat.clamp(-32000, 32000)
    return lat.to(torch.bfloat16), rope.to(torch.bfloat16)


@pytest.mark.parametrize("fmt", FMTS)
def test_append_hard_values_bitexact(fmt):
    n = 200
    lat, rope = _hard_tokens(n, 3)
    table = torch.tensor([[3, 0, 2, 1]], dtype=torch.int32)
    cache = PagedCache(fmt, table, 4)
    cache.append(lat[None].cuda(), rope[None].cuda())
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    ref = np.zeros(4 * qmla_block_bytes(fmt), np.uint8)
    oracle.append(W.FORMATS[fmt], ref, table.numpy(), np.array([0], np.int32), lat[None],
                  rope[None])
    assert np.array_equal(cache.blocks.cpu().numpy(), ref)


@pytest.mark.parametrize("fmt", ["C4R4", "C2R4", "C2R2"])
def test_append_incremental_equals_bulk_gpu(fmt):
    n = 130
    lat, rope = _hard_tokens(n, 4)
    table = torch.tensor([[1, 2, 0]], dtype=torch.int32)
    bulk = PagedCache(fmt, table, 3)
    bulk.append(lat[None].cuda(), rope[None].cuda())
    inc = PagedCache(fmt, table, 3)
    for t in range(n):
        inc.append(lat[None, t:t + 1].cuda(), rope[None, t:t + 1].cuda())
    torch.cuda.synchronize()
    assert torch.equal(bulk.blocks, inc.blocks)


def test_append_batched_multi_token():
    """batch > 1 with several tokens each, sequences at different offsets."""
    B, n = 3, 70
    g = torch.Generator().manual_seed(5)
    lat = torch.randn(B, n, 512, generator=g).to(torch.bfloat16)
    rope = torch.randn(B, n, 64, generator=g).to(torch.bfloat16)
    table = torch.tensor([[0, 5, -1], [4, 1, 6], [2, 3, 7]], dtype=torch.int32)
    pos = torch.tensor([0, 30, 63], dtype=torch.int32)
    cache = PagedCache("C4R4", table, 8)
    cache.seq_lens.copy_(pos)
    cache.append(lat.cuda(), rope.cuda())
    torch.cuda.synchronize()
    assert cache.status.item() == 0
    ref = np.zeros(8 * qmla_block_bytes("C4R4"), np.uint8)
    oracle.append(0, ref, table.numpy(), pos.numpy(), lat, rope)
    assert np.array_equal(cache.blocks.cpu().numpy(), ref)


def test_append_out_of_range_is_flagged_not_faulted():
    lat = torch.zeros(1, 3, 512, dtype=torch.bfloat16, device="cuda")
    rope = torch.zeros(1, 3, 64, dtype=torch.bfloat16, device="cuda")
    bb = qmla_block_bytes("C4R4")
    blocks = torch.zeros(2 * bb, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_table = torch.tensor([[7]], dtype=torch.int32, device="cuda")  # pool has 2 blocks
    qmla_append("C4R4", blocks, bad_table, torch.zeros(1, dtype=torch.int32, device="cuda"),
                lat, rope, status)
    torch.cuda.synchronize()
    assert status.item() & QMLA_STATUS_BAD_BLOCK
    status.zero_()
    table = torch.tensor([[0]], dtype=torch.int32, device="cuda")
    qmla_append("C4R4", blocks, table, torch.tensor([62], dtype=torch.int32, device="cuda"),
                lat, rope, status)  # positions 62, 63 fit, 64 does not
    torch.cuda.synchronize()
    assert status.item() & QMLA_STATUS_BAD_LEN
    assert torch.count_nonzero(blocks[bb:]) == 0


@pytest.mark.parametrize("n_new", [1, 5])
def test_append_advance_matches_append(n_new):
    """qmla_append_advance writes the same bytes as qmla_append and advances
    every position by n_new (one kernel for n_new = 1, two otherwise),
    including a sequence whose block id is out of range."""
    B = 4
    g = torch.Generator().manual_seed(17)
    lat = torch.randn(B, n_new, 512, generator=g).to(torch.bfloat16).cuda()
    rope = torch.randn(B, n_new, 64, generator=g).to(torch.bfloat16).cuda()
    table = torch.tensor([[0, 1], [2, 3], [4, 5], [9, 9]], dtype=torch.int32, device="cuda")
    pos0 = torch.tensor([0, 61, 63, 0], dtype=torch.int32, device="cuda")
    bb = qmla_block_bytes("C4R4")
    ref_blocks = torch.zeros(6 * bb, dtype=torch.uint8, device="cuda")
    ref_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qmla_append("C4R4", ref_blocks, table, pos0, lat, rope, ref_status)
    blocks = torch.zeros_like(ref_blocks)
    status = torch.zeros_like(ref_status)
    pos = pos0.clone()
    qmla_append_advance("C4R4", blocks, table, pos, lat, rope, status)
    torch.cuda.synchronize()
    assert torch.equal(blocks, ref_blocks)
    assert torch.equal(pos, pos0 + n_new)
    assert status.item() == ref_status.item() and status.item() & QMLA_STATUS_BAD_BLOCK
