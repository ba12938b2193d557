"""Shared helpers of the GPU parity tests: build the same cache on both sides
(the GPU through qmla_append, the oracle through its own append) from the
same seeded tokens, and compare decode outputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_mla_kv_qmla_gb300 import workloads as W

# Tolerances of the decode parity: output relative to its largest magnitude,
# LSE absolute.  The operands of the tensor-core kernels are binary16
# (dequantized values and queries rounded to 11 significant bits) with
# binary32 accumulation; P is rounded to binary16 before the P.V product.
O_TOL = 1e-2
LSE_TOL = 1e-3


def oracle_pool_for_seq(w: W.Workload, b: int, L: int, table_row: np.ndarray, nblocks: int,
                        gen_device="cpu"):
    """Oracle-side pool holding sequence b (same block ids as the GPU cache)."""
    fmt = W.FORMATS[w.fmt]
    pool = np.zeros(nblocks * oracle.block_bytes(fmt), np.uint8)
    if L > 0:
        lat, rope = W.tokens(w, b, L, device=gen_device)
        oracle.append(fmt, pool, table_row[None, :].astype(np.int32), np.array([0], np.int32),
                      lat.cpu().unsqueeze(0), rope.cpu().unsqueeze(0))
    return pool


def compare_rows(out, lse, ref_o, ref_l, label=""):
    """out/lse: GPU results for the compared rows; ref_*: oracle (float64)."""
    o = out.float().cpu().numpy().reshape(-1, 512)
    r = np.asarray(ref_o).reshape(-1, 512)
    lg = lse.float().cpu().numpy().reshape(-1)
    lr = np.asarray(ref_l).reshape(-1)
    both_inf = np.isneginf(lg) & np.isneginf(lr)
    assert np.array_equal(np.isneginf(lg), np.isneginf(lr)), f"{label}: -inf LSE mismatch"
    dl = np.abs(lg[~both_inf] - lr[~both_inf])
    assert dl.size == 0 or dl.max() <= LSE_TOL, f"{label}: max |dLSE| = {dl.max():.3e}"
    for i in range(r.shape[0]):
        denom = np.abs(r[i]).max()
        if denom == 0:
            assert np.all(o[i] == 0), f"{label}: row {i} should be zero"
            continue
        err = np.abs(o[i] - r[i]).max() / denom
        assert err <= O_TOL, f"{label}: row {i} max|dO|/max|O| = {err:.3e}"
    return float(dl.max()) if dl.size else 0.0


def sample_heads(H: int, k: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    return sorted(torch.randperm(H, generator=g)[:k].tolist())


def plan_pieces(nblocks, workers: int, piece_cost: int):
    """The decode's split plan, restated on the host: the blocks of all
    sequences, each non-empty sequence preceded by piece_cost virtual blocks,
    cut into min(workers, total) near-equal contiguous ranges.  Returns, per
    sequence, its pieces as (worker, first block, end block)."""
    ext = [n + piece_cost if n > 0 else 0 for n in nblocks]
    N = sum(ext)
    P = min(workers, N)
    out, carry = [], 0
    for n, e in zip(nblocks, ext):
        pcs = []
        if n > 0:
            S = carry + piece_cost
            first = ((S + 1) * P - 1) // N
            last = ((S + n) * P - 1) // N
            for wk in range(first, last + 1):
                w0, w1 = wk * N // P, (wk + 1) * N // P
                pcs.append((wk, max(w0 - S, 0), min(w1 - S, n)))
        out.append(pcs)
        carry += e
    return out


def boundary_sequences(nblocks, workers: int, piece_cost: int, k: int = 2):
    """Sequences whose context a worker boundary cuts into the shortest
    pieces (the split's most ragged merges): the k with the shortest partial
    piece, then the one split over the most workers."""
    plan = plan_pieces(nblocks, workers, piece_cost)
    split = [(min(j1 - j0 for _, j0, j1 in p), b) for b, p in enumerate(plan) if len(p) > 1]
    chosen = [b for _, b in sorted(split)[:k]]
    most = max(range(len(plan)), key=lambda b: len(plan[b]))
    if most not in chosen:
        chosen.append(most)
    return chosen
