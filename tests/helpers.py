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
