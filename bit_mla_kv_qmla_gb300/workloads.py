"""Seeded synthetic workloads for low-bit MLA decode.

This module only draws random numbers and builds block tables; it holds none
of the method's arithmetic (no quantization, no attention).  Both the CUDA
path's tests/benchmark and the CPU oracle draw their inputs from here, so the
two sides see identical bits.

The pages name no dataset, model or request trace ("QuantMLA's INT4/INT2
KV-cache quantization reports 5x long-context throughput over BF16", section
"What the low-bit cache changes", speaks only of a cache-pressure serving
workload at a 128K window).  These synthetic workloads stand in for it: MLA
latents are near-Gaussian with a few outlier channels, which is the regime
the pages' function-aligned transforms are folded for ("QuantMLA: INT4 (and
INT2) for both halves of the MLA cache", section "Key findings").

Recipe (all values drawn in float32 and rounded to bfloat16 nearest-even):
  * queries q_c [B][H][512], q_r [B][H][64] ~ N(0, 1);
  * RoPE keys k_r [B][L][64] ~ N(0, 1);
  * content latents c [B][L][512] ~ N(0, 1), times a per-channel gain:
      "lognormal8"  - 8 seeded channels get gain ~ LogNormal(0, 1);
      "x10pct1"     - 1% of the channels (5 seeded channels) get gain 10;
  * block tables: the blocks of all sequences are a seeded random permutation
    of the pool, so consecutive blocks of a sequence are scattered in memory;
  * sequence lengths: fixed, or uniform integers in [lo, hi] (seeded).
Every sequence b draws its tokens from its own generator seeded by
(seed, b), so one sequence can be regenerated alone (row sampling for the
oracle at full size).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import torch

D_C, D_R, BLOCK = 512, 64, 64
FORMATS = {"C4R4": 0, "C2R4": 1, "BF16": 2, "C4R2": 3, "C2R2": 4}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    fmt: str                # "C4R4" | "C2R4" | "BF16" | "C4R2" | "C2R2"
    batch: int
    heads: int
    seq_len: int            # fixed length, or the upper bound when varlen
    seq_len_lo: int = 0     # > 0: lengths uniform in [seq_len_lo, seq_len]
    latent_outliers: str = "lognormal8"
    n_append: int = 0       # tokens appended per sequence per step
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(192.0)


# The five workloads (the pages' figures are quoted at a 128K window; the
# other sizes span the head counts and context lengths of MLA serving).
WORKLOADS = {
    0: Workload("tiny_c4r4_b1_h16_l256", "C4R4", 1, 16, 256, 0, "lognormal8", 0, 0),
    1: Workload("c4r4_b32_h16_l8192_append1", "C4R4", 32, 16, 8192, 0, "lognormal8", 1, 1),
    2: Workload("c4r4_b16_h128_l32768", "C4R4", 16, 128, 32768, 0, "x10pct1", 0, 2),
    3: Workload("c2r4_b64_h128_l1024to16384", "C2R4", 64, 128, 16384, 1024, "x10pct1", 0, 3),
    4: Workload("c4r4_b4_h128_l131072", "C4R4", 4, 128, 131072, 0, "x10pct1", 0, 4),
}


def with_format(w: Workload, fmt: str) -> Workload:
    return dataclasses.replace(w, fmt=fmt, name=w.name.replace(w.fmt.lower(), fmt.lower(), 1))


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def seq_lens(w: Workload) -> List[int]:
    if w.seq_len_lo <= 0:
        return [w.seq_len] * w.batch
    g = _gen(w.seed * 1000003 + 17)
    return torch.randint(w.seq_len_lo, w.seq_len + 1, (w.batch,), generator=g).tolist()


def channel_gain(w: Workload) -> torch.Tensor:
    """float32 [512] multiplicative gain of the content channels."""
    g = _gen(w.seed * 1000003 + 29)
    gain = torch.ones(D_C, dtype=torch.float32)
    if w.latent_outliers == "lognormal8":
        idx = torch.randperm(D_C, generator=g)[:8]
        gain[idx] = torch.exp(torch.randn(8, generator=g))
    elif w.latent_outliers == "x10pct1":
        idx = torch.randperm(D_C, generator=g)[: max(1, round(0.01 * D_C))]
        gain[idx] = 10.0
    elif w.latent_outliers != "none":
        raise ValueError(w.latent_outliers)
    return gain


def tokens(w: Workload, b: int, n: int, offset_seed: int = 0, device="cpu"):
    """Tokens of sequence b: (latent [n][512] bf16, rope [n][64] bf16).

    ``offset_seed`` selects an independent stream (e.g. tokens appended at
    decode step k use offset_seed = k + 1)."""
    g = _gen((w.seed * 1000003 + 101 + b) * 7919 + offset_seed, device)
    lat = torch.randn(n, D_C, generator=g, device=device, dtype=torch.float32)
    lat *= channel_gain(w).to(device)
    rope = torch.randn(n, D_R, generator=g, device=device, dtype=torch.float32)
    return lat.to(torch.bfloat16), rope.to(torch.bfloat16)


def queries(w: Workload, step: int = 0, device="cpu"):
    """(q_c [B][H][512] bf16, q_r [B][H][64] bf16)."""
    g = _gen(w.seed * 1000003 + 7 + 100003 * step, device)
    qc = torch.randn(w.batch, w.heads, D_C, generator=g, device=device, dtype=torch.float32)
    qr = torch.randn(w.batch, w.heads, D_R, generator=g, device=device, dtype=torch.float32)
    return qc.to(torch.bfloat16), qr.to(torch.bfloat16)


def blocks_needed(lens: Sequence[int], extra_tokens: int = 0) -> List[int]:
    return [(L + extra_tokens + BLOCK - 1) // BLOCK for L in lens]


def block_table(w: Workload, lens: Sequence[int], extra_tokens: int = 0,
                permute: bool = True):
    """(table [B][max_blocks] int32, num_blocks): blocks of every sequence
    drawn from a seeded permutation of the pool; unused entries are -1."""
    need = blocks_needed(lens, extra_tokens)
    total = sum(need)
    maxb = max(max(need), 1)
    if permute:
        perm = torch.randperm(total, generator=_gen(w.seed * 1000003 + 43))
    else:
        perm = torch.arange(total)
    table = torch.full((len(lens), maxb), -1, dtype=torch.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n].to(torch.int32)
        k += n
    return table, max(total, 1)


def exact_grid_group(gen: torch.Generator, bits: int, n: int = 64,
                     scale: float = 0.125, zero: Optional[float] = None):
    """Values code*scale + zero whose group quantizer output is known exactly:
    codes uniform in [0, 2^bits - 1] with 0 and the top code both present.
    Returns (values float32 [n], codes int [n], zero)."""
    levels = (1 << bits) - 1
    if zero is None:
        zero = -1.0 if torch.rand(1, generator=gen).item() < 0.5 else -2.0
    codes = torch.randint(0, levels + 1, (n,), generator=gen)
    perm = torch.randperm(n, generator=gen)
    codes[perm[0]] = 0
    codes[perm[1]] = levels
    vals = codes.to(torch.float32) * scale + zero
    return vals, codes, zero


def orthogonal(n: int, seed: int) -> torch.Tensor:
    """Seeded random orthogonal matrix [n][n] in float64 (Haar-distributed: Q
    of the QR factorization of a standard Gaussian matrix, with the column
    signs that make diag(R) positive).

    Stands in for a transform folded into the weights offline ("QuantMLA:
    INT4 (and INT2) for both halves of the MLA cache", section "Key
    findings"): folding R into the latent's down-projection and into the
    absorbed query projection turns the cached latent c into c R and the
    query q_c into q_c R, which leaves every exact score q_c . c unchanged
    and the output O = P C into O R."""
    g = _gen(seed * 1000003 + 61)
    a = torch.randn(n, n, generator=g, dtype=torch.float64)
    q, r = torch.linalg.qr(a)
    return q * torch.sign(torch.diagonal(r)).unsqueeze(0)


def rotate(x: torch.Tensor, R: torch.Tensor) -> torch.Tensor:
    """x [...][n] (bfloat16) times R [n][n], rounded to bfloat16."""
    return (x.to(torch.float64) @ R.to(x.device)).to(torch.bfloat16)
