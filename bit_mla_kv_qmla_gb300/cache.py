"""Paged low-bit MLA cache held in torch device memory.

Allocation only (torch owns the memory); every byte of the cache is written
by the library's qmla_append and read by its qmla_decode.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import (_fmt, qmla_append_advance, qmla_block_bytes, qmla_decode,
               qmla_decode_multi, qmla_decode_workspace_bytes)
from . import workloads as W


class PagedCache:
    """A pool of 64-token blocks plus a block table and per-sequence lengths."""

    def __init__(self, fmt, block_table: torch.Tensor, num_blocks: int, device="cuda"):
        self.fmt = _fmt(fmt)
        self.device = torch.device(device)
        self.block_bytes = qmla_block_bytes(self.fmt)
        # torch's caching allocator hands out 512-byte aligned storage
        self.blocks = torch.zeros(num_blocks * self.block_bytes, dtype=torch.uint8,
                                  device=self.device)
        self.block_table = block_table.to(self.device, torch.int32).contiguous()
        self.batch = int(block_table.shape[0])
        self.seq_lens = torch.zeros(self.batch, dtype=torch.int32, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    @property
    def num_blocks(self) -> int:
        return self.blocks.numel() // self.block_bytes

    def append(self, latent: torch.Tensor, rope: torch.Tensor, stream=None) -> None:
        """Append latent [B][n][512] / rope [B][n][64] (bf16, device) to every sequence."""
        qmla_append_advance(self.fmt, self.blocks, self.block_table, self.seq_lens, latent, rope,
                            self.status, stream)

    def append_seq(self, b: int, latent: torch.Tensor, rope: torch.Tensor, stream=None) -> None:
        """Append latent [n][512] / rope [n][64] to sequence b only."""
        qmla_append_advance(self.fmt, self.blocks, self.block_table[b:b + 1],
                            self.seq_lens[b:b + 1], latent.unsqueeze(0), rope.unsqueeze(0),
                            self.status, stream)


class Decoder:
    """Pre-allocated outputs and workspace for repeated qmla_decode calls
    (q_len > 1: qmla_decode_multi, q_len query tokens per sequence)."""

    def __init__(self, cache: PagedCache, heads: int, max_seq_len: int, q_len: int = 1):
        self.cache = cache
        self.heads = heads
        self.q_len = int(q_len)
        self.max_seq_len = int(max_seq_len)
        dev = cache.device
        nbytes = qmla_decode_workspace_bytes(cache.fmt, cache.batch, heads * self.q_len,
                                             self.max_seq_len)
        if nbytes == 0:
            raise ValueError("unsupported decode shape")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        # out and lse in one allocation (lse 256-byte aligned after out), so a
        # caller can read the step's result back with a single copy of `io`
        rows = heads * self.q_len
        ob = cache.batch * rows * W.D_C * 2
        lo = (ob + 255) // 256 * 256
        self.io = torch.empty(lo + cache.batch * rows * 4, dtype=torch.uint8, device=dev)
        shape = (cache.batch, heads) if self.q_len == 1 else (cache.batch, self.q_len, heads)
        self.out = self.io[:ob].view(torch.bfloat16).view(*shape, W.D_C)
        self.lse = self.io[lo:].view(torch.float32).view(*shape)

    def __call__(self, q_c: torch.Tensor, q_r: torch.Tensor, scale: float, stream=None):
        c = self.cache
        fn = qmla_decode if self.q_len == 1 else qmla_decode_multi
        fn(c.fmt, c.blocks, c.block_table, c.seq_lens, self.max_seq_len, q_c, q_r, scale,
           self.out, self.lse, self.workspace, c.status, stream)
        return self.out, self.lse


def build_cache(w: W.Workload, device="cuda", extra_tokens: int = 0,
                lens: Optional[Sequence[int]] = None, permute: bool = True,
                gen_device=None) -> PagedCache:
    """Cache of workload w filled through qmla_append with its seeded tokens.

    ``extra_tokens`` reserves room for later appends.  Tokens are drawn on
    ``gen_device`` (default: the cache device) one sequence at a time."""
    lens = list(W.seq_lens(w) if lens is None else lens)
    table, nblocks = W.block_table(w, lens, extra_tokens, permute)
    cache = PagedCache(w.fmt, table, nblocks, device)
    gdev = device if gen_device is None else gen_device
    for b, L in enumerate(lens):
        if L == 0:
            continue
        lat, rope = W.tokens(w, b, L, device=gdev)
        cache.append_seq(b, lat.to(device), rope.to(device))
    return cache
