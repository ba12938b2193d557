"""Low-bit MLA decode for GB300: Python binding of the C ABI in include/qmla.h.

Every function below only marshals arguments (torch tensors -> device
pointers, the current CUDA stream) and calls the function of the same name in
libqmla.so; all computation runs in the library's CUDA kernels.  Errors
returned by the library raise QmlaError.
"""
from __future__ import annotations

import functools

from typing import Optional

from . import _lib

C4R4, C2R4, BF16, C4R2, C2R2 = 0, 1, 2, 3, 4
FORMAT_NAMES = {"C4R4": C4R4, "C2R4": C2R4, "BF16": BF16, "C4R2": C4R2, "C2R2": C2R2}
D_C, D_R, GROUP, BLOCK_TOKENS = 512, 64, 64, 64

QMLA_OK = 0
QMLA_STATUS_BAD_BLOCK, QMLA_STATUS_BAD_LEN, QMLA_STATUS_TIMEOUT = 0x1, 0x2, 0x4
QMLA_STATUS_BAD_QUERY = 0x8


class QmlaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        msg = _lib.load().qmla_error_string(code).decode()
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


def _fmt(f) -> int:
    return FORMAT_NAMES[f] if isinstance(f, str) else int(f)


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _p(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _check(fn: str, code: int) -> None:
    if code != QMLA_OK:
        raise QmlaError(fn, code)


@functools.lru_cache(maxsize=None)
def qmla_block_bytes(fmt) -> int:
    return int(_lib.load().qmla_block_bytes(_fmt(fmt)))


def qmla_error_string(code: int) -> str:
    return _lib.load().qmla_error_string(int(code)).decode()


def qmla_append(fmt, blocks, block_table, positions, latent, rope_k, status,
                stream=None) -> None:
    """Quantize and pack latent [B][n_new][512] / rope_k [B][n_new][64] (bf16,
    device) into the block pool ``blocks`` (uint8, device)."""
    B, n_new = int(latent.shape[0]), int(latent.shape[1])
    if block_table.shape[0] < B or positions.numel() < B:
        raise ValueError("block_table / positions have fewer rows than latent")
    num_blocks = blocks.numel() // qmla_block_bytes(fmt)
    code = _lib.load().qmla_append(
        _fmt(fmt), _p(blocks), num_blocks, _p(block_table), int(block_table.shape[1]),
        _p(positions), B, n_new, _p(latent), _p(rope_k), _p(status), _stream(stream))
    _check("qmla_append", code)


def qmla_append_advance(fmt, blocks, block_table, positions, latent, rope_k, status,
                        stream=None) -> None:
    """qmla_append, then positions[b] += n_new on the device (positions: int32,
    device, written)."""
    B, n_new = int(latent.shape[0]), int(latent.shape[1])
    if block_table.shape[0] < B or positions.numel() < B:
        raise ValueError("block_table / positions have fewer rows than latent")
    num_blocks = blocks.numel() // qmla_block_bytes(fmt)
    code = _lib.load().qmla_append_advance(
        _fmt(fmt), _p(blocks), num_blocks, _p(block_table), int(block_table.shape[1]),
        _p(positions), B, n_new, _p(latent), _p(rope_k), _p(status), _stream(stream))
    _check("qmla_append_advance", code)


def qmla_decode_workspace_bytes(fmt, batch: int, heads: int, max_seq_len: int) -> int:
    return int(_lib.load().qmla_decode_workspace_bytes(_fmt(fmt), int(batch), int(heads),
                                                       int(max_seq_len)))


def qmla_decode(fmt, blocks, block_table, seq_lens, max_seq_len: int, q_c, q_r, scale: float,
                out, lse, workspace, status, stream=None, _entry="qmla_decode") -> None:
    """Absorbed-query MLA decode; writes out [B][H][512] bf16 and lse [B][H] f32."""
    B, H = int(q_c.shape[0]), int(q_c.shape[1])
    if block_table.shape[0] < B or seq_lens.numel() < B or tuple(q_r.shape[:2]) != (B, H):
        raise ValueError("block_table / seq_lens / q_r do not cover the query batch")
    if tuple(out.shape) != (B, H, D_C) or tuple(lse.shape) != (B, H):
        raise ValueError("out / lse shapes do not match the queries")
    num_blocks = blocks.numel() // qmla_block_bytes(fmt)
    code = getattr(_lib.load(), _entry)(
        _fmt(fmt), _p(blocks), num_blocks, _p(block_table), int(block_table.shape[1]),
        _p(seq_lens), int(max_seq_len), B, H, _p(q_c), _p(q_r), float(scale), _p(out), _p(lse),
        _p(workspace), int(workspace.numel() * workspace.element_size()), _p(status),
        _stream(stream))
    _check(_entry, code)


def qmla_decode_timeout_test(fmt, blocks, block_table, seq_lens, max_seq_len: int, q_c, q_r,
                             scale: float, out, lse, workspace, status, stream=None) -> None:
    """Test hook of the bounded device waits (qmla.h): qmla_decode whose
    16-head kernel withholds one barrier arrival, so that its waits run out
    and QMLA_STATUS_TIMEOUT is set; out / lse are not valid afterwards."""
    qmla_decode(fmt, blocks, block_table, seq_lens, max_seq_len, q_c, q_r, scale, out, lse,
                workspace, status, stream, _entry="qmla_decode_timeout_test")


def qmla_decode_multi(fmt, blocks, block_table, seq_lens, max_seq_len: int, q_c, q_r,
                      scale: float, out, lse, workspace, status, stream=None) -> None:
    """Decode of q_len query tokens per sequence with a causal mask: q_c
    [B][q_len][H][512], q_r [B][q_len][H][64]; writes out [B][q_len][H][512]
    bf16 and lse [B][q_len][H] f32."""
    B, Q, H = int(q_c.shape[0]), int(q_c.shape[1]), int(q_c.shape[2])
    if block_table.shape[0] < B or seq_lens.numel() < B or tuple(q_r.shape[:3]) != (B, Q, H):
        raise ValueError("block_table / seq_lens / q_r do not cover the query batch")
    if tuple(out.shape) != (B, Q, H, D_C) or tuple(lse.shape) != (B, Q, H):
        raise ValueError("out / lse shapes do not match the queries")
    num_blocks = blocks.numel() // qmla_block_bytes(fmt)
    code = _lib.load().qmla_decode_multi(
        _fmt(fmt), _p(blocks), num_blocks, _p(block_table), int(block_table.shape[1]),
        _p(seq_lens), int(max_seq_len), B, H, Q, _p(q_c), _p(q_r), float(scale), _p(out),
        _p(lse), _p(workspace), int(workspace.numel() * workspace.element_size()), _p(status),
        _stream(stream))
    _check("qmla_decode_multi", code)


def qmla_decode_noalloc(fmt, blocks, block_table, seq_lens, max_seq_len: int, q_c, q_r,
                        scale: float, out, lse, status, stream=None) -> None:
    """qmla_decode without a workspace argument, for callers that cannot
    allocate: the scratch is the library's fixed per-device array (see
    include/qmla.h); calls that overlap on the GPU race on it."""
    B, H = int(q_c.shape[0]), int(q_c.shape[1])
    if block_table.shape[0] < B or seq_lens.numel() < B or tuple(q_r.shape[:2]) != (B, H):
        raise ValueError("block_table / seq_lens / q_r do not cover the query batch")
    if tuple(out.shape) != (B, H, D_C) or tuple(lse.shape) != (B, H):
        raise ValueError("out / lse shapes do not match the queries")
    num_blocks = blocks.numel() // qmla_block_bytes(fmt)
    code = _lib.load().qmla_decode_noalloc(
        _fmt(fmt), _p(blocks), num_blocks, _p(block_table), int(block_table.shape[1]),
        _p(seq_lens), int(max_seq_len), B, H, _p(q_c), _p(q_r), float(scale), _p(out), _p(lse),
        _p(status), _stream(stream))
    _check("qmla_decode_noalloc", code)


@functools.lru_cache(maxsize=64)
def qmla_decode_step_layout(batch: int, heads: int, n_new: int) -> tuple:
    """Byte offsets of qmla_decode_step's packed host buffers: (latent, rope_k,
    q_c, q_r, input bytes, out, lse, output bytes)."""
    import ctypes
    o = (ctypes.c_size_t * 8)()
    _check("qmla_decode_step_layout",
           _lib.load().qmla_decode_step_layout(int(batch), int(heads), int(n_new), o))
    return tuple(int(x) for x in o)


def qmla_decode_step_workspace_bytes(fmt, batch: int, heads: int, n_new: int,
                                     max_seq_len: int) -> int:
    return int(_lib.load().qmla_decode_step_workspace_bytes(
        _fmt(fmt), int(batch), int(heads), int(n_new), int(max_seq_len)))


def qmla_decode_step(fmt, blocks, block_table, seq_lens, max_seq_len: int, heads: int,
                     n_new: int, h_in, scale: float, h_out, workspace, status,
                     stream=None) -> None:
    """One decode step from host memory to host memory: h_in (host uint8, the
    step's new tokens and queries packed as qmla_decode_step_layout gives) is
    copied in, the tokens appended and seq_lens advanced, the decode run and
    out / lse copied into h_out (host uint8); returns once they are there."""
    B = int(seq_lens.numel())
    o = qmla_decode_step_layout(B, heads, n_new)
    if h_in.numel() * h_in.element_size() < o[4] or h_out.numel() * h_out.element_size() < o[7]:
        raise ValueError("h_in / h_out smaller than qmla_decode_step_layout's sizes")
    if block_table.shape[0] < B:
        raise ValueError("block_table has fewer rows than seq_lens")
    num_blocks = blocks.numel() // qmla_block_bytes(fmt)
    code = _lib.load().qmla_decode_step(
        _fmt(fmt), _p(blocks), num_blocks, _p(block_table), int(block_table.shape[1]),
        _p(seq_lens), int(max_seq_len), B, int(heads), int(n_new), _p(h_in), float(scale),
        _p(h_out), _p(workspace), int(workspace.numel() * workspace.element_size()), _p(status),
        _stream(stream))
    _check("qmla_decode_step", code)


def qmla_read_status(status, stream=None) -> int:
    """Synchronize the stream and return QMLA_OK or QMLA_ERR_DEVICE."""
    return int(_lib.load().qmla_read_status(_p(status), _stream(stream)))
