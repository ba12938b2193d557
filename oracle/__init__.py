"""CPU oracle for the low-bit MLA cache write and decode (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under
``bit_mla_kv_qmla_gb300`` never imports, links or runs it, and it shares no code
with that library: ``qmla_oracle.cpp`` restates the quantizer, the packed block
layout and the attention math from their written specification (the pages
"QuantMLA: INT4 (and INT2) for both halves of the MLA cache", TL;DR, flowchart
and "Key findings"; the parameters the pages leave open are fixed in the
specification comment of ``include/qmla.h``).

The C++ source is compiled here with g++ into ``oracle/_build/liboracle.so``
(``-frounding-math -ffp-contract=off``: the quantizer relies on the FPU's
directed rounding and on unfused multiply/add).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmla_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

C4R4, C2R4, BF16, C4R2, C2R2 = 0, 1, 2, 3, 4
CONTENT_BITS = {C4R4: 4, C2R4: 2, C4R2: 4, C2R2: 2}
ROPE_BITS = {C4R4: 4, C2R4: 4, C4R2: 2, C2R2: 2}
RN, RD, RU = 0, 1, 2
D_C, D_R, GROUP, SLOTS = 512, 64, 64, 64


def build(force: bool = False) -> str:
    """Compile the oracle shared library if it is missing or stale."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-frounding-math", "-ffp-contract=off",
               "-fPIC", "-shared", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f32, f64, u16 = (ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                       ctypes.c_double, ctypes.c_uint16)
            L.oracle_f32_to_f16.argtypes = [f32, i32]
            L.oracle_f32_to_f16.restype = u16
            L.oracle_f16_to_f32.argtypes = [u16]
            L.oracle_f16_to_f32.restype = f32
            L.oracle_f32_sub.argtypes = [f32, f32, i32]
            L.oracle_f32_sub.restype = f32
            L.oracle_f32_div.argtypes = [f32, f32, i32]
            L.oracle_f32_div.restype = f32
            L.oracle_f64_sub.argtypes = [f64, f64, i32]
            L.oracle_f64_sub.restype = f64
            L.oracle_f64_div.argtypes = [f64, f64, i32]
            L.oracle_f64_div.restype = f64
            L.oracle_grid_for.argtypes = [f32, f32, i32, P, P, P]
            L.oracle_grid_for.restype = None
            L.oracle_block_bytes.argtypes = [i32]
            L.oracle_block_bytes.restype = ctypes.c_size_t
            L.oracle_f32_to_f16_array.argtypes = [P, i64, i32, P]
            L.oracle_f32_to_f16_array.restype = None
            L.oracle_quantize_group.argtypes = [P, i32, i32, P, P, P]
            L.oracle_quantize_group.restype = None
            L.oracle_pack_codes.argtypes = [P, i32, i32, P]
            L.oracle_pack_codes.restype = None
            L.oracle_unpack_codes.argtypes = [P, i32, i32, P]
            L.oracle_unpack_codes.restype = None
            L.oracle_append.argtypes = [i32, P, i64, P, i32, P, i32, i32, P, P]
            L.oracle_append.restype = i32
            L.oracle_read_token.argtypes = [i32, P, i32, P]
            L.oracle_read_token.restype = None
            L.oracle_decode.argtypes = [i32, P, P, i32, P, i32, i32, P, P, f64, P, P]
            L.oracle_decode.restype = None
            L.oracle_merge.argtypes = [i32, i32, P, P, P, P]
            L.oracle_merge.restype = None
            L.oracle_decode_split.argtypes = [i32, P, P, i32, i32, P, P, f64, i32, P, P]
            L.oracle_decode_split.restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    """bfloat16 data as raw uint16 bits (accepts uint16 arrays or torch bf16)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy()
                                    .view(np.uint16))
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16
    return a


def block_bytes(fmt: int) -> int:
    return int(lib().oracle_block_bytes(fmt))


def f32_to_f16(x: np.ndarray, mode: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_f16_array(_ptr(x), x.size, mode, _ptr(out))
    return out


def f16_to_f32(h: int) -> float:
    return float(lib().oracle_f16_to_f32(int(h)))


def f32_sub(a: float, b: float, mode: int) -> float:
    return float(lib().oracle_f32_sub(a, b, mode))


def f32_div(a: float, b: float, mode: int) -> float:
    return float(lib().oracle_f32_div(a, b, mode))


def f64_sub(a: float, b: float, mode: int) -> float:
    return float(lib().oracle_f64_sub(a, b, mode))


def f64_div(a: float, b: float, mode: int) -> float:
    return float(lib().oracle_f64_div(a, b, mode))


def grid_for(mn: float, mx: float, levels: int):
    """(E, Z, M) of the binary16-exact grid of a group with range [mn, mx]."""
    E = ctypes.c_int(0)
    Z = ctypes.c_double(0)
    M = ctypes.c_double(0)
    lib().oracle_grid_for(mn, mx, levels, ctypes.byref(E), ctypes.byref(Z), ctypes.byref(M))
    return E.value, Z.value, M.value


def quantize_group(x: np.ndarray, bits: int):
    """Return (scale_bits, zero_bits, codes[n]) for one group of float32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    codes = np.zeros(x.size, np.uint8)
    lib().oracle_quantize_group(_ptr(x), x.size, bits, _ptr(s), _ptr(z), _ptr(codes))
    return int(s[0]), int(z[0]), codes


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(codes.size * bits // 8, np.uint8)
    lib().oracle_pack_codes(_ptr(codes), codes.size, bits, _ptr(out))
    return out


def unpack_codes(packed: np.ndarray, nch: int, bits: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros(nch, np.uint8)
    lib().oracle_unpack_codes(_ptr(packed), nch, bits, _ptr(out))
    return out


def append(fmt: int, blocks: np.ndarray, block_table: np.ndarray, positions: np.ndarray,
           latent, rope) -> int:
    """Quantize-and-pack into ``blocks`` (uint8, modified in place).

    latent: [B][n_new][512] bf16 bits, rope: [B][n_new][64] bf16 bits.
    Returns the number of skipped tokens."""
    lat = _u16(latent)
    rp = _u16(rope)
    assert blocks.dtype == np.uint8 and blocks.flags["C_CONTIGUOUS"]
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    B, n_new = lat.shape[0], lat.shape[1]
    nb = blocks.size // block_bytes(fmt)
    return int(lib().oracle_append(fmt, _ptr(blocks), nb, _ptr(bt), bt.shape[1], _ptr(pos),
                                   B, n_new, _ptr(lat), _ptr(rp)))


def read_token(fmt: int, block: np.ndarray, slot: int) -> np.ndarray:
    block = np.ascontiguousarray(block, dtype=np.uint8)
    out = np.zeros(D_C + D_R, np.float32)
    lib().oracle_read_token(fmt, _ptr(block), slot, _ptr(out))
    return out


def decode(fmt: int, blocks: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray,
           q_c, q_r, scale: float):
    """Return (O [B][H][512] float64, LSE [B][H] float64)."""
    qc = _u16(q_c)
    qr = _u16(q_r)
    B, H = qc.shape[0], qc.shape[1]
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((B, H, D_C), np.float64)
    lse = np.zeros((B, H), np.float64)
    lib().oracle_decode(fmt, _ptr(blocks), _ptr(bt), bt.shape[1], _ptr(sl), B, H, _ptr(qc),
                        _ptr(qr), float(scale), _ptr(out), _ptr(lse))
    return out, lse


def decode_split(fmt: int, blocks: np.ndarray, table_row: np.ndarray, L: int, q_c, q_r,
                 scale: float, nsplit: int):
    """One sequence, context cut into ``nsplit`` ranges and merged.  q: [H][...]."""
    qc = _u16(q_c)
    qr = _u16(q_r)
    H = qc.shape[0]
    row = np.ascontiguousarray(table_row, dtype=np.int32)
    out = np.zeros((H, D_C), np.float64)
    lse = np.zeros(H, np.float64)
    lib().oracle_decode_split(fmt, _ptr(blocks), _ptr(row), int(L), H, _ptr(qc), _ptr(qr),
                              float(scale), int(nsplit), _ptr(out), _ptr(lse))
    return out, lse


def merge(part_o: np.ndarray, part_lse: np.ndarray):
    """part_o [n][H][512], part_lse [n][H] -> (O [H][512], LSE [H])."""
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    n, H = pl.shape
    out = np.zeros((H, D_C), np.float64)
    lse = np.zeros(H, np.float64)
    lib().oracle_merge(n, H, _ptr(po), _ptr(pl), _ptr(out), _ptr(lse))
    return out, lse


def decode_multi(fmt: int, blocks: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray,
                 q_c, q_r, scale: float):
    """Decode of q_len query tokens per sequence, the last q_len tokens of the
    cache (q_c [B][q_len][H][512], q_r [B][q_len][H][64]).  Query i sits at
    position L - q_len + i and attends causally: to tokens 0 .. L - q_len + i,
    i.e. the decode over the first L - q_len + 1 + i tokens (none when that is
    not positive: O = 0, LSE = -inf).  Returns (O [B][q_len][H][512],
    LSE [B][q_len][H]) in float64.  The multi-token query step is not in the
    pages; it is plain causal attention over the same cache, so it reuses
    ``decode`` on each query's prefix."""
    qc = _u16(q_c)
    qr = _u16(q_r)
    B, Q, H = qc.shape[0], qc.shape[1], qc.shape[2]
    lens = np.asarray(seq_lens, dtype=np.int64)
    out = np.zeros((B, Q, H, D_C), np.float64)
    lse = np.full((B, Q, H), -np.inf, np.float64)
    for i in range(Q):
        li = np.maximum(lens - (Q - 1 - i), 0).astype(np.int32)
        o, l = decode(fmt, blocks, block_table, li, qc[:, i], qr[:, i], scale)
        out[:, i] = o
        lse[:, i] = l
    return out, lse
