"""Host-side checks of the C-ABI library (no GPU needed, nothing launched).

The library must load, export every function include/qmla.h declares, and
reject bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmla.h")


@pytest.fixture(scope="module")
def lib():
    from bit_mla_kv_qmla_gb300 import build as B
    B.build()
    from bit_mla_kv_qmla_gb300 import _lib
    return _lib.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(qmla_[a-z_0-9]+)\s*\(", src, re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert names == sorted(["qmla_block_bytes", "qmla_append", "qmla_append_advance",
                            "qmla_decode_workspace_bytes", "qmla_decode_multi",
                            "qmla_decode", "qmla_decode_noalloc", "qmla_decode_timeout_test",
                            "qmla_decode_step_layout", "qmla_decode_step_workspace_bytes",
                            "qmla_decode_step", "qmla_read_status", "qmla_error_string"])


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    # and nothing that looks like the oracle
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    assert "oracle" not in out


def test_block_bytes(lib):
    assert [lib.qmla_block_bytes(f) for f in (0, 1, 2, 3, 4, 5, -1)] == [
        20736, 12544, 73728, 19712, 11520, 0, 0]


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -99):
        assert lib.qmla_error_string(code)


P = ctypes.c_void_p


def _fake(n):
    # aligned host buffer used only as a non-null pointer value; never dereferenced
    buf = ctypes.create_string_buffer(n + 512)
    addr = (ctypes.addressof(buf) + 511) // 512 * 512
    return buf, addr


@pytest.mark.parametrize("entry", ["qmla_append", "qmla_append_advance"])
def test_append_rejects_bad_arguments(lib, entry):
    keep, p = _fake(1024)
    ok_args = dict(format=0, blocks=p, num_blocks=4, table=p, maxb=2, pos=p, batch=1, n_new=1,
                   lat=p, rope=p, status=p, stream=None)
    fn = getattr(lib, entry)

    def call(**kw):
        a = dict(ok_args, **kw)
        return fn(a["format"], a["blocks"], a["num_blocks"], a["table"], a["maxb"], a["pos"],
                  a["batch"], a["n_new"], a["lat"], a["rope"], a["status"], a["stream"])
    assert call(format=7) == -2
    assert call(batch=-1) == -1
    assert call(n_new=-1) == -1
    assert call(num_blocks=0) == -1
    assert call(blocks=None) == -1
    assert call(lat=None) == -1
    assert call(status=None) == -1
    assert call(blocks=p + 16) == -1  # pool must be 256-byte aligned
    assert call(maxb=0) == -1
    assert call(batch=0) == 0  # nothing to do, nothing launched


def test_decode_rejects_bad_arguments(lib):
    keep, p = _fake(4096)

    def call(fmt=0, heads=16, batch=1, blocks=p, ws=p, qc=p, out=p, wsb=1 << 20, maxb=4):
        return lib.qmla_decode(fmt, blocks, 4, p, maxb, p, 256, batch, heads, qc, p,
                               ctypes.c_float(0.1), out, p, ws, wsb, p, None)
    assert call(fmt=5) == -2
    assert call(heads=17) == -2
    assert call(heads=512) == -2
    assert call(batch=-1) == -1
    assert call(blocks=None) == -1
    assert call(qc=p + 8) == -1      # queries must be 16-byte aligned
    assert call(ws=p + 128) == -1    # workspace must be 256-byte aligned
    assert call(maxb=0) == -1
    assert call(batch=0) == 0


def test_decode_multi_rejects_bad_arguments(lib):
    keep, p = _fake(4096)

    def call(heads=16, q_len=2, batch=1, fmt=0):
        return lib.qmla_decode_multi(fmt, p, 4, p, 4, p, 256, batch, heads, q_len, p, p,
                                     ctypes.c_float(0.1), p, p, p, 1 << 20, p, None)
    assert call(q_len=0) == -1
    assert call(heads=0) == -1
    assert call(heads=64, q_len=5) == -2   # 320 query rows: not served
    assert call(heads=17, q_len=1) == -2
    assert call(batch=0) == 0


def test_read_status_null(lib):
    assert lib.qmla_read_status(None, None) == -1


def test_decode_noalloc_rejects_bad_arguments(lib):
    # every rejection below returns before the library touches the device
    keep, p = _fake(4096)

    def call(fmt=0, heads=128, batch=1, blocks=p, qc=p, out=p, lse=p, status=p, maxb=4, nb=4):
        return lib.qmla_decode_noalloc(fmt, blocks, nb, p, maxb, p, 256, batch, heads, qc, p,
                                       ctypes.c_float(0.1), out, lse, status, None)
    assert call(fmt=5) == -2
    assert call(fmt=-1) == -2
    assert call(heads=17) == -2
    assert call(heads=512) == -2
    assert call(batch=-1) == -1
    assert call(nb=0) == -1
    assert call(blocks=None) == -1
    assert call(qc=None) == -1
    assert call(out=None) == -1
    assert call(status=None) == -1
    assert call(blocks=p + 16) == -1   # pool must be 256-byte aligned
    assert call(qc=p + 8) == -1        # queries must be 16-byte aligned
    assert call(lse=p + 2) == -1       # lse must be 4-byte aligned
    assert call(maxb=0) == -1
    assert call(batch=0) == 0          # nothing to do, nothing launched
    # the formats qmla_decode serves are accepted up to the device query
    for fmt in (0, 1, 2, 3, 4):
        assert call(fmt=fmt, batch=0) == 0


def _step_offsets_by_rule(batch, heads, n_new):
    # the packing rule stated in qmla.h: regions in order, each at the first
    # multiple of 256 at or after the end of the previous one
    def up(x):
        return -(-x // 256) * 256
    sizes_in = ([batch * n_new * 512 * 2, batch * n_new * 64 * 2] if n_new else []) + \
        [batch * heads * 512 * 2, batch * heads * 64 * 2]
    offs, end = [], 0
    for n in sizes_in:
        offs.append(up(end))
        end = offs[-1] + n
    lat, rope = (offs[0], offs[1]) if n_new else (0, 0)
    qc, qr = offs[-2], offs[-1]
    out, lse = 0, up(batch * heads * 512 * 2)
    return (lat, rope, qc, qr, end, out, lse, lse + batch * heads * 4)


@pytest.mark.parametrize("batch,heads,n_new", [(4, 128, 1), (32, 16, 1), (3, 16, 0), (1, 128, 5),
                                                (7, 48, 3), (0, 16, 1)])
def test_decode_step_layout_follows_the_stated_rule(lib, batch, heads, n_new):
    o = (ctypes.c_size_t * 8)()
    assert lib.qmla_decode_step_layout(batch, heads, n_new, o) == 0
    assert tuple(o) == _step_offsets_by_rule(batch, heads, n_new)


def test_decode_step_layout_rejects_bad_arguments(lib):
    o = (ctypes.c_size_t * 8)()
    assert lib.qmla_decode_step_layout(-1, 16, 1, o) == -1
    assert lib.qmla_decode_step_layout(1, -16, 1, o) == -1
    assert lib.qmla_decode_step_layout(1, 16, -1, o) == -1
    assert lib.qmla_decode_step_layout(1, 16, 1, None) == -1


def test_decode_step_rejects_bad_arguments(lib):
    # every rejection below returns before the library touches the device
    keep, p = _fake(4096)

    def call(fmt=0, heads=128, batch=1, n_new=1, h_in=p, h_out=p, ws=p, msl=256):
        return lib.qmla_decode_step(fmt, p, 4, p, 4, p, msl, batch, heads, n_new, h_in,
                                    ctypes.c_float(0.1), h_out, ws, 1 << 20, p, None)
    assert call(batch=-1) == -1
    assert call(heads=-16) == -1
    assert call(n_new=-1) == -1
    assert call(h_in=None) == -1
    assert call(h_out=None) == -1
    assert call(ws=None) == -1
    assert call(ws=p + 128) == -1     # workspace must be 256-byte aligned
    assert call(fmt=5) == -2
    assert call(heads=17) == -2
    assert call(msl=-1) == -1
    assert lib.qmla_decode_step_workspace_bytes(0, 1, 16, -1, 256) == 0
    assert lib.qmla_decode_step_workspace_bytes(5, 1, 16, 1, 256) == 0


def test_host_plan_restatement_covers_every_block_once():
    """The tests' host restatement of the split plan (used to pick the
    full-size parity samples at worker boundaries): every block of every
    sequence in exactly one piece, pieces in order, workers in order, and the
    worker count capped by the total extent."""
    import random
    from helpers import boundary_sequences, plan_pieces
    rng = random.Random(5)
    for workers, cost in ((76, 6), (76, 2), (152, 3), (7, 0)):
        nb = [rng.choice([0, 1, 2, 5, 64, 300]) for _ in range(50)]
        plan = plan_pieces(nb, workers, cost)
        seen = []
        for b, pcs in enumerate(plan):
            assert sum(j1 - j0 for _, j0, j1 in pcs) == nb[b]
            pos = 0
            for wk, j0, j1 in pcs:
                assert j0 == pos and j1 > j0
                pos = j1
                seen.append(wk)
        assert seen == sorted(seen) and max(seen) < min(workers, sum(n + cost for n in nb if n))
        bs = boundary_sequences(nb, workers, cost)
        assert all(len(plan[b]) > 1 for b in bs[:-1])
