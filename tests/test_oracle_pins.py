"""Pins of the CPU oracle to facts fixed outside the oracle itself.

The oracle (oracle/qmla_oracle.cpp) is what the CUDA path is compared with,
so it is checked here against: IEEE conversions as numpy and exact rational
arithmetic compute them, the bounds the quantizer must meet by construction,
a brute-force nearest-code search, a hand-worked packing fixture, the
byte-count formula of the layout, exact-grid recovery, library softmax /
log-sum-exp on exactly representable inputs, closed forms (L = 1, q = 0,
identical tokens, a dominant token), and invariances (split/merge, block-table
permutation, bulk vs incremental append, masking of a partial last block).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from bit_mla_kv_qmla_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# binary32 -> binary16 conversion and directed binary32 arithmetic
# ----------------------------------------------------------------------------

def _probe_floats(n_random=400_000, seed=0):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=n_random, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # every finite binary16 value, its binary32 neighbours and the midpoints
    h = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    h = h[np.isfinite(h)].astype(np.float32)
    up = np.nextafter(h, np.float32(np.inf))
    dn = np.nextafter(h, np.float32(-np.inf))
    hs = np.sort(np.unique(h.astype(np.float64)))
    mids = ((hs[1:] + hs[:-1]) / 2).astype(np.float32)
    extra = np.array([65504, 65519.99, 65520, 65536, 1e9, -65520, 5.96e-8, 2.98e-8,
                      6.1e-5, 0.0, -0.0], np.float32)
    return np.concatenate([x, h, up, dn, mids, extra]).astype(np.float32)


def test_f16_round_nearest_matches_numpy():
    x = _probe_floats()
    ours = oracle.f32_to_f16(x, oracle.RN)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_directed_bracket_and_adjacency():
    x = _probe_floats(seed=1)
    rd = oracle.f32_to_f16(x, oracle.RD).view(np.float16).astype(np.float64)
    ru = oracle.f32_to_f16(x, oracle.RU).view(np.float16).astype(np.float64)
    rn = oracle.f32_to_f16(x, oracle.RN).view(np.float16).astype(np.float64)
    xd = x.astype(np.float64)
    assert np.all(rd <= xd) and np.all(ru >= xd)
    exact = rn == xd
    assert np.all(rd[exact] == xd[exact]) and np.all(ru[exact] == xd[exact])
    ne = ~exact
    # adjacent binary16 values: RU is the successor of RD
    succ = np.nextafter(rd[ne].astype(np.float16), np.float16(np.inf)).astype(np.float64)
    assert np.array_equal(succ, ru[ne])
    assert np.all((rn[ne] == rd[ne]) | (rn[ne] == ru[ne]))


def _exact_bracket(exact: Fraction, rd: float, ru: float) -> None:
    assert Fraction(rd) <= exact <= Fraction(ru)
    if Fraction(rd) == exact:
        assert rd == ru
    else:
        assert np.nextafter(np.float32(rd), np.float32(np.inf)) == np.float32(ru)


def test_directed_binary32_sub_div():
    rng = np.random.default_rng(2)
    a = (rng.standard_normal(3000) * np.exp(rng.uniform(-8, 8, 3000))).astype(np.float32)
    b = (rng.standard_normal(3000) * np.exp(rng.uniform(-8, 8, 3000))).astype(np.float32)
    for x, y in zip(a.tolist(), b.tolist()):
        x, y = float(np.float32(x)), float(np.float32(y))
        _exact_bracket(Fraction(x) - Fraction(y), oracle.f32_sub(x, y, oracle.RD),
                       oracle.f32_sub(x, y, oracle.RU))
        if y != 0.0:
            _exact_bracket(Fraction(x) / Fraction(y), oracle.f32_div(x, y, oracle.RD),
                           oracle.f32_div(x, y, oracle.RU))
        rn = oracle.f32_sub(x, y, oracle.RN)
        assert rn == float(np.float32(x) - np.float32(y))


# ----------------------------------------------------------------------------
# the group quantizer
# ----------------------------------------------------------------------------

def _groups(rng, n_groups=600):
    out = []
    for k in range(n_groups):
        kind = k % 7
        if kind == 0:
            x = rng.standard_normal(64)
        elif kind == 1:
            x = rng.standard_normal(64) * np.where(rng.random(64) < 0.05, 30.0, 1.0)
        elif kind == 2:
            x = rng.uniform(-1e-3, 1e-3, 64)
        elif kind == 3:
            x = rng.uniform(100, 3000, 64)
        elif kind == 4:
            x = -np.abs(rng.standard_normal(64)) * 7
        elif kind == 5:
            x = np.full(64, rng.standard_normal())
            x[rng.integers(0, 64)] += rng.choice([0.0, 1e-2])
        else:
            # binary16 subnormal range: bfloat16 values there are mostly not
            # representable in binary16, so the rounding direction matters
            x = rng.uniform(-4e-6, 4e-6, 64)
        # round to bfloat16 like the cache inputs
        t = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float32)
        out.append(t.numpy().astype(np.float32))
    return out


def _f16(bits):
    return float(np.uint16(bits).view(np.float16))


def _dequant(codes, s, z):
    # binary32 multiply then add, each rounded (numpy float32 ops)
    return (codes.astype(np.float32) * np.float32(s)) + np.float32(z)


@pytest.mark.parametrize("bits", [4, 2])
def test_quantizer_bounds_and_roundtrip(bits):
    rng = np.random.default_rng(10 + bits)
    levels = (1 << bits) - 1
    for x in _groups(rng):
        sb, zb, codes = oracle.quantize_group(x, bits)
        s, z = _f16(sb), _f16(zb)
        assert codes.max() <= levels and s > 0
        mn, mx = float(x.min()), float(x.max())
        assert z <= mn
        assert z + levels * s >= mx  # exact in float64 (both binary16 values)
        xh = _dequant(codes, s, z).astype(np.float64)
        span = np.maximum(np.abs(x.astype(np.float64)), abs(z) + levels * s)
        slack = 3 * np.spacing(span.astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(x - xh) <= s / 2 + slack)


@pytest.mark.parametrize("bits", [4, 2])
def test_quantizer_grid_is_binary16_exact(bits):
    """Every dequantized value code*s + z is exactly a binary16 number, so a
    binary16 tensor-core operand carries it without rounding."""
    rng = np.random.default_rng(50 + bits)
    levels = (1 << bits) - 1
    for x in _groups(rng, 400):
        sb, zb, _ = oracle.quantize_group(x, bits)
        s, z = _f16(sb), _f16(zb)
        grid = [Fraction(z) + c * Fraction(s) for c in range(levels + 1)]
        as16 = np.array([float(g) for g in grid]).astype(np.float16)
        assert all(Fraction(float(h)) == g for h, g in zip(as16, grid))


@pytest.mark.parametrize("bits", [4, 2])
def test_quantizer_step_is_close_to_range_over_levels(bits):
    """For groups that contain zero, the grid step is at most (1 + 16/1023)
    times the ideal (max - min) / levels: the power-of-two unit can be no
    coarser than max(|min|, max) / 1023.  The unit cannot go below binary16's
    smallest subnormal 2^-24, which may add up to two such units."""
    rng = np.random.default_rng(60 + bits)
    levels = (1 << bits) - 1
    n = 0
    for x in _groups(rng, 700):
        mn, mx = float(x.min()), float(x.max())
        if not (mn < 0.0 < mx):
            continue
        n += 1
        sb, _, _ = oracle.quantize_group(x, bits)
        ideal = (mx - mn) / levels
        bound = max(ideal * (1 + 16 / 1023), ideal + 2 * 2.0**-24)
        assert _f16(sb) <= bound * (1 + 1e-12)
    assert n > 100


def test_directed_binary64_sub_div():
    rng = np.random.default_rng(4)
    a = rng.standard_normal(2000) * np.exp(rng.uniform(-30, 30, 2000))
    b = rng.standard_normal(2000) * np.exp(rng.uniform(-30, 30, 2000))
    for x, y in zip(a.tolist(), b.tolist()):
        for op, fr in ((oracle.f64_sub, Fraction(x) - Fraction(y)),
                       (oracle.f64_div, Fraction(x) / Fraction(y))):
            rd, ru = op(x, y, oracle.RD), op(x, y, oracle.RU)
            assert Fraction(rd) <= fr <= Fraction(ru)
            if Fraction(rd) == fr:
                assert rd == ru
            else:
                assert np.nextafter(rd, np.inf) == ru


@pytest.mark.parametrize("bits", [4, 2])
def test_quantizer_picks_nearest_code_bruteforce(bits):
    rng = np.random.default_rng(20 + bits)
    levels = (1 << bits) - 1
    for x in _groups(rng, 300):
        sb, zb, codes = oracle.quantize_group(x, bits)
        if sb == 0:
            continue
        s, z = _f16(sb), _f16(zb)
        grid = _dequant(np.arange(levels + 1), s, z).astype(np.float64)
        err_all = np.abs(x.astype(np.float64)[:, None] - grid[None, :])
        best = err_all.min(axis=1)
        chosen = err_all[np.arange(64), codes]
        tol = 2 * np.spacing(np.float32(abs(z) + levels * s)).astype(np.float64)
        assert np.all(chosen <= best + tol)


@pytest.mark.parametrize("bits", [4, 2])
def test_quantizer_recovers_exact_grid(bits):
    g = torch.Generator().manual_seed(30 + bits)
    for _ in range(50):
        vals, codes, zero = W.exact_grid_group(g, bits)
        sb, zb, got = oracle.quantize_group(vals.numpy(), bits)
        assert _f16(sb) == 0.125 and _f16(zb) == zero
        assert np.array_equal(got, codes.numpy().astype(np.uint8))


def test_quantizer_constant_group():
    for v in [0.0, 1.5, -3.25, 1000.0]:
        sb, zb, codes = oracle.quantize_group(np.full(64, v, np.float32), 4)
        assert _f16(sb) > 0 and np.all(_dequant(codes, _f16(sb), _f16(zb)) == np.float32(v))


def test_packing_golden():
    with open(os.path.join(GOLDEN, "packing.txt")) as f:
        rows = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for ln in rows:
        bits, codes, want = [p.strip() for p in ln.split("|")]
        codes = np.array([int(c) for c in codes.split()], np.uint8)
        want = np.array([int(b, 16) for b in want.split()], np.uint8)
        got = oracle.pack_codes(codes, int(bits))
        assert np.array_equal(got, want)
        assert np.array_equal(oracle.unpack_codes(got, codes.size, int(bits)), codes)


@pytest.mark.parametrize("bits", [4, 2])
def test_pack_unpack_roundtrip(bits):
    rng = np.random.default_rng(40 + bits)
    codes = rng.integers(0, 1 << bits, 64).astype(np.uint8)
    assert np.array_equal(oracle.unpack_codes(oracle.pack_codes(codes, bits), 64, bits), codes)


# ----------------------------------------------------------------------------
# block layout
# ----------------------------------------------------------------------------

def test_block_bytes_formula():
    # bytes/token = d_c*b_c/8 + d_r*b_r/8 + 4*(d_c/G + d_r/G)  (fp16 scale + zero per group)
    for fmt, bc, br in [(oracle.C4R4, 4, 4), (oracle.C2R4, 2, 4), (oracle.C4R2, 4, 2),
                        (oracle.C2R2, 2, 2)]:
        per_tok = 512 * bc // 8 + 64 * br // 8 + 4 * (512 // 64 + 64 // 64)
        assert oracle.block_bytes(fmt) == 64 * per_tok
    assert oracle.block_bytes(oracle.BF16) == 64 * 576 * 2
    assert (oracle.block_bytes(oracle.C4R4), oracle.block_bytes(oracle.C2R4)) == (20736, 12544)
    assert (oracle.block_bytes(oracle.C4R2), oracle.block_bytes(oracle.C2R2)) == (19712, 11520)
    ratio = oracle.block_bytes(oracle.BF16) / oracle.block_bytes(oracle.C4R4)
    assert abs(ratio - 3.5556) < 1e-3  # the pages report 3.59x for their own layout
    assert oracle.block_bytes(5) == 0 and oracle.block_bytes(-1) == 0


def _one_token(seed):
    g = torch.Generator().manual_seed(seed)
    lat = torch.randn(1, 1, 512, generator=g).to(torch.bfloat16)
    rope = torch.randn(1, 1, 64, generator=g).to(torch.bfloat16)
    return lat, rope


# (format, content code bytes per group, RoPE code bytes per half, half bytes):
# a half is 4 content groups x 64 tokens, then 64 tokens of RoPE codes, then
# 4 x 64 content scale/zero words
_LAYOUTS = [(oracle.C4R4, 32, 16, 10240), (oracle.C2R4, 16, 16, 6144),
            (oracle.C4R2, 32, 8, 9728), (oracle.C2R2, 16, 8, 5632)]


@pytest.mark.parametrize("fmt,cb,rb,half", _LAYOUTS)
def test_layout_offsets_match_spec(fmt, cb, rb, half):
    """A token written to slot 5 touches exactly the byte ranges the layout
    specification assigns to slot 5, and those ranges hold the quantizer's
    output for the right group."""
    lat, rope = _one_token(7)
    blocks = np.zeros(oracle.block_bytes(fmt), np.uint8)
    slot = 5
    oracle.append(fmt, blocks, np.zeros((1, 1), np.int32), np.array([slot], np.int32), lat, rope)
    touched = np.zeros_like(blocks, dtype=bool)
    xl = lat.float().numpy()[0, 0]
    xr = rope.float().numpy()[0, 0]
    bits, rbits = cb // 8, rb // 4
    assert half == 4 * 64 * cb + 64 * rb + 1024
    for grp in range(8):
        h, gi = divmod(grp, 4)
        c0 = h * half + (gi * 64 + slot) * cb
        sz0 = h * half + 4 * 64 * cb + 64 * rb + (gi * 64 + slot) * 4
        touched[c0:c0 + cb] = True
        touched[sz0:sz0 + 4] = True
        sb, zb, codes = oracle.quantize_group(xl[grp * 64:(grp + 1) * 64], bits)
        assert np.array_equal(blocks[c0:c0 + cb], oracle.pack_codes(codes, bits))
        assert blocks[sz0:sz0 + 4].view(np.uint16).tolist() == [sb, zb]
    sb, zb, codes = oracle.quantize_group(xr, rbits)
    for h in range(2):
        r0 = h * half + 4 * 64 * cb + slot * rb
        touched[r0:r0 + rb] = True
        assert np.array_equal(blocks[r0:r0 + rb],
                              oracle.pack_codes(codes[32 * h:32 * h + 32], rbits))
    rs = 2 * half + slot * 4
    touched[rs:rs + 4] = True
    assert blocks[rs:rs + 4].view(np.uint16).tolist() == [sb, zb]
    assert not np.any(blocks[~touched])


@pytest.mark.parametrize("fmt_r4,fmt_r2", [(oracle.C4R4, oracle.C4R2), (oracle.C2R4, oracle.C2R2)])
def test_rope_int2_changes_only_the_rope_key(fmt_r4, fmt_r2):
    """The RoPE-at-INT2 formats dequantize the content latent exactly as their
    RoPE-INT4 counterparts do; the RoPE key stays within the 2-bit bound
    |x - x_hat| <= s/2 (+ rounding) of its own group."""
    lat, rope = _one_token(11)
    out = {}
    for fmt in (fmt_r4, fmt_r2):
        blocks = np.zeros(oracle.block_bytes(fmt), np.uint8)
        oracle.append(fmt, blocks, np.zeros((1, 1), np.int32), np.array([3], np.int32), lat, rope)
        out[fmt] = oracle.read_token(fmt, blocks, 3)
    assert np.array_equal(out[fmt_r4][:512], out[fmt_r2][:512])
    xr = rope.float().numpy()[0, 0]
    sb, zb, codes = oracle.quantize_group(xr, 2)
    assert codes.max() <= 3
    s = float(np.array([sb], np.uint16).view(np.float16)[0])
    err2 = np.abs(out[fmt_r2][512:] - xr)
    err4 = np.abs(out[fmt_r4][512:] - xr)
    assert np.all(err2 <= s / 2 + 1e-6 * (1 + np.abs(xr)))
    assert err2.max() > err4.max()


def test_layout_offsets_bf16():
    lat, rope = _one_token(8)
    blocks = np.zeros(oracle.block_bytes(oracle.BF16), np.uint8)
    slot = 9
    oracle.append(oracle.BF16, blocks, np.zeros((1, 1), np.int32), np.array([slot], np.int32),
                  lat, rope)
    u = blocks.view(np.uint16)
    lb = lat.view(torch.int16).numpy().view(np.uint16)[0, 0]
    rb = rope.view(torch.int16).numpy().view(np.uint16)[0, 0]
    for grp in range(8):
        h, gi = divmod(grp, 4)
        o = (h * 36864 + (gi * 64 + slot) * 128) // 2
        assert np.array_equal(u[o:o + 64], lb[grp * 64:(grp + 1) * 64])
    for h in range(2):
        o = (h * 36864 + 32768 + slot * 64) // 2
        assert np.array_equal(u[o:o + 32], rb[32 * h:32 * h + 32])


# ----------------------------------------------------------------------------
# decode
# ----------------------------------------------------------------------------

def _build_cache(fmt, lat, rope, lens, seed=0, permute=True):
    """Pool + block table for sequences (lat [B][Lmax][512] bf16)."""
    B = lat.shape[0]
    need = [max(1, (L + 63) // 64) for L in lens]
    total = sum(need)
    perm = (np.random.default_rng(seed).permutation(total) if permute else np.arange(total))
    table = np.full((B, max(need)), -1, np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    blocks = np.zeros(total * oracle.block_bytes(fmt), np.uint8)
    for b, L in enumerate(lens):
        if L:
            oracle.append(fmt, blocks, table[b:b + 1], np.array([0], np.int32),
                          lat[b:b + 1, :L].contiguous(), rope[b:b + 1, :L].contiguous())
    return blocks, table


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def test_decode_bf16_matches_library_softmax():
    from scipy.special import logsumexp, softmax
    B, H, lens = 3, 4, [37, 70, 128]
    lat, rope = _rand((B, 128, 512), 1), _rand((B, 128, 64), 2)
    qc, qr = _rand((B, H, 512), 3), _rand((B, H, 64), 4)
    blocks, table = _build_cache(oracle.BF16, lat, rope, lens)
    scale = 1 / math.sqrt(192)
    O, lse = oracle.decode(oracle.BF16, blocks, table, np.array(lens), qc, qr, scale)
    for b, L in enumerate(lens):
        K = np.concatenate([lat[b, :L].double().numpy(), rope[b, :L].double().numpy()], 1)
        Q = np.concatenate([qc[b].double().numpy(), qr[b].double().numpy()], 1)
        S = (Q @ K.T) * scale
        assert np.allclose(lse[b], logsumexp(S, axis=1), rtol=0, atol=1e-12)
        ref = softmax(S, axis=1) @ lat[b, :L].double().numpy()
        assert np.allclose(O[b], ref, rtol=0, atol=1e-12)


def _grid_tokens(B, L, bits_c, seed, bits_r=4):
    g = torch.Generator().manual_seed(seed)
    lat = torch.empty(B, L, 512)
    rope = torch.empty(B, L, 64)
    for b in range(B):
        for t in range(L):
            for grp in range(8):
                lat[b, t, grp * 64:(grp + 1) * 64] = W.exact_grid_group(g, bits_c)[0]
            rope[b, t] = W.exact_grid_group(g, bits_r)[0]
    return lat.to(torch.bfloat16), rope.to(torch.bfloat16)


@pytest.mark.parametrize("fmt", [oracle.C4R4, oracle.C2R4, oracle.C4R2, oracle.C2R2])
def test_quantized_decode_equals_bf16_on_exact_grid(fmt):
    bits, rbits = oracle.CONTENT_BITS[fmt], oracle.ROPE_BITS[fmt]
    B, H, lens = 2, 3, [70, 5]
    lat, rope = _grid_tokens(B, 70, bits, 50 + bits + (7 if rbits == 2 else 0), rbits)
    qc, qr = _rand((B, H, 512), 5), _rand((B, H, 64), 6)
    bq, tq = _build_cache(fmt, lat, rope, lens)
    bb, tb = _build_cache(oracle.BF16, lat, rope, lens)
    # quantize then dequantize is the identity on the grid
    bbytes = oracle.block_bytes(fmt)
    for t in (0, 3, 64, 69):
        blk = tq[0, t // 64]
        got = oracle.read_token(fmt, bq[blk * bbytes:(blk + 1) * bbytes], t % 64)
        want = np.concatenate([lat[0, t].float().numpy(), rope[0, t].float().numpy()])
        assert np.array_equal(got, want)
    s = 1 / math.sqrt(192)
    O1, l1 = oracle.decode(fmt, bq, tq, np.array(lens), qc, qr, s)
    O2, l2 = oracle.decode(oracle.BF16, bb, tb, np.array(lens), qc, qr, s)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


def test_decode_single_token_closed_form():
    lat, rope = _grid_tokens(1, 1, 4, 60)
    qc, qr = _rand((1, 2, 512), 7), _rand((1, 2, 64), 8)
    blocks, table = _build_cache(oracle.C4R4, lat, rope, [1])
    s = 0.37
    O, lse = oracle.decode(oracle.C4R4, blocks, table, np.array([1]), qc, qr, s)
    x = lat[0, 0].double().numpy()
    for h in range(2):
        assert np.array_equal(O[0, h], x)  # p = 1 exactly
        score = (qc[0, h].double().numpy() @ x + qr[0, h].double().numpy() @
                 rope[0, 0].double().numpy()) * s
        assert abs(lse[0, h] - score) <= 1e-12 * max(1.0, abs(score))


def test_decode_zero_query_is_mean():
    L = 77
    lat, rope = _grid_tokens(1, L, 4, 61)
    qc = torch.zeros(1, 2, 512, dtype=torch.bfloat16)
    qr = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    blocks, table = _build_cache(oracle.C4R4, lat, rope, [L])
    O, lse = oracle.decode(oracle.C4R4, blocks, table, np.array([L]), qc, qr, 0.1)
    mean = lat[0].double().numpy().mean(0)
    assert np.allclose(O[0, 0], mean, rtol=0, atol=1e-12)
    assert abs(lse[0, 0] - math.log(L)) < 1e-12


def test_decode_identical_tokens_weights_sum_to_one():
    L = 130
    one = _grid_tokens(1, 1, 4, 62)
    lat = one[0].repeat(1, L, 1)
    rope = _rand((1, L, 64), 9)  # scores differ, content does not
    qc, qr = _rand((1, 3, 512), 10), _rand((1, 3, 64), 11)
    blocks, table = _build_cache(oracle.C4R4, lat, rope, [L])
    O, _ = oracle.decode(oracle.C4R4, blocks, table, np.array([L]), qc, qr, 0.5)
    x = one[0][0, 0].double().numpy()
    for h in range(3):
        assert np.allclose(O[0, h], x, rtol=1e-12, atol=1e-12)


def test_decode_dominant_token():
    L = 50
    lat, rope = _grid_tokens(1, L, 4, 63)
    t_star = 17
    qc = (lat[:, t_star:t_star + 1].float() * 3.0).to(torch.bfloat16)  # q aligned with token 17
    qr = torch.zeros(1, 1, 64, dtype=torch.bfloat16)
    blocks, table = _build_cache(oracle.C4R4, lat, rope, [L])
    O, _ = oracle.decode(oracle.C4R4, blocks, table, np.array([L]), qc, qr, 1.0)
    x = lat[0].double().numpy()
    scores = x @ qc[0, 0].double().numpy()
    gap = scores[t_star] - np.max(np.delete(scores, t_star))
    assert gap > 30
    assert np.allclose(O[0, 0], x[t_star], atol=1e-9)


@pytest.mark.parametrize("fmt", [oracle.C4R4, oracle.C2R4, oracle.C2R2])
def test_split_merge_equals_unsplit(fmt):
    L = 64 * 7 + 13
    lat, rope = _rand((1, L, 512), 12), _rand((1, L, 64), 13)
    qc, qr = _rand((1, 4, 512), 14), _rand((1, 4, 64), 15)
    blocks, table = _build_cache(fmt, lat, rope, [L])
    s = 1 / math.sqrt(192)
    O, lse = oracle.decode(fmt, blocks, table, np.array([L]), qc, qr, s)
    for ns in (1, 2, 3, 8):
        O2, l2 = oracle.decode_split(fmt, blocks, table[0], L, qc[0], qr[0], s, ns)
        assert np.allclose(O2, O[0], rtol=0, atol=1e-12)
        assert np.allclose(l2, lse[0], rtol=0, atol=1e-12)


def test_block_permutation_invariance():
    L = 64 * 5 + 3
    lat, rope = _rand((1, L, 512), 16), _rand((1, L, 64), 17)
    qc, qr = _rand((1, 2, 512), 18), _rand((1, 2, 64), 19)
    b1, t1 = _build_cache(oracle.C4R4, lat, rope, [L], seed=1)
    b2, t2 = _build_cache(oracle.C4R4, lat, rope, [L], permute=False)
    assert not np.array_equal(t1, t2)
    O1, l1 = oracle.decode(oracle.C4R4, b1, t1, np.array([L]), qc, qr, 0.1)
    O2, l2 = oracle.decode(oracle.C4R4, b2, t2, np.array([L]), qc, qr, 0.1)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("fmt", [oracle.C4R4, oracle.C2R4, oracle.BF16, oracle.C4R2])
def test_incremental_append_equals_bulk(fmt):
    L = 100
    lat, rope = _rand((1, L, 512), 20), _rand((1, L, 64), 21)
    table = np.array([[1, 0]], np.int32)
    bulk = np.zeros(2 * oracle.block_bytes(fmt), np.uint8)
    oracle.append(fmt, bulk, table, np.array([0], np.int32), lat, rope)
    inc = np.zeros_like(bulk)
    for t in range(L):
        oracle.append(fmt, inc, table, np.array([t], np.int32), lat[:, t:t + 1].contiguous(),
                      rope[:, t:t + 1].contiguous())
    assert np.array_equal(bulk, inc)


def test_partial_last_block_is_masked():
    L = 70
    lat, rope = _rand((1, 128, 512), 22), _rand((1, 128, 64), 23)
    qc, qr = _rand((1, 2, 512), 24), _rand((1, 2, 64), 25)
    b1, t1 = _build_cache(oracle.C4R4, lat, rope, [L])
    b2 = b1.copy()
    # garbage in the unused slots 6..63 of the second block
    oracle.append(oracle.C4R4, b2, t1, np.array([L], np.int32),
                  _rand((1, 128 - L, 512), 26, 50.0), _rand((1, 128 - L, 64), 27, 50.0))
    assert not np.array_equal(b1, b2)
    O1, l1 = oracle.decode(oracle.C4R4, b1, t1, np.array([L]), qc, qr, 0.1)
    O2, l2 = oracle.decode(oracle.C4R4, b2, t1, np.array([L]), qc, qr, 0.1)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


def test_empty_sequence():
    lat, rope = _rand((1, 64, 512), 28), _rand((1, 64, 64), 29)
    qc, qr = _rand((1, 2, 512), 30), _rand((1, 2, 64), 31)
    blocks, table = _build_cache(oracle.C4R4, lat, rope, [0])
    O, lse = oracle.decode(oracle.C4R4, blocks, table, np.array([0]), qc, qr, 0.1)
    assert np.all(O == 0) and np.all(np.isneginf(lse))


def test_merge_matches_logaddexp():
    rng = np.random.default_rng(3)
    po = rng.standard_normal((3, 2, 512))
    pl = rng.standard_normal((3, 2)) * 4
    O, lse = oracle.merge(po, pl)
    L = np.logaddexp.reduce(pl, axis=0)
    assert np.allclose(lse, L, atol=1e-12)
    w = np.exp(pl - L)
    assert np.allclose(O, np.einsum("nh,nhc->hc", w, po), atol=1e-12)


def test_decode_multi_matches_explicit_causal_mask():
    """The multi-token query decode against its textbook form: the full score
    matrix of every query against every cached token, with the causal mask
    (query i at position L - q_len + i sees tokens up to it) applied before a
    library softmax; a sequence shorter than q_len leaves its first queries
    with nothing to attend (O = 0, LSE = -inf)."""
    from scipy.special import logsumexp, softmax
    B, Q, H, lens = 3, 3, 2, [70, 5, 1]
    lat, rope = _rand((B, 70, 512), 11), _rand((B, 70, 64), 12)
    qc, qr = _rand((B, Q, H, 512), 13), _rand((B, Q, H, 64), 14)
    blocks, table = _build_cache(oracle.BF16, lat, rope, lens)
    scale = 1 / math.sqrt(192)
    O, lse = oracle.decode_multi(oracle.BF16, blocks, table, np.array(lens), qc, qr, scale)
    for b, L in enumerate(lens):
        K = np.concatenate([lat[b, :L].double().numpy(), rope[b, :L].double().numpy()], 1)
        for i in range(Q):
            pos = L - Q + i  # position of query i
            Qm = np.concatenate([qc[b, i].double().numpy(), qr[b, i].double().numpy()], 1)
            S = (Qm @ K.T) * scale
            S[:, np.arange(L) > pos] = -np.inf
            if pos < 0:
                assert np.all(O[b, i] == 0) and np.all(np.isneginf(lse[b, i]))
                continue
            assert np.allclose(lse[b, i], logsumexp(S, axis=1), rtol=0, atol=1e-12)
            ref = softmax(S, axis=1) @ lat[b, :L].double().numpy()
            assert np.allclose(O[b, i], ref, rtol=0, atol=1e-12)


def _fold_case(fmt, R, lens, w):
    """Oracle decode of workload w's tokens, rotated by R when R is given
    (content latent and content query: c R, q_c R; the output rotated back)."""
    Lm = max(lens)
    lat = torch.stack([W.tokens(w, b, Lm)[0] for b in range(len(lens))])
    rope = torch.stack([W.tokens(w, b, Lm)[1] for b in range(len(lens))])
    qc, qr = W.queries(w)
    if R is not None:
        lat, qc = W.rotate(lat, R), W.rotate(qc, R)
    blocks, table = _build_cache(fmt, lat, rope, lens)
    O, lse = oracle.decode(fmt, blocks, table, np.array(lens), qc, qr, w.scale)
    if R is not None:
        O = O @ R.numpy().T
    return O, lse


def test_folded_rotation_keeps_scores_and_shrinks_quantization_error():
    """The transform-folding mechanism ("QuantMLA: INT4 (and INT2) for both
    halves of the MLA cache", Key findings): an orthogonal R folded into the
    content latent and query leaves the exact attention unchanged (up to the
    bfloat16 rounding of the rotated inputs) and, on latents with outlier
    channels, shrinks the INT2 content cache's error, because it spreads
    each outlier over every 64-channel group."""
    w = W.Workload("fold_x10", "C2R4", 3, 4, 300, 0, "x10pct1", 0, 5)
    R = W.orthogonal(512, 3)
    lens = [300, 257, 64]
    O0, l0 = _fold_case(oracle.BF16, None, lens, w)
    O1, l1 = _fold_case(oracle.BF16, R, lens, w)
    assert np.abs(l1 - l0).max() < 0.05
    assert np.abs(O1 - O0).max() / np.abs(O0).max() < 0.05
    rms = lambda O: np.sqrt(((O - O0) ** 2).mean() / (O0 ** 2).mean())
    for fmt in (oracle.C4R4, oracle.C2R4):
        Op, lp = _fold_case(fmt, None, lens, w)
        Or, lr = _fold_case(fmt, R, lens, w)
        # mean |dLSE| and relative RMS output error against the exact decode
        lse_plain, lse_rot = np.abs(lp - l0).mean(), np.abs(lr - l0).mean()
        assert lse_rot < 0.6 * lse_plain, (fmt, lse_plain, lse_rot)
        assert rms(Or) < 0.75 * rms(Op), (fmt, rms(Op), rms(Or))
