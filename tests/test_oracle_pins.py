"""Pins for the CPU oracle: each test checks it against something other than
itself -- the E2M1 format definition, hand-worked values of the pages' rules,
mathematical characterisations, brute force with exact rational arithmetic.

Rules pinned (amd-mxfp4-mm submissions): the block scale of `hw_pack_mxfp4`
(submission 748756), the E2M1 rounding and nibble packing of "Software MXFP4
quant" (submission 755056), and the `tl.dot_scaled` product."""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


# ----------------------------------------------------------------------------- independent helpers
def e2m1_value_from_fields(code: int) -> float:
    """E2M1 by its bit fields: sign | 2-bit exponent (bias 1) | 1-bit mantissa;
    exponent 0 is subnormal (0.m * 2^0)."""
    sign = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    mag = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return sign * mag


E2M1_GRID = [Fraction(e2m1_value_from_fields(c)) for c in range(8)]


def brute_e2m1(q: Fraction, negative: bool) -> int:
    """Nearest grid magnitude, ties to the even code, above 6 -> code 7."""
    a = abs(q)
    if a > 6:
        c = 7
    else:
        c = min(range(8), key=lambda i: (abs(a - E2M1_GRID[i]), i & 1))
    return c | (8 if negative else 0)


def brute_scale_exp(amax: Fraction) -> int:
    """The block exponent s characterised by the rule's effect: amax * 2^-s lands
    in [3.5, 7) (so the block maximum rounds to 4 or 6), clamped to [-127, 127]."""
    if amax == 0:
        return -127
    s = -140
    while amax / Fraction(2) ** s >= 7:
        s += 1
    return max(-127, min(127, s))


def bf16_values() -> np.ndarray:
    u = np.arange(1 << 16, dtype=np.uint32)
    u = u[((u >> 7) & 0xFF) != 0xFF]  # finite patterns only
    return (u << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def brute_bf16(d: Fraction) -> int:
    """Nearest finite bf16 to an exact rational by enumeration of neighbours,
    ties to the even pattern; beyond the largest finite value by at least half an
    ulp -> infinity."""
    vals = _BF16_SORTED_VALS
    pats = _BF16_SORTED_PATS
    x = float(d)
    i = int(np.searchsorted(vals, x))
    best = None
    for j in (i - 2, i - 1, i, i + 1):
        if 0 <= j < len(vals):
            err = abs(Fraction(float(vals[j])) - d)
            key = (err, int(pats[j]) & 1)
            if best is None or key < best[0]:
                best = (key, int(pats[j]))
    pat = best[1]
    # overflow: beyond max finite + half ulp (2^127 * (2 - 2^-8)) rounds to inf
    if abs(d) >= Fraction(2) ** 128 - Fraction(2) ** 119:
        pat = 0xFF80 if d < 0 else 0x7F80
    if pat == 0 and d < 0:
        pat = 0x8000  # a negative value that rounds to zero keeps its sign
    return pat


_u = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
_exp = (_u >> 7) & 0xFF
_fin = _u[(_exp != 0xFF) & (_u != 0x8000)]  # finite, one zero
_v = (_fin.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
_order = np.argsort(_v, kind="stable")
_BF16_SORTED_VALS = _v[_order]
_BF16_SORTED_PATS = _fin[_order]


def bf16_tensor_from_floats(vals) -> torch.Tensor:
    return torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)


def bf16_to_float(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------- E2M1
def test_e2m1_decode_matches_format_table(oracle_mod):
    for code, value in _rows("e2m1_table.txt"):
        code, value = int(code), float(value)
        assert oracle_mod.e2m1_decode(code) == value
        assert math.copysign(1.0, oracle_mod.e2m1_decode(code)) == math.copysign(1.0, value) or value != 0
        assert e2m1_value_from_fields(code) == value


def test_e2m1_encode_golden_rounding(oracle_mod):
    for q, code in _rows("e2m1_rounding.txt"):
        assert oracle_mod.e2m1_encode(float(q)) == int(code), q


def test_e2m1_encode_brute_force_dense(oracle_mod):
    # every positive finite bf16 value, scaled by 2^j so that it lands in [0, 16),
    # plus its negative: compared with exact rational nearest search.
    vals = bf16_values()
    vals = vals[np.isfinite(vals) & (vals > 0)]
    rng = np.random.default_rng(7)
    qs = []
    for v in vals:
        e = math.frexp(v)[1]
        q = math.ldexp(v, -e + int(rng.integers(-3, 5)))
        qs.append(q)
    qs = np.array(qs + [-q for q in qs[:5000]], dtype=np.float64)
    got = oracle_mod.e2m1_encode_array(qs)
    for q, c in zip(qs.tolist(), got.tolist()):
        assert c == brute_e2m1(Fraction(q), q < 0 or math.copysign(1, q) < 0), q


def test_e2m1_encode_all_midpoints_and_neighbours(oracle_mod):
    grid = [float(g) for g in E2M1_GRID]
    pts = []
    for a, b in zip(grid, grid[1:]):
        mid = (a + b) / 2
        pts += [mid, math.nextafter(mid, 0), math.nextafter(mid, 10)]
    pts += [6.0, math.nextafter(6.0, 10), 1e300, 5e-324]
    pts += [-p for p in pts]
    got = oracle_mod.e2m1_encode_array(np.array(pts))
    for q, c in zip(pts, got.tolist()):
        assert c == brute_e2m1(Fraction(q), q < 0), q


# ----------------------------------------------------------------------------- block scale
def test_scale_byte_golden(oracle_mod):
    for bits, byte in _rows("scale_examples.txt"):
        f = np.array([int(bits, 16)], np.uint32).view(np.float32)[0]
        assert oracle_mod.scale_byte(float(f)) == int(byte), bits


def test_scale_characterisation_every_bf16_amax(oracle_mod):
    # for every non-negative finite bf16 amax, the scale puts amax * 2^-s in
    # [3.5, 7), except where the clamp at -127 applies (then it is below 7).
    u = np.arange(0, 0x7F80, dtype=np.uint32)
    amax = (u << 16).view(np.float32)
    got = oracle_mod.scale_byte_array(amax).astype(np.int64)
    for a, byte in zip(amax.tolist(), got.tolist()):
        s = byte - 127
        assert s == brute_scale_exp(Fraction(a)), a
        r = Fraction(a) / Fraction(2) ** s
        if s > -127:
            assert Fraction(7, 2) <= r < 7
        else:
            assert r < 7
    assert got.max() == 253 and got.min() == 0


# ----------------------------------------------------------------------------- quantize
def brute_quantize_block(vals_f64: list[float]) -> tuple[list[int], int]:
    amax = max(abs(Fraction(v)) for v in vals_f64)
    s = brute_scale_exp(amax)
    codes = [brute_e2m1(Fraction(v) / Fraction(2) ** s, math.copysign(1.0, v) < 0) for v in vals_f64]
    return codes, s + 127


def pack_codes(codes):
    return [codes[2 * i] | (codes[2 * i + 1] << 4) for i in range(len(codes) // 2)]


def test_quantize_brute_force_random_blocks(oracle_mod):
    rng = np.random.default_rng(11)
    rows = []
    for t in range(48):
        kind = t % 6
        v = rng.standard_normal(32).astype(np.float32)
        if kind == 1:
            v *= np.float32(2.0 ** rng.integers(-60, 60))
        elif kind == 2:
            v[rng.integers(0, 32)] *= 100.0
        elif kind == 3:
            v[:] = 0.0
            v[5] = -0.0
        elif kind == 4:
            v *= np.float32(1e-39)  # bf16 subnormals
        elif kind == 5:
            v = -np.abs(v) * np.float32(1e-3)
            v[0] = 0.2
        rows.append(v)
    x = bf16_tensor_from_floats(np.stack(rows))  # [48, 32]
    xu = x.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle_mod.quantize(x)
    for r in range(x.shape[0]):
        vals = bf16_to_float(xu[r]).tolist()
        # keep the sign of -0.0 through bf16_to_float
        signs = [(int(p) >> 15) & 1 for p in xu[r]]
        vals = [(-0.0 if (sg and v == 0) else v) for v, sg in zip(vals, signs)]
        codes, byte = brute_quantize_block(vals)
        assert s[r, 0] == byte, r
        assert q[r].tolist() == pack_codes(codes), r


def test_quantize_multi_block_layout(oracle_mod):
    # several blocks per row and several rows: block b of row r must land in
    # scales[r, b] and bytes q[r, 16b:16b+16], independent of its neighbours
    A, _ = workloads.make_random(5, 1, 96, seed=3)
    A[2, 32:64] *= 1000.0
    q, s = oracle_mod.quantize(A)
    assert q.shape == (5, 48) and s.shape == (5, 3)
    for r in range(5):
        for b in range(3):
            q1, s1 = oracle_mod.quantize(A[r:r + 1, 32 * b:32 * b + 32].contiguous())
            assert s[r, b] == s1[0, 0]
            assert q[r, 16 * b:16 * b + 16].tolist() == q1[0].tolist()


def test_quantize_nibble_order_even_low(oracle_mod):
    # block of exactly representable values with amax 6 (scale byte 127):
    # x[2i] = grid[i % 8], x[2i+1] = -grid[(i+3) % 8]
    vals = []
    for i in range(16):
        vals += [float(E2M1_GRID[i % 8]), -float(E2M1_GRID[(i + 3) % 8])]
    x = bf16_tensor_from_floats([vals])
    q, s = oracle_mod.quantize(x)
    assert s[0, 0] == 127
    expect = [(i % 8) | ((((i + 3) % 8) | 8) << 4) for i in range(16)]
    assert q[0].tolist() == expect


def test_round_trip_exact_blocks(oracle_mod):
    rng = np.random.default_rng(5)
    for t in range(-20, 21):
        codes = rng.integers(0, 16, 32)
        codes[rng.integers(0, 32)] = 7  # amax exactly 6 * 2^t
        vals = [e2m1_value_from_fields(int(c)) * 2.0 ** t for c in codes]
        x = bf16_tensor_from_floats([vals])
        q, s = oracle_mod.quantize(x)
        assert s[0, 0] == 127 + t
        deq = oracle_mod.dequantize(q, s)
        assert deq[0].tolist() == vals


def test_scale_invariance_power_of_two(oracle_mod):
    x = workloads.make_activation(8, 64, seed=9)
    q0, s0 = oracle_mod.quantize(x)
    for j in (-30, -7, -1, 1, 5, 40):
        xj = (x.float() * (2.0 ** j)).to(torch.bfloat16)
        assert torch.equal(xj.float(), x.float() * 2.0 ** j)  # exact scaling
        qj, sj = oracle_mod.quantize(xj)
        assert np.array_equal(qj, q0)
        assert np.array_equal(sj.astype(int), s0.astype(int) + j)


def test_quantize_every_bf16_value_in_context(oracle_mod):
    # Every finite bf16 value, 31 per block behind a block maximum that fixes the
    # scale; compares codes against brute force (exact rationals).
    allv = workloads.all_bf16_patterns().view(torch.int16).numpy().view(np.uint16)
    vals = bf16_to_float(allv)
    anchor_bits = np.uint16(0x7F7F)  # bf16 max: scale byte 253, every value fits below it
    n = len(allv)
    nblk = (n + 30) // 31
    blocks = np.zeros((nblk, 32), np.uint16)
    flat = np.zeros(nblk * 31, np.uint16)
    flat[:n] = allv
    blocks[:, 0] = anchor_bits
    blocks[:, 1:] = flat.reshape(nblk, 31)
    x = torch.from_numpy(blocks.view(np.int16)).view(torch.bfloat16)
    q, s = oracle_mod.quantize(x)
    assert (s == 253).all()
    assert vals.size == n
    codes = np.zeros((nblk, 32), np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    sc = Fraction(2) ** 126
    for i in range(0, nblk, 7):  # a deterministic 1/7 sample keeps this under a few seconds
        for j in range(1, 32):
            p = int(blocks[i, j])
            v = float(bf16_to_float(np.array([p], np.uint16))[0])
            neg = bool(p >> 15)
            assert codes[i, j] == brute_e2m1(Fraction(v) / sc, neg)
    # and with a small anchor (scale byte 125): values above it saturate at code 7
    blocks[:, 0] = np.uint16(0x3F80)
    x = torch.from_numpy(blocks.view(np.int16)).view(torch.bfloat16)
    q2, s2 = oracle_mod.quantize(x)
    amax = np.abs(bf16_to_float(blocks)).max(axis=1)
    for i in range(0, nblk, 97):
        byte = int(s2[i, 0])
        assert byte - 127 == brute_scale_exp(Fraction(float(amax[i])))


# ----------------------------------------------------------------------------- bf16 rounding
def test_bf16_from_f64_brute_force(oracle_mod):
    rng = np.random.default_rng(13)
    ds = list(rng.standard_normal(3000) * np.exp2(rng.integers(-140, 130, 3000)))
    # exact ties between neighbouring bf16 values, both parities
    for p in (0x3F80, 0x3F81, 0x4000, 0x0001, 0x0002, 0x7F7D, 0x7F7E, 0x0080):
        lo = float(bf16_to_float(np.array([p], np.uint16))[0])
        hi = float(bf16_to_float(np.array([p + 1], np.uint16))[0])
        mid = (lo + hi) / 2
        ds += [mid, -mid, math.nextafter(mid, 0), math.nextafter(mid, math.inf)]
    top = 2.0 ** 128 - 2.0 ** 119  # halfway between the largest finite bf16 and 2^128
    ds += [0.0, 1e-50, -1e-50, 3.4e38, 1e39, -1e39, 2.0 ** -134, 2.0 ** -133 * 1.5,
           top, -top, math.nextafter(top, 0)]
    ds = np.array(ds, np.float64)
    got = oracle_mod.bf16_from_f64_array(ds)
    for d, g in zip(ds.tolist(), got.tolist()):
        if d == 0.0:
            assert g == 0
            continue
        assert g == brute_bf16(Fraction(d)), (d, hex(g))


# ----------------------------------------------------------------------------- GEMM
def test_gemm_exact_against_rationals(oracle_mod):
    rng = np.random.default_rng(17)
    M, N, K = 3, 5, 96  # non-square: a transposed operand cannot pass
    aq = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    bq = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    as_ = rng.integers(110, 140, (M, K // 32)).astype(np.uint8)
    bs = rng.integers(110, 140, (N, K // 32)).astype(np.uint8)
    c64, c16 = oracle_mod.gemm(aq, as_, bq, bs)

    def deq(q, s, r, k):
        byte = int(q[r, k // 2])
        code = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
        return Fraction(e2m1_value_from_fields(code)) * Fraction(2) ** (int(s[r, k // 32]) - 127)

    for m in range(M):
        for n in range(N):
            exact = sum(deq(aq, as_, m, k) * deq(bq, bs, n, k) for k in range(K))
            assert Fraction(c64[m, n]) == exact  # the fp64 sum is exact here
            assert int(c16[m, n]) == brute_bf16(exact)


def test_gemm_sampled_matches_full(oracle_mod):
    A, B = workloads.make_random(7, 40, 128, seed=21)
    aq, as_ = oracle_mod.quantize(A)
    bq, bs = oracle_mod.quantize(B)
    c64, c16 = oracle_mod.gemm(aq, as_, bq, bs)
    ms = np.array([0, 6, 3, 6, 1])
    ns = np.array([0, 39, 17, 0, 22])
    s64, s16 = oracle_mod.gemm_sampled(aq, as_, bq, bs, ms, ns)
    assert np.array_equal(s64, c64[ms, ns]) and np.array_equal(s16, c16[ms, ns])


def test_quant_gemm_is_quantize_then_gemm(oracle_mod):
    A, B = workloads.make_random(6, 33, 160, seed=23)
    bq, bs = oracle_mod.quantize(B)
    aq, as_, c64, c16 = oracle_mod.quant_gemm(A, bq, bs)
    aq2, as2 = oracle_mod.quantize(A)
    assert np.array_equal(aq, aq2) and np.array_equal(as_, as2)
    # and against an fp64 matmul of the independently dequantized operands
    da = np.array([[e2m1_value_from_fields(int(c)) for c in row] for row in
                   np.stack([aq & 0xF, aq >> 4], -1).reshape(6, 160)])
    db = np.array([[e2m1_value_from_fields(int(c)) for c in row] for row in
                   np.stack([bq & 0xF, bq >> 4], -1).reshape(33, 160)])
    da *= np.exp2(np.repeat(as_.astype(np.float64) - 127, 32, axis=1))
    db *= np.exp2(np.repeat(bs.astype(np.float64) - 127, 32, axis=1))
    ref = da @ db.T
    np.testing.assert_allclose(c64, ref, rtol=1e-12, atol=1e-12)


def test_workload_recipe_shapes():
    for name, w in workloads.WORKLOADS.items():
        A, B = workloads.make_random(min(w.M, 4), 8, w.K, w.seed, b_std=w.b_std,
                                     outlier_frac=w.outlier_frac)
        assert A.dtype == torch.bfloat16 and A.shape == (min(w.M, 4), w.K)
        assert B.shape == (8, w.K)
    A, _ = workloads.make_inputs("m16_n2112_k7168")
    frac = (A.float().abs() > 20).float().mean().item()
    assert 0.005 < frac < 0.015  # about 1% outliers


def test_blocked_full_gemm_equals_one_call(oracle_mod):
    """The parallel block-wise oracle GEMM used by the full-size GPU tests gives
    exactly the single call's sums (each element is the same k-ordered sum)."""
    from oracle_blocks import gemm_full

    for M, N, K, threads in ((3, 50, 64, 4), (40, 7, 96, 3), (1, 300, 32, 8), (33, 65, 160, 5)):
        A, B = workloads.make_random(M, N, K, seed=M + N + K)
        aq, as_ = oracle_mod.quantize(A)
        bq, bs = oracle_mod.quantize(B)
        c1, _ = oracle_mod.gemm(aq, as_, bq, bs)
        assert np.array_equal(gemm_full(oracle_mod, aq, as_, bq, bs, threads=threads), c1)
