"""Pins of the oracle's method (reduce, residual add, RMSNorm, per-token FP8) against things
other than itself: hand-worked examples, exact integer sums, closed forms, the exact
(high-precision) value of the normalised output, and invariants of the mathematics.

Sources: page "[OUTDATED] perf: optimize fused AllReduce + RMSNorm (custom_all_reduce)",
Technical Details / 2stage (fp32 rank-order sum, one downcast); page "[HIP] fix(custom-ar):
gfx1250 fused all-reduce + RMSNorm", Changes (same rounding as the unfused path, gemma_norm,
per-token FP8 of the rounded output); page "[HIP] [Perf] Specialize partial tiles in
two-stage custom all-reduce", bench_allreduce_tail.py listing (integer-valued inputs with
exact sums).
"""
import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

from tensor_all_reduce_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
TDT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _t(vals, dtype):
    """Exact values -> storage bits, via torch (independent of the oracle)."""
    t = torch.tensor(vals, dtype=torch.float32)
    out = t.to(TDT[dtype])
    assert torch.equal(out.float(), t), "fixture value not exactly representable"
    return synth.bits(out)


def _hexes(a):
    return [int(x, 16) for x in a]


def _dec(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TDT[dtype]).float().numpy()


# ---------------------------------------------------------------------------
# worked examples
# ---------------------------------------------------------------------------

def test_worked_1x8_bf16(orc):
    g = _gold("worked_1x8.json")
    inp, exp = g["inputs"], g["expected"]
    ps = [_t(inp[f"x{r}"], "bf16").reshape(1, 8) for r in range(4)]
    res = _t(inp["residual"], "bf16").reshape(1, 8)
    s = orc.reduce_sum(ps, "bf16")
    assert list(s.ravel()) == _hexes(exp["s_bf16_bits"])
    # the fp32 accumulator itself, through the fp32 reduce-only form
    ps32 = [np.array(inp[f"x{r}"], np.float32) for r in range(4)]
    assert list(orc.reduce_sum(ps32, "fp32")) == exp["acc_f32"]
    for wkey, gemma in (("weight_plain", False), ("weight_gemma", True)):
        w = _t(inp[wkey], "bf16")
        out = orc.fused(ps, res, w, inp["eps"], gemma, True, "bf16")
        assert list(out["res_out"].ravel()) == _hexes(exp["res_out_bf16_bits"])
        assert list(out["y"].ravel()) == _hexes(exp["y_bf16_bits"])
        assert list(out["q"].ravel()) == _hexes(exp["q_e4m3"])
        assert int(out["scale"].view(np.uint32)[0]) == int(exp["scale_f32_bits"], 16)


def test_worked_1x4_fp16(orc):
    g = _gold("worked_fp16_1x4.json")
    inp, exp = g["inputs"], g["expected"]
    ps = [_t(inp[f"x{r}"], "fp16").reshape(1, 4) for r in range(4)]
    res = _t(inp["residual"], "fp16").reshape(1, 4)
    w = _t(inp["weight"], "fp16")
    assert list(orc.reduce_sum(ps, "fp16").ravel()) == _hexes(exp["s_fp16_bits"])
    ps32 = [np.array(inp[f"x{r}"], np.float32) for r in range(4)]
    assert list(orc.reduce_sum(ps32, "fp32")) == exp["acc_f32"]
    out = orc.fused(ps, res, w, inp["eps"], False, False, "fp16")
    assert list(out["res_out"].ravel()) == _hexes(exp["res_out_fp16_bits"])
    assert list(out["y"].ravel()) == _hexes(exp["y_fp16_bits"])


# ---------------------------------------------------------------------------
# reduce: exact integer sums and rank order
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
def test_reduce_integer_inputs_exact(orc, dtype, n):
    numel = 1025 * 3 + 7
    for seed in (1, 2, 100):
        parts = synth.integer_partials(n, numel, dtype, seed)
        exact = sum(p.double() for p in parts).numpy()   # small integers: exact
        got = orc.reduce_sum([synth.bits(p) for p in parts], dtype)
        val = got if dtype == "fp32" else _dec(got, dtype)
        assert np.array_equal(val.astype(np.float64), exact)


def test_reduce_rank_order_is_binary32_sequential(orc):
    # 2^24 + 1 is a binary32 tie that rounds to 2^24: the ones are lost when they are added
    # to 2^24 one at a time (columns 0 and 1) and kept when they meet first (column 2).
    # The exact sum is 2^24 + 2 in every column.
    x0 = np.array([2.0**24, 1.0, 1.0], np.float32)
    x1 = np.array([1.0, 2.0**24, 1.0], np.float32)
    x2 = np.array([1.0, 1.0, 2.0**24], np.float32)
    got = orc.reduce_sum([x0, x1, x2], "fp32")
    assert list(got) == [2.0**24, 2.0**24, 2.0**24 + 2]


def test_reduce_in_place_alias(orc):
    parts = [synth.bits(p) for p in synth.reduce_inputs(3, 999, "bf16", seed=9)]
    ref = orc.reduce_sum(parts, "bf16")
    assert not np.array_equal(ref, parts[1])


# ---------------------------------------------------------------------------
# norm: exact value, closed forms, invariants
# ---------------------------------------------------------------------------

def _neighbours(bits, dtype):
    """The two adjacent representable values of a 16-bit value (as Fractions)."""
    b = int(bits)
    vals = []
    if b & 0x7FFF == 0:        # +-0: neighbours are the smallest subnormals
        cand = [0x0001, 0x8001]
    else:
        cand = [b - 1, b + 1]
    for c in cand:
        v = float(_dec(np.array([c & 0xFFFF], np.uint16), dtype)[0])
        if math.isfinite(v):
            vals.append(Fraction(v))
    return vals


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("gemma", [False, True])
@pytest.mark.parametrize("eps", [1e-6, 0.0, 0.5])
def test_norm_output_is_nearest_to_exact_value(orc, dtype, gemma, eps):
    """y must be a representable value nearest to z * w' / sqrt(mean(z^2) + eps), evaluated
    exactly (Fraction) up to a 60-digit square root."""
    getcontext().prec = 60
    g = torch.Generator().manual_seed(11)
    for h in (1, 2, 3, 5, 8, 16, 33):
        m = 3
        s = torch.randn((m, h), generator=g).to(TDT[dtype])
        res = torch.randn((m, h), generator=g).to(TDT[dtype])
        w = (0.3 * torch.randn((h,), generator=g) + (0.0 if gemma else 1.0)).to(TDT[dtype])
        y, z = orc.add_rmsnorm(synth.bits(s), synth.bits(res), synth.bits(w), eps, gemma, dtype)
        zf = _dec(z, dtype).astype(np.float64)
        wf = _dec(synth.bits(w), dtype).astype(np.float64)
        yf = _dec(y, dtype)
        e32 = Fraction(float(np.float32(eps)))
        for r in range(m):
            ms = sum(Fraction(float(v)) ** 2 for v in zf[r]) / h + e32
            root = Decimal(ms.numerator).sqrt() / Decimal(ms.denominator).sqrt() if ms else None
            for j in range(h):
                fac = Fraction(float(wf[j])) + (1 if gemma else 0)
                num = Fraction(float(zf[r, j])) * fac
                if root is None:
                    continue
                exact = Decimal(num.numerator) / Decimal(num.denominator) / root
                got = Decimal(float(yf[r, j]))
                dist = abs(got - exact)
                for nb in _neighbours(y[r, j], dtype):
                    nbd = abs(Decimal(nb.numerator) / Decimal(nb.denominator) - exact)
                    # binary64 evaluation can only misplace a value sitting within ~2^-45
                    # (relative) of a midpoint
                    assert dist <= nbd + abs(exact) * Decimal(2) ** -45, (h, r, j, got, exact)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_norm_closed_forms(orc, dtype):
    one = _t([1.0] * 4, dtype)
    # constant row: every element normalises to sign(c), for any c (eps = 0)
    for c in (3.0, -0.375, 1024.0, 2.0**-6):
        s = _t([[c] * 4], dtype)
        y, _ = orc.add_rmsnorm(s, None, one, 0.0, False, dtype)
        assert list(_dec(y, dtype).ravel()) == [math.copysign(1.0, c)] * 4
    # single spike: (2c, 0, 0, 0) has mean square c^2, so y = (2 sign c, 0, 0, 0)
    for c in (3.0, -5.0, 0.5):
        s = _t([[2 * c, 0.0, 0.0, 0.0]], dtype)
        y, _ = orc.add_rmsnorm(s, None, one, 0.0, False, dtype)
        assert list(_dec(y, dtype).ravel()) == [math.copysign(2.0, c), 0.0, 0.0, 0.0]
    # (3, 4) -> mean square 12.5; with eps = 12.5 the denominator is exactly 5
    s = _t([[3.0, 4.0]], dtype)
    y, _ = orc.add_rmsnorm(s, None, _t([1.0, 1.0], dtype), 12.5, False, dtype)
    exp = [orc.f64_to_bits(0.6, dtype), orc.f64_to_bits(0.8, dtype)]
    assert list(y.ravel()) == exp
    # weight scales the output elementwise: w = (2, 0.5) on the constant row
    s = _t([[7.0, 7.0]], dtype)
    y, _ = orc.add_rmsnorm(s, None, _t([2.0, 0.5], dtype), 0.0, False, dtype)
    assert list(_dec(y, dtype).ravel()) == [2.0, 0.5]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_norm_rms_invariant(orc, dtype):
    """With w = 1 and eps = 0 the RMS of the output row is 1, up to the rounding of y."""
    inp = synth.fused_inputs(1, 8, 4096, dtype, seed=5)
    s = synth.bits(inp["partials"][0])
    ones = _t([1.0] * 4096, dtype)
    y, _ = orc.add_rmsnorm(s, None, ones, 0.0, False, dtype)
    yf = _dec(y, dtype).astype(np.float64)
    rms = np.sqrt((yf ** 2).mean(axis=1))
    tol = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -10
    assert np.all(np.abs(rms - 1.0) <= tol)
    # gemma with w = 0 is the same thing
    y2, _ = orc.add_rmsnorm(s, None, _t([0.0] * 4096, dtype), 0.0, True, dtype)
    assert np.array_equal(y, y2)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_norm_scale_invariance(orc, dtype):
    """RMSNorm is invariant to scaling the row by a power of two when eps = 0."""
    inp = synth.fused_inputs(1, 4, 512, dtype, seed=6)
    z = inp["partials"][0].float()
    w = synth.bits(inp["weight"])
    base, _ = orc.add_rmsnorm(synth.bits(inp["partials"][0]), None, w, 0.0, False, dtype)
    # fp16 has few exponents below the data's range, so only scale it up
    for k in ((-6, -1, 1, 5) if dtype == "bf16" else (1, 2, 3)):
        zk = (z * 2.0**k).to(TDT[dtype])
        assert torch.equal(zk.float(), z * 2.0**k)
        yk, _ = orc.add_rmsnorm(synth.bits(zk), None, w, 0.0, False, dtype)
        assert np.array_equal(yk, base)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gemma_equals_plain_with_shifted_weight(orc, dtype):
    g = torch.Generator().manual_seed(4)
    k = torch.randint(-60, 60, (256,), generator=g).float()
    wg = (k / 128).to(TDT[dtype])             # 1 + k/128 is exact in both formats
    wp = (1 + k / 128).to(TDT[dtype])
    assert torch.equal(wp.float(), 1 + wg.float())
    inp = synth.fused_inputs(3, 5, 256, dtype, seed=8)
    ps = [synth.bits(p) for p in inp["partials"]]
    res = synth.bits(inp["residual"])
    a = orc.fused(ps, res, synth.bits(wg), 1e-6, True, True, dtype)
    b = orc.fused(ps, res, synth.bits(wp), 1e-6, False, True, dtype)
    for key in ("y", "res_out", "q", "scale"):
        assert np.array_equal(a[key], b[key])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fused_is_the_unfused_composition(orc, dtype):
    inp = synth.fused_inputs(4, 6, 200, dtype, seed=12, gemma=True)
    ps = [synth.bits(p) for p in inp["partials"]]
    res, w = synth.bits(inp["residual"]), synth.bits(inp["weight"])
    out = orc.fused(ps, res, w, 1e-6, True, True, dtype)
    s = orc.reduce_sum(ps, dtype)
    y, ro = orc.add_rmsnorm(s, res, w, 1e-6, True, dtype)
    q, sc = orc.per_token_quant(y, dtype)
    assert np.array_equal(out["res_out"], ro) and np.array_equal(out["y"], y)
    assert np.array_equal(out["q"], q) and np.array_equal(out["scale"], sc)
    # N = 1 is plain add + RMSNorm of the single partial
    one = orc.fused(ps[:1], res, w, 1e-6, True, False, dtype)
    y1, ro1 = orc.add_rmsnorm(ps[0], res, w, 1e-6, True, dtype)
    assert np.array_equal(one["y"], y1) and np.array_equal(one["res_out"], ro1)
    # no residual: res_out is the rounded sum itself
    nores = orc.fused(ps, None, w, 1e-6, True, False, dtype)
    assert np.array_equal(nores["res_out"], s)


# ---------------------------------------------------------------------------
# per-token FP8
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_quant_properties(orc, dtype):
    inp = synth.fused_inputs(4, 16, 1000, dtype, seed=13)
    y = synth.bits(inp["partials"][0])
    y[3, :] = 0                                   # an all-zero row
    q, sc = orc.per_token_quant(y, dtype)
    yf = _dec(y, dtype)
    amax = np.abs(yf).max(axis=1).astype(np.float32)
    # scale is amax / 448 in binary32 (numpy's division)
    assert np.array_equal(sc, (amax / np.float32(448.0)).astype(np.float32))
    assert sc[3] == 0 and (q[3] == 0).all()
    deq = orc.e4m3_to_f32(q)
    for r in range(16):
        if r == 3:
            continue
        j = int(np.argmax(np.abs(yf[r])))
        assert q[r, j] == (0x7E if yf[r, j] > 0 else 0xFE)   # the amax element maps to +-448
        # reconstruction within half an E4M3 spacing (relative 2^-4, or the subnormal step)
        v = yf[r].astype(np.float64) / float(sc[r])
        err = np.abs(deq[r].astype(np.float64) - v)
        assert np.all(err <= np.maximum(np.abs(v) * 2.0**-4, 2.0**-10) * (1 + 1e-6))
    # odd symmetry
    neg = y ^ np.uint16(0x8000)
    qn, scn = orc.per_token_quant(neg, dtype)
    assert np.array_equal(scn, sc)
    nz = q != 0
    assert np.array_equal(qn[nz], q[nz] ^ np.uint8(0x80))


def test_quant_tiny_rows_and_groups(orc):
    """Rows and groups of tiny bf16 magnitude (maxima 2^-133 .. 2^-118), where the binary32
    scale amax / 448 is subnormal: the scale is still the binary32 quotient with gradual
    underflow, and each code the E4M3 rounding of the binary32 quotient y / scale.  Expected
    values from numpy's binary32 arithmetic and torch's E4M3 cast (saturation at 448 applied
    first, as the format's satfinite conversion does), not from the oracle."""
    g = np.random.default_rng(21)
    m, h = 64, 96
    ks = -133 + (np.arange(m) % 16)
    vals = (g.standard_normal((m, h)) * 2.0 ** ks[:, None]).astype(np.float32)
    y = synth.bits(torch.from_numpy(vals).to(torch.bfloat16))
    y[5, :] = 0                                          # an all-zero row among them
    yf = _dec(y, "bf16")
    amax = np.abs(yf).max(axis=1).astype(np.float32)
    sc_exp = amax / np.float32(448.0)
    assert np.count_nonzero((sc_exp > 0) & (sc_exp < np.float32(2.0 ** -126))) > 40   # subnormal scales
    with np.errstate(divide="ignore", invalid="ignore"):
        quo = np.where(amax[:, None] > 0, yf / sc_exp[:, None], np.float32(0.0)).astype(np.float32)
    q_exp = torch.from_numpy(np.clip(quo, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    q, sc = orc.per_token_quant(y, "bf16")
    assert np.array_equal(sc.view(np.uint32), sc_exp.view(np.uint32))
    assert np.array_equal(q, q_exp)
    assert not np.any((q & 0x7F) == 0x7F)               # no NaN code
    # per group: groups of 16 with tiny and normal groups side by side in one row
    yg = y.copy().reshape(m, h // 16, 16)
    big = synth.bits(torch.from_numpy(g.standard_normal((m, h // 16, 16)).astype(np.float32)).to(torch.bfloat16))
    yg[:, 1::2, :] = big[:, 1::2, :]
    yg = yg.reshape(m, h)
    qg, scg = orc.per_group_quant(yg, 16, "bf16")
    yv = _dec(yg, "bf16").reshape(m, h // 16, 16)
    am = np.abs(yv).max(axis=2).astype(np.float32)
    s_exp = am / np.float32(448.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        qq = np.where(am[:, :, None] > 0, yv / s_exp[:, :, None], np.float32(0.0)).astype(np.float32)
    qg_exp = torch.from_numpy(np.clip(qq, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(scg.view(np.uint32), s_exp.reshape(m, -1).view(np.uint32))
    assert np.array_equal(qg, qg_exp.reshape(m, h))


# ---------------------------------------------------------------------------
# options: no normalisation (all-reduce + per-token FP8) and binary32 output
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_skip_norm_is_the_rounded_residual_sum(orc, dtype):
    inp = synth.fused_inputs(4, 9, 300, dtype, seed=31)
    ps = [synth.bits(p) for p in inp["partials"]]
    res = synth.bits(inp["residual"])
    out = orc.fused_ex(ps, res, None, 0.0, False, True, dtype, skip_norm=True, out_fp32=True)
    assert np.array_equal(out["y"], out["res_out"])
    # y32 holds exactly the 16-bit values
    assert np.array_equal(out["y32"], _dec(out["res_out"], dtype))
    s = orc.reduce_sum(ps, dtype)
    _, z = orc.add_rmsnorm(s, res, synth.bits(inp["weight"]), 1e-6, False, dtype)
    assert np.array_equal(out["res_out"], z)
    q, sc = orc.per_token_quant(z, dtype)
    assert np.array_equal(out["q"], q) and np.array_equal(out["scale"], sc)
    # no residual: the output is the reduced sum itself
    out2 = orc.fused_ex(ps, None, None, 0.0, False, False, dtype, skip_norm=True)
    assert np.array_equal(out2["y"], s)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("gemma", [False, True])
def test_fp32_output_is_nearest_binary32_of_exact_value(orc, dtype, gemma):
    getcontext().prec = 60
    g = torch.Generator().manual_seed(17)
    for h in (1, 3, 8, 21):
        ps = [torch.randn((2, h), generator=g).to(TDT[dtype]) for _ in range(3)]
        res = torch.randn((2, h), generator=g).to(TDT[dtype])
        w = (0.3 * torch.randn((h,), generator=g) + (0.0 if gemma else 1.0)).to(TDT[dtype])
        out = orc.fused_ex([synth.bits(p) for p in ps], synth.bits(res), synth.bits(w), 1e-6, gemma, False,
                           dtype, out_fp32=True)
        z = _dec(out["res_out"], dtype).astype(np.float64)
        wf = _dec(synth.bits(w), dtype).astype(np.float64)
        y32 = out["y32"]
        e32 = Fraction(float(np.float32(1e-6)))
        for r in range(2):
            ms = sum(Fraction(float(v)) ** 2 for v in z[r]) / h + e32
            root = Decimal(ms.numerator).sqrt() / Decimal(ms.denominator).sqrt()
            for j in range(h):
                num = Fraction(float(z[r, j])) * (Fraction(float(wf[j])) + (1 if gemma else 0))
                exact = Decimal(num.numerator) / Decimal(num.denominator) / root
                got = Decimal(float(y32[r, j]))
                for nb in (np.nextafter(y32[r, j], np.float32(np.inf)), np.nextafter(y32[r, j], np.float32(-np.inf))):
                    assert abs(got - exact) <= abs(Decimal(float(nb)) - exact) + abs(exact) * Decimal(2) ** -45
        # the 16-bit output is within one 16-bit ulp of the binary32 one
        y = _dec(out["y"], dtype).astype(np.float64)
        assert np.all(np.abs(y - y32) <= np.abs(y32) * (2.0 ** -8 if dtype == "bf16" else 2.0 ** -11) + 1e-30)


def test_fp32_output_closed_forms(orc):
    one = _t([1.0] * 4, "bf16")
    s = _t([[3.0] * 4, [2.0, 0.0, 0.0, 0.0]], "bf16")
    out = orc.fused_ex([s], None, one, 0.0, False, False, "bf16", out_fp32=True)
    assert list(out["y32"][0]) == [1.0] * 4
    assert list(out["y32"][1]) == [2.0, 0.0, 0.0, 0.0]


# ---------------------------------------------------------------------------
# per-group FP8 (groups of G consecutive elements along a row)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("group", [8, 32, 128])
def test_per_group_quant_is_per_token_quant_of_the_groups(orc, dtype, group):
    """Cutting every row into groups and quantising each group as its own token gives the
    per-group result: the per-token routine (pinned above) run on the [m * h / G, G] view."""
    inp = synth.fused_inputs(1, 6, 512, dtype, seed=41)
    y = synth.bits(inp["partials"][0])
    y[2, 64:192] = 0                                   # zero groups
    q, sc = orc.per_group_quant(y, group, dtype)
    q2, sc2 = orc.per_token_quant(y.reshape(-1, group), dtype)
    assert np.array_equal(q, q2.reshape(q.shape))
    assert np.array_equal(sc, sc2.reshape(sc.shape))
    # one group per row is per-token quantisation
    q3, sc3 = orc.per_group_quant(y, 512, dtype)
    q4, sc4 = orc.per_token_quant(y, dtype)
    assert np.array_equal(q3, q4) and np.array_equal(sc3.ravel(), sc4)


def test_per_group_scales_follow_their_own_groups(orc):
    # row 0: groups of 4 with maxima 1, 2, 4, 8 -> scales max/448, and each group's max -> 448
    vals = np.array([[0.5, 1.0, -0.25, 0.75, 2.0, -1.0, 0.0, 1.5, 4.0, 3.0, -2.0, 1.0, -8.0, 0.5, 4.0, 2.0]],
                    np.float32)
    y = _t(vals.tolist(), "bf16")
    q, sc = orc.per_group_quant(y, 4, "bf16")
    assert list(sc[0]) == [np.float32(x) / np.float32(448) for x in (1.0, 2.0, 4.0, 8.0)]
    assert q[0, 1] == 0x7E and q[0, 4] == 0x7E and q[0, 8] == 0x7E and q[0, 12] == 0xFE


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fused_with_per_group_quant(orc, dtype):
    inp = synth.fused_inputs(4, 5, 384, dtype, seed=43, gemma=True)
    ps = [synth.bits(p) for p in inp["partials"]]
    res, w = synth.bits(inp["residual"]), synth.bits(inp["weight"])
    out = orc.fused_ex(ps, res, w, 1e-6, True, True, dtype, group=64)
    q, sc = orc.per_group_quant(out["y"], 64, dtype)
    assert np.array_equal(out["q"], q) and np.array_equal(out["scale"], sc)
    assert out["scale"].shape == (5, 6)
    # the rest of the path is unchanged by the grouping
    ref = orc.fused(ps, res, w, 1e-6, True, True, dtype)
    assert np.array_equal(out["y"], ref["y"]) and np.array_equal(out["res_out"], ref["res_out"])



def test_per_group_hand_worked_row(orc):
    """Per-group FP8 of a hand-worked 1 x 16 bf16 row in two groups of 8
    (tests/golden/worked_group8_1x16.json, derived from the format definitions)."""
    import json
    import os
    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_group8_1x16.json")))
    y = np.array([int(b, 16) for b in fx["inputs"]["y_bf16_bits"]], dtype=np.uint16).reshape(1, 16)
    q, sc = orc.per_group_quant(y, fx["inputs"]["group"], "bf16")
    assert [f"0x{v:08x}" for v in sc.view(np.uint32).ravel()] == fx["expected"]["scale_f32_bits"]
    assert [f"0x{v:02x}" for v in q.ravel()] == fx["expected"]["q_e4m3"]
