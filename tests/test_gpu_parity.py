"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element.

Covers the five workload families at their full sizes (in the launch configuration the
benchmark uses), the shape list of the fused-kernel test on page "[HIP] fix(custom-ar):
gfx1250 fused all-reduce + RMSNorm" (Changes / test command), the tail cases of page "[HIP]
[Perf] Specialize partial tiles in two-stage custom all-reduce" (1023/1024/1025 x 512,
tails of 1/63/64/65/127 packs, byte sizes around 1 MiB), every kernel variant, N = 1..8,
both element types, aliases, misaligned pointers, empty inputs and the maximum sizes (the
longest rows accepted and the first refused; 2^20 rows in one call, checked on sampled rows).
Outputs sit between sentinel guard regions and are poisoned before each call.
"""
import numpy as np
import pytest
import torch

import tensor_all_reduce_gb300 as tar
from tensor_all_reduce_gb300 import synth

from gpu_helpers import (Guarded, TDT, assert_bits_equal, assert_fp8, assert_y_within_ulp, bits_of,
                         decode, to_dev)

pytestmark = pytest.mark.gpu

DT_CODE = {"bf16": tar.AR_DTYPE_BF16, "fp16": tar.AR_DTYPE_F16, "fp32": tar.AR_DTYPE_F32}
TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def ctx(dev):
    c = tar.Context(0)
    yield c
    c.close()


@pytest.fixture(autouse=True)
def _reset_options(request):
    yield
    if "ctx" in request.fixturenames:
        c = request.getfixturevalue("ctx")
        for opt in (tar.AR_OPT_FORCE_VARIANT, tar.AR_OPT_CLUSTER_SIZE, tar.AR_OPT_PACKS_PER_THREAD,
                    tar.AR_OPT_REDUCE_UNROLL, tar.AR_OPT_STAGES):
            c.set_option(opt, 0)
        c.set_option(tar.AR_OPT_PDL, 1)


# ---------------------------------------------------------------------------
# fused path
# ---------------------------------------------------------------------------

def run_fused(ctx, dev, inp, dtype, gemma=False, quant=False, mirror=True, eps=1e-6, res_out=True):
    parts = to_dev(inp["partials"], dev)
    res = inp["residual"].to(dev) if inp["residual"] is not None else None
    w = inp["weight"].to(dev)
    m, h = parts[0].shape
    g_out = Guarded((m, h), TDT[dtype], dev) if (mirror or not quant) else None
    g_ro = Guarded((m, h), TDT[dtype], dev) if res_out else None
    g_q = Guarded((m, h), torch.uint8, dev) if quant else None
    g_s = Guarded((m,), torch.float32, dev) if quant else None
    ctx.fused_reduce_rmsnorm(parts, res, w, eps=eps, gemma=gemma, quant=quant,
                             out=g_out.t if g_out else None, residual_out=g_ro.t if g_ro else None,
                             q_out=g_q.t if g_q else None, scale_out=g_s.t if g_s else None,
                             want_out=g_out is not None, want_residual_out=g_ro is not None)
    torch.cuda.synchronize()
    for g in (g_out, g_ro, g_q, g_s):
        if g is not None:
            assert g.guards_intact(), "a kernel wrote outside its output"
    return {"y": bits_of(g_out.t) if g_out else None, "res_out": bits_of(g_ro.t) if g_ro else None,
            "q": g_q.t.cpu().numpy() if g_q else None, "scale": g_s.t.cpu().numpy() if g_s else None,
            "variant": ctx.last_variant}


def oracle_fused(orc, inp, dtype, gemma=False, quant=False, eps=1e-6):
    return orc.fused([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                     synth.bits(inp["weight"]), eps, gemma, quant, dtype)


def check_fused(orc, got, ref, dtype, quant):
    if got["res_out"] is not None:
        assert_bits_equal(got["res_out"], ref["res_out"], "residual_out")
    if got["y"] is not None:
        assert_y_within_ulp(got["y"], ref["y"], dtype)
    if quant:
        y_for_q = got["y"] if got["y"] is not None else ref["y"]
        if got["y"] is not None:
            assert_fp8(orc, got["q"], got["scale"], y_for_q, dtype, ref)
        else:
            # no mirror: the kernel's y is not visible, so compare with the oracle's own y.
            # Every row's scale is within one 16-bit ulp of amax of the oracle's (the y bar at
            # the amax element), almost every row's scale is equal, and every code is within
            # one code: a scale off by 2^-7 and a y off by one ulp move a quotient by less than
            # half an E4M3 step, so at most one rounding boundary is crossed.
            from gpu_helpers import code_ordinal
            s_g, s_r = got["scale"].astype(np.float64), ref["scale"].astype(np.float64)
            tol = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -10
            assert np.all(np.abs(s_g - s_r) <= tol * s_r * 1.0001), "scale beyond one ulp of amax of the oracle's"
            same = got["scale"] == ref["scale"]
            assert same.mean() > 0.99
            d = np.abs(code_ordinal(got["q"]) - code_ordinal(ref["q"]))
            assert d.max(initial=0) <= 1, f"codes differ from the oracle's by {d.max()} codes"


WORKLOADS = synth.all_fused()


@pytest.mark.parametrize("wl", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_fused_workloads_full_size(ctx, dev, orc, wl, record_property):
    inp = wl.inputs()
    got = run_fused(ctx, dev, inp, wl.dtype, wl.gemma, wl.quant, wl.mirror)
    ref = oracle_fused(orc, inp, wl.dtype, wl.gemma, wl.quant)
    check_fused(orc, got, ref, wl.dtype, wl.quant)
    assert got["variant"].startswith("fused_")
    if wl.quant:
        # rows whose scale takes the one-ulp-of-amax allowance (the kernel's y at the row's
        # largest element one ulp from the oracle's): counted, and bounded at 1 % of rows so
        # that a drift in the norm arithmetic shows up as a number
        n_diff = int(np.count_nonzero(got["scale"] != ref["scale"]))
        record_property("scale_rows_one_ulp_of_amax", f"{n_diff} of {wl.m}")
        print(f"\n{wl.name}: {n_diff} of {wl.m} rows with a scale one ulp of amax from the oracle's")
        assert n_diff <= 0.01 * wl.m


# shape list of the fused AR + RMSNorm test command on the gfx1250 page
PAGE_SHAPES = [(16, 6144), (4, 2880), (384, 6144), (1024, 6144), (2730, 6144), (2800, 6144), (1024, 7168),
               (512, 8192), (1024, 4096), (1024, 2880)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("quant", [False, True])
@pytest.mark.parametrize("m,h", PAGE_SHAPES)
def test_fused_page_shapes(ctx, dev, orc, m, h, dtype, quant):
    inp = synth.fused_inputs(4, m, h, dtype, seed=m * 7 + h, gemma=quant)
    got = run_fused(ctx, dev, inp, dtype, gemma=quant, quant=quant)
    ref = oracle_fused(orc, inp, dtype, gemma=quant, quant=quant)
    check_fused(orc, got, ref, dtype, quant)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("h", [1, 7, 9, 15, 2880, 6143, 6145])
def test_fused_tail_hidden_sizes(ctx, dev, orc, dtype, h):
    for quant in (False, True):
        inp = synth.fused_inputs(3, 5, h, dtype, seed=h, gemma=quant)
        got = run_fused(ctx, dev, inp, dtype, gemma=quant, quant=quant)
        ref = oracle_fused(orc, inp, dtype, gemma=quant, quant=quant)
        check_fused(orc, got, ref, dtype, quant)
        if h % 8:
            assert "scalar" in got["variant"], got["variant"]


VARIANTS = ([("row", {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_ROW, tar.AR_OPT_PACKS_PER_THREAD: p}) for p in (1, 2, 4)]
            + [(f"cluster{c}", {tar.AR_OPT_CLUSTER_SIZE: c}) for c in (2, 4, 8, 16)]
            + [("cluster8_ppt2", {tar.AR_OPT_CLUSTER_SIZE: 8, tar.AR_OPT_PACKS_PER_THREAD: 2})]
            + [("staged", {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_STAGED}),
               ("staged_s2_ppt4", {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_STAGED, tar.AR_OPT_STAGES: 2,
                                   tar.AR_OPT_PACKS_PER_THREAD: 4})]
            + [("scalar", {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_SCALAR}),
               ("scalar_cluster4", {tar.AR_OPT_FORCE_VARIANT: tar.VARIANT_SCALAR, tar.AR_OPT_CLUSTER_SIZE: 4})])


@pytest.mark.parametrize("name,opts", VARIANTS, ids=[v[0] for v in VARIANTS])
@pytest.mark.parametrize("m,h", [(33, 6144), (3, 7168), (2, 2880), (700, 4096)])
def test_fused_every_variant(ctx, dev, orc, name, opts, m, h):
    for k, v in opts.items():
        ctx.set_option(k, v)
    for quant in (False, True):
        inp = synth.fused_inputs(4, m, h, "bf16", seed=m + h, gemma=quant)
        got = run_fused(ctx, dev, inp, "bf16", gemma=quant, quant=quant)
        ref = oracle_fused(orc, inp, "bf16", gemma=quant, quant=quant)
        check_fused(orc, got, ref, "bf16", quant)
        if "cluster" in name:
            assert "cluster" in got["variant"], got["variant"]
        elif name.startswith("staged"):
            assert got["variant"] == "fused_staged"
            assert ctx.device_status() == 0
        elif name == "scalar":
            assert "scalar" in got["variant"]
        else:
            assert got["variant"] == "fused_row_vec"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("m", [151, 152, 153, 256, 304, 305])
def test_fused_one_to_two_rows_per_sm(ctx, dev, orc, m, dtype):
    """Around the one-CTA-per-row regime (one to two rows per SM), where the automatic choice
    switches stage count and, for rows without FP8, packs per thread: every form it picks
    against the oracle, with and without FP8, for 4 and 8 partials."""
    for n, h, quant in ((4, 6144, False), (4, 4096, False), (8, 6144, False), (4, 6144, True)):
        inp = synth.fused_inputs(n, m, h, dtype, seed=m * 3 + h + n, gemma=quant)
        got = run_fused(ctx, dev, inp, dtype, gemma=quant, quant=quant)
        assert got["variant"] == "fused_staged", got["variant"]
        check_fused(orc, got, oracle_fused(orc, inp, dtype, gemma=quant, quant=quant), dtype, quant)


@pytest.mark.parametrize("n", range(1, 9))
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fused_every_n(ctx, dev, orc, n, dtype):
    inp = synth.fused_inputs(n, 40, 1024, dtype, seed=n)
    got = run_fused(ctx, dev, inp, dtype, quant=True, gemma=True)
    ref = oracle_fused(orc, inp, dtype, quant=True, gemma=True)
    check_fused(orc, got, ref, dtype, True)


def test_fused_options(ctx, dev, orc):
    # no residual: residual_out receives the rounded sum
    inp = synth.fused_inputs(4, 20, 6144, "bf16", seed=3, residual=False)
    got = run_fused(ctx, dev, inp, "bf16")
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], None, synth.bits(inp["weight"]), 1e-6, False,
                    False, "bf16")
    check_fused(orc, got, ref, "bf16", False)
    assert_bits_equal(got["res_out"], orc.reduce_sum([synth.bits(p) for p in inp["partials"]], "bf16"), "sum")
    # FP8 without the mirror, and without residual_out
    inp = synth.fused_inputs(4, 64, 6144, "bf16", seed=4, gemma=True)
    got = run_fused(ctx, dev, inp, "bf16", gemma=True, quant=True, mirror=False, res_out=False)
    ref = oracle_fused(orc, inp, "bf16", gemma=True, quant=True)
    check_fused(orc, got, ref, "bf16", True)
    # eps = 0 and a large eps
    for eps in (0.0, 4.0):
        inp = synth.fused_inputs(2, 8, 512, "fp16", seed=5)
        got = run_fused(ctx, dev, inp, "fp16", eps=eps)
        check_fused(orc, got, oracle_fused(orc, inp, "fp16", eps=eps), "fp16", False)


@pytest.mark.parametrize("variant", [tar.VARIANT_ROW, tar.VARIANT_STAGED, tar.VARIANT_CLUSTER, tar.VARIANT_SCALAR])
def test_fp8_codes_exact_given_y(ctx, dev, orc, variant):
    """The kernels quantise with a correctly rounded quotient, so given the kernel's own y
    the codes and scales equal the oracle's exactly (the contract allows one code)."""
    ctx.set_option(tar.AR_OPT_FORCE_VARIANT, variant)
    inp = synth.fused_inputs(4, 700, 4096, "bf16", seed=21, gemma=True)
    # rows spanning many magnitudes, so scales cover many binades
    g = torch.Generator().manual_seed(5)
    mags = (2.0 ** torch.randint(-12, 12, (700, 1), generator=g)).to(torch.float32)
    inp["weight"] = (inp["weight"].float() * 3).to(torch.bfloat16)
    inp["partials"] = [(p.float() * mags).to(torch.bfloat16) for p in inp["partials"]]
    inp["residual"] = (inp["residual"].float() * mags).to(torch.bfloat16)
    got = run_fused(ctx, dev, inp, "bf16", gemma=True, quant=True)
    q_ref, s_ref = orc.per_token_quant(got["y"], "bf16")
    assert np.array_equal(got["scale"].view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(got["q"], q_ref)


def test_fused_zero_row_and_saturation(ctx, dev, orc):
    inp = synth.fused_inputs(4, 6, 2048, "bf16", seed=6, gemma=True)
    for p in inp["partials"]:
        p[2].zero_()
    inp["residual"][2].zero_()
    inp["partials"][0][4, 5] = 1000.0      # one dominant element: its code is +-448
    got = run_fused(ctx, dev, inp, "bf16", gemma=True, quant=True)
    ref = oracle_fused(orc, inp, "bf16", gemma=True, quant=True)
    check_fused(orc, got, ref, "bf16", True)
    assert got["scale"][2] == 0.0 and (got["q"][2] == 0).all()
    assert got["q"][4, 5] in (0x7E, 0xFE)


def test_fused_aliases(ctx, dev, orc):
    inp = synth.fused_inputs(4, 48, 6144, "bf16", seed=7)
    ref = oracle_fused(orc, inp, "bf16")
    parts = to_dev(inp["partials"], dev)
    res = inp["residual"].to(dev)
    w = inp["weight"].to(dev)
    # residual_out written over residual_in, y written over partial 0
    ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6, out=parts[0], residual_out=res)
    torch.cuda.synchronize()
    assert_bits_equal(bits_of(res), ref["res_out"], "residual_out in place")
    assert_y_within_ulp(bits_of(parts[0]), ref["y"], "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("n", [1, 4, 8])
def test_fused_staged_large(ctx, dev, orc, n, dtype):
    """The staged variant on large batches: many rows per CTA, every pipeline stage reused."""
    ctx.set_option(tar.AR_OPT_FORCE_VARIANT, tar.VARIANT_STAGED)
    for quant in (False, True):
        inp = synth.fused_inputs(n, 1500, 6144, dtype, seed=n * 3 + quant, gemma=quant)
        got = run_fused(ctx, dev, inp, dtype, gemma=quant, quant=quant)
        assert got["variant"] == "fused_staged"
        check_fused(orc, got, oracle_fused(orc, inp, dtype, gemma=quant, quant=quant), dtype, quant)
    inp = synth.fused_inputs(n, 777, 4096, dtype, seed=n, residual=False)
    got = run_fused(ctx, dev, inp, dtype)
    ref = orc.fused([synth.bits(p) for p in inp["partials"]], None, synth.bits(inp["weight"]), 1e-6, False,
                    False, dtype)
    check_fused(orc, got, ref, dtype, False)
    assert ctx.device_status() == 0


def test_fused_empty_batch(ctx, dev):
    inp = synth.fused_inputs(2, 0, 128, "bf16", seed=8)
    parts = to_dev(inp["partials"], dev)
    ctx.fused_reduce_rmsnorm(parts, inp["residual"].to(dev), inp["weight"].to(dev))
    assert ctx.last_variant == "none"


def test_fused_misaligned_pointers(ctx, dev, orc):
    m, h = 9, 2048
    inp = synth.fused_inputs(3, m, h, "bf16", seed=9)
    ref = oracle_fused(orc, inp, "bf16")
    parts = []
    for p in inp["partials"]:
        g = Guarded((m, h), torch.bfloat16, dev, offset_elems=1)   # 2 bytes off 16-byte alignment
        g.t.copy_(p.to(dev))
        parts.append(g.t)
    res, w = inp["residual"].to(dev), inp["weight"].to(dev)
    y, ro, _, _ = ctx.fused_reduce_rmsnorm(parts, res, w)
    torch.cuda.synchronize()
    assert "scalar" in ctx.last_variant
    assert_bits_equal(bits_of(ro), ref["res_out"], "residual_out")
    assert_y_within_ulp(bits_of(y), ref["y"], "bf16")


def test_invalid_options_and_device(ctx):
    with pytest.raises(tar.ArError):
        ctx.set_option(tar.AR_OPT_CLUSTER_SIZE, 3)
    with pytest.raises(tar.ArError):
        ctx.set_option(tar.AR_OPT_PACKS_PER_THREAD, 8)
    with pytest.raises(tar.ArError):
        tar.ar_init(10_000)
    assert ctx.info(tar.AR_INFO_SM_COUNT) > 0


# ---------------------------------------------------------------------------
# plain reduce
# ---------------------------------------------------------------------------

def run_reduce(ctx, dev, parts_cpu, dtype, out_offset=0, in_offset=0):
    parts = []
    for p in parts_cpu:
        g = Guarded(p.shape, TORCH[dtype], dev, offset_elems=in_offset)
        g.t.copy_(p.to(dev))
        parts.append(g.t)
    g_out = Guarded(parts_cpu[0].shape, TORCH[dtype], dev, offset_elems=out_offset)
    ctx.reduce_sum(parts, out=g_out.t)
    torch.cuda.synchronize()
    assert g_out.guards_intact(), "reduce wrote outside its output"
    return synth.bits(g_out.t.cpu()), ctx.last_variant


REDUCE_WORKLOADS = synth.reduce_only() + synth.reduce_large()


@pytest.mark.parametrize("wl", REDUCE_WORKLOADS, ids=[w.name for w in REDUCE_WORKLOADS])
def test_reduce_workloads(ctx, dev, orc, wl):
    parts = synth.reduce_inputs(wl.n, wl.numel, wl.dtype, wl.seed)
    got, variant = run_reduce(ctx, dev, parts, wl.dtype)
    assert_bits_equal(got, orc.reduce_sum([synth.bits(p) for p in parts], wl.dtype), wl.name)
    staged = wl.dtype != "fp32" and 4 <= wl.n <= 6 and wl.numel >= 8192 * 16 * ctx.info(tar.AR_INFO_SM_COUNT)
    assert variant == "reduce_staged" if staged else variant.startswith("reduce_vec"), variant


@pytest.mark.parametrize("n", [4, 5, 6])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_reduce_large_through_staged_rows(ctx, dev, orc, n, dtype):
    """Large 16-bit arrays of 4-6 partials run on the staged kernel as rows (no residual, no
    norm): the same bits as the oracle's rank-order fp32 sum, with guard regions intact, in
    place too, and with row lengths other than 8192 (the array length picks the row)."""
    for numel in (4096 * 6144, 7168 * 2999):            # rows of 8192, and of 7168
        parts = synth.reduce_inputs(n, numel, dtype, seed=n + numel % 97)
        ref = orc.reduce_sum([synth.bits(p) for p in parts], dtype)
        got, variant = run_reduce(ctx, dev, parts, dtype)
        assert variant == "reduce_staged", variant
        assert_bits_equal(got, ref, f"{n} x {numel}")
    d = to_dev(parts, dev)
    ctx.reduce_sum(d, out=d[1])
    torch.cuda.synchronize()
    assert ctx.last_variant == "reduce_staged"
    assert_bits_equal(synth.bits(d[1].cpu()), ref, "in place")
    ctx.set_option(tar.AR_OPT_REDUCE_UNROLL, 1)            # the per-thread kernel agrees bit for bit
    got, variant = run_reduce(ctx, dev, parts, dtype)
    ctx.set_option(tar.AR_OPT_REDUCE_UNROLL, 0)
    assert variant.startswith("reduce_vec")
    assert_bits_equal(got, ref, "per-thread kernel")


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_reduce_tail_sweep(ctx, dev, orc, dtype):
    ctx.set_option(tar.AR_OPT_REDUCE_UNROLL, 4)
    tile = ctx.info(tar.AR_INFO_REDUCE_TILE_PACKS)
    pack = 16 // (4 if dtype == "fp32" else 2)
    sizes = []
    for t in (0, 1, 63, 64, 65, 127):
        for r in (0, 1, pack - 1):
            sizes.append(pack * (3 * tile + t) + r)
    sizes += [(2**20 + off) // (4 if dtype == "fp32" else 2) for off in (-64, 0, 64, 63 * 64, 64 * 64, 65 * 64)]
    sizes += [1, 2, pack - 1, pack, pack + 1, tile * pack - 1]
    for unroll in (1, 4):
        ctx.set_option(tar.AR_OPT_REDUCE_UNROLL, unroll)
        for numel in sizes:
            parts = synth.reduce_inputs(4, numel, dtype, seed=numel)
            got, variant = run_reduce(ctx, dev, parts, dtype)
            assert_bits_equal(got, orc.reduce_sum([synth.bits(p) for p in parts], dtype), f"numel={numel}")
            full = numel % pack == 0 and (numel // pack) % (256 * unroll) == 0
            assert variant == ("reduce_vec" if full else "reduce_vec_tail"), (numel, variant)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_reduce_integer_inputs_exact(ctx, dev, dtype):
    for n in (2, 4, 8):
        numel = 1025 * 512
        parts = synth.integer_partials(n, numel, dtype, seed=n)
        got, _ = run_reduce(ctx, dev, parts, dtype)
        exact = sum(p.double() for p in parts).numpy()
        val = got if dtype == "fp32" else decode(got, dtype)
        assert np.array_equal(val.astype(np.float64), exact)


@pytest.mark.parametrize("n", range(1, 9))
def test_reduce_every_n(ctx, dev, orc, n):
    parts = synth.reduce_inputs(n, 300_001, "bf16", seed=n)
    got, _ = run_reduce(ctx, dev, parts, "bf16")
    assert_bits_equal(got, orc.reduce_sum([synth.bits(p) for p in parts], "bf16"), f"n={n}")


def test_reduce_misaligned_and_inplace(ctx, dev, orc):
    parts = synth.reduce_inputs(4, 99_999, "fp16", seed=11)
    ref = orc.reduce_sum([synth.bits(p) for p in parts], "fp16")
    got, variant = run_reduce(ctx, dev, parts, "fp16", out_offset=1)
    assert variant == "reduce_scalar"
    assert_bits_equal(got, ref, "misaligned out")
    got, variant = run_reduce(ctx, dev, parts, "fp16", in_offset=3)
    assert variant == "reduce_scalar"
    assert_bits_equal(got, ref, "misaligned inputs")
    d = to_dev(parts, dev)
    ctx.reduce_sum(d, out=d[2])
    torch.cuda.synchronize()
    assert_bits_equal(synth.bits(d[2].cpu()), ref, "in place")


def test_reduce_empty(ctx, dev):
    parts = [torch.empty(0, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    ctx.reduce_sum(parts)
    assert ctx.last_variant == "none"


# ---------------------------------------------------------------------------
# maximum sizes
# ---------------------------------------------------------------------------

def test_longest_rows(ctx, dev, orc):
    """The longest rows a call accepts: 1024 packs per CTA times the largest cluster (16 CTAs
    where the device allows non-portable clusters, else 8); one pack more is refused."""
    longest = None
    for h in (131072, 65536):
        inp = synth.fused_inputs(2, 3, h, "bf16", seed=h % 997, gemma=True)
        try:
            got = run_fused(ctx, dev, inp, "bf16", gemma=True, quant=True)
        except tar.ArError as e:
            assert e.status == tar.AR_ERR_UNSUPPORTED and h == 131072
            continue
        check_fused(orc, got, oracle_fused(orc, inp, "bf16", gemma=True, quant=True), "bf16", True)
        longest = h
        break
    assert longest is not None
    inp = synth.fused_inputs(2, 2, longest + 8, "bf16", seed=5)
    with pytest.raises(tar.ArError) as e:
        run_fused(ctx, dev, inp, "bf16")
    assert e.value.status == tar.AR_ERR_UNSUPPORTED


def test_tall_call_sampled_rows(ctx, dev, orc):
    """2^20 rows of 64 elements in one call (the persistent staged kernel runs hundreds of rows
    per CTA): rows are independent, so sampled rows are checked against the oracle run on
    those rows alone, FP8 included."""
    m, h, n = 1 << 20, 64, 2
    inp = synth.fused_inputs(n, m, h, "bf16", seed=17, gemma=True)
    got = run_fused(ctx, dev, inp, "bf16", gemma=True, quant=True)
    assert got["variant"] == "fused_staged"
    rows = np.unique(np.concatenate([np.arange(0, m, 4099), np.arange(m - 300, m)]))
    sub = {"partials": [p[rows] for p in inp["partials"]], "residual": inp["residual"][rows],
           "weight": inp["weight"]}
    ref = oracle_fused(orc, sub, "bf16", gemma=True, quant=True)
    pick = {k: (v[rows] if v is not None and k != "variant" else v) for k, v in got.items()}
    check_fused(orc, pick, ref, "bf16", True)


# ---------------------------------------------------------------------------
# L2 prefetch ahead of the grid-dependency wait
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("variant", [tar.VARIANT_AUTO, tar.VARIANT_ROW, tar.VARIANT_STAGED, tar.VARIANT_CLUSTER])
def test_prefetch_changes_no_bit(ctx, dev, variant):
    """The kernels' L2 prefetch of their first inputs (issued before they wait for the previous
    kernel) is a hint only: every output is bit-identical with it on and off, including when
    the previous kernel on the stream writes the inputs of the next call."""
    ctx.set_option(tar.AR_OPT_FORCE_VARIANT, variant)
    inp = synth.fused_inputs(4, 300, 6144, "bf16", seed=41, gemma=True)
    parts = to_dev(inp["partials"], dev)
    res, w = inp["residual"].to(dev), inp["weight"].to(dev)
    outs = {}
    for pf in (0, 1):
        ctx.set_option(tar.AR_OPT_L2_PREFETCH, pf)
        # the first call writes into a partial of the second (a producer right before its consumer)
        p2 = [p.clone() for p in parts]
        ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6, gemma=True, quant=False, out=p2[1], want_residual_out=False)
        y, ro, q, sc = ctx.fused_reduce_rmsnorm(p2, res, w, eps=1e-6, gemma=True, quant=True)
        rs = torch.empty_like(parts[0])
        ctx.reduce_sum(p2, out=rs)
        torch.cuda.synchronize()
        outs[pf] = [bits_of(y), bits_of(ro), q.cpu().numpy(), sc.cpu().numpy(), bits_of(rs)]
    ctx.set_option(tar.AR_OPT_L2_PREFETCH, 1)
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)


def test_prefetch_changes_no_bit_cluster_and_batch(ctx, dev):
    """The same for the staged cluster form (rows split over CTAs, each prefetching its slice)
    and the batched kernel (each CTA prefetching its call's row)."""
    inp = synth.fused_inputs(4, 40, 16384, "bf16", seed=43, gemma=True)
    parts = to_dev(inp["partials"], dev)
    res, w = inp["residual"].to(dev), inp["weight"].to(dev)
    small = [synth.fused_inputs(2, m, 4096, "bf16", seed=44 + m) for m in (3, 17, 1)]
    outs = {}
    for pf in (0, 1):
        ctx.set_option(tar.AR_OPT_L2_PREFETCH, pf)
        y, ro, q, sc = ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6, gemma=True, quant=True)
        assert ctx.last_variant == "fused_staged_cluster"
        calls = [{"partials": to_dev(s["partials"], dev), "residual": s["residual"].to(dev),
                  "weight": s["weight"].to(dev), "quant": True} for s in small]
        res_b = ctx.fused_reduce_rmsnorm_batch(calls)
        assert ctx.last_variant == "fused_batch"
        torch.cuda.synchronize()
        outs[pf] = [bits_of(y), bits_of(ro), q.cpu().numpy(), sc.cpu().numpy()] + \
                   [x.view(torch.uint8).cpu().numpy() for r in res_b for x in r if x is not None]
    ctx.set_option(tar.AR_OPT_L2_PREFETCH, 1)
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
