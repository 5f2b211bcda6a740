"""Seeded random configurations of the fused call against the oracle.

Each case draws the number of partials (1-8), rows (0-600), hidden size (ragged, aligned and
wider than one CTA holds), element type, residual on or off, plain or gemma weighting, the
no-norm and fp32-output forms, per-token or per-group FP8 with or without the mirror, and
padded row strides, and runs it through the automatic choice of kernel.  Bars, as in every
parity test: residual_out bit-exact; y within one ulp of the oracle's (bit-exact without the
norm; fp32 output within 2^-19 relative); FP8 codes and scales exactly the oracle's
quantisation of the kernel's own 16-bit y (with fp32 output, where that row is not an output,
scales within one 16-bit ulp of amax and codes within one code of the oracle's).  Padding
columns of the outputs must stay untouched.

Source of the operation: page "[HIP] fix(custom-ar): gfx1250 fused all-reduce + RMSNorm",
Changes (the fused call's options), and page "[OUTDATED] perf: optimize fused AllReduce +
RMSNorm (custom_all_reduce)", Technical Details (fp32 rank-order reduction).
"""
import numpy as np
import pytest
import torch

import tensor_all_reduce_gb300 as tar
from tensor_all_reduce_gb300 import synth

from gpu_helpers import TDT, assert_bits_equal, assert_y_within_ulp, bits_of, code_ordinal

pytestmark = pytest.mark.gpu

F32_REL_TOL = 2.0 ** -19
CASES = 200


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


def draw(k):
    """The k-th random configuration (seeded, so every run draws the same cases)."""
    g = np.random.default_rng(9000 + k)
    n = int(g.integers(1, 9))
    dtype = ["bf16", "fp16"][int(g.integers(0, 2))]
    kind = g.random()
    if kind < 0.15:
        h = int(g.integers(1, 64))                              # short, mostly ragged rows
    elif kind < 0.75:
        h = int(g.integers(1, 1025)) * 8                        # aligned rows up to 8192
    elif kind < 0.9:
        h = int(g.integers(1, 8193))                            # any length up to 8192
    else:
        h = [12288, 16384, 10240, 9000][int(g.integers(0, 4))]  # wider than one CTA holds
    m_max = max(1, min(600, 3_000_000 // (h * (n + 3))))
    m = int(g.integers(0, m_max + 1)) if g.random() < 0.95 else 0
    skip_norm = g.random() < 0.2
    out_fp32 = (not skip_norm) and g.random() < 0.15
    quant = g.random() < 0.6
    group = 0
    if quant and g.random() < 0.35 and h <= 8192:
        options = [gs for gs in (8, 16, 32, 64, 128, 256) if h % gs == 0]
        group = int(g.choice(options)) if options else 0
    pad_in = [0, 0, 8, 3, 64][int(g.integers(0, 5))]
    pad_out = [0, 0, 16, 5][int(g.integers(0, 4))]
    return dict(n=n, m=m, h=h, dtype=dtype, residual=g.random() < 0.85, gemma=g.random() < 0.5,
                skip_norm=skip_norm, out_fp32=out_fp32, quant=quant, group=group,
                mirror=out_fp32 or not quant or g.random() < 0.8, pad_in=pad_in, pad_out=pad_out,
                seed=100 + k)


def _view(t, pad, dev, fill=None):
    m, h = t.shape
    big = torch.empty((m, h + pad), dtype=t.dtype, device=dev)
    if fill is None:
        big.view(torch.uint8).fill_(0x5A)
        big[:, :h].copy_(t)
    else:
        big.view(torch.uint8).fill_(fill)
    return big, big[:, :h]


def _pads_intact(big, h):
    raw = big[:, h:].contiguous().view(torch.uint8)
    return bool((raw == 0xA5).all().item()) if raw.numel() else True


@pytest.mark.parametrize("k", range(CASES))
def test_random_configuration(ctx, dev, orc, k):
    c = draw(k)
    n, m, h, dt = c["n"], c["m"], c["h"], c["dtype"]
    inp = synth.fused_inputs(n, m, h, dt, seed=c["seed"], gemma=c["gemma"], residual=c["residual"])
    parts = [_view(p, c["pad_in"], dev)[1] for p in inp["partials"]]
    res = _view(inp["residual"], c["pad_in"], dev)[1] if c["residual"] else None
    w = None if c["skip_norm"] else inp["weight"].to(dev)
    t16 = TDT[dt]
    ro_big, ro = _view(torch.empty((m, h), dtype=t16), c["pad_out"], dev, fill=0xA5)
    y_big = y = None
    if c["mirror"]:
        y_big, y = _view(torch.empty((m, h), dtype=torch.float32 if c["out_fp32"] else t16), c["pad_out"], dev,
                         fill=0xA5)
    q_big = q = sc = None
    if c["quant"]:
        q_big, q = _view(torch.empty((m, h), dtype=torch.uint8), c["pad_out"], dev, fill=0xA5)
        sc = torch.full((m, h // c["group"]) if c["group"] else (m,), float("nan"), dtype=torch.float32, device=dev)
    ctx.fused_reduce_rmsnorm(parts, res, w, eps=1e-6, gemma=c["gemma"], quant=c["quant"], out=y, residual_out=ro,
                             q_out=q, scale_out=sc, want_out=c["mirror"], skip_norm=c["skip_norm"],
                             out_fp32=c["out_fp32"], group_size=c["group"])
    torch.cuda.synchronize()
    if m == 0:
        assert ctx.last_variant == "none"
        return
    ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                       None if c["skip_norm"] else synth.bits(inp["weight"]), 1e-6, c["gemma"], c["quant"], dt,
                       skip_norm=c["skip_norm"], out_fp32=c["out_fp32"], group=c["group"])
    what = f"case {k} {c} ({ctx.last_variant})"
    assert_bits_equal(bits_of(ro), ref["res_out"], f"residual_out, {what}")
    assert _pads_intact(ro_big, h), what
    y16 = None
    if c["mirror"]:
        assert _pads_intact(y_big, h), what
        if c["out_fp32"]:
            g32, r32 = y.cpu().numpy().astype(np.float64), ref["y32"].astype(np.float64)
            assert np.all(np.abs(g32 - r32) <= F32_REL_TOL * np.abs(r32) + 1e-30), what
        else:
            y16 = bits_of(y)
            if c["skip_norm"]:
                assert_bits_equal(y16, ref["y"], f"output (= z), {what}")
            else:
                assert_y_within_ulp(y16, ref["y"], dt, f"y, {what}")
    elif c["skip_norm"]:
        y16 = ref["res_out"]          # without the norm the kernel's y is z = residual_out
    if c["quant"]:
        assert _pads_intact(q_big, h), what
        qg, sg = q.cpu().numpy(), sc.cpu().numpy()
        assert not np.any((qg & 0x7F) == 0x7F), f"NaN code, {what}"
        if y16 is not None:
            q_ref, s_ref = (orc.per_group_quant(y16, c["group"], dt) if c["group"]
                            else orc.per_token_quant(y16, dt))
            assert np.array_equal(sg.view(np.uint32), s_ref.view(np.uint32)), f"scales, {what}"
            assert np.array_equal(qg, q_ref), f"codes, {what}"
        else:
            tol = 2.0 ** -7 if dt == "bf16" else 2.0 ** -10
            s_g, s_r = sg.astype(np.float64), ref["scale"].astype(np.float64)
            assert np.all(np.abs(s_g - s_r) <= tol * s_r * 1.0001), f"scales, {what}"
            d = np.abs(code_ordinal(qg) - code_ordinal(ref["q"]))
            assert d.max(initial=0) <= 1, f"codes, {what}"


# ---------------------------------------------------------------------------
# the plain sum: random lengths, partial counts, element types and alignments
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("k", range(60))
def test_random_reduce(ctx, dev, orc, k):
    g = np.random.default_rng(7000 + k)
    n = int(g.integers(1, 9))
    dtype = ["bf16", "fp16", "fp32"][int(g.integers(0, 3))]
    numel = int(g.integers(1, 3_000_000)) if g.random() < 0.8 else int(g.integers(1, 600))
    off_in, off_out = [(0, 0), (0, 0), (1, 0), (0, 1), (3, 5)][int(g.integers(0, 5))]
    t = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dtype]
    parts_cpu = synth.reduce_inputs(n, numel, dtype, seed=500 + k)
    parts = []
    for p in parts_cpu:
        buf = torch.empty(numel + off_in, dtype=t, device=dev)
        buf[off_in:].copy_(p.to(dev))
        parts.append(buf[off_in:])
    out_buf = torch.full((numel + off_out + 64,), float("nan"), dtype=t, device=dev)
    out = out_buf[off_out:off_out + numel]
    in_place = g.random() < 0.1 and off_in == off_out
    if in_place:
        out = parts[int(g.integers(0, n))]
    ctx.reduce_sum(parts, out=out)
    torch.cuda.synchronize()
    ref = orc.reduce_sum([synth.bits(p) for p in parts_cpu], dtype)
    assert_bits_equal(synth.bits(out.cpu()), ref, f"reduce case {k}: n={n} {dtype} numel={numel} "
                                                  f"offsets {off_in},{off_out} ({ctx.last_variant})")
    if not in_place:
        assert bool(torch.isnan(out_buf[off_out + numel:].float()).all())       # nothing past the end


# ---------------------------------------------------------------------------
# batches of independent calls
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("k", range(30))
def test_random_batch(ctx, dev, orc, k):
    g = np.random.default_rng(8000 + k)
    n = int(g.integers(1, 9))
    dtype = ["bf16", "fp16"][int(g.integers(0, 2))]
    quant = g.random() < 0.5
    skip_norm = g.random() < 0.2
    ragged = g.random() < 0.2                     # one call with an unaligned hidden size: separate launches
    count = int(g.integers(1, tar.AR_MAX_BATCH + 1))
    calls, keep = [], []
    for j in range(count):
        m = int(g.integers(0, 40))
        h = int(g.integers(1, 1025)) * 8 if not (ragged and j == 0) else int(g.integers(1, 4000)) * 8 + 3
        gemma = g.random() < 0.5
        inp = synth.fused_inputs(n, m, h, dtype, seed=900 + 31 * k + j, gemma=gemma)
        call = {"partials": [p.to(dev) for p in inp["partials"]], "residual": inp["residual"].to(dev),
                "weight": None if skip_norm else inp["weight"].to(dev), "eps": 1e-6, "gemma": gemma,
                "quant": quant, "skip_norm": skip_norm}
        calls.append(call)
        keep.append((inp, gemma))
    results = ctx.fused_reduce_rmsnorm_batch(calls)
    torch.cuda.synchronize()
    for j, ((inp, gemma), (y, ro, q, sc)) in enumerate(zip(keep, results)):
        if inp["partials"][0].shape[0] == 0:
            continue
        ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                           None if skip_norm else synth.bits(inp["weight"]), 1e-6, gemma, quant, dtype,
                           skip_norm=skip_norm)
        what = f"batch case {k} call {j} ({ctx.last_variant})"
        assert_bits_equal(bits_of(ro), ref["res_out"], f"residual_out, {what}")
        y16 = bits_of(y)
        if skip_norm:
            assert_bits_equal(y16, ref["y"], f"output (= z), {what}")
        else:
            assert_y_within_ulp(y16, ref["y"], dtype, f"y, {what}")
        if quant:
            q_ref, s_ref = orc.per_token_quant(y16, dtype)
            assert np.array_equal(sc.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), what
            assert np.array_equal(q.cpu().numpy(), q_ref), what


# ---------------------------------------------------------------------------
# the other entry points: host buffers and the allocation-free call
# ---------------------------------------------------------------------------

def _check_fused(orc, c, inp, ro, y, q, sc, what):
    """The bars of test_random_configuration for outputs already copied to the host."""
    dt = c["dtype"]
    ref = orc.fused_ex([synth.bits(p) for p in inp["partials"]], synth.bits(inp["residual"]),
                       None if c["skip_norm"] else synth.bits(inp["weight"]), 1e-6, c["gemma"], c["quant"], dt,
                       skip_norm=c["skip_norm"], out_fp32=c["out_fp32"], group=c["group"])
    assert_bits_equal(synth.bits(ro), ref["res_out"], f"residual_out, {what}")
    y16 = None
    if y is not None and c["out_fp32"]:
        g32, r32 = y.numpy().astype(np.float64), ref["y32"].astype(np.float64)
        assert np.all(np.abs(g32 - r32) <= F32_REL_TOL * np.abs(r32) + 1e-30), what
    elif y is not None:
        y16 = synth.bits(y)
        if c["skip_norm"]:
            assert_bits_equal(y16, ref["y"], f"output (= z), {what}")
        else:
            assert_y_within_ulp(y16, ref["y"], dt, f"y, {what}")
    if c["quant"]:
        qg, sg = q.numpy(), sc.numpy()
        if y16 is not None:
            q_ref, s_ref = orc.per_group_quant(y16, c["group"], dt) if c["group"] else orc.per_token_quant(y16, dt)
            assert np.array_equal(sg.view(np.uint32), s_ref.view(np.uint32)), f"scales, {what}"
            assert np.array_equal(qg, q_ref), f"codes, {what}"
        else:
            tol = 2.0 ** -7 if dt == "bf16" else 2.0 ** -10
            s_g, s_r = sg.astype(np.float64), ref["scale"].astype(np.float64)
            assert np.all(np.abs(s_g - s_r) <= tol * s_r * 1.0001), f"scales, {what}"
            assert np.abs(code_ordinal(qg) - code_ordinal(ref["q"])).max(initial=0) <= 1, f"codes, {what}"


@pytest.mark.parametrize("k", range(40))
def test_random_configuration_host_buffers(ctx, dev, orc, k):
    """Random configurations through ar_fused_reduce_rmsnorm_host, every buffer page-locked
    host memory (padded rows included)."""
    c = draw(1000 + k)
    n, m, h, dt = c["n"], c["m"], c["h"], c["dtype"]
    if m == 0:
        return
    m = min(m, 64)                                     # host memory is read across the CPU-GPU link
    inp = synth.fused_inputs(n, m, h, dt, seed=c["seed"], gemma=c["gemma"], residual=c["residual"])

    def pinned(t, pad):
        big = torch.empty((m, h + pad), dtype=t.dtype, pin_memory=True)
        big[:, :h].copy_(t)
        return big[:, :h]

    parts = [pinned(p, c["pad_in"]) for p in inp["partials"]]
    res = pinned(inp["residual"], c["pad_in"]) if c["residual"] else None
    w = None if c["skip_norm"] else inp["weight"].pin_memory()
    t16 = TDT[dt]
    zeros = lambda dtype: torch.zeros((m, h), dtype=dtype)
    ro = pinned(zeros(t16), c["pad_out"])
    y = pinned(zeros(torch.float32 if c["out_fp32"] else t16), c["pad_out"]) if c["mirror"] else None
    q = pinned(zeros(torch.uint8), c["pad_out"]) if c["quant"] else None
    sc = (torch.empty((m, h // c["group"]) if c["group"] else (m,), dtype=torch.float32, pin_memory=True)
          if c["quant"] else None)
    ctx.fused_reduce_rmsnorm_host(parts, res, w, eps=1e-6, gemma=c["gemma"], quant=c["quant"], out=y, residual_out=ro,
                                  q_out=q, scale_out=sc, want_out=c["mirror"], skip_norm=c["skip_norm"],
                                  out_fp32=c["out_fp32"], group_size=c["group"])
    torch.cuda.synchronize()
    what = f"host case {k} {c} m={m} ({ctx.last_variant})"
    if y is None and c["skip_norm"]:
        y = ro
    _check_fused(orc, c, inp, ro.clone(), None if y is None else y.clone(), None if q is None else q.clone(),
                 None if sc is None else sc.clone(), what)


@pytest.mark.parametrize("k", range(40))
def test_random_configuration_noalloc(dev, orc, k):
    """Random configurations (16-byte-aligned rows of at most 8192 elements, what the entry
    takes) through the allocation-free ar_fused_reduce_rmsnorm_noalloc."""
    c = draw(2000 + k)
    n, m, dt = c["n"], c["m"], c["dtype"]
    h = max(8, min(8192, c["h"] // 8 * 8))
    if c["group"] and h % c["group"]:
        c["group"] = 8
    pad_in, pad_out = c["pad_in"] // 8 * 8, c["pad_out"] // 8 * 8
    inp = synth.fused_inputs(n, m, h, dt, seed=c["seed"], gemma=c["gemma"], residual=c["residual"])
    parts = [_view(p, pad_in, dev)[1] for p in inp["partials"]]
    res = _view(inp["residual"], pad_in, dev)[1] if c["residual"] else None
    w = None if c["skip_norm"] else inp["weight"].to(dev)
    t16 = TDT[dt]
    ro = _view(torch.empty((m, h), dtype=t16), pad_out, dev, fill=0xA5)[1]
    y = _view(torch.empty((m, h), dtype=torch.float32 if c["out_fp32"] else t16), pad_out, dev, fill=0xA5)[1] \
        if c["mirror"] else None
    q = _view(torch.empty((m, h), dtype=torch.uint8), pad_out, dev, fill=0xA5)[1] if c["quant"] else None
    sc = (torch.full((m, h // c["group"]) if c["group"] else (m,), float("nan"), dtype=torch.float32, device=dev)
          if c["quant"] else None)
    ptr = lambda t: None if t is None else t.data_ptr()
    code = tar.AR_DTYPE_BF16 if dt == "bf16" else tar.AR_DTYPE_F16
    args = tar.make_fused_args([p.data_ptr() for p in parts], ptr(res), ptr(ro), ptr(w), ptr(y), 1e-6, c["gemma"],
                               c["quant"], ptr(q), ptr(sc), m, h, code, skip_norm=c["skip_norm"],
                               out_fp32=c["out_fp32"], group_size=c["group"], ld_in=h + pad_in, ld_out=h + pad_out)
    tar.ar_fused_reduce_rmsnorm_noalloc(args, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    if m == 0:
        return
    if y is None and c["skip_norm"]:
        y = ro
    _check_fused(orc, c, inp, ro.cpu(), None if y is None else y.cpu(), None if q is None else q.cpu(),
                 None if sc is None else sc.cpu(), f"noalloc case {k} {c} h={h}")
