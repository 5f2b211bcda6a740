"""Host-side checks of the C ABI that need no GPU: the library loads, exports every entry
point include/ar.h declares, and rejects bad arguments before launching anything.

Argument validation runs before the context is consulted, so with ctx = NULL a bad call
returns its argument error and a good call returns AR_ERR_NOT_INITIALIZED.  Pointer values
below are never dereferenced (they are only compared and range-checked on the host).
"""
import ctypes
import os
import re

import pytest

import tensor_all_reduce_gb300 as tar

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ar.h")


@pytest.fixture(scope="module")
def lib():
    from tensor_all_reduce_gb300 import _build
    _build.build()
    return tar.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:ar_status|const char\s*\*)\s*(ar_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ar_init", "ar_reduce_sum", "ar_fused_reduce_rmsnorm", "ar_destroy", "ar_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings(lib):
    for code in range(7):
        assert tar.status_string(code) not in ("", "unknown status")
    assert tar.status_string(99) == "unknown status"


def test_null_context_queries(lib):
    v = ctypes.c_int64()
    assert lib.ar_get_info(None, tar.AR_INFO_SM_COUNT, ctypes.byref(v)) == tar.AR_ERR_NOT_INITIALIZED
    assert lib.ar_set_option(None, tar.AR_OPT_CLUSTER_SIZE, 4) == tar.AR_ERR_NOT_INITIALIZED
    assert lib.ar_set_option(None, tar.AR_OPT_TEST_STALL, 1) == tar.AR_ERR_NOT_INITIALIZED
    assert lib.ar_set_option(None, tar.AR_OPT_L2_PREFETCH, 0) == tar.AR_ERR_NOT_INITIALIZED
    assert lib.ar_destroy(None) == tar.AR_OK
    assert tar.ar_last_variant(None) == ""
    assert lib.ar_init(None, 0, 0) == tar.AR_ERR_INVALID_ARG
    code = ctypes.c_int(-1)
    assert lib.ar_device_status(None, ctypes.byref(code)) == tar.AR_ERR_NOT_INITIALIZED
    assert lib.ar_device_status(None, None) == tar.AR_ERR_INVALID_ARG


BASE = 1 << 40   # fake, well-aligned device addresses; never dereferenced
MB = 1 << 20


def reduce_status(out, parts, numel, dtype=tar.AR_DTYPE_BF16):
    return tar.ar_reduce_sum(None, out, parts, numel, dtype, None, raise_on_error=False)


def test_reduce_validation(lib):
    p = [BASE + i * MB for i in range(4)]
    out = BASE + 16 * MB
    assert reduce_status(out, p, 1000) == tar.AR_ERR_NOT_INITIALIZED           # valid
    assert reduce_status(p[2], p, 1000) == tar.AR_ERR_NOT_INITIALIZED          # exact in-place alias
    assert reduce_status(0, p, 1000) == tar.AR_ERR_INVALID_ARG                 # null out
    assert reduce_status(out, [], 1000) == tar.AR_ERR_INVALID_ARG              # n = 0
    assert reduce_status(out, p * 3, 1000) == tar.AR_ERR_INVALID_ARG           # n = 12 > 8
    assert reduce_status(out, p, -1) == tar.AR_ERR_INVALID_ARG                 # negative numel
    assert reduce_status(out, p, 10, dtype=7) == tar.AR_ERR_INVALID_ARG        # bad dtype
    assert reduce_status(out, p[:1] + [0], 10) == tar.AR_ERR_INVALID_ARG       # null partial
    assert reduce_status(out + 1, p, 10) == tar.AR_ERR_ALIGNMENT               # odd address, bf16
    assert reduce_status(out + 2, p, 10, tar.AR_DTYPE_F32) == tar.AR_ERR_ALIGNMENT
    assert reduce_status(p[1] + 64, p, 1000) == tar.AR_ERR_OVERLAP             # partial overlap
    assert reduce_status(out, p, 0) == tar.AR_ERR_NOT_INITIALIZED              # empty is valid


def fused_args(**kw):
    m, h = kw.pop("m", 16), kw.pop("h", 6144)
    tb = m * h * 2
    d = dict(partials=[BASE + i * 64 * MB for i in range(4)], residual_in=BASE + 4 * 64 * MB,
             residual_out=BASE + 5 * 64 * MB, weight=BASE + 6 * 64 * MB, out=BASE + 7 * 64 * MB,
             eps=1e-6, gemma=False, quant=False, q_out=None, scale_out=None, m=m, h=h,
             dtype=tar.AR_DTYPE_BF16)
    n_override = kw.pop("n", None)
    d.update(kw)
    assert tb < 64 * MB
    a = tar.make_fused_args(**d)
    if n_override is not None:
        a.n = n_override
    return a


def fused(**kw):
    return tar.ar_fused_reduce_rmsnorm(None, fused_args(**kw), None, raise_on_error=False)


def test_fused_validation(lib):
    NI = tar.AR_ERR_NOT_INITIALIZED
    assert fused() == NI
    assert fused(m=0) == NI                                             # empty batch is valid
    assert fused(residual_in=None, residual_out=None) == NI
    assert fused(residual_out=BASE + 4 * 64 * MB) == NI                 # residual_out == residual_in
    assert fused(out=BASE) == NI                                        # out == partials[0] exactly
    assert fused(quant=True, q_out=BASE + 8 * 64 * MB, scale_out=BASE + 9 * 64 * MB) == NI
    assert fused(quant=True, out=None, q_out=BASE + 8 * 64 * MB, scale_out=BASE + 9 * 64 * MB) == NI
    IA = tar.AR_ERR_INVALID_ARG
    assert fused(h=0) == IA
    assert fused(m=-1) == IA
    assert fused(weight=None) == IA
    assert fused(out=None) == IA                                        # no output without quant
    assert fused(quant=True, q_out=None, scale_out=BASE + 9 * 64 * MB) == IA
    assert fused(quant=True, q_out=BASE + 8 * 64 * MB, scale_out=None) == IA
    assert fused(dtype=tar.AR_DTYPE_F32) == IA                          # fused is 16-bit only
    assert fused(eps=float("nan")) == IA
    assert fused(eps=-1.0) == IA
    assert fused(eps=float("inf")) == IA
    assert fused(partials=[]) == IA
    assert fused(n=9) == IA
    assert fused(partials=[BASE, 0, BASE + 64 * MB]) == IA
    AL = tar.AR_ERR_ALIGNMENT
    assert fused(out=BASE + 7 * 64 * MB + 1) == AL
    assert fused(weight=BASE + 6 * 64 * MB + 1) == AL
    assert fused(quant=True, q_out=BASE + 8 * 64 * MB, scale_out=BASE + 9 * 64 * MB + 2) == AL
    # without the norm the weight may be absent; with it, it may not
    assert fused(weight=None, skip_norm=True) == NI
    assert fused(weight=None, skip_norm=False) == IA
    # fp32 output: 4-byte alignment, and never an alias of a 16-bit input
    assert fused(out_fp32=True, out=BASE + 7 * 64 * MB + 2) == AL
    assert fused(out_fp32=True, m=8) == NI
    # per-group FP8: a power-of-two group of 8..256 elements that divides h, rows <= 8192
    QG = dict(quant=True, q_out=BASE + 8 * 64 * MB, scale_out=BASE + 9 * 64 * MB)
    assert fused(group_size=128, **QG) == NI
    assert fused(group_size=100, **QG) == IA
    assert fused(group_size=512, **QG) == IA
    assert fused(group_size=4, **QG) == IA
    assert fused(group_size=128, h=6144 + 64, **QG) == IA
    assert fused(group_size=128, h=16384, m=4, **QG) == tar.AR_ERR_UNSUPPORTED
    # padded rows: strides of at least h
    assert fused(ld_in=6144 + 64, ld_out=6144 + 8) == NI
    assert fused(ld_in=6000) == IA
    assert fused(ld_out=100) == IA
    assert fused(ld_in=-8) == IA
    OV = tar.AR_ERR_OVERLAP
    assert fused(out_fp32=True, out=BASE) == OV                          # fp32 y over partials[0]
    # an output on an input is allowed only with the same row stride
    assert fused(out=BASE, ld_in=6144 + 64, ld_out=6144 + 64) == NI
    assert fused(out=BASE, ld_in=6144 + 64, ld_out=6144) == OV
    # strided extents count: residual_out's 16 rows with stride 4.5M elements span 135 MB
    # and reach `out`, 128 MB further on
    assert fused(ld_out=4_500_000) == OV
    # the per-group scales are m * h / G floats: these would run into the codes
    assert fused(group_size=8, quant=True, q_out=BASE + 8 * 64 * MB + 16 * 6144 // 8 * 4 - 4,
                 scale_out=BASE + 8 * 64 * MB) == OV
    assert fused(out=BASE + 32) == OV                                   # inside partials[0]
    assert fused(residual_out=BASE + 7 * 64 * MB) == OV                 # residual_out == out
    assert fused(out=BASE + 6 * 64 * MB) == OV                          # out on the weight
    assert fused(quant=True, q_out=BASE, scale_out=BASE + 9 * 64 * MB) == OV  # codes over a partial
    assert fused(quant=True, q_out=BASE + 8 * 64 * MB, scale_out=BASE + 8 * 64 * MB + 64) == OV


def test_options_reject_out_of_range_values(lib):
    # ar_set_option checks the context first; the value ranges are exercised on the GPU
    assert lib.ar_set_option(None, 99, 0) == tar.AR_ERR_NOT_INITIALIZED


def test_batch_validation(lib):
    def call(base, **kw):
        d = dict(partials=[base + i * 64 * MB for i in range(4)], residual_in=base + 4 * 64 * MB,
                 residual_out=base + 5 * 64 * MB, weight=BASE + 6 * 64 * MB, out=base + 7 * 64 * MB,
                 eps=1e-6, gemma=False, quant=False, q_out=None, scale_out=None, m=16, h=6144,
                 dtype=tar.AR_DTYPE_BF16)
        d.update(kw)
        return tar.make_fused_args(**d)

    B2 = BASE + (1 << 36)
    NI, IA, OV = tar.AR_ERR_NOT_INITIALIZED, tar.AR_ERR_INVALID_ARG, tar.AR_ERR_OVERLAP
    st = lambda calls: tar.ar_fused_reduce_rmsnorm_batch(None, calls, None, raise_on_error=False)
    assert st([call(BASE), call(B2)]) == NI                         # shared weight is fine
    assert st([]) == IA
    assert st([call(BASE + i * (1 << 33)) for i in range(tar.AR_MAX_BATCH + 1)]) == IA
    assert st([call(BASE), call(B2, partials=[B2, B2 + 64 * MB])]) == IA       # different n
    assert st([call(BASE), call(B2, dtype=tar.AR_DTYPE_F16)]) == IA
    assert st([call(BASE), call(B2, out=BASE)]) == OV               # writes call 0's partial
    assert st([call(BASE), call(B2, residual_out=BASE + 5 * 64 * MB)]) == OV   # same output
    assert st([call(BASE), call(B2, h=0)]) == IA                    # per-call rules apply



def test_host_entry_validates_like_the_device_entry(lib):
    # ar_fused_reduce_rmsnorm_host applies the device entry's argument rules before it looks
    # at what memory the pointers name
    QG = dict(quant=True, q_out=BASE + 8 * 64 * MB, scale_out=BASE + 9 * 64 * MB)
    cases = [dict(), dict(m=0), dict(h=0), dict(m=-1), dict(weight=None), dict(weight=None, skip_norm=True),
             dict(out=None), dict(dtype=tar.AR_DTYPE_F32), dict(eps=float("nan")), dict(n=9),
             dict(out=BASE + 7 * 64 * MB + 1), dict(out=BASE + 32), dict(residual_out=BASE + 7 * 64 * MB),
             dict(group_size=128, **QG), dict(group_size=100, **QG), dict(group_size=128, h=16384, m=4, **QG),
             dict(ld_in=6000), dict(ld_in=6144 + 64, ld_out=6144 + 8), dict(out_fp32=True, out=BASE)]
    for kw in cases:
        a = fused_args(**dict(kw))
        dev_st = tar.ar_fused_reduce_rmsnorm(None, a, None, raise_on_error=False)
        host_st = tar.ar_fused_reduce_rmsnorm_host(None, a, None, raise_on_error=False)
        assert host_st == dev_st, (kw, host_st, dev_st)
    assert lib.ar_fused_reduce_rmsnorm_host(None, None, None) == tar.AR_ERR_INVALID_ARG


def test_binding_has_a_function_for_every_entry_point(lib):
    # the Python binding mirrors the C ABI name for name
    for name in declared_functions():
        assert hasattr(tar, name), f"no binding for {name}"


def test_header_compiles_and_links_as_plain_c(lib, tmp_path):
    """include/ar.h is a C header: a C11 program compiles against it (warnings as errors) and
    links to libar.so; it runs only the calls that need no GPU."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "ar.h"
int main(void) {
  ar_fused_args a;
  memset(&a, 0, sizeof a);
  a.n = 1; a.h = 0; a.dtype = AR_DTYPE_BF16;            /* h = 0: refused before anything else */
  if (ar_fused_reduce_rmsnorm(NULL, &a, NULL) != AR_ERR_INVALID_ARG) return 1;
  if (ar_fused_reduce_rmsnorm_host(NULL, &a, NULL) != AR_ERR_INVALID_ARG) return 2;
  if (ar_destroy(NULL) != AR_OK) return 3;
  if (strcmp(ar_status_string(AR_OK), "success") != 0) return 4;
  if (ar_reduce_sum(NULL, NULL, NULL, 0, 0, AR_DTYPE_F32, NULL) != AR_ERR_INVALID_ARG) return 5;
  printf("ok %d\n", AR_MAX_PARTIALS);
  return 0;
}
''')
    libdir = os.path.dirname(tar.LIB_PATH)
    exe = tmp_path / "abi"
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-lar", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == f"ok {tar.AR_MAX_PARTIALS}", (r.returncode, r.stdout, r.stderr)


def test_binding_constants_match_the_header():
    """Every AR_* constant of the binding has the value include/ar.h gives it, and every valued
    AR_* name of the header (enumerators and #defines) is mirrored in the binding."""
    text = open(os.path.join(ROOT, "include", "ar.h")).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    header = {k: int(v) for k, v in re.findall(r"\b(AR_[A-Z0-9_]+)\s*=\s*(\d+)", text)}
    header.update({k: int(v) for k, v in re.findall(r"#define\s+(AR_[A-Z0-9_]+)\s+(\d+)", text)})
    assert len(header) >= 29
    binding = {k: getattr(tar, k) for k in dir(tar) if k.startswith("AR_") and isinstance(getattr(tar, k), int)}
    missing = sorted(set(header) - set(binding) - {"AR_NOALLOC_SCRATCH_BYTES"})
    assert not missing, f"header constants without a binding mirror: {missing}"
    wrong = {k: (binding[k], header[k]) for k in binding if k in header and binding[k] != header[k]}
    assert not wrong, f"binding constants that differ from the header: {wrong}"
    assert set(binding) <= set(header), sorted(set(binding) - set(header))
