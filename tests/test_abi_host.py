"""Host-side checks of the C-ABI library (no GPU): symbols, validation, knobs."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_smem_gb300 import build as b
    b.build()
    from exact_attention_smem_gb300 import _lib
    return _lib.load()


def _declared(header="fa.h", macro="FA_API"):
    src = open(os.path.join(ROOT, "include", header)).read()
    return re.findall(macro + r"[^;]*?\b(fa_\w+)\s*\(", src)


def _dynamic_symbols(path):
    """Names in the library's dynamic symbol table that start with fa_."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.split()[-1].startswith("fa_")}


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    from exact_attention_smem_gb300 import _lib
    assert set(_lib.exported_symbols()) == set(names)
    # the attention library exports exactly the contract: no test hooks
    assert _dynamic_symbols(_lib.LIB_PATH) == set(names)


def test_test_library_exports_its_header(lib):
    import fa_testing_lib as ft
    tlib = ft.load()
    names = _declared("fa_testing.h", "FA_TEST_API")
    assert len(names) >= 10
    for n in names:
        assert hasattr(tlib, n), n
    assert set(ft.SIGS) == set(names)
    assert _dynamic_symbols(ft.TEST_LIB_PATH) == set(names)
    assert not set(names) & set(_declared())


def test_status_strings(lib):
    for s in range(7):
        assert lib.fa_status_string(s)
    assert lib.fa_status_string(99) == b"unknown status"


FAKE = 0x7f0000000000  # never dereferenced: validation rejects before any CUDA call


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=2, Sq=16, Sk=16, d=128,
             causal=0, scale=0.1, cu=None)
    a.update(kw)
    return lib.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Sq"],
                      a["Sk"], a["d"], a["causal"], a["scale"], a["cu"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), 1), (dict(lse=None), 1), (dict(v=FAKE + 8), 1), (dict(d=96), 2),
    (dict(d=320), 2), (dict(Hq=3, Hkv=2), 1), (dict(Hkv=0), 1), (dict(scale=float("nan")), 1),
    (dict(scale=-1.0), 1), (dict(scale=float("inf")), 1), (dict(Sq=-1), 1),
    (dict(cu=FAKE, Sq=16, Sk=8), 1),
])
def test_forward_validation(lib, kw, status):
    assert _fwd(lib, **kw) == status
    assert lib.fa_last_error()


def test_forward_empty_is_noop(lib):
    assert _fwd(lib, B=0) == 0
    assert _fwd(lib, Sq=0, Sk=0) == 0


def test_backward_validation_and_workspace(lib):
    # fp32 dQ accumulator [T][Hq][d] (used by the one-pass form) + two padded
    # fp32 row arrays [Hq][P], P = round_up(T, 128) + 256 * (nseq + 1), each
    # part rounded up to 256 bytes
    need = lib.fa_bwd_workspace_bytes(2, 4, 100, 128, 0)
    assert need == 200 * 4 * 128 * 4 + 2 * (1024 * 4 * 4) + 256   # + boundary lists (3 ints each)
    assert lib.fa_bwd_workspace_bytes(1, 4, 300, 64, 512) == 512 * 4 * 64 * 4 + 2 * (1024 * 4 * 4) + 256
    args = [FAKE] * 9 + [2, 4, 4, 100, 100, 128, 1, 0.1, None]
    assert lib.fa_bwd(*args, FAKE, need - 1, None) == 5
    assert lib.fa_bwd(*args, FAKE + 16, need, None) == 5      # workspace must be 256-aligned
    assert lib.fa_bwd(*args, None, need, None) == 5
    # head dims outside {64, 128, 192, 256} are rejected before any device work
    big = [FAKE] * 9 + [2, 4, 4, 100, 100, 320, 1, 0.1, None]
    assert lib.fa_bwd(*big, FAKE, 1 << 30, None) == 2
    bad = [FAKE] * 8 + [None] + [2, 4, 4, 100, 100, 128, 1, 0.1, None]
    assert lib.fa_bwd(*bad, FAKE, need, None) == 1


def test_debug_knobs(lib):
    assert lib.fa_debug_set(b"tau", 2.0) == 0
    assert lib.fa_debug_set(b"tau", 0.0) == 0
    assert lib.fa_debug_set(b"tau", -1.0) == 1
    assert lib.fa_debug_set(b"poly8", 3.0) == 1
    assert lib.fa_debug_set(b"nope", 1.0) == 1
    for v in (-1.0, 0.0, 1.0):
        assert lib.fa_debug_set(b"fwd_split_q", v) == 0
    assert lib.fa_debug_set(b"fwd_split_q", 2.0) == 1
    assert lib.fa_debug_set(b"fwd_split_q", -1.0) == 0
    assert lib.fa_debug_set(None, 1.0) == 1


def test_fp8_entry_points_validate_before_any_device_work(lib):
    f = FAKE
    # fa_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale)
    ok = [f] * 8 + [1, 2, 2, 16, 16, 128, 1, 0.1]
    def fwd8(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.fa_fwd_fp8(*a, None)
    assert fwd8(a0=None) == 1 and fwd8(a5=None) == 1 and fwd8(a7=None) == 1
    assert fwd8(a2=f + 4) == 1                      # vt8 not 16-byte aligned
    assert fwd8(a13=64) == 2                        # head dim 128 only
    assert fwd8(a9=3) == 1                          # Hq % Hkv
    assert fwd8(a15=float("nan")) == 1 and fwd8(a15=0.0) == 1
    assert fwd8(a8=0) == 0 and fwd8(a11=0) == 0     # nothing to do
    # fa_quantize_fp8(x, B, S, H, d, layout, codes, scales)
    assert lib.fa_quantize_fp8(None, 1, 16, 1, 128, 0, f, f, None) == 1
    assert lib.fa_quantize_fp8(f, 1, 16, 1, 128, 2, f, f, None) == 1
    assert lib.fa_quantize_fp8(f, 1, 16, 1, 96, 0, f, f, None) == 2
    assert lib.fa_quantize_fp8(f + 8, 1, 16, 1, 128, 1, f, f, None) == 1
    assert lib.fa_quantize_fp8(f, 0, 16, 1, 128, 1, f, f, None) == 0
    assert lib.fa_last_error() is not None


def test_fp8_knobs(lib):
    assert lib.fa_debug_set(b"fp8_tau", 0.0) == 0
    assert lib.fa_debug_set(b"fp8_tau", 1.5) == 0
    assert lib.fa_debug_set(b"fp8_tau", 1.6) == 1     # 2^(7 + tau) must stay below 448
    assert lib.fa_debug_set(b"fp8_poly8", 2.0) == 0
    assert lib.fa_debug_set(b"fp8_poly8", 0.0) == 0
    assert lib.fa_debug_set(b"fp8_poly8", 1.0) == 1


def test_merge_validates_before_any_device_work(lib):
    f = FAKE
    # fa_merge(o_parts, lse_parts, P, B, Hq, S, d, packed, o, lse, stream)
    assert lib.fa_merge(None, f, 2, 1, 1, 16, 128, 0, f, f, None) == 1
    assert lib.fa_merge(f + 2, f, 2, 1, 1, 16, 128, 0, f, f, None) == 1   # 16-byte vectors
    assert lib.fa_merge(f, f, 2, 1, 1, 16, 128, 0, f + 8, f, None) == 1
    assert lib.fa_merge(f, f, 0, 1, 1, 16, 128, 0, f, f, None) == 1
    assert lib.fa_merge(f, f, 65, 1, 1, 16, 128, 0, f, f, None) == 1
    assert lib.fa_merge(f, f, 2, 1, 1, 16, 96, 0, f, f, None) == 2
    assert lib.fa_merge(f, f, 2, 0, 1, 16, 128, 0, f, f, None) == 0      # nothing to do


def test_accumulate_and_conversion_validate_before_any_device_work(lib):
    f = FAKE
    for fn in (lib.fa_accumulate, lib.fa_to_bf16):
        assert fn(None, f, 64, None) == 1
        assert fn(f, None, 64, None) == 1
        assert fn(f + 4, f, 64, None) == 1                 # 16-byte vectors
        assert fn(f, f + 8, 64, None) == 1
        assert fn(f, f, 12, None) == 1                     # whole groups of 8 elements
        assert fn(f, f, -8, None) == 1
        assert fn(f, f, 0, None) == 0                      # nothing to do


def test_every_knob_is_documented_and_accepted(lib):
    """The keys fa_debug_set accepts are exactly the ones fa.h documents."""
    api = open(os.path.join(ROOT, "exact_attention_smem_gb300", "csrc", "api.cu")).read()
    accepted = set(re.findall(r'strcmp\(key, "([a-z_0-9]+)"\)', api))
    hdr = open(os.path.join(ROOT, "include", "fa.h")).read()
    block = hdr[hdr.index("Test and tuning knobs"):hdr.index("FA_API int fa_debug_set")]
    documented = set(re.findall(r'"([a-z_0-9]+)"', block))
    assert accepted == documented
    defaults = {"tau": 0.0, "poly8": 0.0, "bwd_poly8": 0.0, "fp8_poly8": 0.0, "fp8_tau": 1.5,
                "timeout_ms": 2000.0, "grid": 0.0, "bwd_mode": 1.0, "fwd_hblock": 0.0,
                "bwd_hblock": 0.0, "bwd_hblock_q": 0.0, "fwd_split_q": -1.0,
                "bwd_pdl": -1.0}
    assert set(defaults) == accepted
    for k, v in defaults.items():                     # every key takes its default value
        assert lib.fa_debug_set(k.encode(), v) == 0, k
