"""CPU-side checks of the C ABI library: it loads, exports every function that
include/confkv.h declares, and rejects bad arguments before touching a GPU.
Also checks the separation between the product path and the test oracle."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from confidence_gated_kv_logits_gb300 import build as B
    B.build()
    import confidence_gated_kv_logits_gb300 as pkg
    return pkg.load_library()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(confkv_\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    import confidence_gated_kv_logits_gb300 as pkg
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(pkg.EXPORTS)


def test_invalid_arguments_rejected_on_host(lib):
    import confidence_gated_kv_logits_gb300 as pkg
    h = ctypes.c_void_p()
    o = pkg.Opts(1, 1000, 0, 1.0, -1, 0, 0, 0)
    good = (2, 8, 2, 128, 36, 24, 0.5, 4, 16, 0.9)
    bad_cases = [
        (2, 8, 3, 128, 36, 24, 0.5, 4, 16, 0.9),    # Hq % Hkv != 0
        (2, 8, 2, 96, 36, 24, 0.5, 4, 16, 0.9),     # head_dim not 64/128
        (2, 8, 2, 128, 36, 24, 0.5, 4, 2, 0.9),     # W < P
        (2, 8, 2, 128, 3, 24, 0.5, 4, 16, 0.9),     # N_low < P
        (2, 8, 2, 128, 36, 24, 0.5, 0, 16, 0.9),    # P < 1
        (2, 8, 2, 128, 36, 24, 0.5, 4, 16, 1.5),    # ema_decay > 1
        (0, 8, 2, 128, 36, 24, 0.5, 4, 16, 0.9),    # no layers
        (2, 64, 2, 128, 36, 24, 0.5, 4, 16, 0.9),   # group of 32 > 16
    ]
    for args in bad_cases:
        rc = lib.confkv_create(*args, ctypes.byref(o), ctypes.byref(h))
        assert rc == pkg.ERR_INVALID_ARG and not h.value, args
    o_bad = pkg.Opts(1, 1, 0, 1.0, -1, 0, 0, 0)                 # vocab < 2
    assert lib.confkv_create(*good, ctypes.byref(o_bad), ctypes.byref(h)) == pkg.ERR_INVALID_ARG
    o_bad = pkg.Opts(1, 1000, 0, 1.5, -1, 0, 0, 0)              # pyramid factor > 1
    assert lib.confkv_create(*good, ctypes.byref(o_bad), ctypes.byref(h)) == pkg.ERR_INVALID_ARG
    o_bad = pkg.Opts(1, 1000, 0, 1.0, -1, 0, 3, 0)             # unknown kernel choice
    assert lib.confkv_create(*good, ctypes.byref(o_bad), ctypes.byref(h)) == pkg.ERR_INVALID_ARG
    o_bad = pkg.Opts(1, 1000, 0, 1.0, -1, 0, 0, 0, 4)          # unknown ranking policy
    assert lib.confkv_create(*good, ctypes.byref(o_bad), ctypes.byref(h)) == pkg.ERR_INVALID_ARG
    o_bad = pkg.Opts(1, 1000, 0, 1.0, -1, 0, 0, 0, 1, 7)       # unknown INT8 storage mode
    assert lib.confkv_create(*good, ctypes.byref(o_bad), ctypes.byref(h)) == pkg.ERR_INVALID_ARG
    assert lib.confkv_create(*good, ctypes.byref(o), None) == pkg.ERR_INVALID_ARG
    # null contexts
    assert lib.confkv_step(*([None] * 11)) == pkg.ERR_INVALID_ARG
    assert lib.confkv_prefill(None, None, None, 0, None, None) == pkg.ERR_INVALID_ARG
    assert lib.confkv_stats(None, None) == pkg.ERR_INVALID_ARG
    assert lib.confkv_last_error(None) == b"null context"
    assert lib.confkv_attention_path(None) == pkg.ERR_INVALID_ARG
    g, w = ctypes.c_int(), ctypes.c_double()
    assert lib.confkv_selftest_bounded_wait(0, 0, ctypes.byref(g), ctypes.byref(w)) == pkg.ERR_INVALID_ARG
    assert lib.confkv_selftest_bounded_wait(0, 2000000, ctypes.byref(g), ctypes.byref(w)) == pkg.ERR_INVALID_ARG
    assert lib.confkv_selftest_bounded_wait(0, 100, None, ctypes.byref(w)) == pkg.ERR_INVALID_ARG
    lib.confkv_free(None)


def test_product_never_imports_the_oracle():
    pkg_dir = os.path.join(ROOT, "confidence_gated_kv_logits_gb300")
    for f in glob.glob(os.path.join(pkg_dir, "**", "*"), recursive=True):
        if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            txt = open(f).read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", txt, flags=re.M), f
            assert "confkv_oracle" not in txt and "orc_" not in txt, f
    for f in glob.glob(os.path.join(ROOT, "oracle", "*")):
        if f.endswith((".py", ".cpp")):
            txt = open(f).read()
            assert "confidence_gated_kv_logits_gb300" not in txt and "confkv.h" not in txt, f


def test_missing_library_fails_loudly(tmp_path):
    import confidence_gated_kv_logits_gb300 as pkg
    saved = pkg._lib
    try:
        pkg._lib = None
        with pytest.raises(ImportError):
            pkg.load_library(str(tmp_path / "nope.so"))
    finally:
        pkg._lib = saved
