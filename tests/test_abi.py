"""The C-ABI library builds, loads without a GPU and exports what include/spd.h declares."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spd.h")


@pytest.fixture(scope="module")
def libspd():
    from sparse_attention_decode_pages_gb300 import _build
    _build.build()
    import sparse_attention_decode_pages_gb300 as spd
    return spd


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    keywords = {"sizeof", "if", "while", "for", "return"}
    return sorted({n for n in names if n not in keywords})


def test_header_declares_the_five_calls():
    fns = declared_functions()
    for f in ("pages_summarize", "pages_score_select", "sparse_decode_attn", "dense_verify_attn",
              "lse_merge"):
        assert f in fns


def test_library_exports_every_declared_symbol(libspd):
    L = ctypes.CDLL(libspd.LIB_PATH)
    missing = [f for f in declared_functions() if not hasattr(L, f)]
    assert not missing, missing
    assert L.spd_version() == 100


def test_validation_rejects_bad_shapes_without_touching_the_gpu(libspd):
    L = libspd.lib()
    d = libspd.dims_of(2, 4, 2, 96, 16, 8, 16)          # head dim 96 unsupported
    assert L.pages_summarize(ctypes.byref(d), None, None, None, None, 0, None, None) == 2
    assert b"head dim" in L.spd_last_error()
    d = libspd.dims_of(2, 6, 4, 64, 16, 8, 16)          # H_q not a multiple of H_kv
    assert L.pages_summarize(ctypes.byref(d), None, None, None, None, 0, None, None) == 1
    d = libspd.dims_of(2, 36, 4, 64, 16, 8, 16)         # GQA group 9 > 8
    assert L.pages_summarize(ctypes.byref(d), None, None, None, None, 0, None, None) == 2
    d = libspd.dims_of(2, 4, 2, 64, 24, 8, 16)          # page size 24
    assert L.pages_summarize(ctypes.byref(d), None, None, None, None, 0, None, None) == 2
    d = libspd.dims_of(2, 4, 2, 64, 16, 8, 16)
    assert L.pages_summarize(ctypes.byref(d), None, None, None, None, 0, None, None) == 1  # NULLs
    assert L.pages_summarize(None, None, None, None, None, 0, None, None) == 1
    pol = libspd.Policy(0, 8, 0, 0, 1, 0, 1, 1, 1, 4)
    # k_max below sink + local
    assert L.pages_score_select(ctypes.byref(d), None, None, None, ctypes.byref(pol), None,
                                None, 3, None, None, 0, None) == 1
    pol_tp = libspd.Policy(3, 0, 0, 1, 0, 0, 1, 1, 1, 1, 1.5, 0.1)  # top_p > 1
    assert L.pages_score_select(ctypes.byref(d), None, None, None, ctypes.byref(pol_tp), None,
                                None, 8, None, None, 0, None) == 1
    pol_tp = libspd.Policy(3, 0, 0, 1, 0, 0, 1, 1, 1, 1, 0.5, 0.0)  # score_scale = 0
    assert L.pages_score_select(ctypes.byref(d), None, None, None, ctypes.byref(pol_tp), None,
                                None, 8, None, None, 0, None) == 1
    pol_bad = libspd.Policy(1, 0, 0, 1, 0, 0, 1, 1, 1, 1)  # slope_den = 0
    assert L.pages_score_select(ctypes.byref(d), None, None, None, ctypes.byref(pol_bad),
                                None, None, 8, None, None, 0, None) == 1
    assert L.lse_merge(0, 4, 64, None, None, None, None, None) == 1
    assert L.lse_merge(2, 4, 80, None, None, None, None, None) == 2
    d = libspd.dims_of(2, 4, 2, 64, 16, 8, 16)
    assert L.dense_verify_attn(ctypes.byref(d), 0, None, None, None, None, None, 0, 0.1, None,
                               None, None, 0, None) == 2   # T = 0
    assert L.dense_verify_attn(ctypes.byref(d), 40, None, None, None, None, None, 0, 0.1, None,
                               None, None, 0, None) == 2   # T*G = 80 > 64
    assert L.kv_append_refresh(ctypes.byref(d), 0, None, None, None, None, None, None, None,
                               None) == 1                   # T = 0
    assert L.kv_append_refresh(ctypes.byref(d), 1, None, None, None, None, None, None, None,
                               None) == 1                   # NULL pointers
    assert L.pages_append_score_select(ctypes.byref(d), None, None, None, None, None, None, None, None,
                                       ctypes.byref(pol), None, None, 8, None, None, 0, None) == 1
    assert L.sparse_decode_step(ctypes.byref(d), None, None, None, None, None, None, None, None,
                                ctypes.byref(pol), None, None, 8, ctypes.c_float(0.1), None, None, None, 0,
                                None) == 1
    assert L.spec_accept(4, 0, 100, None, None, None, None, None, None, None, None) == 2   # k = 0
    assert L.spec_accept(4, 33, 100, None, None, None, None, None, None, None, None) == 2  # k > 32
    assert L.spec_accept(4, 6, 0, None, None, None, None, None, None, None, None) == 2    # empty vocab
    assert L.spec_accept(4, 6, 100, None, None, None, None, None, None, None, None) == 1  # NULLs
    assert L.spec_accept(0, 6, 100, None, None, None, None, None, None, None, None) == 0  # B = 0


def test_empty_batch_is_a_no_op(libspd):
    L = libspd.lib()
    d = libspd.dims_of(0, 4, 2, 64, 16, 8, 0)
    assert L.pages_summarize(ctypes.byref(d), None, None, None, None, 0, None, None) == 0
    assert L.lse_merge(2, 0, 64, None, None, None, None, None) == 0


def test_product_path_does_not_reference_the_oracle():
    pkg = os.path.join(ROOT, "sparse_attention_decode_pages_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "liboracle" not in text, f


def test_wait_limit_setting(libspd):
    """The limit of the kernels' bounded waits is a setting (no GPU needed to set it)."""
    L = libspd.lib()
    assert libspd.spd_wait_limit_ns() == 2_000_000_000
    assert L.spd_set_wait_limit_ns(0) == 1 and b"wait limit" in L.spd_last_error()
    try:
        libspd.spd_set_wait_limit_ns(1_000_000)
        assert libspd.spd_wait_limit_ns() == 1_000_000
    finally:
        libspd.spd_set_wait_limit_ns(2_000_000_000)
