"""The C ABI library builds, loads and exports every entry point include/cvr.h declares (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "cvr.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cvr_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import cvr_ranking_model_gb300 as cvr
    return cvr.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "cvr_create" in names and "cvr_score" in names and "cvr_destroy" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(8):
        assert lib.cvr_status_string(code)
    assert lib.cvr_status_string(3) == b"id out of table range"


def test_create_rejects_bad_arguments_without_touching_the_gpu(lib):
    import cvr_ranking_model_gb300 as cvr
    h = ctypes.c_void_p()
    cfg = cvr.make_config(seq_len=(16, 16, 16), n_layers=1, user_rows=[10] * 8, item_rows=[10] * 8, seq_rows=10)
    w = cvr.Weights()
    # null weights / config / out
    assert lib.cvr_create(None, ctypes.byref(cfg), None, ctypes.byref(h)) == 1
    assert lib.cvr_create(ctypes.byref(w), None, None, ctypes.byref(h)) == 1
    assert lib.cvr_create(ctypes.byref(w), ctypes.byref(cfg), None, None) == 1
    # unsupported dimensions, bad sizes
    for field, value in (("token_dim", 64), ("n_layers", 0), ("n_layers", 5), ("heads", 8), ("tau", 0.0)):
        c = cvr.make_config(seq_len=(16, 16, 16), n_layers=1, user_rows=[10] * 8, item_rows=[10] * 8, seq_rows=10)
        setattr(c, field, value)
        assert lib.cvr_create(ctypes.byref(w), ctypes.byref(c), None, ctypes.byref(h)) == 1, field
    c = cvr.make_config(seq_len=(0, 16, 16), n_layers=1, user_rows=[10] * 8, item_rows=[10] * 8, seq_rows=10)
    assert lib.cvr_create(ctypes.byref(w), ctypes.byref(c), None, ctypes.byref(h)) == 1
    # valid config, but every weight pointer is NULL
    assert lib.cvr_create(ctypes.byref(w), ctypes.byref(cfg), None, ctypes.byref(h)) == 1
    assert not h.value


def test_null_handle_calls_are_rejected(lib):
    assert lib.cvr_score(None, 1, 1, None, None, None, None, None) == 1
    assert lib.cvr_set_option(None, 0, 1) == 1
    assert lib.cvr_last_launch_count(None) == 0
    lib.cvr_destroy(None)
