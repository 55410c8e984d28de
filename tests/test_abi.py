"""The C-ABI library loads and exports every entry point that include/mk.h declares;
host-only planning works without a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import synth
from persistent_moe_decode_cta_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = B.load_library()
    names = declared_functions()
    assert "mk_create" in names and "mk_decode_step" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.EXPORTS) == names
    assert lib.mk_version() == 1


def test_config_validation_without_device():
    cfg = dict(synth.model_config("tiny_b1_64"))
    cfg["head_dim"] = 48
    with pytest.raises(B.MkError) as e:
        B.mk_plan_dry(cfg, 1, 8)
    assert e.value.code == B.MK_ERR_UNSUPPORTED
    cfg = synth.model_config("tiny_b1_64")
    with pytest.raises(B.MkError) as e:
        B.mk_plan_dry(cfg, 9, 8)
    assert e.value.code == B.MK_ERR_INVALID


def test_null_arguments_are_rejected():
    lib = B.load_library()
    assert lib.mk_create(None, None, None, None) == B.MK_ERR_INVALID
    h = ctypes.c_void_p()
    assert lib.mk_create(None, None, None, ctypes.byref(h)) == B.MK_ERR_INVALID
    assert lib.mk_plan(None, 1, None, None, 1, 1) == B.MK_ERR_INVALID
    assert lib.mk_decode_step(None, None, None, None, None, None) == B.MK_ERR_INVALID
    lib.mk_destroy(None)
