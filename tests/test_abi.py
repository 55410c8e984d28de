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
    return sorted(set(re.findall(r"\b(mk_[a-z0-9_]+)\s*\(", src)))


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
    assert lib.mk_read_expert_fp8(None, 0, 0, None, 0) == B.MK_ERR_INVALID


def test_fp8_expert_configs_without_device():
    # FP8 items are 64 rows of d_ff: scales (2 * 64 gate/up rows + d down rows, f32) +
    # 3 * 64 * d codes
    for wl in ("tiny_fp8_b1_64", "small_fp8_b1_2k", "pages_fp8_b1_8k"):
        cfg = synth.model_config(wl)
        _, _, _, info = B.mk_plan_dry(cfg, 1, 8)
        d = cfg["d_model"]
        assert info[30] == B.MK_EXPERT_FP8
        assert info[31] == (2 * 64 + d) * 4 + 3 * 64 * d
        assert info[5] == cfg["d_ff"] // 64 and info[8] == 64
    # handles for batches below 4 take 32-row FP8 items
    cfg = synth.model_config("pages_fp8_b1_8k")
    _, _, _, info = B.mk_plan_dry(cfg, 1, 8, max_batch=2)
    assert info[8] == 32 and info[31] == (2 * 32 + 2048) * 4 + 3 * 32 * 2048
    _, _, _, info = B.mk_plan_dry(synth.model_config("tiny_b1_64"), 1, 8)
    assert info[30] == B.MK_EXPERT_BF16 and info[31] == 3 * 32 * 256 * 2
    # FP8 experts need f-slices of 64 and no dense layers; an unknown dtype is invalid
    with pytest.raises(B.MkError) as e:
        B.mk_plan_dry(dict(synth.model_config("tiny_fp8_b1_64"), d_ff=176), 1, 8, max_batch=2)
    assert e.value.code == B.MK_ERR_UNSUPPORTED
    for bad, code in ((dict(d_ff=160), B.MK_ERR_UNSUPPORTED),):
        cfg = dict(synth.model_config("tiny_fp8_b1_64"), **bad)
        with pytest.raises(B.MkError) as e:
            B.mk_plan_dry(cfg, 1, 8)
        assert e.value.code == code, bad
    # FP8 experts beside dense layers: the dense FFN items stay bf16 slices of 32 rows
    cfg = synth.model_config("small_dense_fp8_b1_2k")
    _, _, _, info = B.mk_plan_dry(cfg, 1, 8)
    assert info[30] == B.MK_EXPERT_FP8 and info[27] == cfg["dense_ff"] // 32 and info[8] == 64
    c = B.make_config(synth.model_config("tiny_b1_64"))
    c.expert_dtype = 7
    info = np.zeros(32, dtype=np.int32)
    assert B.load_library().mk_plan_dry(ctypes.byref(c), 1, 8, None, 0, None, None, 0,
                                        info.ctypes.data) == B.MK_ERR_INVALID
