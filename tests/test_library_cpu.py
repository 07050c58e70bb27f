"""The C-ABI library builds, loads and exports every declared entry point.

No compute calls: these run without a GPU.  Host-side validation that needs
no device (bad configurations, NULL handles) is exercised too.
"""
import ctypes
import os
import re

import pytest

import __graft_entry__
from dual_ar_decode_gb300 import binding
from synth import FULL, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return binding.lib()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "tf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tf_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert {"tf_create", "tf_load_weights", "tf_prefill", "tf_decode_frame", "tf_destroy"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(binding.EXPORTS)


def test_library_is_built_for_sm103a_only():
    from dual_ar_decode_gb300 import build as b
    assert "arch=compute_103a,code=sm_103a" in " ".join(b.NVCC_FLAGS)


def test_destroy_null_and_last_error(L):
    L.tf_destroy(None)
    assert isinstance(L.tf_last_error(None), bytes)


@pytest.mark.parametrize("change,needle", [
    (dict(head_dim=96), b"head_dim"),
    (dict(n_kv_heads=3), b"multiple of n_kv_heads"),
    (dict(n_codebooks=8), b"n_codebooks"),
    (dict(semantic_vocab=10_000), b"semantic_vocab"),
    (dict(max_seq_len=5), b"max_seq_len"),
    (dict(max_batch=0), b"max_batch"),
    (dict(max_batch=33), b"max_batch"),
    (dict(hidden=250), b"hidden"),
    (dict(flags=16), b"flags"),
])
def test_create_rejects_bad_config_before_touching_a_device(L, change, needle):
    cfg = binding.config_from_dims(TINY)
    for k, v in change.items():
        setattr(cfg, k, v)
    h = ctypes.c_void_p()
    st = L.tf_create(ctypes.byref(cfg), 0, ctypes.byref(h))
    assert st == 1 and not h.value
    assert needle in L.tf_last_error(None)


def test_create_without_device_fails_cleanly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    cfg = binding.config_from_dims(FULL)
    h = ctypes.c_void_p()
    assert L.tf_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == 1
    assert b"device" in L.tf_last_error(None)


def test_op_argument_validation_is_host_side(L):
    s = binding.TfSampling(0, 1.0, 0, 1.0, 1.0, 0)
    assert L.tf_op_select(None, 1, 64, ctypes.byref(s), 0, 0, 0, None, 0, None, None) == 1
    ok = ctypes.c_void_p(16)   # never dereferenced: the arguments are refused first
    bad_p = binding.TfSampling(30, 1.0, 0, 1.5, 1.0, 0)
    assert L.tf_op_select(ok, 1, 64, ctypes.byref(bad_p), 0, 0, 0, None, 0, ok, None) == 1
    assert L.tf_op_select(ok, 1, 64, ctypes.byref(s), 0, 0, 0, None, 3, ok, None) == 1   # window, no ids
    assert L.tf_op_select(ok, 1, 64, ctypes.byref(s), 0, 0, 0, ok, 65, ok, None) == 1    # window > 64
    assert L.tf_op_quantize_fp8(None, 1, 16, None, None, None) == 1
    assert L.tf_test_inject(None, 1) == 1
    assert L.tf_op_gemv(None, 0, None, 1, 16, None, None, 1, None, None) == 1
    assert L.tf_op_gemm_skinny(None, None, 16, 256, 256, None, None) == 1
    assert L.tf_op_gemm_skinny(1, 1, 65, 256, 256, 1, None) == 1   # more than 64 rows
    assert L.tf_op_gemm_skinny(1, 1, 16, 255, 256, 1, None) == 1   # odd N
    assert L.tf_op_gemm_skinny(1, 1, 16, 256, 100, 1, None) == 1   # K not a multiple of 8
