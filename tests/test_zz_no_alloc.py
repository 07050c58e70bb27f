"""The allocation-free attention entry point, through the C ABI.

tf_op_attention_noalloc serves callers that cannot allocate device memory
while they run (allocator-free real-time loops, hosts that own all device
memory in their own pool, plugins kept off the CUDA allocator).  It must give
the same results as tf_op_attention, which allocates its scratch, and keep
doing so on back-to-back calls that reuse its fixed scratch array.  This file
is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from dual_ar_decode_gb300 import binding
from synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TF_E_INVAL = 1


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    return binding.lib()


def _inputs(Hq, Hkv, D, T, rows, seed):
    rng = np.random.default_rng(seed)
    q = torch.from_numpy(rng.standard_normal((rows, Hq * D)).astype(np.float32)).to(DEV)
    K = f32_to_bf16_bits(rng.standard_normal((Hkv, T, D)).astype(np.float32))
    V = f32_to_bf16_bits(rng.standard_normal((Hkv, T, D)).astype(np.float32))
    Kd = torch.from_numpy(K.view(np.int16)).to(DEV)
    Vd = torch.from_numpy(V.view(np.int16)).to(DEV)
    return q, Kd, Vd


def _run(fn, q, K, V, T, Hq, Hkv, D, rows, pos0, splits):
    out = torch.full((rows, Hq * D), float("nan"), dtype=torch.float32, device=DEV)
    st = fn(q.data_ptr(), K.data_ptr(), V.data_ptr(), T, Hq, Hkv, D, rows, pos0, splits,
            out.data_ptr(), None)
    return st, out


def test_noalloc_attention_matches_allocating_entry_point(L):
    cases = [  # two calls in a row with different shapes and split counts
        dict(Hq=32, Hkv=8, D=128, T=1024, rows=2, pos0=900, splits=38, seed=1),
        dict(Hq=32, Hkv=8, D=128, T=1024, rows=1, pos0=400, splits=19, seed=2),
    ]
    for c in cases:
        q, K, V = _inputs(c["Hq"], c["Hkv"], c["D"], c["T"], c["rows"], c["seed"])
        args = (q, K, V, c["T"], c["Hq"], c["Hkv"], c["D"], c["rows"], c["pos0"], c["splits"])
        st_ref, ref = _run(L.tf_op_attention, *args)
        st, got = _run(L.tf_op_attention_noalloc, *args)
        assert st_ref == 0 and st == 0
        assert torch.allclose(got, ref, rtol=1e-5, atol=1e-6)
        assert torch.isfinite(got).all()


def test_noalloc_attention_refuses_sizes_beyond_its_scratch(L):
    q, K, V = _inputs(32, 8, 128, 1024, 4, 3)
    # 4 rows x 32 heads x 64 splits x 130 floats exceeds the fixed 2 MiB
    st, _ = _run(L.tf_op_attention_noalloc, q, K, V, 1024, 32, 8, 128, 4, 900, 64)
    assert st == TF_E_INVAL
