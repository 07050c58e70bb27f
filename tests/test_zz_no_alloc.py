"""The allocation-free attention entry point, through the C ABI.

tf_op_attention_noalloc serves callers that cannot allocate device memory
while they run (allocator-free real-time loops, hosts that own all device
memory in their own pool, plugins kept off the CUDA allocator).  It must give
the same results as tf_op_attention, which allocates its scratch, and as the
oracle's attention, and keep doing so on back-to-back calls that reuse its
fixed scratch array.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
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


def _inputs(Hq, Hkv, D, T, rows, seed, device=DEV):
    rng = np.random.default_rng(seed)
    qh = rng.standard_normal((rows, Hq * D)).astype(np.float32)
    K = f32_to_bf16_bits(rng.standard_normal((Hkv, T, D)).astype(np.float32))
    V = f32_to_bf16_bits(rng.standard_normal((Hkv, T, D)).astype(np.float32))
    q = torch.from_numpy(qh).to(device)
    Kd = torch.from_numpy(K.view(np.int16)).to(device)
    Vd = torch.from_numpy(V.view(np.int16)).to(device)
    return q, Kd, Vd, (qh, K, V)


def _run(fn, q, K, V, T, Hq, Hkv, D, rows, pos0, splits):
    out = torch.full((rows, Hq * D), float("nan"), dtype=torch.float32, device=q.device)
    st = fn(q.data_ptr(), K.data_ptr(), V.data_ptr(), T, Hq, Hkv, D, rows, pos0, splits,
            out.data_ptr(), None)
    return st, out


def _oracle_rows(host, Hq, D, rows, pos0):
    qh, K, V = host
    Kf, Vf = oracle.bf16_bits_to_f64(K), oracle.bf16_bits_to_f64(V)
    return np.stack([oracle.attention_row(qh[m].reshape(Hq, D).astype(np.float64), Kf, Vf,
                                          pos0 + m + 1).reshape(-1) for m in range(rows)])


CASES = [  # back-to-back calls with different shapes, groups and split counts
    dict(Hq=32, Hkv=8, D=128, T=1024, rows=2, pos0=900, splits=38, seed=1),
    dict(Hq=32, Hkv=8, D=128, T=1024, rows=1, pos0=400, splits=19, seed=2),
    dict(Hq=4, Hkv=4, D=64, T=300, rows=3, pos0=250, splits=7, seed=4),     # D = 64, G = 1
    dict(Hq=8, Hkv=1, D=64, T=700, rows=2, pos0=600, splits=20, seed=5),    # G = 8
    dict(Hq=32, Hkv=8, D=128, T=1024, rows=1, pos0=1000, splits=1, seed=6),  # one slice after many
]


def test_noalloc_attention_matches_allocating_entry_point_and_oracle(L):
    for c in CASES:
        q, K, V, host = _inputs(c["Hq"], c["Hkv"], c["D"], c["T"], c["rows"], c["seed"])
        args = (q, K, V, c["T"], c["Hq"], c["Hkv"], c["D"], c["rows"], c["pos0"], c["splits"])
        st_ref, ref = _run(L.tf_op_attention, *args)
        st, got = _run(L.tf_op_attention_noalloc, *args)
        assert st_ref == 0 and st == 0
        assert torch.isfinite(got).all()
        # the same kernel on the same inputs: equal up to the order in which
        # the slices' partials are read back (the merge is in slice order)
        assert torch.allclose(got, ref, rtol=1e-5, atol=1e-6)
        want = _oracle_rows(host, c["Hq"], c["D"], c["rows"], c["pos0"])
        assert np.allclose(got.cpu().numpy(), want, rtol=1e-4, atol=1e-5)


def test_noalloc_attention_refuses_sizes_beyond_its_scratch(L):
    q, K, V, _ = _inputs(32, 8, 128, 1024, 4, 3)
    # 4 rows x 32 heads x 64 splits x 130 floats exceeds the fixed 2 MiB
    st, _ = _run(L.tf_op_attention_noalloc, q, K, V, 1024, 32, 8, 128, 4, 900, 64)
    assert st == TF_E_INVAL
    # 129 rows x 8 KV heads needs more than the 1024 tickets
    q, K, V, _ = _inputs(32, 8, 64, 200, 129, 7)
    st, _ = _run(L.tf_op_attention_noalloc, q, K, V, 200, 32, 8, 64, 129, 0, 1)
    assert st == TF_E_INVAL
    # and the entry point still works afterwards
    q, K, V, host = _inputs(4, 2, 64, 64, 1, 8)
    st, got = _run(L.tf_op_attention_noalloc, q, K, V, 64, 4, 2, 64, 1, 40, 2)
    assert st == 0
    assert np.allclose(got.cpu().numpy(), _oracle_rows(host, 4, 64, 1, 40), rtol=1e-4, atol=1e-5)


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs a second GPU")
def test_noalloc_attention_on_a_second_device(L):
    dev1 = torch.device("cuda", 1)
    q, K, V, host = _inputs(32, 8, 128, 512, 1, 9, device=dev1)
    with torch.cuda.device(dev1):
        st, got = _run(L.tf_op_attention_noalloc, q, K, V, 512, 32, 8, 128, 1, 500, 16)
    assert st == 0
    assert np.allclose(got.cpu().numpy(), _oracle_rows(host, 32, 128, 1, 500), rtol=1e-4, atol=1e-5)
