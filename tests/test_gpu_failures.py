"""Failure paths on the GPU, made without faulting it.

A bounded device wait is made to run out by a test hook that keeps one
weight copy from being issued (the wait's 200 ms budget expires, the kernel
raises its error bit and returns); a device allocation is refused by a
host-side hook.  The context must report TF_E_TIMEOUT / TF_E_NOMEM, refuse
further work after the timeout, free everything on tf_destroy, and leave
the device usable for a new context.
"""
import time

import numpy as np
import pytest
import torch

from dual_ar_decode_gb300 import Decoder, TfError, binding
from synth import TINY, make_prompt, make_weights

from gpu_helpers import BF16_TOL, TeacherForced

pytestmark = pytest.mark.gpu

TF_TEST_SKIP_ONE_COPY = 1


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def test_expired_wait_poisons_the_context_and_the_device_stays_usable():
    w = make_weights(TINY, seed=21)
    dec = Decoder(TINY, "bf16")
    dec.load_weights(w)
    dec.prefill(make_prompt(TINY, 8, seed=1))
    dec.decode_frame()
    assert binding.lib().tf_test_inject(dec.h, TF_TEST_SKIP_ONE_COPY) == 0
    t0 = time.monotonic()
    with pytest.raises(TfError, match="TIMEOUT"):
        dec.decode_frame()
    assert time.monotonic() - t0 < 5.0          # two 200 ms waits, not a hang
    with pytest.raises(TfError, match="STATE"):  # poisoned from here on
        dec.decode_frame()
    with pytest.raises(TfError, match="STATE"):
        dec.prefill(make_prompt(TINY, 8, seed=1))
    dec.close()
    # the CUDA context is intact: a new decoder matches the oracle
    tf = TeacherForced(TINY, "bf16", weights=w)
    tf.prefill(make_prompt(TINY, 8, seed=2))
    tf.decode()
    tf.check(BF16_TOL)
    tf.dec.close()


def test_copy_skip_needs_a_batch_one_context():
    dec = Decoder(TINY, "bf16", max_batch=2)
    assert binding.lib().tf_test_inject(dec.h, TF_TEST_SKIP_ONE_COPY) == 1   # TF_E_INVAL
    assert binding.lib().tf_test_inject(dec.h, 99) == 1
    dec.close()


def test_refused_allocations_return_nomem_and_free_everything():
    L = binding.lib()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    refused = 0
    try:
        for n in (1, 2, 3, 7, 12, 20, 40, 400):
            L.tf_test_fail_alloc(n)
            try:
                dec = Decoder(TINY, "bf16", max_batch=2)
            except TfError as e:
                assert "NOMEM" in str(e) and "refused" in str(e)
                refused += 1
            else:
                dec.close()       # n beyond the allocations tf_create makes
            L.tf_test_fail_alloc(0)
    finally:
        L.tf_test_fail_alloc(0)
    assert refused >= 5
    torch.cuda.synchronize()
    # everything the refused creates had allocated was freed again
    assert abs(torch.cuda.mem_get_info()[0] - free0) <= 64 << 20
    dec = Decoder(TINY, "bf16")
    dec.load_weights(make_weights(TINY, seed=22))
    f, _ = dec.prefill(make_prompt(TINY, 4, seed=3))
    assert f.shape == (1, 10)
    dec.close()
