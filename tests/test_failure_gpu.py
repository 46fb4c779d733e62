"""Failure detection on the GPU without a fault.

Every wait in the kernels is bounded: a wait that runs out latches a bit in
the device status word and the kernel winds down instead of trapping or
hanging.  The self-test entry point runs that same bounded wait on a barrier
nothing completes (a 50 ms limit instead of the kernels' 2 s); the status
must read FA_ERR_TIMEOUT, be cleared by reading it, and the context must
still compute correct results afterwards.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from exact_attention_21_gb300.inputs import make_qkv
from tests.gpu_util import assert_fwd_close, f64, fa_module, run_fwd

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_the_context_survives(cuda_device):
    fa = fa_module()
    fa.fa_stream_status()  # starts clean
    t0 = time.perf_counter()
    fa.fa_selftest_wait_timeout(50)
    with pytest.raises(fa.FAError) as e:
        fa.fa_stream_status()
    elapsed = time.perf_counter() - t0
    assert e.value.code == fa.FA_ERR_TIMEOUT
    assert "timed out" in str(e.value)
    assert 0.04 <= elapsed < 5.0, elapsed
    fa.fa_stream_status()  # reading the word cleared it
    t = make_qkv(300, 2, 2, 64, seed=40)
    o, lse = run_fwd(t["q"], t["k"], t["v"], True)
    o_ref, lse_ref = oracle.attention_forward(f64(t["q"]), f64(t["k"]), f64(t["v"]), [0, 300], 0.125, True)
    assert_fwd_close(o, lse, o_ref, lse_ref)


def test_timeouts_on_two_streams_are_both_seen(cuda_device):
    """The word is per device: a timeout on any stream is reported once."""
    fa = fa_module()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    fa.fa_selftest_wait_timeout(20, stream=s1)
    fa.fa_selftest_wait_timeout(20, stream=s2)
    torch.cuda.synchronize()
    with pytest.raises(fa.FAError) as e:
        fa.fa_stream_status()
    assert e.value.code == fa.FA_ERR_TIMEOUT
    fa.fa_stream_status()
