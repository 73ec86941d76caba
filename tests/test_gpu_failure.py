"""Failure detection on the GPU without a fault: a bounded wait runs out, the
kernel records GQA_ERR_TIMEOUT and returns, and the context stays usable."""
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import assert_parity, to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    try:
        G.set_wait_timeout_ns(5_000_000)          # 5 ms
        st, ns = G.selftest_wait_timeout()
        assert st == 4                            # GQA_ERR_TIMEOUT
        assert 5_000_000 <= ns < 1_000_000_000, ns
        assert G.last_device_status() == 0        # read-and-clear
    finally:
        G.set_wait_timeout_ns(2_000_000_000)
    # the context still runs real work correctly
    x = S.make_prefill(1, 8, 2, 100, seed=3)
    out = G.prefill(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.g.cuda())
    assert G.last_device_status() == 0
    ref = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g))[0]
    assert_parity(out, ref, "after timeout")
