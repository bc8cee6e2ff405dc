"""The failure path on the GPU, without a fault: a bounded wait is made to run out (the test
hook has the attention's first CTA withhold its first scores, a signal nothing else sends),
the launch gives up on its own, the device status reports the timeout, and the next launch
on the same context is correct."""
import numpy as np
import pytest
import torch

import oracle
import topology_scheduled_gb300 as tsa
from topology_scheduled_gb300.workloads import WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    w = WORKLOADS["s1024"]
    q, k, v = make_qkv(w, seed=0, device="cpu")
    qd, kd, vd = (x.to(DEV) for x in (q, k, v))
    rp, ci = tsa.tsa_dense_causal_csr(w.S, w.block)
    assert tsa.tsa_last_device_status() == 0
    tsa.tsa_debug_set_wait_injection(True)
    try:
        tsa.tsa_scheduled_attention(qd, kd, vd, rp, ci, w.scale)
        assert tsa.tsa_last_device_status() == 7  # TSA_ERR_TIMEOUT
    finally:
        tsa.tsa_debug_set_wait_injection(False)
    # the same context: a normal launch afterwards is complete and correct
    out = tsa.tsa_scheduled_attention(qd, kd, vd, rp, ci, w.scale)
    assert tsa.tsa_last_device_status() == 0
    rp_o, ci_o = oracle.dense_causal_csr(w.nb)
    ref = oracle.attention(q, k, v, rp_o, ci_o, w.block, w.scale)
    err = float(np.max(np.abs(out.cpu().double().numpy().reshape(ref.shape) - ref)))
    assert err <= 2e-3


def test_injection_switch_rejects_other_values():
    assert tsa.lib().tsa_debug_set_wait_injection(2) == 1  # TSA_ERR_INVALID_ARGUMENT
    assert tsa.lib().tsa_debug_set_wait_injection(0) == 0
