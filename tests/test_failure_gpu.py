"""The bounded-wait failure path, exercised without faulting or hanging the GPU.

Every pipeline wait in the kernels gives up after a time limit, records a
status bit and lets its kernel return; attn_device_status reports it.  The
library's self-test kernel waits on a barrier that nothing arrives on, with no
copy or tensor-core work in flight and a 1 ms limit, so the wait must run out.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from exact_transformer_attention_flashattention_b300.inputs import prefill_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_transformer_attention_flashattention_b300 import binding
    return binding


def test_wait_that_runs_out_is_reported_once_and_cleared(fa):
    assert fa.device_status() == 0
    fa.selftest_bounded_wait(1_000_000)  # 1 ms
    assert fa.device_status() == fa.ERR_TIMEOUT
    assert "self-test" in fa.last_error()
    assert fa.device_status() == 0
    # the context stays usable: a normal call afterwards matches the oracle
    q, k, v = prefill_inputs(1, 2, 2, 300, 128, seed=3)
    O, L = fa.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, out_dtype=torch.float32)
    assert fa.device_status() == 0
    O_ref, L_ref = oracle.attention(q, k, v, causal=True, scale=1.0 / math.sqrt(128))
    assert np.abs(O.double().cpu().numpy() - O_ref).max() <= 1e-2
    assert np.abs(L.double().cpu().numpy() - L_ref).max() <= 1e-3


def test_selftest_rejects_limits_out_of_range(fa):
    for bad in (0, 999, 100_000_001):
        with pytest.raises(fa.B300AttnError):
            fa.selftest_bounded_wait(bad)
    assert fa.device_status() == 0
