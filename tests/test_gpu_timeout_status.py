"""Failure detection without a GPU fault: a bounded device-side wait that runs
out is reported to the host as ATTN_ERR_TIMEOUT, the status word is cleared by
reading it, and the CUDA context keeps working."""
import math

import numpy as np
import pytest
import torch

from optimal_tiling_gb300 import attn, inputs

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives(oracle_mod):
    assert attn.attn_device_status() == attn.ATTN_OK          # nothing pending
    attn.attn_selftest_timeout(20000)                          # 20 ms wait that nothing completes
    assert attn.attn_device_status() == attn.ATTN_ERR_TIMEOUT
    assert attn.attn_device_status() == attn.ATTN_OK          # reading cleared it
    # the context still runs the real kernels correctly
    x = inputs.make_inputs(1, 1, 256, 64, torch.bfloat16, seed=3, with_do=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = attn.attn_fwd(q, k, v, 1.0 / math.sqrt(64))
    assert attn.attn_device_status() == attn.ATTN_OK
    Or, _ = oracle_mod.fwd_naive(x["q"], x["k"], x["v"], 1.0 / math.sqrt(64))
    assert np.max(np.abs(o.float().cpu().numpy() - Or)) <= 1e-2
