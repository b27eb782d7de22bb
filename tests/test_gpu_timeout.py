"""The bounded wait of the pipelined kernels runs out cleanly: a wait on a
barrier that nothing arrives at ends after its 2 s limit with
MOE_ERR_TIMEOUT in the workspace's error word (read by moe_check, which then
clears it), and the same context then runs a forward pass that matches the
oracle."""
import time

import numpy as np
import pytest
import torch

from parity_util import check_against_oracle, oracle_full, prepared_inputs, run_forward, to_dev
from sparsely_gated_mixture_top_b300 import binding as B
from sparsely_gated_mixture_top_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_the_context_stays_usable():
    w = wl.Workload("after_timeout", T=64, d=128, h=256, n=8, k=2, bias_std=0.1, seed=70)
    s = B.shape_of(w)
    ws = B.workspace(s)
    t0 = time.time()
    B.moe_selftest_timeout(ws)
    status = B.moe_check(ws)          # synchronises
    elapsed = time.time() - t0
    assert status == B.MOE_ERR_TIMEOUT
    assert 1.5 < elapsed < 30.0
    assert B.moe_check(ws) == B.MOE_OK   # cleared by the first read
    inp = prepared_inputs(w)
    out, _ = run_forward(w, to_dev(inp))
    check_against_oracle(w, out, oracle_full(w, inp))
