"""Failure detection without a GPU fault.

A bounded wait that runs out (a barrier nothing completes) sets
WEDLM_DEV_TIMEOUT and lets the kernel return, and non-finite scores (NaN
weights) set WEDLM_DEV_NUMERIC; after either, the same process runs a clean
step that matches the oracle, so the CUDA context stayed usable."""
import numpy as np
import pytest
import torch

from tests.gpu_common import dev, run_step
from tests.test_gpu_tiny import check_step, ctx_for, make_case

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    from serving_wedlm_step_gb300 import binding as B
    word = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    err, gave_up = B.selftest_bounded_wait(word)
    assert gave_up == 1
    assert err & B.DEV_TIMEOUT
    assert word.cpu().tolist() == [err, 1]
    s, wl, w_np, st, pools_np = make_case(batch=2, seed=31)
    check_step(s, wl, w_np, st, pools_np)


def test_nan_weights_set_the_numeric_bit():
    from serving_wedlm_step_gb300 import binding as B
    s, wl, w_np, st, pools_np = make_case(batch=2, seed=37)
    bad = dict(w_np)
    bad["final_norm"] = w_np["final_norm"].copy()
    bad["final_norm"][0] = np.nan  # every masked row's logits become NaN
    ctx = ctx_for(s, bad, wl.window, wl.batch, st["max_pages"])
    pools = [dev(p) for p in pools_np]
    run_step(ctx, st, pools, st["num_pages"], 0.01, 1.0)
    assert ctx.status() & B.DEV_NUMERIC
    ctx.close()
    check_step(s, wl, w_np, st, pools_np)
