"""LM head with the fused streaming-softmax epilogue (bf16, vocab 151936,
hidden 4096) against the oracle at several row counts: 16, 24 (not a
multiple of 16), 128, 256, 512 rows (one and two activation chunks of the
tensor-core GEMM).  Logits (debug output) and the per-row records
(argmax, entropy, p_max, lse) are compared on sampled rows."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import make_weights_torch, plant_bias_for, qwen3_layers
from tests.gpu_common import MARGIN, top2_gap
from serving_wedlm_step_gb300.binding import rows_to_numpy

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module")
def model():
    s = qwen3_layers(1)
    w = make_weights_torch(s, seed=2, norm_jitter=0.2)
    lm = w["lm_head"].float().cpu().numpy().astype(np.float64)
    norm = w["final_norm"].float().cpu().numpy()
    return s, w, lm, norm


@pytest.mark.parametrize("B,W", [(1, 16), (3, 8), (8, 16), (16, 16), (32, 16)])
def test_lm_head_matches_oracle(model, B, W):
    from serving_wedlm_step_gb300.binding import WedlmContext
    s, w, lm, norm = model
    ctx = WedlmContext(s, w, window=W, max_batch=B, max_pages_per_seq=4)
    M = B * W
    g = torch.Generator(device="cuda")
    g.manual_seed(M)
    x = (torch.randn(M, s.hidden, generator=g, device="cuda") * 0.7).to(torch.bfloat16)
    plant = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    plant[::3] = 1000 + torch.arange(0, M, 3, device="cuda", dtype=torch.int32) % 200
    bias = plant_bias_for(s.vocab)
    rows = torch.empty(M, 4, dtype=torch.int32, device="cuda")
    logits = torch.empty(M, s.vocab, dtype=torch.float32, device="cuda")
    ctx.lm_head(B, x, rows, plant_token=plant, plant_bias=bias, logits=logits)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    am, H, pm, lse = rows_to_numpy(rows)
    xs = x.float().cpu().numpy()
    pl = plant.cpu().numpy()
    sample = sorted(set([0, M - 1, M // 2] + list(range(1, M, max(1, M // 6)))))
    h = O.bf16_round(O.rmsnorm(xs[sample], norm, s.rms_eps))
    z = O.lm_head_logits(h, lm, s.mask_id, pl[sample], bias)
    sc = O.softmax_scores(z)
    zg = logits.cpu().numpy()[sample]
    fin = np.isfinite(z)
    assert np.array_equal(np.isfinite(zg), fin)
    err = np.abs(zg[fin] - z[fin]).max()
    print(f"M={M}: logits max err {err:.2e}")
    assert err <= TOL
    for name, gv, rv in (("lse", lse[sample], sc.lse), ("entropy", H[sample], sc.entropy),
                         ("p_max", pm[sample], sc.p_max)):
        e = np.abs(gv - rv).max()
        print(f"  {name} max err {e:.2e}")
        assert e <= TOL, name
    gaps = top2_gap(z)
    for i, r in enumerate(sample):
        if gaps[i] >= MARGIN:
            assert am[r] == sc.argmax[i]
    # records of every row agree with the logits the kernel wrote
    zall = logits.cpu().numpy().astype(np.float64)
    ref_all = O.softmax_scores(zall)
    assert np.abs(lse - ref_all.lse).max() < 1e-3
    ctx.close()
