"""GPU parity on the tiny fp32 single-layer shape (hidden 256, 4 q / 2 kv
heads of 64, vocab 1024, RoPE theta 1e4, W = 8): every output of the step
against the CPU oracle, through the C ABI.  Tolerance 1e-4 (fp32)."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import TINY, WORKLOADS, Workload, make_pool_np, make_state_np, make_weights_np
from tests.gpu_common import (Stats, check_pool_writes, compare_seq, dev, pool_bits,
                              pool_np, run_step, teacher_forced_scores, weights_np_to_torch)

pytestmark = pytest.mark.gpu
TOL = 1e-4


def make_case(batch=1, prefix=128, masked=5, seed=0, qk_norm=True, W=8, shuffled=False,
              extra_pages=2, all_masked=False):
    s = TINY.replace(qk_norm=qk_norm)
    wl = Workload("t", s, batch=batch, window=W, prefix=prefix, masked=masked,
                  shuffled_pages=shuffled, seed=seed, extra_pages=extra_pages,
                  all_masked_start=all_masked)
    w_np = make_weights_np(s, seed=seed, norm_jitter=0.2)
    st = make_state_np(wl)
    pools_np = [make_pool_np(s, st["num_pages"], seed, l) for l in range(s.n_layers)]
    return s, wl, w_np, st, pools_np


def ctx_for(s, w_np, W, max_batch, max_pages):
    from serving_wedlm_step_gb300.binding import WedlmContext
    return WedlmContext(s, weights_np_to_torch(w_np, torch.float32), window=W,
                        max_batch=max_batch, max_pages_per_seq=max_pages)


def check_step(s, wl, w_np, st, pools_np, alpha=0.01, tau=1.0, logits=True, graphs=True,
               ctx=None):
    ctx = ctx or ctx_for(s, w_np, wl.window, wl.batch, st["max_pages"])
    ctx.set_graphs(graphs)
    pools = [dev(p) for p in pools_np]
    before = [pool_bits(p) for p in pools]
    gpu = run_step(ctx, st, pools, st["num_pages"], alpha, tau, logits=logits)
    assert ctx.status() == 0
    ref_pools = [p.astype(np.float64) for p in pools_np]
    refs = O.oracle_step(s, w_np, st, ref_pools, alpha, tau)
    stats = Stats()
    W = wl.window
    for b, ref in enumerate(refs):
        compare_seq(gpu, b, W, ref, st, alpha, tau, TOL, stats, s.mask_id,
                    tf=teacher_forced_scores(gpu, b, W, w_np, s))
        if logits:
            # logits of the masked rows (the physical suffix); observed rows
            # have none
            n_obs = int(st["obs"][b].sum())
            z = gpu["logits"].numpy()[b * W + n_obs:(b + 1) * W]
            zr = ref.scores.logits[n_obs:]
            fin = np.isfinite(zr)
            assert np.array_equal(np.isfinite(z), fin)
            e = np.abs(z[fin] - zr[fin]).max() if fin.any() else 0.0
            stats.err("logits", e)
            assert e <= TOL
    after = [pool_bits(p) for p in pools]
    for l in range(s.n_layers):
        seqs = [(st["page_table"][b], int(st["seq_len"][b]), ref.n_commit,
                 ref.k_win[l][ref.inv[:ref.n_commit]], ref.v_win[l][ref.inv[:ref.n_commit]])
                for b, ref in enumerate(refs)]
        check_pool_writes(before[l], after[l], pool_np(pools[l]), seqs, s, TOL, stats)
    return gpu, refs, stats


def test_tiny_step_matches_oracle():
    s, wl, w_np, st, pools_np = make_case()
    _, refs, stats = check_step(s, wl, w_np, st, pools_np)
    print(stats)


def test_tiny_step_eager_equals_graph_bitwise():
    s, wl, w_np, st, pools_np = make_case(seed=3, batch=2)
    ctx = ctx_for(s, w_np, wl.window, wl.batch, st["max_pages"])
    outs = []
    for graphs in (False, True, True):
        ctx.set_graphs(graphs)
        pools = [dev(p) for p in pools_np]
        outs.append(run_step(ctx, st, pools, st["num_pages"], 0.01, 1.0))
    for k in ("hidden", "rows", "new_tokens", "committed"):
        assert torch.equal(outs[0][k], outs[1][k]) and torch.equal(outs[1][k], outs[2][k]), k


@pytest.mark.parametrize("qk_norm", [False, True])
def test_tiny_ragged_batch_shuffled_pages(qk_norm):
    # prefixes 0, 1, 15, 16, 17, 100, 128 (page tails), shuffled page ids
    s, wl, w_np, st, pools_np = make_case(batch=7, seed=5, qk_norm=qk_norm, shuffled=True)
    lens = np.array([0, 1, 15, 16, 17, 100, 128], np.int32)
    wl2 = Workload("t", s, batch=7, window=8, prefix=0, masked=(0, 8), shuffled_pages=True,
                   seed=5, extra_pages=2)
    st = make_state_np(wl2, prefix_override=lens)
    pools_np = [make_pool_np(s, st["num_pages"], 5, l) for l in range(s.n_layers)]
    _, _, stats = check_step(s, wl2, w_np, st, pools_np)
    print(stats)


def test_tiny_all_observed_patterns_w8():
    """All 2^8 observed/masked patterns (32 batches of 8 sequences)."""
    s = TINY.replace(qk_norm=True)
    w_np = make_weights_np(s, seed=7, norm_jitter=0.2)
    wl = Workload("t", s, batch=8, window=8, prefix=24, masked=4, seed=7, extra_pages=1)
    base = make_state_np(wl)
    pools_np = [make_pool_np(s, base["num_pages"], 7, l) for l in range(s.n_layers)]
    ctx = ctx_for(s, w_np, 8, 8, base["max_pages"])
    stats_all = Stats()
    for chunk in range(32):
        st = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in base.items()}
        for b in range(8):
            bits = chunk * 8 + b
            obs = np.array([(bits >> j) & 1 for j in range(8)], np.uint8)
            st["obs"][b] = obs
            st["tokens"][b] = np.where(obs == 1, 10 + 3 * np.arange(8) + b, s.mask_id)
        _, _, stats = check_step(s, wl, w_np, st, pools_np, logits=False, ctx=ctx)
        stats_all.checked_select += stats.checked_select
        stats_all.excluded_select += stats.excluded_select
    print(stats_all)


def test_tiny_empty_prefix_and_all_masked():
    s, wl, w_np, st, pools_np = make_case(batch=3, prefix=0, all_masked=True, seed=9)
    check_step(s, wl, w_np, st, pools_np)


def test_tiny_low_threshold_many_fills():
    """tau above every entropy: every masked slot is filled in one step."""
    s, wl, w_np, st, pools_np = make_case(batch=2, seed=11)
    gpu, refs, _ = check_step(s, wl, w_np, st, pools_np, alpha=0.0, tau=100.0)
    for b, ref in enumerate(refs):
        assert len(ref.fill) == int((st["obs"][b] == 0).sum())


def test_tiny_streaming_steps_teacher_forced():
    """Several steps on the device, each compared with the oracle on the
    GPU's own input state (window, lengths and pages copied back)."""
    s, wl, w_np, st, pools_np = make_case(batch=2, seed=13, all_masked=True, extra_pages=4)
    ctx = ctx_for(s, w_np, wl.window, wl.batch, st["max_pages"])
    pools = [dev(p) for p in pools_np]
    state = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    total = 0
    for step in range(8):
        ref_pools = [pool_np(p) for p in pools]
        before = [pool_bits(p) for p in pools]
        gpu = run_step(ctx, state, pools, state["num_pages"], 0.05, 3.0)
        refs = O.oracle_step(s, w_np, state, ref_pools, 0.05, 3.0)
        stats = Stats()
        for b, ref in enumerate(refs):
            compare_seq(gpu, b, wl.window, ref, state, 0.05, 3.0, TOL, stats, s.mask_id,
                        tf=teacher_forced_scores(gpu, b, wl.window, w_np, s))
            total += ref.n_commit
        after = [pool_bits(p) for p in pools]
        seqs = [(state["page_table"][b], int(state["seq_len"][b]), ref.n_commit,
                 ref.k_win[0][ref.inv[:ref.n_commit]], ref.v_win[0][ref.inv[:ref.n_commit]])
                for b, ref in enumerate(refs)]
        check_pool_writes(before[0], after[0], pool_np(pools[0]), seqs, s, TOL, stats)
        # next input state = the GPU's output window
        state["tokens"] = gpu["new_tokens"].numpy().copy()
        state["pos"] = gpu["new_pos"].numpy().copy()
        state["obs"] = gpu["new_observed"].numpy().copy()
        state["seq_len"] = gpu["seq_len"].copy()
    assert total > 0


def test_tiny_prefill_by_all_observed_steps_equals_ar_prefill():
    """A prompt prefilled with all-observed windows (the step's commit path)
    leaves exactly the autoregressive K/V in the pages (Key claims §5.2)."""
    s = TINY.replace(qk_norm=True)
    w_np = make_weights_np(s, seed=17, norm_jitter=0.2)
    W, T = 8, 40
    rng = np.random.default_rng(17)
    prompt = rng.integers(0, s.vocab - 1, T).astype(np.int32)
    num_pages = 4
    page_row = np.array([2, 0, 3, 1], np.int32)
    ctx = ctx_for(s, w_np, W, 1, num_pages)
    pools = [torch.zeros(num_pages * 2 * s.n_kv_heads * 16 * s.head_dim, device="cuda")]
    st = {"page_table": page_row[None, :], "num_pages": num_pages}
    L = 0
    for c0 in range(0, T, W):
        st.update(tokens=prompt[None, c0:c0 + W], pos=(c0 + np.arange(W))[None].astype(np.int32),
                  obs=np.ones((1, W), np.uint8), seq_len=np.array([L], np.int32))
        gpu = run_step(ctx, st, pools, num_pages, 0.01, 1.0)
        assert int(gpu["n_committed"][0]) == W
        L += W
    ks, vs, _ = O.oracle_prefill(s, w_np, prompt)
    k, v = O.pool_gather(pool_np(pools[0]), page_row, T, s)
    assert np.abs(k - ks[0]).max() <= TOL and np.abs(v - vs[0]).max() <= TOL


def test_device_error_word_on_bad_inputs():
    """Bad page ids, out-of-range tokens, negative lengths and capacity
    overflow set bits of the device error word; the kernels skip the
    offending accesses (checked before each access) and the context stays
    usable."""
    from serving_wedlm_step_gb300 import binding as B
    s, wl, w_np, st, pools_np = make_case(batch=2, seed=19)
    ctx = ctx_for(s, w_np, wl.window, wl.batch, st["max_pages"])
    pools = [dev(p) for p in pools_np]
    bad = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    bad["page_table"][0, 0] = st["num_pages"] + 5
    run_step(ctx, bad, pools, st["num_pages"], 0.01, 1.0)
    assert ctx.status() & B.DEV_BAD_PAGE
    bad = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    bad["tokens"][1, 0] = s.vocab + 3
    run_step(ctx, bad, pools, st["num_pages"], 0.01, 1.0)
    assert ctx.status() & B.DEV_BAD_TOKEN
    bad = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    bad["seq_len"][0] = st["max_pages"] * 16
    run_step(ctx, bad, pools, st["num_pages"], 0.01, 1.0)
    assert ctx.status() & B.DEV_CAPACITY
    bad = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    bad["seq_len"][1] = -4
    run_step(ctx, bad, pools, st["num_pages"], 0.01, 1.0)
    assert ctx.status() & B.DEV_BAD_SEQLEN
    # a clean step afterwards still matches the oracle
    check_step(s, wl, w_np, st, pools_np, ctx=ctx)


def test_host_argument_errors():
    from serving_wedlm_step_gb300 import binding as B
    s, wl, w_np, st, pools_np = make_case(batch=1)
    ctx = ctx_for(s, w_np, wl.window, 1, st["max_pages"])
    pools = [dev(p) for p in pools_np]
    big = {k: (np.concatenate([v, v]) if isinstance(v, np.ndarray) and v.ndim >= 1 else v)
           for k, v in st.items()}
    with pytest.raises(B.WedlmError) as e:
        run_step(ctx, big, pools, st["num_pages"], 0.01, 1.0)
    assert e.value.code == B.ERR_INVALID_ARG
    # unsupported shapes are refused at create
    with pytest.raises(B.WedlmError):
        ctx_for(s.replace(head_dim=48), w_np, 8, 1, 4)
    with pytest.raises(B.WedlmError):
        ctx_for(s, w_np, 100, 1, 4)


def test_packed_outputs_match_separate_outputs():
    """make_outputs(packed=True) puts the window and commit results in one
    byte buffer (one copy back for a caller); the step writes the same
    values as into separate tensors, and the host-side views of a copy of
    the buffer read them back."""
    from serving_wedlm_step_gb300 import binding as B
    from tests.gpu_common import state_to_dev
    s, wl, w_np, st, pools_np = make_case(batch=3, seed=41)
    ctx = ctx_for(s, w_np, wl.window, wl.batch, st["max_pages"])
    res = []
    for packed in (False, True):
        d = state_to_dev(st)
        pools = [dev(p) for p in pools_np]
        out = ctx.make_outputs(wl.batch, packed=packed)
        ctx.step(d["tokens"], d["pos"], d["obs"], d["seq_len"], d["page_table"], pools,
                 st["num_pages"], 0.01, 1.0, out)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        if packed:
            host = out["packed"].cpu()
            views = B.step_result_views(host, wl.batch, wl.window)
            assert host.numel() == B.step_result_bytes(wl.batch, wl.window)
        else:
            views = {k: out[k].cpu() for k in ("new_tokens", "new_pos", "committed",
                                               "n_committed", "new_observed")}
        res.append(views)
    for k in res[0]:
        assert torch.equal(res[0][k], res[1][k]), k
