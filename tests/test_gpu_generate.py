"""GPU parity of the rows around the window step: prompt prefill into the
paged cache (chunks larger than the window, Qwen3-8B-shaped bf16 and the
tiny fp32 shape), the streaming decode loop run on the device (a CUDA graph
with a conditional while node) against host-driven steps and, step by step,
the CPU oracle; per-sequence stop; the pages' window size N = 64 (256 query
rows per kv head at 32/8 heads: two row blocks of the tensor-core
attention); and the confidence reading of Eq. 11 (score -ln p_max).

bud-325 summary page, Method: the decoder keeps a window of W slots and runs
"a causal forward on top of the persistent KV cache"; the committed prefix is
immediately cache-valid; Key claims §5.2: Eq. 11 and the fixed-size sliding
window, compatible with CUDA Graphs; Results: window N = 64."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from synth import (TINY, Workload, make_pool_torch, make_state_np, make_weights_np,
                   make_weights_torch, plant_bias_for, plant_targets, qwen3_layers)
from tests.gpu_common import (Stats, compare_seq, dev, pool_bits, pool_np, run_step,
                              teacher_forced_scores, weights_torch_to_np, within)

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _ctx(s, w, W, max_batch, max_pages):
    from serving_wedlm_step_gb300.binding import WedlmContext
    return WedlmContext(s, w, window=W, max_batch=max_batch, max_pages_per_seq=max_pages)


def _paged(s, B, length, seed, dtype=torch.bfloat16, layers=1):
    """Zeroed pools and a shuffled page table with room for `length`
    positions per sequence."""
    rng = np.random.default_rng(seed)
    max_pages = length // 16 + 2
    num_pages = B * max_pages
    ids = rng.permutation(num_pages).astype(np.int32)
    pt = ids.reshape(B, max_pages)
    n = num_pages * 2 * s.n_kv_heads * 16 * s.head_dim
    pools = [torch.zeros(n, dtype=dtype, device="cuda") for _ in range(layers)]
    return pt, num_pages, max_pages, pools


# ---------------------------------------------------------------------------
# prompt prefill
# ---------------------------------------------------------------------------
def test_prefill_bf16_chunks_match_oracle_prefill():
    """A 512-token prompt through two Qwen3-8B-shaped bf16 layers in chunks of
    128, 128 and 256 tokens (4 and 8 row blocks of the attention, one and two
    window tiles).  Layer 0's K/V in the pages equal oracle_prefill's
    (autoregressive-order causal forward); layer 1's equal the oracle layer
    applied to the GPU's own layer-0 output (teacher forcing; that output
    comes from a one-layer context over the same weights, whose pages must be
    bit-identical to layer 0's), both within 2e-2 plus two bf16 ulps; no
    page element beyond the prompt is written."""
    s = qwen3_layers(2).replace(vocab=4096)
    w = make_weights_torch(s, seed=3, norm_jitter=0.2)
    w_np = weights_torch_to_np(w)
    rng = np.random.default_rng(3)
    T, chunks = 512, (128, 128, 256)
    prompt = rng.integers(0, s.vocab - 1, size=(1, T)).astype(np.int32)
    pt, num_pages, max_pages, pools = _paged(s, 1, T + 32, 3, layers=2)
    _, _, _, pool1 = _paged(s, 1, T + 32, 3, layers=1)
    s1 = s.replace(n_layers=1)
    w1 = {"embed": w["embed"], "final_norm": w["final_norm"], "lm_head": w["lm_head"],
          "layers": [w["layers"][0]]}
    ctx = _ctx(s, w, 32, 8, max_pages)
    ctx1 = _ctx(s1, w1, 32, 8, max_pages)
    seq_len = dev(np.zeros(1, np.int32))
    seq_len1 = dev(np.zeros(1, np.int32))
    pt_d = dev(pt)
    x0 = []
    o = 0
    for chunk in chunks:
        tok = dev(prompt[:, o:o + chunk])
        ctx.prefill(tok, seq_len, pt_d, pools, num_pages)
        hid = torch.empty(chunk, s.hidden, dtype=torch.bfloat16, device="cuda")
        ctx1.prefill(tok, seq_len1, pt_d, pool1, num_pages, hidden=hid)
        x0.append(hid)
        o += chunk
    torch.cuda.synchronize()
    assert ctx.status() == 0 and ctx1.status() == 0
    assert int(seq_len.cpu()[0]) == T and int(seq_len1.cpu()[0]) == T
    assert torch.equal(pools[0], pool1[0]), "layer 0 differs between the two contexts"
    x0 = torch.cat(x0).float().cpu().numpy().astype(np.float64)
    ks, vs, _ = O.oracle_prefill(s1, w_np, prompt[0])
    cos, sin = O.rope_cos_sin(np.arange(T), s.head_dim, s.rope_theta)
    z = np.zeros((0, s.n_kv_heads, s.head_dim))
    _, k1, v1, _ = O.layer_forward(s, w_np["layers"][1], x0, cos, sin, z, z, O.storer("bf16"))
    for l, (kr, vr) in enumerate(((ks[0], vs[0]), (k1, v1))):
        vals = pool_np(pools[l])
        k, v = O.pool_gather(vals, pt[0], T, s)
        ek, okk = within(k, kr, TOL, True, name=f"prefill_k{l}")
        ev, okv = within(v, vr, TOL, True, name=f"prefill_v{l}")
        assert okk and okv, (l, ek, ev)
        # positions T.. of the sequence's pages are untouched (still zero)
        kk, vv = O.pool_gather(vals, pt[0], max_pages * 16, s)
        assert not np.any(kk[T:]) and not np.any(vv[T:])
    ctx.close()
    ctx1.close()


def test_prefill_fp32_chunk_larger_than_window():
    """The tiny fp32 shape (window 8) prefilled in chunks of 64 and 36 tokens
    for two sequences at once: K/V in the pages equal oracle_prefill's within
    1e-4, and the final hidden state of the last chunk equals the oracle's."""
    s = TINY
    w_np = make_weights_np(s, seed=4, norm_jitter=0.2)
    w = {"embed": dev(w_np["embed"]), "final_norm": dev(w_np["final_norm"]),
         "lm_head": dev(w_np["lm_head"]),
         "layers": [{k: dev(v) for k, v in lw.items()} for lw in w_np["layers"]]}
    rng = np.random.default_rng(4)
    B, T = 2, 100
    prompt = rng.integers(0, s.vocab - 1, size=(B, T)).astype(np.int32)
    pt, num_pages, max_pages, pools = _paged(s, B, T + 8, 4, dtype=torch.float32)
    ctx = _ctx(s, w, 8, 16, max_pages)  # 128 workspace rows: 2 x 64
    seq_len = dev(np.zeros(B, np.int32))
    hid = torch.empty(B * 36, s.hidden, dtype=torch.float32, device="cuda")
    ctx.prefill(dev(prompt[:, :64]), seq_len, dev(pt), pools, num_pages)
    ctx.prefill(dev(prompt[:, 64:]), seq_len, dev(pt), pools, num_pages, hidden=hid)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    assert seq_len.cpu().tolist() == [T, T]
    vals = pool_np(pools[0])
    for b in range(B):
        ks, vs, x = O.oracle_prefill(s, w_np, prompt[b])
        k, v = O.pool_gather(vals, pt[b], T, s)
        ek, okk = within(k, ks[0], 1e-4, name="prefill_k")
        ev, okv = within(v, vs[0], 1e-4, name="prefill_v")
        eh, okh = within(hid.cpu().numpy()[b * 36:(b + 1) * 36], x[64:], 1e-4,
                         name="prefill_hidden")
        assert okk and okv and okh, (b, ek, ev, eh)
    ctx.close()


# ---------------------------------------------------------------------------
# the streaming loop on the device
# ---------------------------------------------------------------------------
def _stream_setup(B=2, W=16, prompt_len=48, seed=7, steps=24):
    """One Qwen3-8B-shaped bf16 layer with an 8192-token vocabulary, a
    prompt prefilled in chunks of W, an all-masked window after it, and the
    planted counting bias (different targets per sequence) so that many
    slots commit per step."""
    s = qwen3_layers(1).replace(vocab=8192)
    w = make_weights_torch(s, seed=seed, norm_jitter=0.2)
    rng = np.random.default_rng(seed)
    prompt = rng.integers(0, s.vocab - 1, size=(B, prompt_len)).astype(np.int32)
    length = prompt_len + (steps + 2) * W
    pt, num_pages, max_pages, pools = _paged(s, B, length, seed)
    ctx = _ctx(s, w, W, B, max_pages)
    seq_len = dev(np.zeros(B, np.int32))
    for o in range(0, prompt_len, W):
        ctx.prefill(dev(prompt[:, o:o + W]), seq_len, dev(pt), pools, num_pages)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    pos = (prompt_len + np.arange(W))[None, :].repeat(B, 0).astype(np.int32)
    st = {"tokens": np.full((B, W), s.mask_id, np.int32), "pos": pos,
          "obs": np.zeros((B, W), np.uint8), "seq_len": np.full(B, prompt_len, np.int32),
          "page_table": pt, "num_pages": num_pages, "max_pages": max_pages}
    plant = (plant_targets(pos, 17) + 50 * np.arange(B)[:, None]).astype(np.int32)
    return s, w, ctx, st, pools, plant, plant_bias_for(s.vocab)


def _host_steps(ctx, s, st, pools, plant, bias, n, alpha, tau, oracle_w=None, stats=None):
    """n host-driven wedlm_step calls; with oracle_w, every step is compared
    with the oracle on the same input state and pages (teacher forcing).
    Returns the final state and the committed tokens of every step."""
    st = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st.items()}
    committed = []
    for _ in range(n):
        ref_pools = [pool_np(p) for p in pools] if oracle_w is not None else None
        gpu = run_step(ctx, st, pools, st["num_pages"], alpha, tau, plant=plant,
                       plant_bias=bias)
        assert ctx.status() == 0
        if oracle_w is not None:
            refs = O.oracle_step(s, oracle_w, st, ref_pools, alpha, tau, plant_tok=plant,
                                 plant_bias=bias)
            for b in range(st["tokens"].shape[0]):
                W = st["tokens"].shape[1]
                tf = teacher_forced_scores(gpu, b, W, oracle_w, s,
                                           plant[b][refs[b].perm], bias)
                compare_seq(gpu, b, W, refs[b], st, alpha, tau, TOL, stats, s.mask_id,
                            bf16_stored=True, tf=tf, e2e_scores=False)
        committed.append([gpu["committed"].numpy()[b][:int(gpu["n_committed"].numpy()[b])]
                          .tolist() for b in range(st["tokens"].shape[0])])
        st["tokens"] = gpu["new_tokens"].numpy().copy()
        st["pos"] = gpu["new_pos"].numpy().copy()
        st["obs"] = gpu["new_observed"].numpy().copy()
        st["seq_len"] = gpu["seq_len"].copy()
    return st, committed


def _device_loop(ctx, st, pools, plant, bias, max_steps, alpha, tau, stop_len=None,
                 stop_token=-1, out_cap=512):
    B = st["tokens"].shape[0]
    d = {k: dev(st[k]) for k in ("tokens", "pos", "obs", "seq_len", "page_table")}
    done = dev(np.zeros(B, np.int32))
    out = torch.full((B, out_cap), -1, dtype=torch.int32, device="cuda")
    base = dev(st["seq_len"].astype(np.int32))
    steps_run = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.generate(d["tokens"], d["pos"], d["obs"], d["seq_len"], d["page_table"], pools,
                 st["num_pages"], alpha, tau, max_steps, done,
                 stop_len=None if stop_len is None else dev(np.asarray(stop_len, np.int32)),
                 stop_token=stop_token, out_tokens=out, out_base=base, plant_token=dev(plant),
                 plant_bias=bias, steps_run=steps_run)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    return ({k: d[k].cpu().numpy() for k in ("tokens", "pos", "obs", "seq_len")},
            done.cpu().numpy(), out.cpu().numpy(), int(steps_run.cpu()[0]))


def test_streaming_loop_on_device_matches_steps_and_oracle():
    """16 streaming steps after a prompt prefill: host-driven wedlm_step calls
    match the oracle step by step (teacher forced, bit-exact decisions and
    commits, 2e-2 on the scores), and the device loop (one wedlm_generate
    call) reproduces them bit for bit: window, lengths, every page of the
    pool and the transcript of committed tokens."""
    alpha, tau, n = 0.01, 2.0, 16
    s, w, ctx, st0, pools, plant, bias = _stream_setup()
    w_np = weights_torch_to_np(w)
    pools0 = [p.clone() for p in pools]
    stats = Stats()
    st_h, committed = _host_steps(ctx, s, st0, pools, plant, bias, n, alpha, tau,
                                  oracle_w=w_np, stats=stats)
    print(stats)
    assert stats.checked_select > 0
    total = sum(len(c[b]) for c in committed for b in range(2))
    assert total > 2 * n, "the planted regime commits more than one token per step"
    host_bits = [pool_bits(p) for p in pools]
    # the same 16 steps as one device loop, from the same start
    pools_d = [p.clone() for p in pools0]
    fin, done, out, steps = _device_loop(ctx, st0, pools_d, plant, bias, n, alpha, tau)
    assert steps == n and not done.any()
    for k in ("tokens", "pos", "obs", "seq_len"):
        assert np.array_equal(fin[k], st_h[k]), k
    for a, b in zip(host_bits, pools_d):
        assert np.array_equal(a, pool_bits(b)), "pool differs between loop and steps"
    for b in range(2):
        want = [t for c in committed for t in c[b]]
        assert out[b][:len(want)].tolist() == want
        assert np.all(out[b][len(want):] == -1)
    ctx.close()


def test_streaming_loop_stops_each_sequence():
    """Per-sequence stop on the device: sequence 1 stops after committing a
    given token, sequence 0 on its length budget; each stops right after the
    step that reached its condition, is left unchanged afterwards, and the
    loop ends as soon as both have stopped.  The reference is a host-driven
    run that applies the same rules and freezes a stopped sequence by
    feeding its window back unchanged (the other sequences then see the same
    cached lengths as on the device, so the runs agree bit for bit)."""
    alpha, tau, n = 0.01, 2.0, 24
    s, w, ctx, st0, pools, plant, bias = _stream_setup(seed=8)
    pools0 = [p.clone() for p in pools]
    # a free run picks the stop conditions
    st, lens, committed = st0, [], []
    for _ in range(n):
        st, c = _host_steps(ctx, s, st, pools, plant, bias, 1, alpha, tau)
        committed += c
        lens.append(st["seq_len"].copy())
    lens = np.array(lens)
    budget0 = int(lens[12, 0])
    # sequence 1 stops on the first token it commits (its planted targets
    # are disjoint from sequence 0's, so sequence 0 never commits it)
    first1 = next(k for k, c in enumerate(committed) if c[1])
    stop_tok = committed[first1][1][0]
    assert all(stop_tok not in c[0] for c in committed)
    assert first1 < 10
    # the reference: the same rules on the host, stopped sequences frozen
    pools_h = [p.clone() for p in pools0]
    st = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in st0.items()}
    done = [False, False]
    stop_at, trans = [None, None], [[], []]
    for k in range(n):
        prev = {key: st[key].copy() for key in ("tokens", "pos", "obs", "seq_len")}
        st, c = _host_steps(ctx, s, st, pools_h, plant, bias, 1, alpha, tau)
        for b in range(2):
            if done[b]:
                for key in prev:
                    st[key][b] = prev[key][b]
                continue
            trans[b] += c[0][b]
            if (b == 0 and int(st["seq_len"][0]) >= budget0) or (stop_tok in c[0][b]):
                done[b], stop_at[b] = True, k
        if all(done):
            break
    assert all(done) and stop_at[1] < stop_at[0], stop_at
    fin, done_d, out, steps = _device_loop(ctx, st0, [p.clone() for p in pools0], plant, bias,
                                           n, alpha, tau, stop_len=[budget0, 1 << 30],
                                           stop_token=stop_tok)
    assert done_d.tolist() == [1, 1]
    assert steps == max(stop_at) + 1
    for key in ("tokens", "pos", "obs", "seq_len"):
        assert np.array_equal(fin[key], st[key]), key
    for b in range(2):
        assert out[b][:len(trans[b])].tolist() == trans[b]
        assert np.all(out[b][len(trans[b]):] == -1)
    ctx.close()


# ---------------------------------------------------------------------------
# the pages' window N = 64 and the confidence score
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,masked,seed", [(8, (36, 60), 2), (5, (8, 40), 3), (8, (0, 0), 4)])
def test_step_above_256_rows_matches_oracle(B, masked, seed):
    """More than 256 window rows (B x 64): the projections and the LM head
    run on SM pairs with two 256-row blocks, and the LM head loads and
    multiplies only the row blocks holding masked rows (B = 8 with 36..60
    masked slots of 64: more than 256 rows; B = 5 with 8..40: at most 200
    of 320; B = 8 with none masked: an all-observed window, no LM-head row
    live).  The whole step on one Qwen3-8B-shaped layer, 8192-token
    vocabulary, against the oracle."""
    s = qwen3_layers(1).replace(vocab=8192)
    w = make_weights_torch(s, seed=seed, norm_jitter=0.2)
    w_np = weights_torch_to_np(w)
    wl = Workload("w64-wide", s, batch=B, window=64, prefix=(100, 400), masked=masked,
                  shuffled_pages=True, seed=seed)
    st = make_state_np(wl)
    pool = make_pool_torch(s, st["num_pages"], seed, 0)
    ref_pools = [pool_np(pool)]
    ctx = _ctx(s, w, 64, B, st["max_pages"])
    gpu = run_step(ctx, st, [pool], st["num_pages"], 0.01, 1.0)
    assert ctx.status() == 0
    n_masked = int((st["obs"][:B] == 0).sum())
    if masked[1] == 0:
        assert n_masked == 0
    else:
        assert n_masked > 256 if B == 8 else n_masked <= 256
    refs = O.oracle_step(s, w_np, st, ref_pools, 0.01, 1.0)
    stats = Stats()
    for b in range(B):
        tf = teacher_forced_scores(gpu, b, 64, w_np, s)
        compare_seq(gpu, b, 64, refs[b], st, 0.01, 1.0, TOL, stats, s.mask_id,
                    bf16_stored=True, tf=tf, e2e_scores=False)
    print(stats)
    ctx.close()


@pytest.mark.parametrize("B,prefix,seed", [(1, 700, 0), (3, (200, 1500), 1)])
def test_window_64_step_matches_oracle(B, prefix, seed):
    """A window of 64 slots (the pages' N) at 32 q / 8 kv heads: 256 query
    rows per kv head, two row blocks of the attention; the whole step on one
    Qwen3-8B-shaped layer with an 8192-token vocabulary against the oracle."""
    s = qwen3_layers(1).replace(vocab=8192)
    w = make_weights_torch(s, seed=seed, norm_jitter=0.2)
    w_np = weights_torch_to_np(w)
    wl = Workload("w64", s, batch=B, window=64, prefix=prefix, masked=(16, 48),
                  shuffled_pages=True, seed=seed)
    st = make_state_np(wl)
    st["obs"][0, :5] = 1
    st["tokens"][0, :5] = [21, 22, 23, 24, 25]
    pool = make_pool_torch(s, st["num_pages"], seed, 0)
    ref_pools = [pool_np(pool)]
    ctx = _ctx(s, w, 64, B, st["max_pages"])
    gpu = run_step(ctx, st, [pool], st["num_pages"], 0.01, 1.0)
    assert ctx.status() == 0
    refs = O.oracle_step(s, w_np, st, ref_pools, 0.01, 1.0)
    stats = Stats()
    for b in range(B):
        tf = teacher_forced_scores(gpu, b, 64, w_np, s)
        compare_seq(gpu, b, 64, refs[b], st, 0.01, 1.0, TOL, stats, s.mask_id,
                    bf16_stored=True, tf=tf, e2e_scores=False)
    print(stats)
    ctx.close()


def test_window_64_attention_matches_oracle():
    """The attention alone at W = 64, G = 4 (two row blocks per kv head),
    ragged prefixes and shuffled pages: flat 2e-2 and deterministic."""
    from tests.test_gpu_bf16 import _pack_window
    s = qwen3_layers(1)
    B, W = 4, 64
    wl = Workload("a64", s, batch=B, window=W, prefix=(100, 5000), masked=(16, 48),
                  shuffled_pages=True, seed=9)
    st = make_state_np(wl)
    nq, nkv, hd = s.n_q_heads, s.n_kv_heads, s.head_dim
    pool = make_pool_torch(s, st["num_pages"], 9, 0)
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    q = torch.randn(B * W, nq, hd, generator=g, device="cuda").to(torch.bfloat16)
    kw = torch.randn(B, W, nkv, hd, generator=g, device="cuda").to(torch.bfloat16)
    vw = torch.randn(B, W, nkv, hd, generator=g, device="cuda").to(torch.bfloat16)
    kw_np, vw_np = kw.float().cpu().numpy(), vw.float().cpu().numpy()
    win = dev(_pack_window(kw_np, vw_np, W), torch.bfloat16)
    w = make_weights_torch(s, seed=0)
    ctx = _ctx(s, w, W, B, st["max_pages"])
    o = torch.empty(B * W, nq * hd, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o)
    for out in (o, o2):
        ctx.attention(q, pool, dev(st["page_table"]), dev(st["seq_len"]), st["num_pages"], win,
                      out)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    assert torch.equal(o, o2), "attention is not deterministic"
    o_np = o.float().cpu().numpy().reshape(B, W, nq, hd)
    q_np = q.float().cpu().numpy().reshape(B, W, nq, hd)
    pool_f = pool_np(pool)
    ok_all = True
    for b in range(B):
        kp, vp = O.pool_gather(pool_f, st["page_table"][b], int(st["seq_len"][b]), s)
        ref = O.window_attention(q_np[b], kp, vp, kw_np[b], vw_np[b])
        _, ok = within(o_np[b], ref, TOL, name="attn_w64")
        ok_all = ok_all and ok
    assert ok_all
    ctx.close()


def test_confidence_score_step_matches_oracle():
    """Eq. 11 on -ln p_max (score_mode = NEGLOGP): some slots planted with a
    peaked distribution (score ~0.05), the rest near-uniform (score ~8.5);
    fills and window against the oracle in the same reading."""
    s = qwen3_layers(1).replace(vocab=8192)
    w = make_weights_torch(s, seed=12, norm_jitter=0.2)
    w_np = weights_torch_to_np(w)
    wl = Workload("conf", s, batch=2, window=16, prefix=(300, 900), masked=(6, 12),
                  shuffled_pages=True, seed=12)
    st = make_state_np(wl)
    plant = plant_targets(st["pos"], 5)
    plant[:, ::3] = -1  # every third slot without a planted peak
    bias = plant_bias_for(s.vocab)
    pool = make_pool_torch(s, st["num_pages"], 12, 0)
    ref_pools = [pool_np(pool)]
    ctx = _ctx(s, w, 16, 2, st["max_pages"])
    gpu = run_step(ctx, st, [pool], st["num_pages"], 0.05, 1.0, plant=plant, plant_bias=bias,
                   score_mode=O.SCORE_NEGLOGP)
    assert ctx.status() == 0
    refs = O.oracle_step(s, w_np, st, ref_pools, 0.05, 1.0, plant_tok=plant, plant_bias=bias,
                         score_mode=O.SCORE_NEGLOGP)
    stats = Stats()
    n_fill = 0
    for b in range(2):
        tf = teacher_forced_scores(gpu, b, 16, w_np, s, plant[b][refs[b].perm], bias)
        compare_seq(gpu, b, 16, refs[b], st, 0.05, 1.0, TOL, stats, s.mask_id,
                    bf16_stored=True, tf=tf, score_mode=O.SCORE_NEGLOGP,
                    e2e_scores=False)
        n_fill += len(refs[b].fill)
    assert n_fill >= 2
    print(stats)
    ctx.close()


# ---------------------------------------------------------------------------
# Dual-Stream Masking attention
# ---------------------------------------------------------------------------
def _pages_in_order(k, v):
    """[n][nkv][hd] K and V -> n/16 pages in order, the paged layout
    ([page][2][nkv][16 tokens][hd], 8x8 tiles inside each (page, K|V, head))."""
    n, nkv, hd = k.shape
    off = O.page_elem_offset(np.arange(16)[:, None], np.arange(hd)[None, :], hd)
    pool = np.zeros((n // 16, 2, nkv, 16 * hd), np.float32)
    for p in range(n // 16):
        for h in range(nkv):
            pool[p, 0, h][off] = k[16 * p:16 * p + 16, h]
            pool[p, 1, h][off] = v[16 * p:16 * p + 16, h]
    return pool.reshape(-1)


def _blocks(k, v, block):
    """[n][nkv][hd] -> [n/block][2][nkv][block*hd] window blocks (tiles)."""
    from tests.test_gpu_bf16 import _pack_window
    n, nkv, hd = k.shape
    return _pack_window(k.reshape(n // block, block, nkv, hd),
                        v.reshape(n // block, block, nkv, hd), block)


@pytest.mark.parametrize("n,block", [(512, 32), (512, 64), (256, 16)])
def test_dual_stream_attention_matches_oracle(n, block):
    """Memory stream (causal) and prediction stream (blocks of `block`,
    each seeing the memory before it and itself causally) at 32 q / 8 kv
    heads of 128: flat 2e-2 against the oracle's explicit Dual-Stream mask,
    and deterministic."""
    s = qwen3_layers(1).replace(vocab=1024)
    nq, nkv, hd = s.n_q_heads, s.n_kv_heads, s.head_dim
    g = torch.Generator(device="cuda")
    g.manual_seed(n + block)
    q = torch.randn(2 * n, nq, hd, generator=g, device="cuda").to(torch.bfloat16)
    kv = [torch.randn(n, nkv, hd, generator=g, device="cuda").to(torch.bfloat16).float()
          .cpu().numpy() for _ in range(4)]
    km, vm, kp, vp = kv
    pool = dev(_pages_in_order(km, vm), torch.bfloat16)
    win = dev(np.concatenate([_blocks(km, vm, block), _blocks(kp, vp, block)]), torch.bfloat16)
    w = make_weights_torch(s, seed=0)
    ctx = _ctx(s, w, 16, 32, 4)  # 512 workspace rows: room for the partials
    o = torch.empty(2 * n, nq * hd, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o)
    ctx.dual_stream_attention(n, block, q, pool, win, o)
    ctx.dual_stream_attention(n, block, q, pool, win, o2)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    assert torch.equal(o, o2), "dual-stream attention is not deterministic"
    ref = O.dual_stream_attention(q.float().cpu().numpy(), km, vm, kp, vp, block)
    e, ok = within(o.float().cpu().numpy().reshape(2 * n, nq, hd), ref, TOL, name="dual_stream")
    assert ok, e
    ctx.close()


def test_dual_stream_attention_at_benchmark_size_sampled_rows():
    """The benchmark's Dual-Stream call (n = 4096 tokens per stream, blocks of
    32, 32 q / 8 kv heads of 128), in its own launch configuration: sampled
    memory and prediction rows (both ends of the streams and of blocks, and
    random ones) at flat 2e-2 against the oracle evaluated on those rows."""
    from serving_wedlm_step_gb300.binding import WedlmContext
    n, block = 4096, 32
    s = qwen3_layers(1).replace(vocab=1024)
    nq, nkv, hd = s.n_q_heads, s.n_kv_heads, s.head_dim
    g = torch.Generator(device="cuda")
    g.manual_seed(4096)
    q = torch.randn(2 * n, nq, hd, generator=g, device="cuda").to(torch.bfloat16)
    kv = [torch.randn(n, nkv, hd, generator=g, device="cuda").to(torch.bfloat16).float()
          .cpu().numpy() for _ in range(4)]
    km, vm, kp, vp = kv
    pool = dev(_pages_in_order(km, vm), torch.bfloat16)
    win = dev(np.concatenate([_blocks(km, vm, block), _blocks(kp, vp, block)]), torch.bfloat16)
    w = make_weights_torch(s, seed=0)
    # the benchmark's context: 512 workspace rows for the partials
    ctx = WedlmContext(s, w, window=1, max_batch=512, max_pages_per_seq=4)
    o = torch.empty(2 * n, nq * hd, dtype=torch.bfloat16, device="cuda")
    ctx.dual_stream_attention(n, block, q, pool, win, o)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    rng = np.random.default_rng(3)
    rows = sorted(set([0, 1, 31, 32, 2047, n - 1, n, n + 31, n + 32, n + 2048, 2 * n - 1]
                      + list(rng.integers(0, 2 * n, 13))))
    ref = O.dual_stream_attention_rows(q.float().cpu().numpy(), km, vm, kp, vp, block, rows)
    got = o.float().cpu().numpy().reshape(2 * n, nq, hd)[rows]
    e, ok = within(got, ref, TOL, name="dual_stream_4096")
    assert ok, e
    ctx.close()


def test_dual_stream_attention_rejects_beyond_workspace():
    from serving_wedlm_step_gb300 import binding as Bd
    s = qwen3_layers(1).replace(vocab=1024)
    w = make_weights_torch(s, seed=0)
    ctx = _ctx(s, w, 16, 1, 4)  # 16 workspace rows
    n, block = 4096, 16        # 512 blocks x 8 kv heads: more units than it holds
    q = torch.zeros(2 * n, 32, 128, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(n * 8 * 128 * 2, dtype=torch.bfloat16, device="cuda")
    win = torch.zeros(2 * n * 2 * 8 * 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(2 * n, 32 * 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Bd.WedlmError) as e:
        ctx.dual_stream_attention(n, block, q, pool, win, o)
    assert e.value.code == Bd.ERR_CAPACITY
    with pytest.raises(Bd.WedlmError) as e:
        ctx.dual_stream_attention(100, 24, q, pool, win, o)  # block not a multiple of 16
    assert e.value.code == Bd.ERR_INVALID_ARG
    ctx.close()
