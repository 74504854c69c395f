"""Pins for the CPU oracle against what the WeDLM pages and mathematics fix.

Each test checks the oracle against something other than itself: values
worked by hand (tests/golden), closed forms, invariants the pages state
(Key claims §3.2/§4.1/§5.2 and Method of the bud-325 summary page),
independent library routines (torch's bf16 cast, scipy's logsumexp and
entropy, torch's scaled_dot_product_attention), and brute force on tiny
inputs.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import oracle as O
from synth import TINY, Workload, make_state_np, make_weights_np, make_pool_np
from synth import plant_bias_for

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# bf16 rounding: against torch's float32 -> bfloat16 cast (nearest-even)
# ---------------------------------------------------------------------------
def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 20000),
        np.array([0.0, -0.0, 1.0, -1.0, 1.00390625, 1.001953125, 3.0e38, -3.0e38,
                  np.inf, -np.inf, 1e-40], np.float32),
    ]).astype(np.float32)
    # exact ties: values halfway between two bf16 neighbours
    ties = (np.arange(1, 200, dtype=np.uint32) << 16) | 0x8000
    x = np.concatenate([x, ties.view(np.float32)])
    ours = O.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)
    assert np.isnan(O.bf16_round(np.array([np.nan]))[0])


# ---------------------------------------------------------------------------
# RMSNorm closed forms
# ---------------------------------------------------------------------------
def test_rmsnorm_closed_forms():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 64))
    y = O.rmsnorm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, -1)), 1.0, rtol=1e-12)
    # scale invariance and gain
    g = rng.uniform(0.5, 2, 64)
    np.testing.assert_allclose(O.rmsnorm(7.0 * x, g, 0.0), O.rmsnorm(x, g, 0.0) , rtol=1e-12)
    np.testing.assert_allclose(O.rmsnorm(x, g, 0.0), y * g, rtol=1e-12)
    # constant row c: c / sqrt(c^2 + eps)
    c = np.full((1, 8), 3.0)
    np.testing.assert_allclose(O.rmsnorm(c, np.ones(8), 1.0), 3.0 / math.sqrt(10.0))


# ---------------------------------------------------------------------------
# RoPE: rotate-half equals complex multiplication by e^{i p w_k};
# dot products depend only on the position difference
# ---------------------------------------------------------------------------
def test_rope_is_complex_rotation():
    rng = np.random.default_rng(3)
    hd, theta = 64, 1e4
    x = rng.standard_normal((7, 3, hd))
    pos = rng.integers(0, 5000, 7)
    cos, sin = O.rope_cos_sin(pos, hd, theta)
    y = O.rope_apply(x, cos, sin)
    half = hd // 2
    w = theta ** (-(np.arange(half) * 2.0) / hd)
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * pos[:, None, None] * w)
    np.testing.assert_allclose(y[..., :half], z.real, atol=1e-10)
    np.testing.assert_allclose(y[..., half:], z.imag, atol=1e-10)


def test_rope_relative_position_property():
    rng = np.random.default_rng(4)
    hd, theta = 128, 1e6
    q = rng.standard_normal((1, 1, hd))
    k = rng.standard_normal((1, 1, hd))

    def dot(p, s):
        cq, sq = O.rope_cos_sin(np.array([p]), hd, theta)
        ck, sk = O.rope_cos_sin(np.array([s]), hd, theta)
        return float(np.sum(O.rope_apply(q, cq, sq) * O.rope_apply(k, ck, sk)))
    base = dot(50, 30)
    for shift in (1, 17, 4096, 30000):
        assert abs(dot(50 + shift, 30 + shift) - base) < 1e-8
    # norm preserved
    c, s = O.rope_cos_sin(np.array([12345]), hd, theta)
    assert abs(np.linalg.norm(O.rope_apply(q, c, s)) - np.linalg.norm(q)) < 1e-12


# ---------------------------------------------------------------------------
# Topological Reordering: exhaustive over all 2^8 observed patterns
# ---------------------------------------------------------------------------
def test_reorder_exhaustive_w8():
    W = 8
    for bits in range(1 << W):
        obs = [(bits >> j) & 1 for j in range(W)]
        perm, inv = O.topological_reorder(obs)
        assert sorted(perm.tolist()) == list(range(W))
        assert np.all(perm[inv] == np.arange(W))
        n_obs = sum(obs)
        # observed first, masked after, each group in ascending slot order
        assert all(obs[j] for j in perm[:n_obs])
        assert not any(obs[j] for j in perm[n_obs:])
        assert list(perm[:n_obs]) == sorted(perm[:n_obs])
        assert list(perm[n_obs:]) == sorted(perm[n_obs:])
        # the pages' invariant: under the causal mask on physical order every
        # masked slot sees every observed slot, and no observed slot sees a
        # masked one
        for j in range(W):
            for k in range(W):
                sees = inv[k] <= inv[j]
                if not obs[j] and obs[k]:
                    assert sees
                if obs[j] and not obs[k]:
                    assert not sees


# ---------------------------------------------------------------------------
# page layout: hand-worked offsets; gather/scatter round trip
# ---------------------------------------------------------------------------
def test_page_layout_golden():
    rows = np.loadtxt(os.path.join(GOLDEN, "page_layout_offsets.txt"),
                      dtype=np.int64, comments="#")
    for hd, t, d, off in rows:
        assert int(O.page_elem_offset(t, d, hd)) == off
    # a block is a bijection onto 0..blk*hd-1
    for hd in (64, 128):
        t, d = np.meshgrid(np.arange(16), np.arange(hd), indexing="ij")
        offs = O.page_elem_offset(t, d, hd).reshape(-1)
        assert sorted(offs.tolist()) == list(range(16 * hd))


def test_pool_roundtrip():
    s = TINY
    rng = np.random.default_rng(5)
    num_pages = 9
    pool = np.zeros(num_pages * 2 * s.n_kv_heads * s.page_block * s.head_dim)
    row = rng.permutation(num_pages)
    positions = np.array([0, 3, 15, 16, 17, 40, 127 % 144])
    k = rng.standard_normal((positions.size, s.n_kv_heads, s.head_dim))
    v = rng.standard_normal((positions.size, s.n_kv_heads, s.head_dim))
    O.pool_scatter(pool, row, positions, k, v, s)
    kk, vv = O.pool_gather(pool, row, 128, s)
    np.testing.assert_array_equal(kk[positions], k)
    np.testing.assert_array_equal(vv[positions], v)
    # untouched positions stay zero
    mask = np.ones(128, bool)
    mask[positions] = False
    assert np.all(kk[mask] == 0) and np.all(vv[mask] == 0)


# ---------------------------------------------------------------------------
# attention special cases reduce to library routines
# ---------------------------------------------------------------------------
def _sdpa(q, k, v, mask):
    # torch SDPA on [heads][rows][hd] in float64
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(mask))
    return out.numpy()


def test_attention_l0_all_observed_is_causal_self_attention():
    rng = np.random.default_rng(6)
    W, nq, nkv, hd = 9, 4, 2, 16
    q = rng.standard_normal((W, nq, hd))
    k = rng.standard_normal((W, nkv, hd))
    v = rng.standard_normal((W, nkv, hd))
    z = np.zeros((0, nkv, hd))
    ours = O.window_attention(q, z, z, k, v)
    kk = np.repeat(k, nq // nkv, axis=1).transpose(1, 0, 2)
    vv = np.repeat(v, nq // nkv, axis=1).transpose(1, 0, 2)
    ref = _sdpa(q.transpose(1, 0, 2), kk, vv, np.tril(np.ones((W, W), bool)))
    np.testing.assert_allclose(ours, ref.transpose(1, 0, 2), atol=1e-12)


def test_attention_w1_is_single_query_decode():
    rng = np.random.default_rng(7)
    L, nq, nkv, hd = 37, 8, 2, 32
    q = rng.standard_normal((1, nq, hd))
    kp = rng.standard_normal((L, nkv, hd))
    vp = rng.standard_normal((L, nkv, hd))
    kw = rng.standard_normal((1, nkv, hd))
    vw = rng.standard_normal((1, nkv, hd))
    ours = O.window_attention(q, kp, vp, kw, vw)
    K = np.concatenate([kp, kw])
    V = np.concatenate([vp, vw])
    for h in range(nq):
        g = h // (nq // nkv)
        s = K[:, g] @ q[0, h] / math.sqrt(hd)
        ref = scipy.special.softmax(s) @ V[:, g]
        np.testing.assert_allclose(ours[0, h], ref, atol=1e-12)


# ---------------------------------------------------------------------------
# softmax statistics: library routines and closed forms
# ---------------------------------------------------------------------------
def test_softmax_scores_match_scipy():
    rng = np.random.default_rng(8)
    z = rng.standard_normal((6, 300)) * 3
    z[:, 299] = -np.inf
    sc = O.softmax_scores(z)
    np.testing.assert_allclose(sc.lse, scipy.special.logsumexp(z, axis=1), rtol=1e-13)
    p = scipy.special.softmax(z, axis=1)
    np.testing.assert_allclose(sc.entropy, scipy.stats.entropy(p, axis=1), rtol=1e-12)
    np.testing.assert_allclose(sc.p_max, p.max(1), rtol=1e-13)
    assert np.all(sc.argmax == np.argmax(z, 1))
    # tie: lowest id
    zt = np.zeros((1, 10))
    zt[0, [3, 7]] = 5.0
    assert O.softmax_scores(zt).argmax[0] == 3


def test_entropy_closed_forms_and_planted_peak():
    V = 1024
    h = np.zeros((1, 8))
    w = np.zeros((V, 8))
    # uniform over the V-1 non-mask tokens
    sc = O.softmax_scores(O.lm_head_logits(h, w, V - 1))
    assert abs(sc.entropy[0] - math.log(V - 1)) < 1e-12
    assert abs(sc.p_max[0] - 1.0 / (V - 1)) < 1e-15
    assert abs(sc.lse[0] - math.log(V - 1)) < 1e-12
    # planted bias b = ln(19 (V-1)) on token 1003 over zero logits, with the
    # mask token excluded: p_top = e^b / (e^b + V - 2) (about 0.95)
    b = plant_bias_for(V)
    sc = O.softmax_scores(O.lm_head_logits(h, w, V - 1, np.array([1003 % V]), b))
    assert sc.argmax[0] == 1003 % V
    p_top = 19.0 * (V - 1) / (19.0 * (V - 1) + V - 2)
    assert abs(sc.p_max[0] - p_top) < 1e-12 and abs(p_top - 0.95) < 1e-4
    # two-point + uniform-rest entropy closed form
    p_rest = (1.0 - p_top) / (V - 2)
    H = -(p_top * math.log(p_top) + (V - 2) * p_rest * math.log(p_rest))
    assert abs(sc.entropy[0] - H) < 1e-10


# ---------------------------------------------------------------------------
# Eq. 11 selection + commit + refill: hand-worked golden cases
# ---------------------------------------------------------------------------
def _parse_cases():
    cases, cur, mask_id = [], None, None
    for line in open(os.path.join(GOLDEN, "eq11_commit_refill_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        key, *vals = line.split()
        if key == "mask_id":
            mask_id = int(vals[0])
        elif key == "case":
            cur = {"name": vals[0]}
            cases.append(cur)
        else:
            cur[key] = vals
    return mask_id, cases


def _ints(vals, mask_id):
    return np.array([mask_id if v == "M" else (-1 if v == "-" else int(v))
                     for v in vals], np.int32)


def _floats(vals):
    return np.array([np.nan if v in ("-", "nan") else float(v) for v in vals])


@pytest.mark.parametrize("case", _parse_cases()[1], ids=lambda c: c["name"])
def test_eq11_commit_refill_golden(case):
    mask_id = _parse_cases()[0]
    toks = _ints(case["tokens"], mask_id)
    pos = _ints(case["pos"], mask_id)
    obs = _ints(case["obs"], mask_id).astype(np.uint8)
    H = _floats(case["H"])
    am = _ints(case["argmax"], mask_id)
    L = int(case["seq_len"][0])
    fill, ht = O.select_eq11(H, pos, obs, float(case["alpha"][0]),
                             float(case["tau"][0]))
    assert fill == [int(v) for v in case["expect_fill"]]
    c = O.commit_run(obs, pos, L)
    assert c == int(case["expect_commit"][0])
    assert toks[:c].tolist() == [int(v) for v in case["expect_committed"]]
    nt, npos, nobs = O.refill(toks, pos, obs, fill, am, c, mask_id)
    assert nt.tolist() == _ints(case["expect_new_tokens"], mask_id).tolist()
    assert npos.tolist() == _ints(case["expect_new_pos"], mask_id).tolist()
    assert nobs.tolist() == _ints(case["expect_new_obs"], mask_id).tolist()
    assert L + c == int(case["expect_seq_len"][0])


def test_eq11_matches_brute_force_definition():
    """Sort-based restatement: the fill set is {H~ < tau} if non-empty, else
    the first element of the masked slots sorted by (H~, slot)."""
    rng = np.random.default_rng(9)
    for trial in range(3000):
        W = int(rng.integers(1, 17))
        obs = (rng.random(W) < 0.4).astype(np.uint8)
        L = int(rng.integers(0, 100))
        pos = L + np.arange(W)
        H = rng.choice([0.0, 0.5, 1.0, 2.0, 4.0, 8.0], W) + rng.integers(0, 4, W) * 0.25
        alpha = float(rng.choice([0.0, 0.125, 0.25, 1.0]))
        tau = float(rng.choice([0.25, 1.0, 3.0]))
        fill, _ = O.select_eq11(H, pos, obs, alpha, tau)
        masked = [j for j in range(W) if not obs[j]]
        if not masked:
            assert fill == []
            continue
        # exact arithmetic suffices: every value is a dyadic rational
        ht = {j: H[j] + alpha * (pos[j] - pos[masked[0]]) for j in masked}
        below = sorted(j for j in masked if ht[j] < tau)
        expect = below if below else [sorted(masked, key=lambda j: (ht[j], j))[0]]
        assert fill == expect


def test_commit_refill_invariants_exhaustive_w8():
    W, L, mask_id = 8, 50, 999
    for bits in range(1 << W):
        obs = np.array([(bits >> j) & 1 for j in range(W)], np.uint8)
        toks = np.where(obs == 1, 100 + np.arange(W), mask_id).astype(np.int32)
        pos = (L + np.arange(W)).astype(np.int32)
        c = O.commit_run(obs, pos, L)
        # c = number of leading observed slots
        lead = 0
        while lead < W and obs[lead]:
            lead += 1
        assert c == lead
        fill = [j for j in range(W) if not obs[j]][:1]
        nt, npos, nobs = O.refill(toks, pos, obs, fill, np.full(W, 7), c, mask_id)
        assert nt.size == W and npos.size == W                # fixed window
        assert np.all(npos == L + c + np.arange(W))            # contiguous
        assert np.all(nt[W - c:] == mask_id) and np.all(nobs[W - c:] == 0)


# ---------------------------------------------------------------------------
# whole-step invariants on the tiny shape
# ---------------------------------------------------------------------------
def _tiny(prefix=40, W=8, seed=0, dtype="fp32", jitter=0.3):
    s = TINY.replace(dtype=dtype, qk_norm=True)
    w = make_weights_np(s, seed=seed, norm_jitter=jitter)
    wl = Workload("t", s, batch=1, window=W, prefix=prefix, masked=(2, 5), seed=seed)
    st = make_state_np(wl)
    pools = [make_pool_np(s, st["num_pages"], seed, l) * 0.5 for l in range(s.n_layers)]
    return s, w, st, pools


def test_reordered_step_equals_logical_step_with_visibility_mask():
    """Key claims §4.1: the reordered causal forward, mapped back to slot
    order, equals a forward in logical order whose window mask is
    visibility(j, k) = [phys(k) <= phys(j)]."""
    s, w, st, pools = _tiny()
    for trial in range(4):
        rng = np.random.default_rng(trial)
        W = 8
        obs = (rng.random(W) < 0.5).astype(np.uint8)
        toks = st["tokens"][0].copy()
        toks[obs == 0] = s.mask_id
        pos = st["pos"][0]
        L = int(st["seq_len"][0])
        row = st["page_table"][0]
        perm, inv = O.topological_reorder(obs)
        store = O.storer(s.dtype)
        x_phys, k_phys, _, _ = O.forward_window(s, w, toks[perm], pos[perm], pools, row, L, store)
        vis = inv[None, :] <= inv[:, None]
        x_log, k_log, _, _ = O.forward_window(s, w, toks, pos, pools, row, L, store, visible=vis)
        np.testing.assert_allclose(x_phys[inv], x_log, atol=1e-10, rtol=0)
        np.testing.assert_allclose(k_phys[0][inv], k_log[0], atol=1e-10, rtol=0)


def test_masked_slots_do_not_influence_observed_rows():
    s, w, st, pools = _tiny(seed=1)
    toks, pos, obs = st["tokens"][0], st["pos"][0], st["obs"][0]
    L, row = int(st["seq_len"][0]), st["page_table"][0]
    a = O.oracle_step_seq(s, w, toks, pos, obs, L, row, [p.copy() for p in pools], 0.01, 1.0)
    # replace the masked slots' tokens by other ids: observed rows unchanged
    t2 = toks.copy()
    t2[obs == 0] = 3
    b = O.oracle_step_seq(s, w, t2, pos, obs, L, row, [p.copy() for p in pools], 0.01, 1.0)
    n_obs = int(obs.sum())
    np.testing.assert_array_equal(a.x_final[:n_obs], b.x_final[:n_obs])
    assert not np.allclose(a.x_final[n_obs:], b.x_final[n_obs:])
    # changing an observed token changes every masked row
    j = int(np.nonzero(obs)[0][0])
    t3 = toks.copy()
    t3[j] = (t3[j] + 1) % (s.vocab - 1)
    c = O.oracle_step_seq(s, w, t3, pos, obs, L, row, [p.copy() for p in pools], 0.01, 1.0)
    for p in range(n_obs, 8):
        assert not np.allclose(a.x_final[p], c.x_final[p])


def test_all_observed_window_equals_autoregressive_prefill():
    """Every-slot-observed window on top of cached KV made by a plain AR
    prefill gives the same K/V and hidden states as one AR prefill over the
    concatenation (Key claims §5.2: the step is a small causal prefill)."""
    s = TINY.replace(qk_norm=True)
    w = make_weights_np(s, seed=3, norm_jitter=0.3)
    rng = np.random.default_rng(3)
    T0, W = 37, 8
    toks = rng.integers(0, s.vocab - 1, T0 + W).astype(np.int32)
    ks, vs, x_all = O.oracle_prefill(s, w, toks)
    num_pages = 8
    row = np.arange(num_pages)[::-1].copy()
    pools = [np.zeros(num_pages * 2 * s.n_kv_heads * s.page_block * s.head_dim)
             for _ in range(s.n_layers)]
    ks0, vs0, _ = O.oracle_prefill(s, w, toks[:T0])
    for l in range(s.n_layers):
        O.pool_scatter(pools[l], row, np.arange(T0), ks0[l], vs0[l], s)
    r = O.oracle_step_seq(s, w, toks[T0:], T0 + np.arange(W), np.ones(W, np.uint8),
                          T0, row, pools, 0.01, 1.0)
    np.testing.assert_allclose(r.x_final, x_all[T0:], atol=1e-10, rtol=0)
    assert r.n_commit == W and r.fill == []
    # the committed K/V equals the AR K/V and lands at positions T0..T0+W-1
    for l in range(s.n_layers):
        kk, vv = O.pool_gather(pools[l], row, T0 + W, s)
        np.testing.assert_allclose(kk, ks[l], atol=1e-10, rtol=0)
        np.testing.assert_allclose(vv, vs[l], atol=1e-10, rtol=0)


def test_committed_kv_is_cache_valid_and_never_recomputed():
    """Method: the committed prefix is cache-valid at once.  K/V written for
    committed slots equals AR prefill K/V over prefix || committed tokens,
    whatever the masked slots hold, and later steps leave it bit-unchanged."""
    s = TINY.replace(qk_norm=True)
    w = make_weights_np(s, seed=4, norm_jitter=0.3)
    rng = np.random.default_rng(4)
    T0, W = 21, 8
    prompt = rng.integers(0, s.vocab - 1, T0).astype(np.int32)
    ks0, vs0, _ = O.oracle_prefill(s, w, prompt)
    num_pages = 12
    row = rng.permutation(num_pages)
    pools = [np.zeros(num_pages * 2 * s.n_kv_heads * s.page_block * s.head_dim)
             for _ in range(s.n_layers)]
    for l in range(s.n_layers):
        O.pool_scatter(pools[l], row, np.arange(T0), ks0[l], vs0[l], s)
    toks = rng.integers(0, s.vocab - 1, W).astype(np.int32)
    obs = np.array([1, 1, 1, 0, 1, 0, 0, 1], np.uint8)
    toks[obs == 0] = s.mask_id
    pos = T0 + np.arange(W)
    r = O.oracle_step_seq(s, w, toks, pos, obs, T0, row, pools, 0.01, 1.0)
    assert r.n_commit == 3
    ks, vs, _ = O.oracle_prefill(s, w, np.concatenate([prompt, toks[:3]]))
    for l in range(s.n_layers):
        kk, vv = O.pool_gather(pools[l], row, T0 + 3, s)
        np.testing.assert_allclose(kk, ks[l], atol=1e-10, rtol=0)
        np.testing.assert_allclose(vv, vs[l], atol=1e-10, rtol=0)
    snapshot = [p.copy() for p in pools]
    # continue streaming: committed positions are never rewritten
    st_t, st_p, st_o, L = r.new_tokens, r.new_pos, r.new_obs, r.new_seq_len
    for _ in range(5):
        rr = O.oracle_step_seq(s, w, st_t, st_p, st_o, L, row, pools, 0.01, 1.0)
        for l in range(s.n_layers):
            a, _ = O.pool_gather(snapshot[l], row, T0 + 3, s)
            b, _ = O.pool_gather(pools[l], row, T0 + 3, s)
            np.testing.assert_array_equal(a, b)
        assert rr.new_tokens.size == W
        st_t, st_p, st_o, L = rr.new_tokens, rr.new_pos, rr.new_obs, rr.new_seq_len


def test_window_position_shift_invariance_without_prefix():
    """RoPE is relative: with no cached prefix, shifting every logical
    position of the window by a constant leaves all outputs unchanged."""
    s = TINY.replace(qk_norm=True)
    w = make_weights_np(s, seed=5, norm_jitter=0.3)
    rng = np.random.default_rng(5)
    W = 8
    toks = rng.integers(0, s.vocab - 1, W).astype(np.int32)
    obs = np.array([1, 0, 1, 1, 0, 0, 1, 0], np.uint8)
    toks[obs == 0] = s.mask_id
    perm, _ = O.topological_reorder(obs)
    store = O.storer("fp32")
    pools = [np.zeros(2 * 2 * s.n_kv_heads * s.page_block * s.head_dim)]
    row = np.array([0, 1])
    a, _, _, _ = O.forward_window(s, w, toks[perm], np.arange(W)[perm], pools, row, 0, store)
    b, _, _, _ = O.forward_window(s, w, toks[perm], 777 + np.arange(W)[perm], pools, row, 0, store)
    np.testing.assert_allclose(a, b, atol=1e-9, rtol=0)


def test_layer_forward_matches_torch_formulation():
    """The pre-norm decoder layer (RMSNorm, q/k/v, QK-norm, RoPE at logical
    positions, GQA attention over prefix || window, O-proj, SwiGLU FFN,
    residuals) against the same layer written with torch.nn.functional
    routines in float64 and RoPE as complex multiplication."""
    import torch.nn.functional as F
    s = TINY.replace(qk_norm=True)
    w = make_weights_np(s, seed=6, norm_jitter=0.3)
    lw = w["layers"][0]
    rng = np.random.default_rng(6)
    W, L = 8, 19
    x = rng.standard_normal((W, s.hidden)) * 0.5
    pos = L + rng.permutation(W)                 # arbitrary logical positions
    kp = rng.standard_normal((L, s.n_kv_heads, s.head_dim))
    vp = rng.standard_normal((L, s.n_kv_heads, s.head_dim))
    cos, sin = O.rope_cos_sin(pos, s.head_dim, s.rope_theta)
    ours, k_o, v_o, _ = O.layer_forward(s, lw, x, cos, sin, kp, vp, O.storer("fp32"))

    T = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    eps = s.rms_eps
    xt = T(x)
    h = F.rms_norm(xt, (s.hidden,), T(lw["attn_norm"]), eps)
    q = F.linear(h, T(lw["w_q"])).view(W, s.n_q_heads, s.head_dim)
    k = F.linear(h, T(lw["w_k"])).view(W, s.n_kv_heads, s.head_dim)
    v = F.linear(h, T(lw["w_v"])).view(W, s.n_kv_heads, s.head_dim)
    q = F.rms_norm(q, (s.head_dim,), T(lw["q_norm"]), eps)
    k = F.rms_norm(k, (s.head_dim,), T(lw["k_norm"]), eps)
    half = s.head_dim // 2
    freq = torch.tensor(s.rope_theta, dtype=torch.float64) ** (
        -torch.arange(half, dtype=torch.float64) * 2 / s.head_dim)
    rot = torch.polar(torch.ones(W, half, dtype=torch.float64),
                      torch.from_numpy(pos.astype(np.float64))[:, None] * freq)

    def rope(t):
        z = torch.complex(t[..., :half], t[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)
    q, k = rope(q), rope(k)
    keys = torch.cat([T(kp), k], 0).repeat_interleave(s.n_q_heads // s.n_kv_heads, 1)
    vals = torch.cat([T(vp), v], 0).repeat_interleave(s.n_q_heads // s.n_kv_heads, 1)
    mask = torch.ones(W, L + W, dtype=torch.bool)
    mask[:, L:] = torch.tril(torch.ones(W, W, dtype=torch.bool))
    o = F.scaled_dot_product_attention(q.transpose(0, 1), keys.transpose(0, 1),
                                       vals.transpose(0, 1), attn_mask=mask)
    xt = xt + F.linear(o.transpose(0, 1).reshape(W, -1), T(lw["w_o"]))
    h2 = F.rms_norm(xt, (s.hidden,), T(lw["ffn_norm"]), eps)
    xt = xt + F.linear(F.silu(F.linear(h2, T(lw["w_gate"]))) * F.linear(h2, T(lw["w_up"])),
                       T(lw["w_down"]))
    np.testing.assert_allclose(ours, xt.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(k_o, k.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(v_o, v.numpy(), atol=1e-11, rtol=0)


# ---------------------------------------------------------------------------
# the confidence reading of Eq. 11: score = -ln p_max
# ---------------------------------------------------------------------------
def test_negative_log_confidence_closed_forms():
    rng = np.random.default_rng(11)
    z = rng.standard_normal((6, 300)) * 3.0
    sc = O.softmax_scores(z)
    got = O.slot_score(sc, O.SCORE_NEGLOGP)
    # -ln p_max = logsumexp(z) - max z (scipy's logsumexp, not the oracle's lse)
    want = scipy.special.logsumexp(z, axis=1) - z.max(axis=1)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    assert np.all(got >= 0)
    # uniform logits over V tokens: p_max = 1/V, score ln V (= the entropy)
    V = 1000
    u = O.softmax_scores(np.zeros((1, V)))
    assert abs(O.slot_score(u, O.SCORE_NEGLOGP)[0] - math.log(V)) < 1e-12
    assert abs(O.slot_score(u, O.SCORE_ENTROPY)[0] - math.log(V)) < 1e-12
    # planted peak with p_top = 0.95 over equal other logits: score ln(1/0.95)
    Vp = 151936
    zp = np.zeros((1, Vp))
    zp[0, 7] = plant_bias_for(Vp)
    p = O.softmax_scores(zp)
    assert abs(O.slot_score(p, O.SCORE_NEGLOGP)[0] - math.log(1 / 0.95)) < 1e-9
    # the entropy reading is the default and equals the entropy field
    np.testing.assert_array_equal(O.slot_score(sc, O.SCORE_ENTROPY), sc.entropy)
    with pytest.raises(ValueError):
        O.slot_score(sc, 7)


def test_score_mode_changes_only_the_selection_score():
    """A whole oracle step in the confidence reading: the forward, the
    commit and the scores are those of the entropy reading; the fills are
    Eq. 11 applied to -ln p_max (the definition, re-evaluated here through
    the brute-force sort of all masked slots)."""
    s = TINY
    wl = Workload("t", s, batch=2, window=8, prefix=(40, 70), masked=(3, 6), seed=5)
    st = make_state_np(wl)
    w = make_weights_np(s, seed=5)
    pools = [make_pool_np(s, st["num_pages"], 5, 0).astype(np.float64)]
    ent = O.oracle_step(s, w, st, [p.copy() for p in pools], 0.05, 5.0)
    neg = O.oracle_step(s, w, st, [p.copy() for p in pools], 0.05, 5.0,
                        score_mode=O.SCORE_NEGLOGP)
    for a, b, bb in zip(ent, neg, range(2)):
        assert a.n_commit == b.n_commit and np.array_equal(a.scores.lse, b.scores.lse)
        obs = st["obs"][bb].astype(bool)
        pos = st["pos"][bb]
        score = -np.log(b.scores.p_max[b.inv])
        masked = [j for j in range(8) if not obs[j]]
        m0 = masked[0]
        ht = {j: np.float32(np.float32(score[j]) + np.float32(np.float32(0.05) *
                                                            np.float32(pos[j] - pos[m0])))
              for j in masked}
        ordered = sorted(masked, key=lambda j: (float(ht[j]), j))
        below = [j for j in ordered if ht[j] < np.float32(5.0)]
        want = sorted(below) if below else [ordered[0]]
        assert b.fill == want


# ---------------------------------------------------------------------------
# Dual-Stream Masking (Key claims §4.2, Eq. 8-10; Method)
# ---------------------------------------------------------------------------
def test_dual_stream_memory_rows_are_causal_self_attention():
    """The memory stream is plain causal self-attention: torch's
    scaled_dot_product_attention with is_causal over the memory tokens."""
    rng = np.random.default_rng(21)
    n, nq, nkv, hd, block = 48, 4, 2, 16, 16
    q = rng.standard_normal((2 * n, nq, hd))
    km, vm, kp, vp = (rng.standard_normal((n, nkv, hd)) for _ in range(4))
    out = O.dual_stream_attention(q, km, vm, kp, vp, block)
    qt = torch.from_numpy(q[:n]).permute(1, 0, 2)
    kt = torch.from_numpy(np.repeat(km, nq // nkv, axis=1)).permute(1, 0, 2)
    vt = torch.from_numpy(np.repeat(vm, nq // nkv, axis=1)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    np.testing.assert_allclose(out[:n], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_dual_stream_prediction_block_is_an_inference_window_step():
    """A prediction block attends exactly as the inference-time window step
    does with the memory before the block as its cached prefix (the point of
    Dual-Stream Masking: training sees the prefix-conditioned setting of
    inference): window_attention(q_block, memory K/V of positions < j*block,
    the block's own K/V) with the causal mask in the block's order.  The
    first block sees no memory at all; blocks never see each other."""
    rng = np.random.default_rng(22)
    n, nq, nkv, hd, block = 64, 4, 2, 16, 16
    q = rng.standard_normal((2 * n, nq, hd))
    km, vm, kp, vp = (rng.standard_normal((n, nkv, hd)) for _ in range(4))
    out = O.dual_stream_attention(q, km, vm, kp, vp, block)
    for j in range(n // block):
        rows = slice(j * block, (j + 1) * block)
        ref = O.window_attention(q[n:][rows], km[:j * block], vm[:j * block], kp[rows], vp[rows])
        np.testing.assert_allclose(out[n:][rows], ref, rtol=0, atol=1e-12)
    # perturbing another block's prediction K/V changes nothing in block 1
    kp2 = kp.copy()
    kp2[2 * block:] += 5.0
    out2 = O.dual_stream_attention(q, km, vm, kp2, vp, block)
    np.testing.assert_array_equal(out2[n + block:n + 2 * block], out[n + block:n + 2 * block])
    # and memory rows never see the prediction stream
    np.testing.assert_array_equal(out2[:n], out[:n])


def test_dual_stream_visibility_counts():
    """Closed form: memory rows see r+1 keys; prediction row i of block j at
    physical index p sees j*block + p + 1 keys."""
    n, block = 48, 16
    vis = O.dual_stream_visibility(n, block)
    assert vis.sum(1)[:n].tolist() == [r + 1 for r in range(n)]
    assert vis.sum(1)[n:].tolist() == [(i // block) * block + i % block + 1 for i in range(n)]
    # no prediction row sees a memory token at or after its block's start
    for i in range(n):
        assert not vis[n + i, (i // block) * block:n].any()


def test_dual_stream_rows_equal_the_whole_call():
    """The row-restricted Dual-Stream attention (used to check sampled rows
    of large calls) is the whole call's rows: memory rows, prediction rows at
    every position of a block, both ends."""
    rng = np.random.default_rng(7)
    n, block, nq, nkv, hd = 24, 8, 4, 2, 16
    q = rng.standard_normal((2 * n, nq, hd))
    km, vm, kp, vp = (rng.standard_normal((n, nkv, hd)) for _ in range(4))
    full = O.dual_stream_attention(q, km, vm, kp, vp, block)
    rows = [0, 5, n - 1, n, n + 3, n + 7, n + 8, 2 * n - 1]
    part = O.dual_stream_attention_rows(q, km, vm, kp, vp, block, rows)
    assert np.allclose(part, full[rows], rtol=1e-12, atol=1e-12)
