"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare with the CPU oracle on the same seeded inputs.

Decision rule (integer outputs decided by floating point): token ids,
permutations, commit counts, windows and page placement must be bit-exact.
Where the ORACLE's own scores leave a decision inside a 1e-3 margin (top-2
logit gap, |H~ - tau|, or the gap between the two smallest H~ when the
fallback argmin decides), that decision is excluded and counted.  In
addition the CUDA path's decisions must equal the oracle's decision rule
applied to the CUDA path's own scores, with no margin at all.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from serving_wedlm_step_gb300.binding import WedlmContext, rows_to_numpy

MARGIN = 1e-3


def bf16_tol(ref, base=2e-2):
    """Tolerance for a tensor both sides store in bf16: `base` absolute plus
    two bf16 ulps of the value (|ref| * 2^-6 bounds two ulps).  When the
    GPU's fp32 value and the oracle's fp64 value fall on two sides of a bf16
    rounding boundary the stored values differ by one ulp, which for |x| >= 4
    exceeds any fixed absolute bound of 2e-2; the residual stream is rounded
    twice per layer (after the O projection and after the FFN), so two such
    flips can add up."""
    return base + np.abs(ref) * 2.0 ** -6


def within(got, ref, tol, bf16_stored, row_scaled=False, tail=0.0):
    """max |got - ref| and whether it is inside the tolerance; on failure
    prints the worst offending elements.

    row_scaled: for the residual stream, whose absolute error is set by the
    size of the terms summed into it (attention and FFN outputs) rather than
    by the final value, the absolute part of the tolerance is scaled by the
    row's RMS when that exceeds 1.

    tail: fraction of elements allowed beyond the bound, provided every
    element stays within 5x the bound (the residual stream after a whole
    layer, where one-ulp differences of several bf16-stored intermediates
    pass through the FFN)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(got - ref)
    if row_scaled and ref.ndim >= 1 and ref.size:
        tol = tol * np.maximum(1.0, np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True)))
    bound = bf16_tol(ref, tol) if bf16_stored else tol
    over = d > bound
    ok = bool(np.all(d <= 5 * bound)) and over.mean() <= tail if tail else not over.any()
    if not ok:
        bad = np.argwhere(d > bound)
        print(f"  {len(bad)} of {d.size} elements outside the tolerance; worst:")
        excess = (d - bound)[tuple(bad.T)]
        for i in np.argsort(-excess)[:8]:
            ix = tuple(bad[i])
            print(f"    at {ix}: got {got[ix]:.6g} ref {ref[ix]:.6g} diff {d[ix]:.3g}")
    return float(d.max()) if d.size else 0.0, ok


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def weights_np_to_torch(w, dtype):
    cv = lambda a: dev(a, dtype)
    return {"embed": cv(w["embed"]), "final_norm": cv(w["final_norm"]),
            "lm_head": cv(w["lm_head"]),
            "layers": [{k: cv(v) for k, v in lw.items()} for lw in w["layers"]]}


def weights_torch_to_np(w, layers=None):
    cv = lambda t: t.float().cpu().numpy()
    idx = range(len(w["layers"])) if layers is None else layers
    out = {"embed": cv(w["embed"]), "final_norm": cv(w["final_norm"]),
           "lm_head": cv(w["lm_head"]), "layers": [None] * len(w["layers"])}
    for l in idx:
        out["layers"][l] = {k: cv(v) for k, v in w["layers"][l].items()}
    return out


def pool_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def pool_bits(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy()
    return t.view(torch.int32).cpu().numpy()


def state_to_dev(st):
    return {"tokens": dev(st["tokens"]), "pos": dev(st["pos"]), "obs": dev(st["obs"]),
            "seq_len": dev(st["seq_len"]), "page_table": dev(st["page_table"])}


def run_step(ctx, st, pools, num_pages, alpha, tau, plant=None, plant_bias=0.0,
             logits=False, hidden=True):
    d = state_to_dev(st)
    out = ctx.make_outputs(st["tokens"].shape[0], rows=True, perm=True, logits=logits,
                           hidden=hidden)
    ctx.step(d["tokens"], d["pos"], d["obs"], d["seq_len"], d["page_table"], pools,
             num_pages, alpha, tau, out,
             plant_token=None if plant is None else dev(plant), plant_bias=plant_bias)
    torch.cuda.synchronize()
    res = {k: v.cpu() for k, v in out.items()}
    res["seq_len"] = d["seq_len"].cpu().numpy()
    am, H, pm, lse = rows_to_numpy(res["rows"])
    res.update(argmax=am, entropy=H, p_max=pm, lse=lse)
    return res


def top2_gap(z):
    zz = np.sort(np.where(np.isfinite(z), z, -np.inf), axis=1)
    return zz[:, -1] - zz[:, -2]


class Stats:
    def __init__(self):
        self.excluded_argmax = 0
        self.excluded_select = 0
        self.checked_argmax = 0
        self.checked_select = 0
        self.max_err = {}

    def err(self, name, v):
        self.max_err[name] = max(self.max_err.get(name, 0.0), float(v))

    def __repr__(self):
        return (f"Stats(argmax checked {self.checked_argmax} excluded {self.excluded_argmax}; "
                f"select checked {self.checked_select} excluded {self.excluded_select}; "
                f"max_err {self.max_err})")


def teacher_forced_scores(gpu, b, W, weights, shape, plant_phys=None, plant_bias=0.0):
    """The oracle's LM head and softmax statistics applied to the GPU's own
    final hidden state of sequence b (physical rows)."""
    store = O.storer(shape.dtype)
    hid = gpu["hidden"].float().numpy()[b * W:(b + 1) * W].astype(np.float64)
    h = store(O.rmsnorm(hid, weights["final_norm"], shape.rms_eps))
    return O.softmax_scores(O.lm_head_logits(h, weights["lm_head"], shape.mask_id,
                                             plant_phys, plant_bias))


def compare_seq(gpu, b, W, ref: O.SeqStep, st, alpha, tau, tol, stats: Stats,
                mask_id, check_hidden=True, bf16_stored=False, tf=None):
    """Compare sequence b of a GPU step result with the oracle's SeqStep.

    Continuous outputs are compared end to end with the oracle (`ref`).
    Token decisions (argmax, fill set, window) are judged against the
    oracle's scores `tf` computed from the GPU's own LM-head input (teacher
    forcing; see teacher_forced_scores), so that a decision only differs
    when float32 vs float64 accumulation puts it inside the 1e-3 margin."""
    if tf is None:
        tf = ref.scores
    rows = slice(b * W, (b + 1) * W)
    obs = st["obs"][b].astype(bool)
    # permutation and the score-independent integers: bit-exact
    assert gpu["perm"].numpy()[b].tolist() == ref.perm.tolist()
    assert int(gpu["n_committed"].numpy()[b]) == ref.n_commit
    assert gpu["committed"].numpy()[b][:ref.n_commit].tolist() == ref.committed.tolist()
    assert np.all(gpu["committed"].numpy()[b][ref.n_commit:] == -1)
    assert gpu["new_pos"].numpy()[b].tolist() == ref.new_pos.tolist()
    assert int(gpu["seq_len"][b]) == ref.new_seq_len
    # floating point: within tolerance
    if check_hidden:
        e, ok = within(gpu["hidden"].float().numpy()[rows], ref.x_final, tol, bf16_stored,
                       row_scaled=bf16_stored, tail=1e-4 if bf16_stored else 0.0)
        stats.err("hidden", e)
        assert ok, f"hidden err {e}"
    sc = ref.scores
    for name, g, r in (("lse", gpu["lse"][rows], sc.lse), ("entropy", gpu["entropy"][rows], sc.entropy),
                       ("p_max", gpu["p_max"][rows], sc.p_max)):
        e = np.abs(g - r).max()
        stats.err(name, e)
        assert e <= tol, f"{name} err {e}"
    # argmax per physical row, excluding oracle near-ties
    gaps = top2_gap(tf.logits)
    for p in range(W):
        if gaps[p] < MARGIN:
            stats.excluded_argmax += 1
            continue
        stats.checked_argmax += 1
        assert gpu["argmax"][b * W + p] == tf.argmax[p], (b, p)
    # teacher-forced: the GPU's decisions = the rule applied to the GPU's own
    # scores (fp32, no margin)
    inv = ref.inv
    gH = np.where(obs, np.nan, gpu["entropy"][b * W + inv])
    g_fill, _ = O.select_eq11(gH, st["pos"][b], st["obs"][b], alpha, tau)
    g_filled = np.nonzero(gpu["filled"].numpy()[b])[0].tolist()
    assert g_filled == g_fill, (b, g_filled, g_fill)
    # and the GPU window equals the refill rule applied to the GPU's own fills
    g_am = gpu["argmax"][b * W + inv]
    nt, _, nobs = O.refill(st["tokens"][b], st["pos"][b], st["obs"][b], g_fill, g_am,
                           ref.n_commit, mask_id)
    assert gpu["new_tokens"].numpy()[b].tolist() == nt.tolist()
    assert gpu["new_observed"].numpy()[b].tolist() == nobs.tolist()
    # oracle decisions (on the teacher-forced scores) with margins
    masked = [j for j in range(W) if not obs[j]]
    tf_H = np.where(obs, np.nan, tf.entropy[inv])
    tf_fill, ht = O.select_eq11(tf_H, st["pos"][b], st["obs"][b], alpha, tau)
    tf_nt, _, tf_nobs = O.refill(st["tokens"][b], st["pos"][b], st["obs"][b], tf_fill,
                                 tf.argmax[inv], ref.n_commit, mask_id)
    near = any(abs(float(ht[j]) - tau) < MARGIN for j in masked)
    below = [j for j in masked if ht[j] < np.float32(tau)]
    if not below and len(masked) >= 2:
        v = np.sort(np.array([ht[j] for j in masked], np.float64))
        near = near or (v[1] - v[0] < MARGIN)
    if near:
        stats.excluded_select += 1
    else:
        stats.checked_select += 1
        assert g_filled == tf_fill, (b, g_filled, tf_fill)
        fill_gaps_ok = all(gaps[inv[j]] >= MARGIN for j in tf_fill)
        if fill_gaps_ok:
            assert gpu["new_tokens"].numpy()[b].tolist() == tf_nt.tolist()
            assert gpu["new_observed"].numpy()[b].tolist() == tf_nobs.tolist()


def check_pool_writes(before_bits, after_bits, after_vals, seqs, shape, tol, stats,
                      name="kv", bf16_stored=False):
    """Placement bit-exact: across the whole pool only the committed
    positions change.  `seqs` lists (page_row, L, c, ref_k, ref_v) per
    sequence; the values at positions L..L+c-1 must be within tol of the
    oracle's committed K/V ([c][nkv][hd])."""
    changed = before_bits != after_bits
    hd, blk, nkv = shape.head_dim, shape.page_block, shape.n_kv_heads
    expect = np.zeros_like(changed)
    pv_exp = expect.reshape(-1, 2, nkv, blk * hd)
    heads = np.arange(nkv)
    for page_row, L, c, _, _ in seqs:
        if not c:
            continue
        positions = L + np.arange(c)
        pages = np.asarray(page_row)[positions // blk]
        off = O.page_elem_offset((positions % blk)[:, None], np.arange(hd)[None, :], hd)
        pv_exp[pages[:, None, None], :, heads[None, :, None], off[:, None, :]] = True
    # every changed element is an expected one (values equal to the old
    # ones may legitimately appear unchanged)
    assert not np.any(changed & ~expect), f"{name}: writes outside the committed positions"
    for page_row, L, c, ref_k, ref_v in seqs:
        if not c:
            continue
        k, v = O.pool_gather(after_vals, page_row, L + c, shape)
        ek, okk = within(k[L:], ref_k, tol, bf16_stored)
        ev, okv = within(v[L:], ref_v, tol, bf16_stored)
        stats.err(name, max(ek, ev))
        assert okk and okv, f"{name} err {ek} {ev}"
