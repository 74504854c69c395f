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


# every comparison made through `within` in this process: the test, the
# tensor, and the measured error against the bound (printed in the pytest
# terminal summary; also appended as JSON lines to $WEDLM_PARITY_LOG)
PARITY_LOG = []


def _log_parity(name, d, ref, bound):
    import json
    import os
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" (")[0]
    a = np.abs(ref)
    # one bf16 ulp of the reference value (2^(e-7) for |x| in [2^e, 2^(e+1)))
    ulp = np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7)
    rec = {"test": test, "name": name, "n": int(d.size),
           "max_abs": float(d.max()) if d.size else 0.0,
           "max_over_bound": float((d / bound).max()) if d.size else 0.0,
           "n_over_bound": int((d > bound).sum()),
           "max_ulps": float((d / ulp).max()) if d.size else 0.0}
    if ref.ndim >= 1 and ref.size:
        rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
        rec["max_over_row_rms"] = float((d / np.maximum(rms, 1e-30)).max())
    PARITY_LOG.append(rec)
    path = os.environ.get("WEDLM_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
    return rec


def resid_bound(x_out, x_mid, tol):
    """Elementwise bound for the bf16 residual stream after one decoder layer
    whose input is identical on both sides (x_mid: the oracle's residual
    after the attention block, x_out: after the FFN):

        tol + 2^-6 max(|x_mid|, |x_out|) + 2^-5 rms_row(x_out - x_mid)

    * two bf16 ulps of the largest value the element held: each side rounds
      x_mid and x_out to bf16, and where the GPU's fp32 sum and the oracle's
      fp64 sum fall on two sides of a rounding boundary the stored values
      differ by one ulp; a flip of x_mid carries into x_out unchanged
      (|x| 2^-7 bounds one ulp of x);
    * 2^-5 of the row RMS of the FFN term: the FFN reads RMSNorm(x_mid),
      which rescales the whole row to unit size, so a relative error e of
      x_mid (in the row-RMS sense) becomes a relative error of about e of
      the FFN term.  The attention output is ~1% off the fp64 value (P is
      rounded to bf16 for the P.V MMA, on the GPU only), and where x_mid is
      small next to the FFN term (the first layers of a random-init stack:
      x_mid ~0.03 RMS, FFN term ~2 RMS) that 1% reaches the output; measured
      max |error| / rms(FFN term) = 0.029 over the bf16 layer tests.
    """
    x_out = np.asarray(x_out, np.float64)
    x_mid = np.asarray(x_mid, np.float64)
    ffn = x_out - x_mid
    ffn_rms = np.sqrt(np.mean(ffn * ffn, axis=-1, keepdims=True))
    return tol + np.maximum(np.abs(x_mid), np.abs(x_out)) * 2.0 ** -6 + ffn_rms * 2.0 ** -5


def within(got, ref, tol, bf16_stored=False, name="", bound=None):
    """max |got - ref| and whether every element is inside the bound; the
    measured error is logged (see PARITY_LOG) and, on failure, the worst
    offending elements are printed.

    bf16_stored: both sides store this tensor in bf16, so the bound is `tol`
    plus two bf16 ulps of the value (bf16_tol).  Without it the bound is the
    flat absolute `tol` (attention outputs, logits and softmax statistics).
    `bound`, when given, is an elementwise bound used instead (resid_bound)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(got - ref)
    if bound is None:
        bound = bf16_tol(ref, tol) if bf16_stored else np.full_like(ref, tol)
    bound = np.broadcast_to(np.asarray(bound, np.float64), ref.shape)
    _log_parity(name, d, ref, bound)
    over = d > bound
    ok = not over.any()
    if not ok:
        bad = np.argwhere(over)
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
             logits=False, hidden=True, score_mode=0):
    d = state_to_dev(st)
    out = ctx.make_outputs(st["tokens"].shape[0], rows=True, perm=True, logits=logits,
                           hidden=hidden)
    ctx.step(d["tokens"], d["pos"], d["obs"], d["seq_len"], d["page_table"], pools,
             num_pages, alpha, tau, out,
             plant_token=None if plant is None else dev(plant), plant_bias=plant_bias,
             score_mode=score_mode)
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


def gpu_slot_score(gpu, score_mode):
    """The score the CUDA path's selection used, per physical row, from its
    own records (fp32): the entropy, or -ln p_max (computed here in float64
    from the fp32 p_max; the kernel's logf may differ by an ulp)."""
    if score_mode == O.SCORE_NEGLOGP:
        return -np.log(np.asarray(gpu["p_max"], np.float64))
    return np.asarray(gpu["entropy"])


def _check_decisions(gpu, b, W, ref, scores, st, alpha, tau, stats, mask_id, kind,
                     score_mode=0):
    """The CUDA path's argmax, fill set and new window against the oracle's
    decision rule applied to `scores`, skipping the decisions that those
    scores leave inside the 1e-3 margin (counted in `stats`)."""
    obs = st["obs"][b].astype(bool)
    inv = ref.inv
    gaps = top2_gap(scores.logits)
    n_obs = int(obs.sum())
    for p in range(n_obs, W):  # masked rows: the physical suffix
        if gaps[p] < MARGIN:
            stats.excluded_argmax += 1
            continue
        stats.checked_argmax += 1
        assert gpu["argmax"][b * W + p] == scores.argmax[p], (kind, b, p)
    g_filled = np.nonzero(gpu["filled"].numpy()[b])[0].tolist()
    masked = [j for j in range(W) if not obs[j]]
    H = np.where(obs, np.nan, O.slot_score(scores, score_mode)[inv])
    fill, ht = O.select_eq11(H, st["pos"][b], st["obs"][b], alpha, tau)
    nt, _, nobs = O.refill(st["tokens"][b], st["pos"][b], st["obs"][b], fill,
                           scores.argmax[inv], ref.n_commit, mask_id)
    near = any(abs(float(ht[j]) - tau) < MARGIN for j in masked)
    below = [j for j in masked if ht[j] < np.float32(tau)]
    if not below and len(masked) >= 2:
        v = np.sort(np.array([ht[j] for j in masked], np.float64))
        near = near or (v[1] - v[0] < MARGIN)
    if near:
        stats.excluded_select += 1
        return
    stats.checked_select += 1
    assert g_filled == fill, (kind, b, g_filled, fill)
    if all(gaps[inv[j]] >= MARGIN for j in fill):
        assert gpu["new_tokens"].numpy()[b].tolist() == nt.tolist(), (kind, b)
        assert gpu["new_observed"].numpy()[b].tolist() == nobs.tolist(), (kind, b)


def compare_seq(gpu, b, W, ref: O.SeqStep, st, alpha, tau, tol, stats: Stats,
                mask_id, check_hidden=True, bf16_stored=False, tf=None, score_mode=0,
                e2e_scores=True):
    """Compare sequence b of a GPU step result with the oracle's SeqStep.

    Continuous outputs are compared end to end with the oracle (`ref`):
    softmax statistics at the flat `tol`, the final hidden state at `tol`
    (a bf16 residual stream when bf16_stored: resid_bound over the last
    layer).
    Token decisions (argmax, fill set, window) are judged three ways:
      * against the oracle's end-to-end scores, 1e-3 margin;
      * when `tf` is given, also against the oracle's scores computed from
        the GPU's own LM-head input (teacher forcing; see
        teacher_forced_scores), 1e-3 margin;
      * the CUDA path's fills and window equal the oracle's rule applied to
        the CUDA path's own records, with no margin.
    e2e_scores=False (with `tf`): the softmax statistics and decisions are
    judged against the teacher-forced scores only.  End to end the logits
    carry the whole layer's bf16 error (the hidden state within
    resid_bound); under a planted peak the entropy moves by ~0.57 per unit
    of top-logit error, and near-uniform rows flip their argmax on top-2
    gaps just above the margin, so the LM head is held to its own input."""
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
        rb = resid_bound(ref.x_final, ref.x_mid[-1], tol) if bf16_stored else None
        e, ok = within(gpu["hidden"].float().numpy()[rows], ref.x_final, tol, bf16_stored,
                       name="hidden", bound=rb)
        stats.err("hidden", e)
        assert ok, f"hidden err {e}"
    sc = ref.scores
    assert e2e_scores or tf is not None
    cmp = sc if e2e_scores else tf
    tag = "" if e2e_scores else "_tf"
    # the LM head runs on the masked rows only (the physical suffix
    # n_obs..W-1); observed rows carry no record (argmax -1, NaN)
    n_obs = int(obs.sum())
    mrows = slice(b * W + n_obs, (b + 1) * W)
    assert np.all(gpu["argmax"][b * W:b * W + n_obs] == -1)
    assert np.all(np.isnan(gpu["entropy"][b * W:b * W + n_obs]))
    for name, g, r in (("lse", gpu["lse"][mrows], cmp.lse[n_obs:]),
                       ("entropy", gpu["entropy"][mrows], cmp.entropy[n_obs:]),
                       ("p_max", gpu["p_max"][mrows], cmp.p_max[n_obs:])):
        e, ok = within(g, r, tol, name=name + tag)
        stats.err(name, e)
        assert ok, f"{name} err {e}"
    # the CUDA path's decisions = the rule applied to its own records (fp32,
    # no margin), and its window = the refill rule on its own fills
    inv = ref.inv
    gH = np.where(obs, np.nan, gpu_slot_score(gpu, score_mode)[b * W + inv])
    g_fill, g_ht = O.select_eq11(gH, st["pos"][b], st["obs"][b], alpha, tau)
    g_filled = np.nonzero(gpu["filled"].numpy()[b])[0].tolist()
    # (the confidence score is recomputed here in float64: a rule decision
    # within 1e-6 of tau may go either way)
    edge = score_mode == O.SCORE_NEGLOGP and bool(
        np.any(np.abs(g_ht[~obs].astype(np.float64) - tau) < 1e-6))
    assert g_filled == g_fill or edge, (b, g_filled, g_fill)
    g_am = gpu["argmax"][b * W + inv]
    nt, _, nobs = O.refill(st["tokens"][b], st["pos"][b], st["obs"][b], g_fill, g_am,
                           ref.n_commit, mask_id)
    assert gpu["new_tokens"].numpy()[b].tolist() == nt.tolist()
    assert gpu["new_observed"].numpy()[b].tolist() == nobs.tolist()
    # the oracle's decisions, end to end and (when given) teacher forced
    if e2e_scores:
        _check_decisions(gpu, b, W, ref, sc, st, alpha, tau, stats, mask_id, "end-to-end",
                         score_mode)
    if tf is not None:
        _check_decisions(gpu, b, W, ref, tf, st, alpha, tau, stats, mask_id, "teacher-forced",
                         score_mode)


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
        ek, okk = within(k[L:], ref_k, tol, bf16_stored, name=f"{name}_k")
        ev, okv = within(v[L:], ref_v, tol, bf16_stored, name=f"{name}_v")
        stats.err(name, max(ek, ev))
        assert okk and okv, f"{name} err {ek} {ev}"
