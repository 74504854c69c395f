"""CPU oracle for one WeDLM window decode step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module;
only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
shares no code with the CUDA path (no kernels, headers, tables or helpers):
it is a plain, slow restatement of what one decoding step computes, in
float64, written from the WeDLM pages ("WeDLM: Reconciling Diffusion
Language Models with Standard Causal Attention for Fast Inference"; the
bud-325 summary's Key claims and Method sections carry the only formulas).

The step, in the order the Method section gives it:
  1. Topological Reordering: observed slots take the physical prefix, masked
     slots the physical suffix; RoPE keeps each token's logical position
     (Key claims, "Topological Reordering ... §4.1, Eq. 5-6").
  2. A causal forward of the reordered window on top of the cached prefix
     K/V, with an unmodified lower-triangular mask (Key claims, §3.2 and
     §5.2: "a small causal prefill over the active window").
  3. Per masked slot: softmax over the vocabulary, its entropy H_j and
     argmax (Method: "distance-penalized entropy").
  4. Selection with the distance-penalised entropy H~_j = H_j + alpha*d_j,
     d_j the distance from slot j to the leftmost remaining mask (Method;
     called Eq. 11 in Key claims, §5.2).
  5. Commit the leftmost contiguous filled prefix into the KV cache and
     refill the freed slots with [M] (Method; Key claims §5.2).

Readings where the pages are silent (each is listed in the design notes):
  * score = entropy in nats; fill every masked slot with H~ < tau, and if
    none qualifies the single argmin (ties: lowest slot);
  * d_j = pos_j - pos_{m0}, m0 the leftmost masked slot before this step's
    fills;
  * commit set = the longest run of slots 0..c-1 observed *at input* whose
    logical positions continue the committed prefix (pos = L + i); slots
    filled this step are committed in a later step;
  * the prediction for slot j is the output row of slot j itself (mask
    recovery, not next-token shifted);
  * [M] = `mask_id`; its logit is set to -inf; argmax ties go to the lowest
    token id;
  * backbone: pre-norm RMSNorm, no biases, optional per-head QK-RMSNorm,
    rotate-half RoPE with inv_freq_i = theta^(-2i/hd), SwiGLU FFN, untied
    LM head, final RMSNorm before the LM head;
  * when the CUDA path stores a tensor in bf16, the oracle rounds the same
    tensor to bf16 (round to nearest, ties to even); all other arithmetic
    is float64.  For fp32 storage no rounding is mirrored.
  * the selection compares H~ in float32, as the kernel does, so that both
    sides take the integer decision in the same precision.

Parity pins for every function here live in tests/test_oracle_*.py.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

# ---------------------------------------------------------------------------
# storage rounding
# ---------------------------------------------------------------------------


def bf16_round(x):
    """Round to the nearest bfloat16 value (ties to even), as float64.

    bfloat16 is the top 16 bits of an IEEE binary32.  The value is first
    rounded to binary32 (numpy, nearest-even), then the low 16 bits are
    rounded away: add 0x7FFF plus the lowest kept bit, truncate.  NaN stays
    NaN; values beyond the bf16 range become +-inf.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)) << np.uint64(16)
    out = r.astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(f)
    if np.any(nan):
        out = np.where(nan, np.nan, out)
    return out


def storer(dtype: str):
    """The rounding applied where the CUDA path stores a tensor."""
    if dtype == "bf16":
        return bf16_round
    return lambda a: np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# backbone pieces
# ---------------------------------------------------------------------------


def rmsnorm(x, gain, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gain."""
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gain, np.float64)


def rope_cos_sin(pos, head_dim, theta):
    """cos/sin of the rotation angles at (logical) positions `pos`.

    Angle for pair i (0 <= i < head_dim/2) at position p:
    p * theta^(-2i/head_dim), computed in float64.
    """
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = np.power(float(theta), -2.0 * i / head_dim)
    ang = np.asarray(pos, np.float64)[..., None] * inv_freq
    return np.cos(ang), np.sin(ang)


def rope_apply(x, cos, sin):
    """Rotate-half RoPE on the last axis: pairs (i, i + hd/2).

    x: [..., n_heads, hd]; cos/sin: [..., hd/2] (broadcast over heads).
    """
    half = x.shape[-1] // 2
    c = cos[..., None, :]
    s = sin[..., None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


# ---------------------------------------------------------------------------
# Topological Reordering (Key claims §4.1; Method)
# ---------------------------------------------------------------------------


def topological_reorder(observed):
    """Stable partition of the W window slots: observed first, then masked.

    Returns (perm, inv): perm[p] is the slot placed at physical index p,
    inv[j] is the physical index of slot j.  Inside each group the slots
    keep ascending slot (= logical) order.
    """
    obs = [bool(o) for o in np.asarray(observed).reshape(-1)]
    perm = [j for j in range(len(obs)) if obs[j]] + \
           [j for j in range(len(obs)) if not obs[j]]
    perm = np.asarray(perm, np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm), dtype=np.int32)
    return perm, inv


# ---------------------------------------------------------------------------
# paged KV pool format
# ---------------------------------------------------------------------------


def page_elem_offset(t, d, head_dim):
    """Offset of (token t, dim d) inside one (page, K|V, kv-head) block.

    The block is stored as 8x8 tiles (8 tokens x 8 dims, row = token),
    tiles ordered by token group first, then dim group.
    """
    t = np.asarray(t)
    d = np.asarray(d)
    return ((t // 8) * (head_dim // 8) + d // 8) * 64 + (t % 8) * 8 + (d % 8)


def pool_view(pool, shape):
    """A flat pool as [num_pages][2][n_kv][page_block*head_dim]."""
    blockn = shape.page_block * shape.head_dim
    return np.asarray(pool).reshape(-1, 2, shape.n_kv_heads, blockn)


def pool_gather(pool, page_row, length, shape):
    """Cached K and V of positions 0..length-1: two [length][n_kv][hd]."""
    hd, blk, nkv = shape.head_dim, shape.page_block, shape.n_kv_heads
    if length == 0:
        z = np.zeros((0, nkv, hd))
        return z, z.copy()
    pv = pool_view(pool, shape)
    t = np.arange(length)
    pages = np.asarray(page_row)[t // blk]
    off = page_elem_offset((t % blk)[:, None], np.arange(hd)[None, :], hd)
    heads = np.arange(nkv)
    k = pv[pages[:, None, None], 0, heads[None, :, None], off[:, None, :]]
    v = pv[pages[:, None, None], 1, heads[None, :, None], off[:, None, :]]
    return np.asarray(k, np.float64), np.asarray(v, np.float64)


def pool_scatter(pool, page_row, positions, k, v, shape):
    """Write K/V rows ([n][n_kv][hd]) at sequence positions `positions`."""
    hd, blk, nkv = shape.head_dim, shape.page_block, shape.n_kv_heads
    positions = np.asarray(positions, np.int64)
    if positions.size == 0:
        return
    pv = pool_view(pool, shape)
    pages = np.asarray(page_row)[positions // blk]
    off = page_elem_offset((positions % blk)[:, None], np.arange(hd)[None, :], hd)
    heads = np.arange(nkv)
    pv[pages[:, None, None], 0, heads[None, :, None], off[:, None, :]] = k
    pv[pages[:, None, None], 1, heads[None, :, None], off[:, None, :]] = v


# ---------------------------------------------------------------------------
# attention: causal over [cached prefix || window] (Key claims §3.2, §5.2)
# ---------------------------------------------------------------------------


def window_attention(q, k_pre, v_pre, k_win, v_win, visible=None):
    """Softmax attention of the window queries.

    q: [W][nq][hd]; k_pre/v_pre: [L][nkv][hd]; k_win/v_win: [W][nkv][hd].
    Every query sees the whole prefix.  Among window keys, row p sees key
    j iff visible[p][j]; the default is the lower-triangular causal mask on
    physical indices (j <= p).  Query head h uses kv head h // (nq/nkv).
    Scale 1/sqrt(hd).
    """
    W, nq, hd = q.shape
    L = k_pre.shape[0]
    nkv = k_win.shape[1]
    group = nq // nkv
    if visible is None:
        visible = np.tril(np.ones((W, W), bool))
    vis = np.concatenate([np.ones((W, L), bool), np.asarray(visible, bool)], 1)
    out = np.zeros((W, nq, hd))
    for h in range(nq):
        g = h // group
        keys = np.concatenate([k_pre[:, g], k_win[:, g]], 0)
        vals = np.concatenate([v_pre[:, g], v_win[:, g]], 0)
        s = (q[:, h] @ keys.T) / np.sqrt(hd)
        s = np.where(vis, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h] = p @ vals
    return out


def dual_stream_visibility(n, block):
    """Visibility of Dual-Stream Masking over the 2n keys [memory stream ||
    prediction stream] for the 2n query rows in the same order (Key claims
    §4.2, Eq. 8-10; Method: "prediction-stream tokens in block i attend to
    memory-stream tokens whose logical positions precede i").  Memory row r
    (logical position r) sees memory keys 0..r.  Prediction row n+i lies in
    block j = i // block at physical index p = i % block of the block's
    topologically reordered order; it sees the memory keys at positions
    before the block, 0..j*block-1, and the keys of its own block at physical
    index <= p (causal in the reordered order)."""
    vis = np.zeros((2 * n, 2 * n), bool)
    for r in range(2 * n):
        vis[r] = dual_stream_visible_row(n, block, r)
    return vis


def dual_stream_visible_row(n, block, r):
    """Row r of the Dual-Stream visibility above (same rule, one query row):
    a memory row sees the memory up to itself, a prediction row the memory
    before its block and its own block causally."""
    v = np.zeros(2 * n, bool)
    if r < n:
        v[:r + 1] = True
    else:
        j, p = divmod(r - n, block)
        v[:j * block] = True
        v[n + j * block:n + j * block + p + 1] = True
    return v


def dual_stream_attention(q, k_mem, v_mem, k_pred, v_pred, block):
    """Attention of both streams under Dual-Stream Masking.

    q: [2n][nq][hd] (memory rows, then prediction rows); k/v of each stream:
    [n][nkv][hd].  Softmax with scale 1/sqrt(hd) over the visible keys;
    query head h reads kv head h // (nq/nkv).  Returns [2n][nq][hd]."""
    q = np.asarray(q, np.float64)
    n2, nq, hd = q.shape
    n = n2 // 2
    keys = np.concatenate([k_mem, k_pred], 0).astype(np.float64)
    vals = np.concatenate([v_mem, v_pred], 0).astype(np.float64)
    nkv = keys.shape[1]
    group = nq // nkv
    vis = dual_stream_visibility(n, block)
    out = np.zeros((n2, nq, hd))
    for h in range(nq):
        g = h // group
        s = (q[:, h] @ keys[:, g].T) / np.sqrt(hd)
        s = np.where(vis, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h] = p @ vals[:, g]
    return out


def dual_stream_attention_rows(q, k_mem, v_mem, k_pred, v_pred, block, rows):
    """dual_stream_attention for the query rows `rows` only (indices into the
    2n rows; q holds all 2n): the same softmax over each row's visible keys,
    for checking sampled rows of a call too large to evaluate whole.
    Returns [len(rows)][nq][hd]."""
    q = np.asarray(q, np.float64)
    n2, nq, hd = q.shape
    n = n2 // 2
    keys = np.concatenate([k_mem, k_pred], 0).astype(np.float64)
    vals = np.concatenate([v_mem, v_pred], 0).astype(np.float64)
    group = nq // keys.shape[1]
    out = np.zeros((len(rows), nq, hd))
    for i, r in enumerate(rows):
        vis = dual_stream_visible_row(n, block, r)
        for h in range(nq):
            g = h // group
            s = (keys[vis, g] @ q[r, h]) / np.sqrt(hd)
            p = np.exp(s - s.max())
            out[i, h] = (p / p.sum()) @ vals[vis, g]
    return out


def _f64(a):
    return np.asarray(a, np.float64)


def qkv_project(shape, lw, x, cos, sin, store):
    """RMSNorm -> q, k, v -> optional QK-norm -> RoPE (logical positions).

    x: [W][H] (rows in physical order).  Returns (xn, q, k, v) as stored.
    """
    s = shape
    W = x.shape[0]
    xn = store(rmsnorm(x, lw["attn_norm"], s.rms_eps))
    q = (xn @ _f64(lw["w_q"]).T).reshape(W, s.n_q_heads, s.head_dim)
    k = (xn @ _f64(lw["w_k"]).T).reshape(W, s.n_kv_heads, s.head_dim)
    v = (xn @ _f64(lw["w_v"]).T).reshape(W, s.n_kv_heads, s.head_dim)
    if s.qk_norm:
        q = rmsnorm(q, lw["q_norm"], s.rms_eps)
        k = rmsnorm(k, lw["k_norm"], s.rms_eps)
    q = store(rope_apply(q, cos, sin))
    k = store(rope_apply(k, cos, sin))
    v = store(v)
    return xn, q, k, v


def layer_forward(shape, lw, x, cos, sin, k_pre, v_pre, store, visible=None, mid=None):
    """One pre-norm decoder layer over the window rows.

    Returns (x_out, k_win, v_win, attn_out).  When `mid` is a list, the
    residual stream between the attention block and the FFN (as stored) is
    appended to it.
    """
    s = shape
    W = x.shape[0]
    _, q, k, v = qkv_project(s, lw, x, cos, sin, store)
    o = store(window_attention(q, k_pre, v_pre, k, v, visible))
    x = store(x + o.reshape(W, -1) @ _f64(lw["w_o"]).T)
    if mid is not None:
        mid.append(x)
    xn = store(rmsnorm(x, lw["ffn_norm"], s.rms_eps))
    g = xn @ _f64(lw["w_gate"]).T
    u = xn @ _f64(lw["w_up"]).T
    a = store(silu(g) * u)
    x = store(x + a @ _f64(lw["w_down"]).T)
    return x, k, v, o


# ---------------------------------------------------------------------------
# LM head + softmax statistics (Method: entropy H_j per masked slot)
# ---------------------------------------------------------------------------


@dataclass
class SlotScores:
    argmax: np.ndarray   # int32 token id (lowest id among equal maxima)
    entropy: np.ndarray  # H_j in nats
    p_max: np.ndarray    # probability of the argmax token
    lse: np.ndarray      # log-sum-exp of the logits
    logits: Optional[np.ndarray] = None


def lm_head_logits(h_final, lm_head, mask_id, plant_tok=None, plant_bias=0.0):
    """z = h W_lm^T (+ planted bias on one token per row); z[mask_id] = -inf."""
    z = _f64(h_final) @ _f64(lm_head).T
    if plant_tok is not None:
        pt = np.asarray(plant_tok).reshape(-1)
        rows = np.nonzero(pt >= 0)[0]
        z[rows, pt[rows]] += plant_bias
    z[:, mask_id] = -np.inf
    return z


def softmax_scores(z):
    """argmax, entropy, p_max and lse of softmax(z) per row, from the
    definitions (materialised probabilities)."""
    a = np.argmax(z, axis=1).astype(np.int32)
    m = z[np.arange(z.shape[0]), a]
    e = np.exp(z - m[:, None])
    ssum = e.sum(axis=1)
    p = e / ssum[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        plogp = np.where(p > 0, p * np.log(np.where(p > 0, p, 1.0)), 0.0)
    ent = -plogp.sum(axis=1)
    return SlotScores(argmax=a, entropy=ent, p_max=p.max(axis=1),
                      lse=m + np.log(ssum), logits=z)


# ---------------------------------------------------------------------------
# Eq. 11 selection and the commit / refill (Method)
# ---------------------------------------------------------------------------


SCORE_ENTROPY, SCORE_NEGLOGP = 0, 1


def slot_score(scores, mode):
    """The per-row score that Eq. 11 penalises by distance: the entropy H_j
    of the row's softmax (Method: "distance-penalized entropy"), or, for
    the confidence reading (Key claims §5.2: "distance-penalized confidence
    rule"), the negative log of the row's top probability, -ln p_max.
    Lower is more certain in both readings."""
    if mode == SCORE_ENTROPY:
        return np.asarray(scores.entropy, np.float64)
    if mode == SCORE_NEGLOGP:
        return -np.log(np.asarray(scores.p_max, np.float64))
    raise ValueError(f"unknown score mode {mode}")


def select_eq11(entropy, pos, observed, alpha, tau):
    """Distance-penalised entropy selection for one window.

    Among masked slots: d_j = pos_j - pos_{m0} (m0 = leftmost masked slot),
    H~_j = H_j + alpha * d_j, evaluated in float32 (multiply, then add, each
    rounded).  Fill every masked j with H~_j < tau; if none qualifies, fill
    the single masked slot with the smallest H~ (ties -> lowest slot; NaN
    counts as +inf).  Returns (fill list, H~ array with NaN at observed).
    """
    obs = np.asarray(observed).astype(bool)
    W = obs.size
    ht = np.full(W, np.nan, np.float32)
    masked = [j for j in range(W) if not obs[j]]
    if not masked:
        return [], ht
    m0 = masked[0]
    a32 = np.float32(alpha)
    t32 = np.float32(tau)
    for j in masked:
        d = np.float32(int(pos[j]) - int(pos[m0]))
        ht[j] = np.float32(np.float32(entropy[j]) + np.float32(a32 * d))
    fill = [j for j in masked if ht[j] < t32]
    if not fill:
        def key(j):
            v = ht[j]
            return (np.inf if np.isnan(v) else float(v), j)
        fill = [min(masked, key=key)]
    return fill, ht


def commit_run(observed, pos, seq_len):
    """Length c of the leftmost contiguous observed run continuing the
    committed prefix: slots 0..c-1 observed with pos = seq_len + i."""
    c = 0
    W = len(observed)
    while c < W and observed[c] and int(pos[c]) == int(seq_len) + c:
        c += 1
    return c


def refill(tokens, pos, observed, fill, fill_tokens, c, mask_id):
    """Window after the step: fills applied, the first c slots dropped,
    c new [M] slots appended at the next logical positions."""
    tok = np.array(tokens, np.int32)
    obs = np.array(observed, np.uint8)
    for j in fill:
        tok[j] = fill_tokens[j]
        obs[j] = 1
    W = tok.size
    last = int(pos[W - 1])
    new_tok = np.concatenate([tok[c:], np.full(c, mask_id, np.int32)])
    new_pos = np.concatenate([np.asarray(pos, np.int32)[c:],
                              last + 1 + np.arange(c, dtype=np.int32)])
    new_obs = np.concatenate([obs[c:], np.zeros(c, np.uint8)])
    return new_tok, new_pos.astype(np.int32), new_obs


# ---------------------------------------------------------------------------
# the whole step
# ---------------------------------------------------------------------------


@dataclass
class SeqStep:
    perm: np.ndarray
    inv: np.ndarray
    scores: SlotScores            # per PHYSICAL row
    slot_entropy: np.ndarray      # per slot (NaN at observed slots)
    slot_argmax: np.ndarray
    ht: np.ndarray                # H~ per slot (float32, NaN at observed)
    fill: List[int]
    n_commit: int
    committed: np.ndarray
    new_tokens: np.ndarray
    new_pos: np.ndarray
    new_obs: np.ndarray
    new_seq_len: int
    x_final: np.ndarray           # residual stream after the last layer
    h_final: np.ndarray           # final-norm LM-head input
    k_win: list = field(default_factory=list)   # per layer [W][nkv][hd]
    v_win: list = field(default_factory=list)
    attn_out: list = field(default_factory=list)
    x_mid: list = field(default_factory=list)   # per layer: residual after attention


def forward_window(shape, weights, tokens_phys, pos_phys, pools, page_row,
                   seq_len, store, visible=None, layers=None, mid=None):
    """Causal forward of the reordered window on top of the cached prefix.

    Returns (x_final, k_win per layer, v_win per layer, attn_out per layer);
    `mid` (a list, optional) receives each layer's residual stream between
    its attention block and its FFN.
    """
    s = shape
    x = store(_f64(weights["embed"])[np.asarray(tokens_phys)])
    cos, sin = rope_cos_sin(pos_phys, s.head_dim, s.rope_theta)
    ks, vs, os_ = [], [], []
    for l in (range(s.n_layers) if layers is None else layers):
        kp, vp = pool_gather(pools[l], page_row, seq_len, s)
        x, k, v, o = layer_forward(s, weights["layers"][l], x, cos, sin,
                                   kp, vp, store, visible, mid)
        ks.append(k)
        vs.append(v)
        os_.append(o)
    return x, ks, vs, os_


def oracle_step_seq(shape, weights, tokens, pos, observed, seq_len, page_row,
                    pools, alpha, tau, plant_tok=None, plant_bias=0.0,
                    write_pools=True, score_mode=SCORE_ENTROPY):
    """One window decode step of one sequence.  `pools` (list of flat
    per-layer arrays) are updated in place with the committed K/V when
    `write_pools` is set.  `score_mode` picks the score Eq. 11 penalises
    (slot_score)."""
    s = shape
    store = storer(s.dtype)
    tokens = np.asarray(tokens, np.int32)
    pos = np.asarray(pos, np.int32)
    obs = np.asarray(observed).astype(np.uint8)
    perm, inv = topological_reorder(obs)
    mids = []
    x, ks, vs, os_ = forward_window(s, weights, tokens[perm], pos[perm],
                                    pools, page_row, int(seq_len), store, mid=mids)
    h = store(rmsnorm(x, weights["final_norm"], s.rms_eps))
    pt = None if plant_tok is None else np.asarray(plant_tok)[perm]
    sc = softmax_scores(lm_head_logits(h, weights["lm_head"], s.mask_id,
                                       pt, plant_bias))
    W = tokens.size
    slot_H = np.where(obs.astype(bool), np.nan, slot_score(sc, score_mode)[inv])
    slot_a = sc.argmax[inv]
    fill, ht = select_eq11(slot_H, pos, obs, alpha, tau)
    c = commit_run(obs, pos, seq_len)
    if write_pools and c > 0:
        rows = inv[:c]
        for l in range(s.n_layers):
            pool_scatter(pools[l], page_row, int(seq_len) + np.arange(c),
                         ks[l][rows], vs[l][rows], s)
    nt, npos, nobs = refill(tokens, pos, obs, fill, slot_a, c, s.mask_id)
    return SeqStep(perm=perm, inv=inv, scores=sc, slot_entropy=slot_H,
                   slot_argmax=slot_a, ht=ht, fill=fill, n_commit=c,
                   committed=tokens[:c].copy(), new_tokens=nt, new_pos=npos,
                   new_obs=nobs, new_seq_len=int(seq_len) + c, x_final=x,
                   h_final=h, k_win=ks, v_win=vs, attn_out=os_, x_mid=mids)


def oracle_step(shape, weights, state, pools, alpha, tau, plant_tok=None,
                plant_bias=0.0, write_pools=True, score_mode=SCORE_ENTROPY):
    """One window decode step of a batch; per-sequence results."""
    out = []
    for b in range(state["tokens"].shape[0]):
        out.append(oracle_step_seq(
            shape, weights, state["tokens"][b], state["pos"][b],
            state["obs"][b], int(state["seq_len"][b]),
            state["page_table"][b], pools, alpha, tau,
            None if plant_tok is None else plant_tok[b], plant_bias,
            write_pools, score_mode))
    return out


def oracle_prefill(shape, weights, tokens):
    """Plain autoregressive-order causal forward over `tokens` at positions
    0..T-1 with an empty cache.  Returns per-layer K and V ([T][nkv][hd])
    as stored, and the final residual stream."""
    s = shape
    store = storer(s.dtype)
    tokens = np.asarray(tokens, np.int32)
    T = tokens.size
    empty = [np.zeros(0)] * s.n_layers
    x = store(_f64(weights["embed"])[tokens])
    cos, sin = rope_cos_sin(np.arange(T), s.head_dim, s.rope_theta)
    ks, vs = [], []
    z = np.zeros((0, s.n_kv_heads, s.head_dim))
    for l in range(s.n_layers):
        x, k, v, _ = layer_forward(s, weights["layers"][l], x, cos, sin, z, z,
                                   store)
        ks.append(k)
        vs.append(v)
    return ks, vs, x
