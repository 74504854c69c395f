"""The allocation-free attention entry point (wedlm_attention_static).

Callers that cannot allocate device memory (a host framework that owns all
allocations, a memory-capped service) use this entry point: its scratch is a
static device array of the library.  It runs the same kernel as
wedlm_attention with the same grid and the same slot-order merge, so its
output must be bit-identical to wedlm_attention's, on two calls in a row (the
second reuses the array with the first call's contents still in it).  This
file is collected last on purpose."""
import numpy as np
import pytest
import torch

from synth import Workload, make_pool_torch, make_state_np, make_weights_torch, qwen3_layers

pytestmark = pytest.mark.gpu


def test_attention_static_matches_wedlm_attention_twice():
    from serving_wedlm_step_gb300 import binding as Bd
    from tests.gpu_common import dev
    s = qwen3_layers(1)
    B, W = 8, 16
    wl = Workload("t", s, batch=B, window=W, prefix=(300, 2500), masked=(4, 12),
                  shuffled_pages=True, seed=21)
    st = make_state_np(wl)
    pool = make_pool_torch(s, st["num_pages"], 21, 0)
    g = torch.Generator(device="cuda")
    g.manual_seed(21)
    w = make_weights_torch(s, seed=21)
    ctx = Bd.WedlmContext(s, w, window=W, max_batch=B, max_pages_per_seq=st["max_pages"])
    pt, sl = dev(st["page_table"]), dev(st["seq_len"])
    outs_ref, outs_static = [], []
    for call in range(2):
        q = torch.randn(B * W, s.n_q_heads, s.head_dim, generator=g, device="cuda").to(torch.bfloat16)
        win = (torch.randn(B, 2, s.n_kv_heads, 16 * s.head_dim, generator=g, device="cuda")
               .to(torch.bfloat16))
        o_ref = torch.empty(B * W, s.n_q_heads * s.head_dim, dtype=torch.bfloat16, device="cuda")
        o_st = torch.full_like(o_ref, float("nan"))
        ctx.attention(q, pool, pt, sl, st["num_pages"], win, o_ref)
        Bd.attention_static(W, s.n_q_heads, s.n_kv_heads, st["max_pages"], st["num_pages"],
                            q, pool, pt, sl, win, o_st)
        torch.cuda.synchronize()
        assert ctx.status() == 0
        assert Bd.attention_static_status() == 0
        outs_ref.append(o_ref.float().cpu().numpy())
        outs_static.append(o_st.float().cpu().numpy())
    for a, b in zip(outs_ref, outs_static):
        assert np.isfinite(b).all()
        assert np.array_equal(a, b), float(np.abs(a - b).max())
    # the two calls really computed different things
    assert np.abs(outs_static[0] - outs_static[1]).max() > 0.1
    ctx.close()


def test_attention_static_status_reports_bad_page_ids():
    """A page id outside [0, num_pages) reads as zeros and sets
    WEDLM_DEV_BAD_PAGE in the static array's error word, which the status
    call reads back; the next clean call clears it and matches
    wedlm_attention bit for bit."""
    from serving_wedlm_step_gb300 import binding as Bd
    from tests.gpu_common import dev
    s = qwen3_layers(1)
    B, W = 4, 16
    wl = Workload("t", s, batch=B, window=W, prefix=(200, 900), masked=(4, 12),
                  shuffled_pages=True, seed=23)
    st = make_state_np(wl)
    pool = make_pool_torch(s, st["num_pages"], 23, 0)
    g = torch.Generator(device="cuda")
    g.manual_seed(23)
    w = make_weights_torch(s, seed=23)
    ctx = Bd.WedlmContext(s, w, window=W, max_batch=B, max_pages_per_seq=st["max_pages"])
    q = torch.randn(B * W, s.n_q_heads, s.head_dim, generator=g, device="cuda").to(torch.bfloat16)
    win = (torch.randn(B, 2, s.n_kv_heads, 16 * s.head_dim, generator=g, device="cuda")
           .to(torch.bfloat16))
    bad_pt = st["page_table"].copy()
    bad_pt[1, 0] = st["num_pages"] + 5
    o = torch.empty(B * W, s.n_q_heads * s.head_dim, dtype=torch.bfloat16, device="cuda")
    Bd.attention_static(W, s.n_q_heads, s.n_kv_heads, st["max_pages"], st["num_pages"],
                        q, pool, dev(bad_pt), dev(st["seq_len"]), win, o)
    assert Bd.attention_static_status() & Bd.DEV_BAD_PAGE
    pt, sl = dev(st["page_table"]), dev(st["seq_len"])
    o_ref = torch.empty_like(o)
    ctx.attention(q, pool, pt, sl, st["num_pages"], win, o_ref)
    Bd.attention_static(W, s.n_q_heads, s.n_kv_heads, st["max_pages"], st["num_pages"],
                        q, pool, pt, sl, win, o)
    assert Bd.attention_static_status() == 0
    assert ctx.status() == 0
    assert torch.equal(o, o_ref)
    ctx.close()


def test_attention_static_rejects_oversized_batch():
    from serving_wedlm_step_gb300 import binding as Bd
    from tests.gpu_common import dev
    # the partials need (SMs + sequences x kv heads) segments of G*W rows x
    # 130 floats; with G*W = 128 rows each segment is 66560 bytes, and 32
    # sequences x 8 kv heads = 256 segments already exceed the 16 MiB array
    # whatever the SM count; fewer sequences suffice on larger GPUs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nq, nkv, W = 64, 8, 16
    seg = 128 * 130 * 4
    need_units = (16 << 20) // seg + 1 - sms
    B = int(min(32, max(1, -(-need_units // nkv))))
    assert (sms + B * nkv) * seg > (16 << 20)
    q = torch.zeros(B * W, nq, 128, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(2 * 2 * nkv * 16 * 128, dtype=torch.bfloat16, device="cuda")
    win = torch.zeros(B, 2, nkv, 16 * 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(B * W, nq * 128, dtype=torch.bfloat16, device="cuda")
    pt = dev(np.zeros((B, 2), np.int32))
    sl = dev(np.zeros(B, np.int32))
    with pytest.raises(Bd.WedlmError) as e:
        Bd.attention_static(W, nq, nkv, 2, 2, q, pool, pt, sl, win, o)
    assert e.value.code == Bd.ERR_CAPACITY
