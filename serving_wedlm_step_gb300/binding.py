"""ctypes binding of libwedlm (include/wedlm.h): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels; this
module only turns torch tensors into device pointers and checks return
codes.  Importing it loads the in-tree libwedlm.so and fails loudly when the
library is missing (there is no fallback of any kind).
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_void_p

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libwedlm.so")

# error codes and device error bits (mirror include/wedlm.h)
OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_CUDA, ERR_NUMERIC, ERR_TIMEOUT, ERR_DEVICE = range(7)
DEV_BAD_PAGE, DEV_CAPACITY, DEV_BAD_TOKEN, DEV_NUMERIC, DEV_TIMEOUT, DEV_BAD_SEQLEN = (
    1, 2, 4, 8, 16, 32)
BF16, FP32 = 0, 1
SCORE_ENTROPY, SCORE_NEGLOGP = 0, 1
KINDS = ["reorder", "rmsnorm", "gemm_qkv", "attn", "attn_merge", "gemm_o",
         "gemm_gateup", "gemm_down", "lmhead", "lmhead_merge", "select", "commit"]

EXPORTED = ["wedlm_create", "wedlm_destroy", "wedlm_last_error", "wedlm_get_status",
            "wedlm_set_graphs", "wedlm_set_timing", "wedlm_get_timings",
            "wedlm_launches_per_step", "wedlm_step", "wedlm_reorder_embed",
            "wedlm_layer", "wedlm_attention", "wedlm_lm_head", "wedlm_attention_static",
            "wedlm_attention_static_status", "wedlm_selftest_bounded_wait",
            "wedlm_prefill", "wedlm_generate", "wedlm_dual_stream_attention"]


class Config(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in (
        "n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
        "window", "page_block", "max_batch", "max_pages_per_seq", "dtype", "qk_norm",
        "mask_id")] + [("rope_theta", c_float), ("rms_eps", c_float)]


_LAYER_FIELDS = ("attn_norm", "w_q", "w_k", "w_v", "q_norm", "k_norm", "w_o",
                 "ffn_norm", "w_gate", "w_up", "w_down")


class Weights(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("final_norm", c_void_p), ("lm_head", c_void_p)] + [
        (n, POINTER(c_void_p)) for n in _LAYER_FIELDS]


class SlotRec(ctypes.Structure):
    _fields_ = [("argmax", c_int32), ("entropy", c_float), ("p_max", c_float),
                ("lse", c_float)]


class StepIn(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("num_pages", c_int32), ("tokens", c_void_p),
                ("pos", c_void_p), ("observed", c_void_p), ("seq_len", c_void_p),
                ("page_table", c_void_p), ("kv_pools", POINTER(c_void_p)),
                ("plant_token", c_void_p), ("plant_bias", c_float), ("alpha", c_float),
                ("tau", c_float), ("score_mode", c_int32)]


class GenIn(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("num_pages", c_int32), ("tokens", c_void_p),
                ("pos", c_void_p), ("observed", c_void_p), ("seq_len", c_void_p),
                ("page_table", c_void_p), ("kv_pools", POINTER(c_void_p)),
                ("plant_token", c_void_p), ("plant_bias", c_float), ("alpha", c_float),
                ("tau", c_float), ("score_mode", c_int32), ("max_steps", c_int32),
                ("done", c_void_p), ("stop_len", c_void_p), ("stop_token", c_int32),
                ("out_tokens", c_void_p), ("out_base", c_void_p), ("out_cap", c_int32),
                ("steps_run", c_void_p)]


class StepOut(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in (
        "new_tokens", "new_pos", "new_observed", "committed", "n_committed", "perm",
        "filled", "rows", "logits", "hidden")]


def load_library(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(
            f"libwedlm.so not found at {path}: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    lib.wedlm_create.argtypes = [POINTER(Config), POINTER(Weights), POINTER(c_void_p)]
    lib.wedlm_destroy.argtypes = [c_void_p]
    lib.wedlm_destroy.restype = None
    lib.wedlm_last_error.argtypes = [c_void_p]
    lib.wedlm_last_error.restype = ctypes.c_char_p
    lib.wedlm_get_status.argtypes = [c_void_p, POINTER(c_int32)]
    lib.wedlm_set_graphs.argtypes = [c_void_p, ctypes.c_int]
    lib.wedlm_set_timing.argtypes = [c_void_p, ctypes.c_int]
    lib.wedlm_get_timings.argtypes = [c_void_p, POINTER(c_float), POINTER(c_int32), ctypes.c_int]
    lib.wedlm_launches_per_step.argtypes = [c_void_p, c_int32]
    lib.wedlm_step.argtypes = [c_void_p, POINTER(StepIn), POINTER(StepOut), c_void_p]
    lib.wedlm_reorder_embed.argtypes = [c_void_p, c_int32] + [c_void_p] * 8
    lib.wedlm_layer.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_int32] + [c_void_p] * 5
    lib.wedlm_attention.argtypes = [c_void_p, c_int32, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_int32, c_void_p, c_void_p, c_void_p]
    lib.wedlm_lm_head.argtypes = [c_void_p, c_int32, c_void_p, c_void_p, c_float,
                                  c_void_p, c_void_p, c_void_p]
    lib.wedlm_attention_static.argtypes = [c_int32] * 6 + [c_void_p] * 7
    lib.wedlm_attention_static_status.argtypes = [c_void_p, POINTER(c_int32)]
    lib.wedlm_selftest_bounded_wait.argtypes = [c_void_p, POINTER(c_int32), POINTER(c_int32),
                                                c_void_p]
    lib.wedlm_prefill.argtypes = [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                  c_int32, POINTER(c_void_p), c_void_p, c_void_p]
    lib.wedlm_generate.argtypes = [c_void_p, POINTER(GenIn), c_void_p]
    lib.wedlm_dual_stream_attention.argtypes = [c_void_p, c_int32, c_int32] + [c_void_p] * 5
    return lib


_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        _LIB = load_library()
    return _LIB


class WedlmError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libwedlm error {code}: {msg}")
        self.code = code


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class WedlmContext:
    """One libwedlm context over a set of torch weight tensors.

    `weights` is a dict: embed, final_norm, lm_head and `layers`, a list of
    dicts with attn_norm, w_q, w_k, w_v, q_norm, k_norm, w_o, ffn_norm,
    w_gate, w_up, w_down (contiguous CUDA tensors of the context dtype).
    """

    def __init__(self, shape, weights, window, max_batch, max_pages_per_seq):
        import torch
        self._lib = lib()
        self.shape = shape
        self.window = window
        self.max_batch = max_batch
        self.max_pages_per_seq = max_pages_per_seq
        dt = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
        self.torch_dtype = dt
        self._keep = []

        def dev(t):
            assert t.is_cuda and t.dtype == dt and t.is_contiguous(), "bad weight tensor"
            self._keep.append(t)
            return t.data_ptr()

        cfg = Config(n_layers=shape.n_layers, hidden=shape.hidden,
                     n_q_heads=shape.n_q_heads, n_kv_heads=shape.n_kv_heads,
                     head_dim=shape.head_dim, ffn=shape.ffn, vocab=shape.vocab,
                     window=window, page_block=shape.page_block, max_batch=max_batch,
                     max_pages_per_seq=max_pages_per_seq,
                     dtype=BF16 if shape.dtype == "bf16" else FP32,
                     qk_norm=int(shape.qk_norm), mask_id=shape.mask_id,
                     rope_theta=shape.rope_theta, rms_eps=shape.rms_eps)
        arrays = {}
        for f in _LAYER_FIELDS:
            arr = (c_void_p * shape.n_layers)()
            for l, lw in enumerate(weights["layers"]):
                t = lw.get(f)
                arr[l] = dev(t) if t is not None else None
            arrays[f] = arr
        self._arrays = arrays
        w = Weights(embed=dev(weights["embed"]), final_norm=dev(weights["final_norm"]),
                    lm_head=dev(weights["lm_head"]),
                    **{f: ctypes.cast(arrays[f], POINTER(c_void_p)) for f in _LAYER_FIELDS})
        self._cfg = cfg
        h = c_void_p()
        rc = self._lib.wedlm_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))
        if rc != OK:
            raise WedlmError(rc, "wedlm_create failed (unsupported shape or CUDA error)")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            self._lib.wedlm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc):
        if rc != OK:
            raise WedlmError(rc, self._lib.wedlm_last_error(self._h).decode())

    # -- control -----------------------------------------------------------
    def status(self):
        word = c_int32(0)
        rc = self._lib.wedlm_get_status(self._h, ctypes.byref(word))
        if rc not in (OK, ERR_DEVICE):
            self._check(rc)
        return word.value

    def set_graphs(self, enable):
        self._check(self._lib.wedlm_set_graphs(self._h, int(enable)))

    def set_timing(self, enable):
        self._check(self._lib.wedlm_set_timing(self._h, int(enable)))

    def timings(self):
        ms = (c_float * len(KINDS))()
        n = (c_int32 * len(KINDS))()
        self._check(self._lib.wedlm_get_timings(self._h, ms, n, len(KINDS)))
        return {k: (ms[i], n[i]) for i, k in enumerate(KINDS)}

    def launches_per_step(self, batch):
        return self._lib.wedlm_launches_per_step(self._h, batch)

    # -- the step ------------------------------------------------------------
    def make_outputs(self, batch, rows=False, logits=False, perm=False, hidden=False,
                     device="cuda", packed=False):
        """Output tensors of a step.  packed=True places the window and commit
        results in one byte buffer (out["packed"], the layout of
        step_result_views), so that a caller reads them back with one copy."""
        import torch
        W = self.window
        if packed:
            buf = torch.empty(step_result_bytes(batch, W), dtype=torch.uint8, device=device)
            out = step_result_views(buf, batch, W)
            out["packed"] = buf
            out["filled"] = torch.empty(batch, W, dtype=torch.uint8, device=device)
        else:
            out = {
                "new_tokens": torch.empty(batch, W, dtype=torch.int32, device=device),
                "new_pos": torch.empty(batch, W, dtype=torch.int32, device=device),
                "new_observed": torch.empty(batch, W, dtype=torch.uint8, device=device),
                "committed": torch.empty(batch, W, dtype=torch.int32, device=device),
                "n_committed": torch.empty(batch, dtype=torch.int32, device=device),
                "filled": torch.empty(batch, W, dtype=torch.uint8, device=device),
            }
        if perm:
            out["perm"] = torch.empty(batch, W, dtype=torch.int32, device=device)
        if rows:
            out["rows"] = torch.empty(batch * W, 4, dtype=torch.int32, device=device)
        if logits:
            out["logits"] = torch.empty(batch * W, self.shape.vocab, dtype=torch.float32,
                                        device=device)
        if hidden:
            out["hidden"] = torch.empty(batch * W, self.shape.hidden,
                                        dtype=self.torch_dtype, device=device)
        return out

    def step(self, tokens, pos, observed, seq_len, page_table, pools, num_pages,
             alpha, tau, out, plant_token=None, plant_bias=0.0, stream=None,
             score_mode=SCORE_ENTROPY):
        """Enqueue one window decode step.  All tensors are CUDA tensors:
        tokens/pos int32 [B][W], observed uint8 [B][W], seq_len int32 [B]
        (updated in place), page_table int32 [B][max_pages_per_seq], pools a
        list of per-layer pool tensors; `out` from make_outputs()."""
        B = tokens.shape[0]
        pool_arr = (c_void_p * len(pools))(*[p.data_ptr() for p in pools])
        sin = StepIn(batch=B, num_pages=num_pages, tokens=tokens.data_ptr(),
                     pos=pos.data_ptr(), observed=observed.data_ptr(),
                     seq_len=seq_len.data_ptr(), page_table=page_table.data_ptr(),
                     kv_pools=ctypes.cast(pool_arr, POINTER(c_void_p)),
                     plant_token=None if plant_token is None else plant_token.data_ptr(),
                     plant_bias=plant_bias, alpha=alpha, tau=tau, score_mode=score_mode)
        sout = StepOut(**{k: (out[k].data_ptr() if k in out else None)
                          for k, _ in StepOut._fields_})
        self._check(self._lib.wedlm_step(self._h, ctypes.byref(sin), ctypes.byref(sout),
                                         _stream_handle(stream)))
        return out

    def prefill(self, tokens, seq_len, page_table, pools, num_pages, hidden=None, stream=None):
        """Enqueue a prompt prefill: tokens int32 [B][chunk] at positions
        seq_len[b].. (seq_len advanced in place); K/V of every layer to the
        pages.  hidden: optional [B*chunk][hidden] output."""
        B, C = tokens.shape
        pool_arr = (c_void_p * len(pools))(*[p.data_ptr() for p in pools])
        self._check(self._lib.wedlm_prefill(
            self._h, B, C, _ptr(tokens), _ptr(seq_len), _ptr(page_table), num_pages,
            ctypes.cast(pool_arr, POINTER(c_void_p)), _ptr(hidden), _stream_handle(stream)))

    def generate(self, tokens, pos, observed, seq_len, page_table, pools, num_pages, alpha,
                 tau, max_steps, done, stop_len=None, stop_token=-1, out_tokens=None,
                 out_base=None, plant_token=None, plant_bias=0.0, score_mode=SCORE_ENTROPY,
                 steps_run=None, stream=None):
        """Enqueue the streaming loop on the device (up to max_steps steps,
        window tensors updated in place; see wedlm_generate)."""
        B = tokens.shape[0]
        pool_arr = (c_void_p * len(pools))(*[p.data_ptr() for p in pools])
        gin = GenIn(batch=B, num_pages=num_pages, tokens=tokens.data_ptr(), pos=pos.data_ptr(),
                    observed=observed.data_ptr(), seq_len=seq_len.data_ptr(),
                    page_table=page_table.data_ptr(),
                    kv_pools=ctypes.cast(pool_arr, POINTER(c_void_p)),
                    plant_token=None if plant_token is None else plant_token.data_ptr(),
                    plant_bias=plant_bias, alpha=alpha, tau=tau, score_mode=score_mode,
                    max_steps=max_steps, done=done.data_ptr(),
                    stop_len=None if stop_len is None else stop_len.data_ptr(),
                    stop_token=stop_token,
                    out_tokens=None if out_tokens is None else out_tokens.data_ptr(),
                    out_base=None if out_base is None else out_base.data_ptr(),
                    out_cap=0 if out_tokens is None else out_tokens.shape[1],
                    steps_run=None if steps_run is None else steps_run.data_ptr())
        self._check(self._lib.wedlm_generate(self._h, ctypes.byref(gin), _stream_handle(stream)))

    # -- single rows of the step --------------------------------------------
    def reorder_embed(self, tokens, pos, observed, perm, inv, x_out, pos_phys, stream=None):
        self._check(self._lib.wedlm_reorder_embed(
            self._h, tokens.shape[0], _ptr(tokens), _ptr(pos), _ptr(observed), _ptr(perm),
            _ptr(inv), _ptr(x_out), _ptr(pos_phys), _stream_handle(stream)))

    def layer(self, layer, x, pos_phys, seq_len, page_table, num_pages, pool,
              kv_win_out=None, q_out=None, attn_out=None, stream=None):
        B = seq_len.shape[0]
        self._check(self._lib.wedlm_layer(
            self._h, layer, B, _ptr(x), _ptr(pos_phys), _ptr(seq_len), _ptr(page_table),
            num_pages, _ptr(pool), _ptr(kv_win_out), _ptr(q_out), _ptr(attn_out),
            _stream_handle(stream)))

    def attention(self, q, pool, page_table, seq_len, num_pages, kv_win, o, stream=None):
        self._check(self._lib.wedlm_attention(
            self._h, seq_len.shape[0], _ptr(q), _ptr(pool), _ptr(page_table),
            _ptr(seq_len), num_pages, _ptr(kv_win), _ptr(o), _stream_handle(stream)))

    def dual_stream_attention(self, n, block, q, mem_pool, win, o, stream=None):
        """Dual-Stream Masking attention (see wedlm_dual_stream_attention)."""
        self._check(self._lib.wedlm_dual_stream_attention(
            self._h, n, block, _ptr(q), _ptr(mem_pool), _ptr(win), _ptr(o),
            _stream_handle(stream)))

    def lm_head(self, batch, x, rows_out, plant_token=None, plant_bias=0.0, logits=None,
                stream=None):
        self._check(self._lib.wedlm_lm_head(
            self._h, batch, _ptr(x), _ptr(plant_token), plant_bias, _ptr(rows_out),
            _ptr(logits), _stream_handle(stream)))


def _aligned(n, a=256):
    return (n + a - 1) // a * a


def step_result_bytes(batch, W):
    """Bytes of the packed step results: int32 new_tokens, new_pos and
    committed [B][W], int32 n_committed [B], uint8 new_observed [B][W], each
    starting on a 256-byte boundary."""
    n = batch * W
    return 3 * _aligned(4 * n) + _aligned(4 * batch) + _aligned(n)


def step_result_views(buf, batch, W):
    """Views of a packed step-result byte buffer (device or host) by name."""
    import torch
    n = batch * W
    o, views = 0, {}
    for name, nbytes, dt, shape in (("new_tokens", 4 * n, torch.int32, (batch, W)),
                                    ("new_pos", 4 * n, torch.int32, (batch, W)),
                                    ("committed", 4 * n, torch.int32, (batch, W)),
                                    ("n_committed", 4 * batch, torch.int32, (batch,)),
                                    ("new_observed", n, torch.uint8, (batch, W))):
        views[name] = buf[o:o + nbytes].view(dt).view(*shape)
        o += _aligned(nbytes)
    return views


def attention_static(window, n_q_heads, n_kv_heads, max_pages_per_seq, num_pages, q, kv_pool,
                     page_table, seq_len, kv_win, o, stream=None):
    """wedlm_attention_static: the window attention with no device
    allocation at all (scratch in the library's static device array).
    Raises WedlmError on a non-zero return code."""
    rc = lib().wedlm_attention_static(
        seq_len.shape[0], window, n_q_heads, n_kv_heads, max_pages_per_seq, num_pages,
        _ptr(q), _ptr(kv_pool), _ptr(page_table), _ptr(seq_len), _ptr(kv_win), _ptr(o),
        _stream_handle(stream))
    if rc != OK:
        raise WedlmError(rc, "wedlm_attention_static failed")


def selftest_bounded_wait(word, stream=None):
    """wedlm_selftest_bounded_wait: a kernel waits on a barrier nothing
    completes until its bounded wait gives up (about 2 s).  word: device
    int32 tensor of 2.  Returns (device error bits, 1 if the wait gave up)."""
    err, gave = c_int32(0), c_int32(0)
    rc = lib().wedlm_selftest_bounded_wait(_ptr(word), ctypes.byref(err), ctypes.byref(gave),
                                           _stream_handle(stream))
    if rc != OK:
        raise WedlmError(rc, "wedlm_selftest_bounded_wait failed")
    return int(err.value), int(gave.value)


def attention_static_status(stream=None):
    """wedlm_attention_static_status: the WEDLM_DEV_* bits the last
    attention_static call on the current device set (waits for the stream)."""
    word = c_int32(0)
    rc = lib().wedlm_attention_static_status(_stream_handle(stream), ctypes.byref(word))
    if rc != OK:
        raise WedlmError(rc, "wedlm_attention_static_status failed")
    return int(word.value)


def rows_to_numpy(rows_tensor):
    """[N][4] int32 view of wedlm_slot_rec -> (argmax, entropy, p_max, lse)."""
    import numpy as np
    a = rows_tensor.cpu().numpy()
    f = a.view(np.float32)
    return a[:, 0].copy(), f[:, 1].copy(), f[:, 2].copy(), f[:, 3].copy()
