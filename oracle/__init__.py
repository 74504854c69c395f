"""CPU oracle for the WeDLM window decode step (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  It shares no code with the CUDA path.
"""
from .wedlm_oracle import *  # noqa: F401,F403
from .wedlm_oracle import (bf16_round, storer, rmsnorm, rope_cos_sin,  # noqa
                           rope_apply, silu, topological_reorder,
                           page_elem_offset, pool_view, pool_gather,
                           pool_scatter, window_attention, qkv_project,
                           layer_forward, lm_head_logits, softmax_scores,
                           select_eq11, commit_run, refill, forward_window,
                           oracle_step_seq, oracle_step, oracle_prefill,
                           SlotScores, SeqStep)
