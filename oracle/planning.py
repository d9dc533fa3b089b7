"""The pages' bookkeeping formulas, restated plainly -- TEST INFRASTRUCTURE ONLY.

These pin the library's host planner (work decomposition, folding, workspace
sizing) against the worked examples the pages print.  Each function follows
one passage and nothing else; none of it is imported by the CUDA library.
"""
from __future__ import annotations

import math


def task_mapping(task: int, num_kv_heads: int, group: int):
    """task -> (batch, kv_head, q_head_begin).

    "Writing Page Attention with PyPTO", section 1.3: one task is one batch row
    plus one KV head plus its group of query heads; batch = task // Hkv,
    kv_head = task % Hkv, q_head_begin = kv_head * G.
    """
    return task // num_kv_heads, task % num_kv_heads, (task % num_kv_heads) * group


def page_count(seq_len: int, page_size: int) -> int:
    """Pages a sequence covers: ceil(n / page_size) (PyPTO section 5.1)."""
    return -(-seq_len // page_size)


def stack_count(seq_len: int, stack_tokens: int = 512) -> int:
    """Pipeline stacks of 4 pages x 128 tokens: ceil(n / 512) (PyPTO section 5.1)."""
    return -(-seq_len // stack_tokens)


def last_stack_tokens(seq_len: int, stack_tokens: int = 512) -> int:
    """Valid tokens in the final stack (PyPTO section 1.4: n = 700 leaves 188)."""
    c = stack_count(seq_len, stack_tokens)
    return seq_len - (c - 1) * stack_tokens if c else 0


def grid_stride_tasks(core: int, num_tasks: int, num_cores: int) -> list:
    """Tasks a core processes in order: core, core + cores, ... (PyPTO section 3.3)."""
    return list(range(core, num_tasks, num_cores))


def fold_factor(num_heads: int, q_len: int, max_rows: int = 128) -> int:
    """Largest F with q_len % F == 0 and num_heads * F <= max_rows.

    "TokenSpeed-MLA 2.0.1", decode section on grouping q_seqlen and num_heads
    into BMM1 M: without such a factor above one the kernel does not fold.
    """
    best = 1
    for f in range(1, q_len + 1):
        if q_len % f == 0 and num_heads * f <= max_rows:
            best = f
    return best


def packed_q_tiles(num_heads: int, q_len: int, rows: int = 128) -> int:
    """Query tiles when rows are packed as query_token * H + head: ceil(H * q_len / 128)."""
    return -(-(num_heads * q_len) // rows)


def split_workspace_bytes(batch: int, num_heads: int, q_len: int, split_kv: int,
                          head_dim_v: int = 512) -> int:
    """Split-KV workspace: B * 128 * ceil(H*q_len/128) * split_kv * (Dv + 1) * 4 bytes.

    "TokenSpeed-MLA 2.0.1", packed-query paragraph: one FP32 partial output row
    of Dv values plus one LSE value per row per split (513 floats at D512), and
    zero bytes when split_kv is one.
    """
    if split_kv <= 1:
        return 0
    return batch * 128 * packed_q_tiles(num_heads, q_len) * split_kv * (head_dim_v + 1) * 4


def static_anchor_tau(num_keys: int, v_max: float = 2.0 ** 12, delta: float = 2.0,
                      fp32_log_max: float = 88.7) -> float:
    """tau = 88.7 - ln N - ln Vmax - delta ("Flywheel Attention", appendix A)."""
    return fp32_log_max - math.log(num_keys) - math.log(v_max) - delta


def rescale_fifo_schedule(num_stacks: int):
    """Which rescale factor each delayed PV collection uses.

    "Writing Page Attention with PyPTO", sections 8.1 and 8.4: ticks run over
    [0, num_stacks + 2); tick t first collects stack t - 2 (for t >= 2) using
    pending0, then the softmax of stack t (for t < num_stacks) pushes r_t, so
    the pair moves (1, 1) -> (1, r0) -> (r0, r1) -> ...  The pair shifts on
    every tick (a tick with no softmax pushes 1).  Returns a list of
    (tick, collected_stack, factor) with factor a label "r<i>" or "1".
    """
    pending = ["1", "1"]
    out = []
    for tick in range(num_stacks + 2):
        if tick >= 2:
            out.append((tick, tick - 2, pending[0]))
        pending = [pending[1], f"r{tick}" if tick < num_stacks else "1"]
    return out
