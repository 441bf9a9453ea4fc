"""Host-side sizing rules: the dense baseline's logits budget and the byte and
flop models used for roofline reporting.

Dense chunking follows vLLM pull request #60618, section "Motivation: what
materializing the scores costs": the dense path writes fp32 logits for every
(row, key) pair, the default budget is 512 MiB, so one logits call covers
2**27 / keys rows (point 1 of that section) and a 16,384-row chunk needs
ceil(rows / rows_per_call) call pairs.
"""
from __future__ import annotations

FLOP_PER_PAIR = 2 * 32 * 128  # one multiply-add per head and dimension (32 heads)


def flop_per_pair(heads: int = 32) -> int:
    """Tensor FLOPs per scored (row, key) pair: one multiply-add per head and
    dimension (head_dim 128)."""
    return 2 * heads * 128
LOGIT_BYTES = 4


def dense_logits_bytes(rows: int, keys: int) -> int:
    return rows * keys * LOGIT_BYTES


def dense_logits_traffic_bytes(rows: int, keys: int) -> int:
    """Write once, read once."""
    return 2 * dense_logits_bytes(rows, keys)


def dense_rows_per_call(keys: int, budget_bytes: int) -> int:
    return max(1, budget_bytes // (keys * LOGIT_BYTES))


def dense_calls(rows: int, keys: int, budget_bytes: int) -> int:
    per = dense_rows_per_call(keys, budget_bytes)
    return -(-rows // per)


def algorithmic_bytes(rows: int, keys: int, topk: int, heads: int = 32, dim: int = 128) -> int:
    """Bytes the fused op must move at least once: q, k (read once), key
    scales, weights, starts/ends and the int32 output."""
    return rows * heads * dim + keys * dim + keys * 4 + rows * heads * 4 + rows * 8 + rows * topk * 4
