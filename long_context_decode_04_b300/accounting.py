"""Byte and FLOP accounting for the roofline figures.

Algorithmic bytes are what the computation must move at least once: the
attended K and V rows for decode; Q, K, V, O and lse for prefill.  FLOPs
count one multiply-add as two operations.
"""
from __future__ import annotations


def kv_cache_bytes(seq_len: int, head_dim: int, heads: int = 1, layers: int = 1,
                   bytes_per_elem: int = 2) -> int:
    """Bytes of a K plus V cache: 2 tensors x seq_len x head_dim x elem size x heads x layers.

    ThriftAttention page (hyperion-consulting.io), section on the long-context
    crisis, sizes an FP16 cache this way (131072 x 128 -> 67 MB per head).
    """
    return 2 * seq_len * head_dim * bytes_per_elem * heads * layers


def decode_kv_bytes(B: int, Hkv: int, D: int, lengths, bytes_per_elem: int) -> int:
    """KV bytes one decode call must read: every attended key row of every KV head, once.

    ``lengths`` is an int (all sequences) or a sequence of B per-sequence lengths.
    """
    total_len = lengths * B if isinstance(lengths, int) else int(sum(int(x) for x in lengths))
    return 2 * Hkv * D * bytes_per_elem * total_len


def decode_flops(B: int, Hq: int, D: int, lengths) -> int:
    """2 FLOP per multiply-add for q.k and for p.v: 4*D per (query head, attended key)."""
    total_len = lengths * B if isinstance(lengths, int) else int(sum(int(x) for x in lengths))
    return 4 * Hq * D * total_len


def partial_bytes(B: int, Hq: int, n_split: int, D: int) -> int:
    """fp32 (m, l, o[D]) partials written by split-KV decode and read back by the combine."""
    return 2 * 4 * B * Hq * n_split * (D + 2)


def prefill_causal_flops(B: int, H: int, S: int, D: int) -> int:
    """Causal QK^T plus PV: 4*D FLOP per (query i, key j <= i) pair."""
    return 4 * B * H * D * (S * (S + 1) // 2)


def prefill_bytes(B: int, H: int, Hkv: int, S: int, D: int, bytes_per_elem: int = 2) -> int:
    """Q, K, V read once, O written once (all bf16) and lse written (fp32)."""
    return bytes_per_elem * D * S * B * (2 * H + 2 * Hkv) + 4 * B * H * S
