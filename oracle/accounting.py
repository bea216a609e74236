"""The pages' KV byte and block accounting, written from their definitions.

Test infrastructure (part of the oracle package); see ``oracle/__init__``.

* Eq. (1) of "Serving Language Models Within a Memory Budget" and of
  "PagedAttention and Online Inference": uncompressed KV bytes are
  2 * L * H_kv * d * b per retained token, times the retained tokens.
* Eq. (2) of "PagedAttention and Online Inference": a sequence of length n
  in blocks of B slots is allocated A_B(n) = B * ceil(n / B) slots, of which
  W_B(n) = A_B(n) - n are tail waste; with a fixed reservation of M slots the
  waste is M - n.  Eq. (2) of the budget page bounds the total tail waste of
  N nonempty requests by N (B - 1).
* Eq. (3) of the budget page: for lengths uniform on 1..M with B dividing M,
  the mean tail waste is (B - 1) / 2.  ``mean_tail_waste`` computes the mean
  by enumeration, so the closed form is a check, not an input.
* Eq. (3) of "PagedAttention and Online Inference": position utilisation
  U = sum_i n_i / sum_i B ceil(n_i / B).
"""
from __future__ import annotations

from fractions import Fraction
from typing import Iterable, Sequence


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_scalar: int) -> int:
    """2 * L * H_kv * d * b: keys and values of one retained token."""
    return 2 * layers * kv_heads * head_dim * bytes_per_scalar


def kv_bytes(layers: int, kv_heads: int, head_dim: int, bytes_per_scalar: int,
             lengths: Iterable[int]) -> int:
    """Eq. (1): per-token bytes times the sum of retained lengths."""
    return kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_scalar) * sum(lengths)


def blocks_needed(n: int, block_size: int) -> int:
    """ceil(n / B) blocks hold n tokens (0 for an empty sequence)."""
    if n < 0 or block_size <= 0:
        raise ValueError("n must be >= 0 and block_size > 0")
    return -(-n // block_size)


def allocated_slots(n: int, block_size: int) -> int:
    """A_B(n) = B * ceil(n / B)."""
    return block_size * blocks_needed(n, block_size)


def tail_waste(n: int, block_size: int) -> int:
    """W_B(n) = A_B(n) - n, between 0 and B - 1 for n >= 1."""
    return allocated_slots(n, block_size) - n


def reservation_waste(n: int, reserved: int) -> int:
    """Waste of a fixed reservation of M slots: M - n."""
    if n > reserved:
        raise ValueError("request longer than its reservation")
    return reserved - n


def total_tail_waste(lengths: Sequence[int], block_size: int) -> int:
    return sum(tail_waste(n, block_size) for n in lengths)


def utilisation(lengths: Sequence[int], block_size: int) -> Fraction:
    """U = sum n_i / sum B ceil(n_i / B), exact."""
    return Fraction(sum(lengths), sum(allocated_slots(n, block_size) for n in lengths))


def reservation_utilisation(lengths: Sequence[int], reserved: int) -> Fraction:
    """Useful positions over a fixed reservation of ``reserved`` slots each."""
    return Fraction(sum(lengths), reserved * len(lengths))


def mean_tail_waste(block_size: int, max_len: int) -> Fraction:
    """Mean of W_B(n) over n uniform on 1..max_len, by enumeration."""
    return Fraction(sum(tail_waste(n, block_size) for n in range(1, max_len + 1)), max_len)


def mean_reservation_waste(reserved: int, max_len: int) -> Fraction:
    """Mean of M - n over n uniform on 1..max_len, by enumeration."""
    return Fraction(sum(reservation_waste(n, reserved) for n in range(1, max_len + 1)), max_len)
