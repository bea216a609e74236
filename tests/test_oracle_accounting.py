"""Pins of the oracle's accounting formulas to values the pages print.

Every expected number here is read from a golden fixture that cites its
page, or is a closed form of the mathematics; none is computed by the code
under test.
"""
import json
import os
from fractions import Fraction

import pytest

from oracle import accounting as acc


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_bytes_per_token_budget_page(golden_dir):
    g = _load(golden_dir, "kv_bytes.json")["budget_page"]
    per_token = acc.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"],
                                       g["bytes_per_scalar"])
    assert per_token == g["bytes_per_token"] == 128 * 1024
    request = acc.kv_bytes(g["layers"], g["kv_heads"], g["head_dim"], g["bytes_per_scalar"],
                           [g["request_tokens"]])
    assert request == g["request_gib"] * 2**30
    alt = acc.kv_bytes(g["layers"], g["alt_kv_heads"], g["head_dim"], g["bytes_per_scalar"],
                       [g["request_tokens"]])
    assert alt == g["alt_request_gib"] * 2**30


def test_bytes_per_token_opt13b(golden_dir):
    g = _load(golden_dir, "kv_bytes.json")["opt13b"]
    two, hidden, layers, b = g["factors"]
    # hidden 5120 = 40 heads x head dim 128 for every layer.
    per_token = acc.kv_bytes_per_token(layers, 40, hidden // 40, b)
    assert two == 2 and per_token == 2 * hidden * layers * b
    assert per_token == g["bytes_per_token_kib"] * 1024
    request = acc.kv_bytes(layers, 40, hidden // 40, b, [g["request_tokens"]])
    assert round(request / 2**30, 1) == g["request_gb_one_decimal"]


def test_witness_bytes_per_token(golden_dir):
    w = _load(golden_dir, "witness.json")
    assert acc.kv_bytes_per_token(32, 8, 128, 2) == w["bytes_per_token"]


def test_worked_example_positions_and_utilisation(golden_dir):
    g = _load(golden_dir, "worked_example.json")
    lengths = g["lengths"]
    assert sum(lengths) == g["useful_positions"]
    assert g["fixed_reservation"] * len(lengths) == g["fixed_reservation_positions"]
    for bs, positions in g["paged_positions"].items():
        assert sum(acc.allocated_slots(n, int(bs)) for n in lengths) == positions
        u = acc.utilisation(lengths, int(bs))
        assert round(float(u) * 100, 2) == g["utilisation_percent_rounded"][bs]
    u_fixed = acc.reservation_utilisation(lengths, g["fixed_reservation"])
    assert round(float(u_fixed) * 100, 2) == g["utilisation_percent_rounded"]["fixed_512"]


def test_block_counts_from_the_ceiling_definition():
    # ceil(n/B) blocks; the final block wastes at most B - 1 positions
    # (PagedAttention and Online Inference, section 2).
    assert [acc.blocks_needed(n, 16) for n in (37, 91, 128, 201, 511)] == [3, 6, 8, 13, 32]
    assert [acc.blocks_needed(n, 32) for n in (37, 91, 128, 201, 511)] == [2, 3, 4, 7, 16]
    assert [acc.tail_waste(n, 16) for n in (37, 91, 128, 201, 511)] == [11, 5, 0, 7, 1]
    assert [acc.tail_waste(n, 32) for n in (37, 91, 128, 201, 511)] == [27, 5, 0, 23, 1]
    assert acc.blocks_needed(0, 16) == 0
    for bs in (1, 2, 3, 16, 32):
        for n in range(1, 200):
            assert 0 <= acc.tail_waste(n, bs) <= bs - 1
            assert (acc.blocks_needed(n, bs) - 1) * bs < n <= acc.blocks_needed(n, bs) * bs


def test_tail_bound(golden_dir):
    _load(golden_dir, "tail_waste.json")
    lengths = [37, 91, 128, 201, 511]
    for bs in (4, 16, 32, 64):
        assert acc.total_tail_waste(lengths, bs) <= len(lengths) * (bs - 1)
    # equality when every request wastes B - 1 (length 1 mod B)
    assert acc.total_tail_waste([17, 33, 1], 16) == 3 * 15


def test_mean_tail_waste_closed_form(golden_dir):
    g = _load(golden_dir, "tail_waste.json")
    m = g["max_len"]
    for bs in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512):
        assert acc.mean_tail_waste(bs, m) == Fraction(bs - 1, 2)
    assert acc.mean_reservation_waste(512, m) == Fraction(g["fixed_512_mean_waste"])
    # a page size that does not divide 512 breaks the closed form (constructed check)
    assert acc.mean_tail_waste(3, m) != Fraction(2, 2)


def test_invalid_arguments():
    with pytest.raises(ValueError):
        acc.blocks_needed(-1, 16)
    with pytest.raises(ValueError):
        acc.reservation_waste(600, 512)
