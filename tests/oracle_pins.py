"""Pins of the attention / cache-op oracle to facts outside the oracle.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
a value fixed by the pages or by the mathematics.  ``test_oracle_pins.py``
runs them; ``test_oracle_mutations.py`` runs them against deliberately
broken copies of the oracle to show that every planted mistake fails one.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
from scipy.special import softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
DT = {"float16": torch.float16, "bfloat16": torch.bfloat16}


def to_bits(values, dtype):
    """float values -> 16-bit patterns of the storage dtype (torch rounding)."""
    t = torch.as_tensor(np.asarray(values, dtype=np.float32)).to(DT[dtype])
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def widen(bits, dtype):
    """16-bit patterns -> float64 through torch (a library conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(DT[dtype])
    return t.to(torch.float64).numpy()


def build_pool(tokens_k, tokens_v, tables, block_size, num_blocks, dtype, fill=0.0):
    """Place per-sequence token rows [n][H][d] into pools through block tables.

    Written as explicit loops over (sequence, token): logical token t sits in
    physical block tables[s][t // B], slot t % B.
    """
    H, d = tokens_k[0].shape[1], tokens_k[0].shape[2]
    kc = np.full((num_blocks, H, block_size, d), fill, dtype=np.float32)
    vc = np.full_like(kc, fill)
    for s, (ks, vs) in enumerate(zip(tokens_k, tokens_v)):
        for t in range(ks.shape[0]):
            b = tables[s][t // block_size]
            kc[b, :, t % block_size, :] = ks[t]
            vc[b, :, t % block_size, :] = vs[t]
    max_blocks = max(len(t) for t in tables)
    bt = np.zeros((len(tables), max_blocks), dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = t
    return to_bits(kc, dtype), to_bits(vc, dtype), bt


def random_case(rng, lengths, H_q, H_kv, d, block_size, dtype, spare=3):
    """Random tokens for each sequence, blocks scattered over a shuffled pool."""
    need = [max(1, -(-n // block_size)) for n in lengths]
    nb = sum(need) + spare
    perm = rng.permutation(nb)
    tables, pos = [], 0
    for k in need:
        tables.append([int(b) for b in perm[pos:pos + k]])
        pos += k
    ks = [rng.standard_normal((n, H_kv, d)).astype(np.float32) for n in lengths]
    vs = [rng.standard_normal((n, H_kv, d)).astype(np.float32) for n in lengths]
    kc, vc, bt = build_pool(ks, vs, tables, block_size, nb, dtype,
                            fill=float(rng.standard_normal()))
    q = to_bits(rng.standard_normal((len(lengths), H_q, d)), dtype)
    return q, kc, vc, bt, np.asarray(lengths, dtype=np.int32), tables


# ---------------------------------------------------------------------------
# fp16 / bf16 widening
# ---------------------------------------------------------------------------
def pin_f16_widening_all_patterns():
    patterns = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = patterns.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in patterns])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got)), "binary16 widening differs from numpy"
    assert np.all(np.signbit(ref[~both_nan]) == np.signbit(got[~both_nan]))


def pin_bf16_widening_all_patterns():
    patterns = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = widen(patterns, "bfloat16")
    got = np.array([oracle.bf16_to_f64(int(b)) for b in patterns])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got)), "bfloat16 widening differs from torch"


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------
def pin_hand_example():
    """d = 2, scale = ln 2, two query heads sharing one KV head (GQA g = 2).

    Keys (1,0), (0,0), (2,0); values (7,0), (0,7), (-7,14).
    Head 0, q = (1,0): scores ln2 * (1, 0, 2), exp -> (2, 1, 4), weights
    (2, 1, 4) / 7, output (14 - 28, 7 + 56) / 7 = (-2, 9).
    Head 1, q = (0,0): equal weights, output = mean of values = (0, 7).
    The three tokens sit in blocks of 2 at physical blocks 5 and 2.
    """
    for dtype in ("float16", "bfloat16"):
        ks = [np.array([[[1, 0]], [[0, 0]], [[2, 0]]], dtype=np.float32)]
        vs = [np.array([[[7, 0]], [[0, 7]], [[-7, 14]]], dtype=np.float32)]
        kc, vc, bt = build_pool(ks, vs, [[5, 2]], 2, 6, dtype, fill=99.0)
        q = to_bits([[[1, 0], [0, 0]]], dtype)
        out = oracle.attention(q, kc, vc, bt, [3], math.log(2.0), dtype)
        assert np.allclose(out[0, 0], [-2.0, 9.0], rtol=0, atol=1e-13), out
        assert np.allclose(out[0, 1], [0.0, 7.0], rtol=0, atol=1e-13), out


def pin_single_token_is_value_row():
    rng = np.random.default_rng(1)
    for dtype in ("float16", "bfloat16"):
        q, kc, vc, bt, lens, tables = random_case(rng, [1, 1, 1], 4, 2, 16, 4, dtype)
        out = oracle.attention(q, kc, vc, bt, lens, 0.25, dtype)
        for s in range(3):
            b = tables[s][0]
            for i in range(4):
                expect = widen(vc[b, i // 2, 0], dtype)
                assert np.array_equal(out[s, i], expect), "n = 1 must return V_0 exactly"


def pin_zero_query_is_mean_of_values():
    rng = np.random.default_rng(2)
    lengths = [5, 17, 33]
    q, kc, vc, bt, lens, tables = random_case(rng, lengths, 2, 1, 8, 4, "bfloat16")
    q = np.zeros_like(q)
    out = oracle.attention(q, kc, vc, bt, lens, 0.3, "bfloat16")
    for s, n in enumerate(lengths):
        rows = np.stack([widen(vc[tables[s][t // 4], 0, t % 4], "bfloat16") for t in range(n)])
        assert np.allclose(out[s, 0], rows.mean(axis=0), rtol=1e-13, atol=1e-14)


def pin_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    n, d = 11, 8
    key = rng.standard_normal(d).astype(np.float32)
    ks = [np.tile(key, (n, 1, 1))]
    vs = [rng.standard_normal((n, 1, d)).astype(np.float32)]
    kc, vc, bt = build_pool(ks, vs, [[3, 0, 2]], 4, 4, "float16")
    q = to_bits(rng.standard_normal((1, 1, d)), "float16")
    out = oracle.attention(q, kc, vc, bt, [n], 1.0, "float16")
    mean = widen(to_bits(vs[0][:, 0], "float16"), "float16").mean(axis=0)
    assert np.allclose(out[0, 0], mean, rtol=1e-13, atol=1e-14)


def pin_extreme_logits_are_one_hot():
    """Scores up to +-1.0e4 must neither overflow nor lose the argmax."""
    n, d = 9, 16
    for dtype in ("float16", "bfloat16"):
        ks = np.zeros((n, 1, d), dtype=np.float32)
        ks[:, 0, 0] = [-40, 0, 3, -40, 0, 40, 1, -40, 2]  # token 5 dominates
        vs = np.arange(n * d, dtype=np.float32).reshape(n, 1, d) / 7.0
        kc, vc, bt = build_pool([ks], [vs], [[2, 0, 1]], 4, 3, dtype)
        qv = np.zeros((1, 1, d), dtype=np.float32)
        qv[0, 0, 0] = 256.0  # score of token 5: 256 * 40 = 10240
        out = oracle.attention(to_bits(qv, dtype), kc, vc, bt, [n], 1.0, dtype)
        assert np.all(np.isfinite(out))
        expect = widen(vc[bt[0, 5 // 4], 0, 5 % 4], dtype)  # token 5: block 0, slot 1
        assert np.array_equal(out[0, 0], expect)
        # negated query: the three keys of -40 tie at +10240 and share the weight
        qv[0, 0, 0] = -256.0
        out = oracle.attention(to_bits(qv, dtype), kc, vc, bt, [n], 1.0, dtype)
        assert np.all(np.isfinite(out))
        rows = [t for t in range(n) if ks[t, 0, 0] == -40]
        mean = np.mean([widen(vc[bt[0, t // 4], 0, t % 4], dtype) for t in rows], axis=0)
        assert len(rows) == 3 and np.allclose(out[0, 0], mean, rtol=1e-13, atol=1e-13)


def pin_gqa_equals_replicated_mha():
    rng = np.random.default_rng(4)
    lengths = [7, 20, 1]
    H_q, H_kv, d, B = 8, 2, 16, 4
    q, kc, vc, bt, lens, _ = random_case(rng, lengths, H_q, H_kv, d, B, "bfloat16")
    gqa = oracle.attention(q, kc, vc, bt, lens, 0.2, "bfloat16")
    kc_rep = np.repeat(kc, H_q // H_kv, axis=1).copy()
    vc_rep = np.repeat(vc, H_q // H_kv, axis=1).copy()
    mha = oracle.attention(q, kc_rep, vc_rep, bt, lens, 0.2, "bfloat16")
    assert np.array_equal(gqa, mha), "GQA must equal MHA over replicated KV heads"
    # MQA: one KV head serves every query head
    q1, kc1, vc1, bt1, lens1, _ = random_case(rng, lengths, 4, 1, d, B, "float16")
    mqa = oracle.attention(q1, kc1, vc1, bt1, lens1, 0.2, "float16")
    mha1 = oracle.attention(q1, np.repeat(kc1, 4, axis=1).copy(), np.repeat(vc1, 4, axis=1).copy(),
                            bt1, lens1, 0.2, "float16")
    assert np.array_equal(mqa, mha1)


def pin_paging_invariance():
    """Any physical placement of the same logical blocks gives the same output."""
    rng = np.random.default_rng(5)
    lengths = [13, 40, 4]
    H, d, B = 2, 8, 4
    ks = [rng.standard_normal((n, H, d)).astype(np.float32) for n in lengths]
    vs = [rng.standard_normal((n, H, d)).astype(np.float32) for n in lengths]
    need = [-(-n // B) for n in lengths]
    nb = sum(need) + 2
    q = to_bits(rng.standard_normal((3, H, d)), "float16")
    outs = []
    for trial in range(3):
        perm = rng.permutation(nb)
        tables, pos = [], 0
        for k in need:
            tables.append([int(b) for b in perm[pos:pos + k]])
            pos += k
        kc, vc, bt = build_pool(ks, vs, tables, B, nb, "float16", fill=float(trial))
        outs.append(oracle.attention(q, kc, vc, bt, lengths, 0.35, "float16"))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def pin_shared_prefix_equals_private_copies():
    rng = np.random.default_rng(6)
    H, d, B = 1, 8, 4
    prefix_k = rng.standard_normal((8, H, d)).astype(np.float32)
    prefix_v = rng.standard_normal((8, H, d)).astype(np.float32)
    tail_k = [rng.standard_normal((3, H, d)).astype(np.float32) for _ in range(2)]
    tail_v = [rng.standard_normal((3, H, d)).astype(np.float32) for _ in range(2)]
    ks = [np.concatenate([prefix_k, t]) for t in tail_k]
    vs = [np.concatenate([prefix_v, t]) for t in tail_v]
    q = to_bits(rng.standard_normal((2, H, d)), "bfloat16")
    # private: every block its own
    kc, vc, bt = build_pool(ks, vs, [[0, 1, 2], [3, 4, 5]], B, 6, "bfloat16")
    private = oracle.attention(q, kc, vc, bt, [11, 11], 0.4, "bfloat16")
    # shared: both sequences map their two prefix blocks onto blocks 4 and 1
    kc2, vc2, bt2 = build_pool(ks, vs, [[4, 1, 0], [4, 1, 3]], B, 6, "bfloat16")
    shared = oracle.attention(q, kc2, vc2, bt2, [11, 11], 0.4, "bfloat16")
    assert np.array_equal(private, shared)


def pin_online_recurrence_equals_two_pass():
    """Eq. (4) over any chunking equals dense softmax (witness: 2.2e-16 scale)."""
    with open(os.path.join(GOLDEN, "witness.json")) as f:
        witness = json.load(f)
    rng = np.random.default_rng(7)
    lengths = [1, 16, 37, 91]
    q, kc, vc, bt, lens, _ = random_case(rng, lengths, 4, 2, 32, 16, "bfloat16")
    dense = oracle.attention(q, kc, vc, bt, lens, 1 / math.sqrt(32), "bfloat16")
    worst = 0.0
    cases = 0
    for chunk in (1, 3, 7, 16, 64, 1000):
        online = oracle.online_attention(q, kc, vc, bt, lens, 1 / math.sqrt(32), "bfloat16", chunk)
        worst = max(worst, float(np.max(np.abs(online - dense))))
        cases += 1
    assert cases >= 1 and worst <= 64 * witness["largest_absolute_error"], worst


def pin_partition_merge_equals_two_pass():
    rng = np.random.default_rng(8)
    lengths = [0, 5, 48, 100]
    q, kc, vc, bt, lens, _ = random_case(rng, lengths, 4, 4, 16, 8, "float16")
    dense = oracle.attention(q, kc, vc, bt, lens, 0.25, "float16")
    for part in (8, 16, 40, 128):
        parts = -(-max(lengths) // part)
        m, l, acc = oracle.partition_stats(q, kc, vc, bt, lens, 0.25, "float16", part, parts)
        merged = oracle.merge_partitions(m, l, acc)
        assert np.max(np.abs(merged - dense)) <= 1e-14
    # a single partition covering everything: l is the softmax denominator
    m, l, acc = oracle.partition_stats(q, kc, vc, bt, lens, 0.25, "float16", 128, 1)
    assert np.allclose(acc[:, :, 0, :] / np.where(l > 0, l, 1.0), dense, rtol=0, atol=1e-15)


def pin_brute_force_against_library_softmax():
    """Tiny random cases against scipy's softmax on explicitly gathered rows."""
    rng = np.random.default_rng(9)
    for dtype, B in (("float16", 2), ("bfloat16", 3)):
        lengths = [1, 2, 5]
        q, kc, vc, bt, lens, tables = random_case(rng, lengths, 2, 1, 4, B, dtype)
        out = oracle.attention(q, kc, vc, bt, lens, 0.5, dtype)
        for s, n in enumerate(lengths):
            K = np.stack([widen(kc[tables[s][t // B], 0, t % B], dtype) for t in range(n)])
            V = np.stack([widen(vc[tables[s][t // B], 0, t % B], dtype) for t in range(n)])
            for i in range(2):
                w = softmax(0.5 * (K @ widen(q[s, i], dtype)))
                assert np.allclose(out[s, i], w @ V, rtol=1e-12, atol=1e-13)


def pin_empty_sequence_is_zero():
    rng = np.random.default_rng(10)
    q, kc, vc, bt, lens, _ = random_case(rng, [0, 3], 2, 2, 8, 4, "bfloat16")
    out = oracle.attention(q, kc, vc, bt, lens, 1.0, "bfloat16")
    assert np.array_equal(out[0], np.zeros_like(out[0])) and np.any(out[1] != 0)


# ---------------------------------------------------------------------------
# kv_write and copy_blocks
# ---------------------------------------------------------------------------
def pin_kv_write_slot_arithmetic():
    """slot = physical block * B + offset; negative slots are padding."""
    H, d, B, nb = 2, 4, 4, 5
    kc = np.zeros((nb, H, B, d), dtype=np.uint16)
    vc = np.zeros_like(kc)
    k = np.arange(3 * H * d, dtype=np.uint16).reshape(3, H, d) + 1
    v = k + 1000
    # token 0 -> block 1 slot 2 (slot 6); token 1 padding; token 2 -> block 4 slot 3 (slot 19)
    kc2, vc2, status = oracle.kv_write(k, v, [6, -1, 19], kc, vc)
    assert status == 0
    assert np.array_equal(kc2[1, :, 2, :], k[0]) and np.array_equal(vc2[1, :, 2, :], v[0])
    assert np.array_equal(kc2[4, :, 3, :], k[2]) and np.array_equal(vc2[4, :, 3, :], v[2])
    changed = np.argwhere(kc2 != 0)
    assert len(changed) == 2 * H * d  # nothing else touched, padding skipped
    # a slot past the pool is reported and skipped
    kc3, _, status = oracle.kv_write(k[:1], v[:1], [nb * B], kc, vc)
    assert status != 0 and not kc3.any()


def pin_kv_write_then_read_back():
    """A token written at the next slot is the one a length-1 read returns."""
    rng = np.random.default_rng(11)
    H, d, B, nb = 2, 8, 4, 6
    kc = to_bits(rng.standard_normal((nb, H, B, d)), "bfloat16")
    vc = to_bits(rng.standard_normal((nb, H, B, d)), "bfloat16")
    k = to_bits(rng.standard_normal((1, H, d)), "bfloat16")
    v = to_bits(rng.standard_normal((1, H, d)), "bfloat16")
    slot = 3 * B  # first slot of block 3
    kc2, vc2, _ = oracle.kv_write(k, v, [slot], kc, vc)
    q = to_bits(rng.standard_normal((1, H, d)), "bfloat16")
    out = oracle.attention(q, kc2, vc2, np.array([[3]], dtype=np.int32), [1], 1.0, "bfloat16")
    assert np.array_equal(out[0], widen(v[0], "bfloat16"))


def pin_copy_blocks_copies_whole_blocks():
    rng = np.random.default_rng(12)
    H, d, B, nb = 2, 4, 4, 6
    kc = rng.integers(0, 65535, (nb, H, B, d), dtype=np.uint16)
    vc = rng.integers(0, 65535, (nb, H, B, d), dtype=np.uint16)
    kc2, vc2, status = oracle.copy_blocks(kc, vc, [(1, 4), (2, 0)])
    assert status == 0
    assert np.array_equal(kc2[4], kc[1]) and np.array_equal(vc2[4], vc[1])
    assert np.array_equal(kc2[0], kc[2]) and np.array_equal(vc2[0], vc[2])
    for b in (1, 2, 3, 5):
        assert np.array_equal(kc2[b], kc[b]) and np.array_equal(vc2[b], vc[b])
    _, _, status = oracle.copy_blocks(kc, vc, [(1, nb)])
    assert status != 0


def pin_transfer_blocks_between_pools():
    """Swap out then back in restores the bytes; only the paired blocks move."""
    rng = np.random.default_rng(13)
    H, d, B = 2, 4, 4
    dev_k = rng.integers(0, 65535, (6, H, B, d), dtype=np.uint16)
    dev_v = rng.integers(0, 65535, (6, H, B, d), dtype=np.uint16)
    host_k = np.zeros((3, H, B, d), dtype=np.uint16)
    host_v = np.zeros_like(host_k)
    hk, hv, status = oracle.transfer_blocks(dev_k, dev_v, host_k, host_v, [(4, 0), (1, 2)])
    assert status == 0
    assert np.array_equal(hk[0], dev_k[4]) and np.array_equal(hv[2], dev_v[1])
    assert not hk[1].any() and not hv[1].any()
    # back in, to different device blocks
    back_k, back_v, status = oracle.transfer_blocks(hk, hv, np.zeros_like(dev_k),
                                                    np.zeros_like(dev_v), [(0, 5), (2, 3)])
    assert status == 0
    assert np.array_equal(back_k[5], dev_k[4]) and np.array_equal(back_v[3], dev_v[1])
    assert not back_k[0].any()
    _, _, status = oracle.transfer_blocks(dev_k, dev_v, host_k, host_v, [(0, 3)])
    assert status != 0


# ---------------------------------------------------------------------------
# Paged prefill (causal, many query tokens per sequence)
# ---------------------------------------------------------------------------
def pin_prefill_hand_example():
    """The hand example as a 3-token prompt (ctx 0), one query head per KV head.

    Query 0 sees only token 0: output (7, 0).  Query 1, q = (1, 0), sees keys
    (1,0), (0,0): scores ln2 * (1, 0), weights (2, 1) / 3, output (14/3, 7/3).
    Query 2, q = (1, 0), sees all three: output (-2, 9).
    """
    for dtype in ("float16", "bfloat16"):
        ks = [np.array([[[1, 0]], [[0, 0]], [[2, 0]]], dtype=np.float32)]
        vs = [np.array([[[7, 0]], [[0, 7]], [[-7, 14]]], dtype=np.float32)]
        kc, vc, bt = build_pool(ks, vs, [[5, 2]], 2, 6, dtype, fill=99.0)
        q = to_bits([[[1, 0]], [[1, 0]], [[1, 0]]], dtype)
        out = oracle.prefill(q, [0, 3], kc, vc, bt, [3], math.log(2.0), dtype)
        assert np.allclose(out[0, 0], [7.0, 0.0], rtol=0, atol=1e-13), out
        assert np.allclose(out[1, 0], [14 / 3, 7 / 3], rtol=0, atol=1e-13), out
        assert np.allclose(out[2, 0], [-2.0, 9.0], rtol=0, atol=1e-13), out


def pin_prefill_single_query_is_decode():
    """One query per sequence (its last token) is exactly the decode attention."""
    rng = np.random.default_rng(14)
    lengths = [1, 9, 40, 77]
    q, kc, vc, bt, lens, _ = random_case(rng, lengths, 8, 2, 16, 8, "bfloat16")
    dec = oracle.attention(q, kc, vc, bt, lens, 0.3, "bfloat16")
    pre = oracle.prefill(q, np.arange(len(lengths) + 1), kc, vc, bt, lens, 0.3, "bfloat16")
    assert np.array_equal(dec, pre)


def pin_prefill_is_causal():
    """Changing keys and values after a query's position leaves its output unchanged."""
    rng = np.random.default_rng(15)
    n, q_len, H, d, B = 30, 12, 2, 8, 4
    ks = rng.standard_normal((n, H, d)).astype(np.float32)
    vs = rng.standard_normal((n, H, d)).astype(np.float32)
    tables = [[int(b) for b in rng.permutation(8)]]
    kc, vc, bt = build_pool([ks], [vs], tables, B, 8, "float16")
    q = to_bits(rng.standard_normal((q_len, 2 * H, d)), "float16")
    base = oracle.prefill(q, [0, q_len], kc, vc, bt, [n], 0.4, "float16")
    ctx = n - q_len
    for cut in (0, 5, q_len - 1):
        ks2, vs2 = ks.copy(), vs.copy()
        ks2[ctx + cut + 1:] = rng.standard_normal(ks2[ctx + cut + 1:].shape)
        vs2[ctx + cut + 1:] = rng.standard_normal(vs2[ctx + cut + 1:].shape)
        kc2, vc2, _ = build_pool([ks2], [vs2], tables, B, 8, "float16")
        out = oracle.prefill(q, [0, q_len], kc2, vc2, bt, [n], 0.4, "float16")
        assert np.array_equal(out[:cut + 1], base[:cut + 1])
        if cut + 1 < q_len:
            assert not np.array_equal(out[cut + 1:], base[cut + 1:])


def pin_prefill_brute_force_against_library_softmax():
    rng = np.random.default_rng(16)
    lengths, q_lens = [5, 9], [3, 9]
    H_q, H_kv, d, B = 4, 2, 4, 4
    q_all, kc, vc, bt, lens, tables = random_case(rng, lengths, H_q, H_kv, d, B, "bfloat16")
    q = to_bits(rng.standard_normal((sum(q_lens), H_q, d)), "bfloat16")
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    out = oracle.prefill(q, cu, kc, vc, bt, lens, 0.7, "bfloat16")
    for s, (n, ql) in enumerate(zip(lengths, q_lens)):
        for i in range(ql):
            pos = n - ql + i
            for qh in range(H_q):
                h = qh // (H_q // H_kv)
                K = np.stack([widen(kc[tables[s][t // B], h, t % B], "bfloat16") for t in range(pos + 1)])
                V = np.stack([widen(vc[tables[s][t // B], h, t % B], "bfloat16") for t in range(pos + 1)])
                w = softmax(0.7 * (K @ widen(q[cu[s] + i, qh], "bfloat16")))
                assert np.allclose(out[cu[s] + i, qh], w @ V, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# 8-bit (E4M3) pools: code = E4M3(x / scale) from the binary32 quotient,
# read back as code * scale
# ---------------------------------------------------------------------------
def e4m3_values():
    """Value of every E4M3 code through torch's float8_e4m3fn (a library conversion)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e4m3_codes(x):
    """binary32 values (|x| <= 448) -> E4M3 codes through torch (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_decode_all_codes():
    ref = e4m3_values()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    # the format's landmarks: largest finite 448 (S.1111.110), smallest normal
    # 2^-6, smallest subnormal 2^-9, NaN only at S.1111.111
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9
    assert got[0x38] == 1.0 and got[0xB8] == -1.0
    assert set(np.flatnonzero(np.isnan(got)).tolist()) == {0x7F, 0xFF}


def pin_e4m3_encode_round_trip_and_ties():
    vals = e4m3_values()
    for c in range(256):
        if c not in (0x7F, 0xFF):
            assert oracle.e4m3_from_f32(vals[c]) == c, hex(c)
    for c in range(0x7E):  # neighbouring positive codes c, c + 1
        mid = np.float32((vals[c] + vals[c + 1]) / 2)  # exact: at most 5 significant bits
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_from_f32(mid) == even and oracle.e4m3_from_f32(-mid) == 0x80 | even
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(np.inf))
        assert oracle.e4m3_from_f32(below) == c and oracle.e4m3_from_f32(above) == c + 1


def pin_e4m3_encode_against_library_and_saturation():
    rng = np.random.default_rng(31)
    x = (rng.standard_normal(20000) * 10.0 ** rng.uniform(-4.0, 2.6, 20000)).astype(np.float32)
    x = x[np.abs(x) <= 464]  # torch turns larger magnitudes into NaN instead of saturating
    got = np.array([oracle.e4m3_from_f32(v) for v in x], dtype=np.uint8)
    assert np.array_equal(got, e4m3_codes(x))
    for v, code in ((465.0, 0x7E), (1e30, 0x7E), (np.inf, 0x7E), (-np.inf, 0xFE), (-1000.0, 0xFE),
                    (0.0, 0x00), (-0.0, 0x80)):
        assert oracle.e4m3_from_f32(v) == code, (v, code)
    assert oracle.e4m3_from_f32(np.nan) == 0x7F


def pin_kv_write_fp8_codes():
    """Slots as kv_write; every element stored as E4M3 of the binary32 x / scale."""
    rng = np.random.default_rng(32)
    H, d, B, nb = 2, 8, 4, 5
    k_scale, v_scale = 0.0371, 3.3
    for dtype in ("float16", "bfloat16"):
        k = to_bits(rng.standard_normal((3, H, d)) * 4, dtype)
        v = to_bits(rng.standard_normal((3, H, d)) * 4, dtype)
        kc = np.zeros((nb, H, B, d), dtype=np.uint8)
        vc = np.zeros_like(kc)
        kc2, vc2, status = oracle.kv_write_fp8(k, v, dtype, [6, -1, 19], kc, vc, k_scale, v_scale)
        assert status == 0

        def expect(bits, scale):
            quotient = widen(bits, dtype).astype(np.float32) / np.float32(scale)  # binary32
            return e4m3_codes(np.clip(quotient, -448, 448))

        assert np.array_equal(kc2[1, :, 2], expect(k[0], k_scale))
        assert np.array_equal(vc2[1, :, 2], expect(v[0], v_scale))
        assert np.array_equal(kc2[4, :, 3], expect(k[2], k_scale))
        assert np.array_equal(vc2[4, :, 3], expect(v[2], v_scale))
        untouched = np.ones(nb, dtype=bool)
        untouched[[1, 4]] = False
        assert not kc2[untouched].any() and not vc2[untouched].any()
        assert not kc2[1, :, [0, 1, 3]].any() and not kc2[4, :, :3].any()
    # hand values, keys at scale 0.5: 1 / 0.5 = 2 = 1.0 * 2^(8-7) -> 0x40; -3 / 0.5 = -1.5 * 2^(9-7)
    # -> 0xcc; 1000 / 0.5 saturates to 448 -> 0x7e.  Values at scale 1: 1 -> 0x38, -3 -> 0xc4.
    one = to_bits(np.array([[[1.0, -3.0, 1000.0, 0.0]]]), "bfloat16")
    kc2, vc2, _ = oracle.kv_write_fp8(one, one, "bfloat16", [0], np.zeros((1, 1, 1, 4), np.uint8),
                                      np.zeros((1, 1, 1, 4), np.uint8), 0.5, 1.0)
    assert kc2[0, 0, 0].tolist() == [0x40, 0xCC, 0x7E, 0x00]
    assert vc2[0, 0, 0].tolist() == [0x38, 0xC4, 0x7E, 0x00]
    _, _, status = oracle.kv_write_fp8(one, one, "bfloat16", [1], np.zeros((1, 1, 1, 4), np.uint8),
                                       np.zeros((1, 1, 1, 4), np.uint8), 1.0, 1.0)
    assert status != 0  # slot past the pool


def pin_kv_write_fp8_rounds_the_binary32_quotient():
    """Where the binary32 quotient lands exactly on a midpoint of two codes but
    the exact quotient does not, the stored code follows the binary32 value."""
    from fractions import Fraction
    vals = e4m3_values()

    def exact_nearest(q):
        best = min(range(0x7F), key=lambda c: (abs(Fraction(float(vals[c])) - q), c % 2))
        return best

    differ = 0
    for x in (1.0, 1.5, 3.0, 0.75):
        for c in range(0x30, 0x48):
            mid = (Fraction(float(vals[c])) + Fraction(float(vals[c + 1]))) / 2
            s0 = np.float32(float(Fraction(x) / mid))
            for s in (np.nextafter(s0, np.float32(0)), s0, np.nextafter(s0, np.float32(np.inf))):
                k = to_bits(np.array([[[x]]]), "bfloat16")
                kc, _, _ = oracle.kv_write_fp8(k, k, "bfloat16", [0], np.zeros((1, 1, 1, 1), np.uint8),
                                               np.zeros((1, 1, 1, 1), np.uint8), float(s), 1.0)
                binary32 = int(e4m3_codes([np.float32(x) / s])[0])
                assert int(kc[0, 0, 0, 0]) == binary32, (x, float(s))
                differ += binary32 != exact_nearest(Fraction(x) / Fraction(float(s)))
    assert differ > 0  # the cases above do separate the two readings


def fp8_case(rng, lengths, H_q, H_kv, d, B, spare=2):
    """Random E4M3 pools (NaN codes excluded) and scattered block tables."""
    need = [max(1, -(-n // B)) for n in lengths]
    nb = sum(need) + spare
    perm = rng.permutation(nb)
    tables, pos = [], 0
    for n in need:
        tables.append([int(b) for b in perm[pos:pos + n]])
        pos += n
    kc = rng.integers(0, 256, size=(nb, H_kv, B, d)).astype(np.uint8)
    vc = rng.integers(0, 256, size=(nb, H_kv, B, d)).astype(np.uint8)
    for pool in (kc, vc):
        pool[(pool & 0x7F) == 0x7F] = 0x3C
        pool[(pool & 0x78) >= 0x60] &= 0xC7  # keep magnitudes small: exponent field below 12
    bt = np.zeros((len(lengths), max(need)), dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, :len(t)] = t
    return kc, vc, bt, np.asarray(lengths, dtype=np.int32), tables


def pin_fp8_attention_equals_16bit_on_the_same_values():
    """With power-of-two scales the read-back values are exact in bfloat16, so
    attention over the codes equals attention over those bfloat16 values."""
    rng = np.random.default_rng(33)
    kc, vc, bt, lens, _ = fp8_case(rng, [1, 7, 20], 4, 2, 16, 4)
    vals = e4m3_values()
    k16 = to_bits(vals[kc] * 2.0, "bfloat16")
    v16 = to_bits(vals[vc] * 0.25, "bfloat16")
    assert np.array_equal(widen(k16, "bfloat16"), vals[kc] * 2.0)
    q = to_bits(rng.standard_normal((3, 4, 16)), "bfloat16")
    a = oracle.attention_fp8(q, kc, vc, bt, lens, 0.3, 2.0, 0.25, "bfloat16")
    b = oracle.attention(q, k16, v16, bt, lens, 0.3, "bfloat16")
    assert np.array_equal(a, b)


def pin_fp8_attention_brute_force_against_library_softmax():
    rng = np.random.default_rng(34)
    k_scale, v_scale = 0.0371, 3.3
    vals = e4m3_values()
    for dtype in ("float16", "bfloat16"):
        kc, vc, bt, lens, tables = fp8_case(rng, [0, 1, 5, 9], 4, 2, 8, 4)
        q = to_bits(rng.standard_normal((4, 4, 8)), dtype)
        out = oracle.attention_fp8(q, kc, vc, bt, lens, 0.5, k_scale, v_scale, dtype)
        assert not out[0].any()
        for s, n in enumerate(lens):
            for i in range(4):
                h = i // 2
                K = np.stack([vals[kc[tables[s][t // 4], h, t % 4]] for t in range(n)]) if n else None
                if n == 0:
                    continue
                V = np.stack([vals[vc[tables[s][t // 4], h, t % 4]] for t in range(n)])
                w = softmax(0.5 * ((K * np.float64(np.float32(k_scale))) @ widen(q[s, i], dtype)))
                ref = w @ (V * np.float64(np.float32(v_scale)))
                assert np.allclose(out[s, i], ref, rtol=1e-12, atol=1e-13)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
