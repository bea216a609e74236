"""Plain, slow, obviously correct CPU oracle for the paged-KV decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference arm of ``bench.py`` may import this package.
The product path (``paged_kv_cache_242_gb300``) never imports it, and it
imports nothing from the product: the two share no code.

Contents
--------
* ``attention``            dense two-pass fp64 attention after gathering each
                           sequence's blocks into contiguous rows
                           (``oracle_paged_attention`` in ``pkv_oracle.c``).
* ``online_attention``     the same result by the running-max / running-sum
                           recurrence, Eq. (4) of "Serving Language Models
                           Within a Memory Budget".
* ``partition_stats`` / ``merge_partitions``  per-partition (m, l, acc)
                           statistics and their Eq. (4) merge.
* ``kv_write`` / ``copy_blocks``  byte-exact slot scatter and block copy.
* ``e4m3_to_f64`` / ``e4m3_from_f32`` / ``kv_write_fp8`` / ``attention_fp8``
                           the 8-bit cache variant: E4M3 codes with one
                           scale per pool (stored E4M3(x / scale), read
                           back as code * scale).
* ``accounting``           the pages' byte / block / waste / utilisation
                           formulas (pure Python).

Parity pins (tests/test_oracle_*.py) tie every function to values the
pages print or to closed forms of the mathematics.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import accounting  # noqa: F401  (re-exported)
from .build_oracle import LIBRARY, build

DTYPE_CODES = {"float16": 0, "bfloat16": 1}

_lib = None


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    f64p = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = ctypes.c_double
    common = [u16p, i, i, i, u16p, u16p, i, i, i, i, i32p, i, i32p, ctypes.c_double]
    lib.oracle_paged_attention.argtypes = common + [f64p, i]
    lib.oracle_paged_attention.restype = i
    lib.oracle_online_attention.argtypes = common + [i, f64p]
    lib.oracle_online_attention.restype = i
    lib.oracle_partition_stats.argtypes = common + [i, i, f64p, f64p, f64p]
    lib.oracle_partition_stats.restype = i
    lib.oracle_merge_partitions.argtypes = [f64p, f64p, f64p, ctypes.c_longlong, i, i, f64p]
    lib.oracle_merge_partitions.restype = i
    lib.oracle_kv_write.argtypes = [u16p, u16p, i64p, i, u16p, u16p, i, i, i, i]
    lib.oracle_kv_write.restype = i
    lib.oracle_copy_blocks.argtypes = [u16p, u16p, i, i, i, i, i64p, i]
    lib.oracle_copy_blocks.restype = i
    lib.oracle_paged_prefill.argtypes = [u16p, i32p, i, i, i, u16p, u16p, i, i, i, i, i32p, i,
                                         i32p, ctypes.c_double, f64p, i]
    lib.oracle_paged_prefill.restype = i
    lib.oracle_transfer_blocks.argtypes = [u16p, u16p, i, u16p, u16p, i, i, i, i, i64p, i]
    lib.oracle_transfer_blocks.restype = i
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f32 = ctypes.c_float
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f64.restype = ctypes.c_double
    lib.oracle_e4m3_from_f32.argtypes = [f32]
    lib.oracle_e4m3_from_f32.restype = ctypes.c_uint8
    lib.oracle_kv_write_fp8.argtypes = [u16p, u16p, i, i64p, i, u8p, u8p, i, i, i, i, f32, f32]
    lib.oracle_kv_write_fp8.restype = i
    lib.oracle_paged_attention_fp8.argtypes = [u16p, i, i, i, u8p, u8p, i, i, i, i, i32p, i, i32p,
                                               ctypes.c_double, f32, f32, f64p, i]
    lib.oracle_paged_attention_fp8.restype = i
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


def _ptr(array: np.ndarray, ctype):
    assert array.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return array.ctypes.data_as(ctypes.POINTER(ctype))


def _bits(array: np.ndarray) -> np.ndarray:
    """View a 16-bit array (uint16 bit patterns) as contiguous uint16."""
    a = np.ascontiguousarray(array)
    if a.dtype.itemsize != 2:
        raise TypeError(f"expected 16-bit storage, got {a.dtype}")
    return a.view(np.uint16)


def _check(status: int, what: str) -> None:
    if status != 0:
        raise ValueError(f"oracle {what} failed with status {status}")


def max_threads() -> int:
    return _load().oracle_max_threads()


def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(bits)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits)


def e4m3_to_f64(code: int) -> float:
    """Exact value of one E4M3 code (NaN for 0x7f / 0xff)."""
    return _load().oracle_e4m3_to_f64(int(code) & 0xFF)


def e4m3_from_f32(x: float) -> int:
    """Nearest E4M3 code of a binary32 value (ties to even, saturating at 448)."""
    return int(_load().oracle_e4m3_from_f32(float(np.float32(x))))


def _codes(array: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(array)
    if a.dtype.itemsize != 1:
        raise TypeError(f"expected 8-bit codes, got {a.dtype}")
    return a.view(np.uint8)


def kv_write_fp8(k, v, dtype, slot_mapping, k_cache, v_cache, k_scale, v_scale):
    """Quantising slot scatter into copies of E4M3 pools; returns (kc, vc, status)."""
    lib = _load()
    k, v = _bits(k), _bits(v)
    kc, vc = _codes(k_cache).copy(), _codes(v_cache).copy()
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    nb, hkv, bs, d = _geometry(kc)
    status = lib.oracle_kv_write_fp8(
        _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), DTYPE_CODES[dtype],
        _ptr(sm, ctypes.c_int64), int(sm.shape[0]), _ptr(kc, ctypes.c_uint8),
        _ptr(vc, ctypes.c_uint8), nb, hkv, bs, d, float(k_scale), float(v_scale))
    return kc, vc, status


def attention_fp8(q, k_cache, v_cache, block_tables, seq_lens, scale, k_scale, v_scale, dtype,
                  num_threads=1):
    """Dense fp64 attention over E4M3 pools read back as code * scale.

    q: [S, H_q, d] 16-bit patterns of ``dtype``; k_cache, v_cache: [NB, H_kv, B, d]
    uint8 codes.  Returns float64 [S, H_q, d].
    """
    lib = _load()
    q = _bits(q)
    kc, vc = _codes(k_cache), _codes(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    num_seqs, num_q_heads, head_dim = q.shape
    nb, hkv, bs, d = _geometry(kc)
    assert d == head_dim and vc.shape == kc.shape and bt.shape[0] == num_seqs
    out = np.zeros((num_seqs, num_q_heads, head_dim), dtype=np.float64)
    _check(lib.oracle_paged_attention_fp8(
        _ptr(q, ctypes.c_uint16), DTYPE_CODES[dtype], num_seqs, num_q_heads,
        _ptr(kc, ctypes.c_uint8), _ptr(vc, ctypes.c_uint8), nb, hkv, bs, d,
        _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(sl, ctypes.c_int32), float(scale),
        float(k_scale), float(v_scale), _ptr(out, ctypes.c_double), int(num_threads)),
        "attention_fp8")
    return out


def _geometry(k_cache):
    num_blocks, num_kv_heads, block_size, head_dim = k_cache.shape
    return num_blocks, num_kv_heads, block_size, head_dim


def attention(q, k_cache, v_cache, block_tables, seq_lens, scale, dtype, num_threads=1):
    """Dense fp64 attention of one query token per sequence.

    q: [S, H_q, d] 16-bit patterns; k_cache, v_cache: [NB, H_kv, B, d];
    block_tables: [S, max_blocks] int32; seq_lens: [S] int32.
    Returns float64 [S, H_q, d].
    """
    lib = _load()
    q = _bits(q)
    kc, vc = _bits(k_cache), _bits(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    num_seqs, num_q_heads, head_dim = q.shape
    nb, hkv, bs, d = _geometry(kc)
    assert d == head_dim and vc.shape == kc.shape and bt.shape[0] == num_seqs
    out = np.zeros((num_seqs, num_q_heads, head_dim), dtype=np.float64)
    _check(lib.oracle_paged_attention(
        _ptr(q, ctypes.c_uint16), DTYPE_CODES[dtype], num_seqs, num_q_heads,
        _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16), nb, hkv, bs, d,
        _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(sl, ctypes.c_int32), float(scale),
        _ptr(out, ctypes.c_double), int(num_threads)), "attention")
    return out


def online_attention(q, k_cache, v_cache, block_tables, seq_lens, scale, dtype, chunk):
    """Eq. (4) recurrence over consecutive chunks of ``chunk`` tokens (fp64)."""
    lib = _load()
    q = _bits(q)
    kc, vc = _bits(k_cache), _bits(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    num_seqs, num_q_heads, head_dim = q.shape
    nb, hkv, bs, d = _geometry(kc)
    out = np.zeros((num_seqs, num_q_heads, head_dim), dtype=np.float64)
    _check(lib.oracle_online_attention(
        _ptr(q, ctypes.c_uint16), DTYPE_CODES[dtype], num_seqs, num_q_heads,
        _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16), nb, hkv, bs, d,
        _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(sl, ctypes.c_int32), float(scale),
        int(chunk), _ptr(out, ctypes.c_double)), "online_attention")
    return out


def partition_stats(q, k_cache, v_cache, block_tables, seq_lens, scale, dtype,
                    partition_size, num_partitions):
    """Per-partition (m, l, acc) in natural-log units, fp64.

    Returns m, l: [S, H_q, NP]; acc: [S, H_q, NP, d].
    """
    lib = _load()
    q = _bits(q)
    kc, vc = _bits(k_cache), _bits(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    num_seqs, num_q_heads, head_dim = q.shape
    nb, hkv, bs, d = _geometry(kc)
    m = np.zeros((num_seqs, num_q_heads, num_partitions), dtype=np.float64)
    l = np.zeros_like(m)
    acc = np.zeros((num_seqs, num_q_heads, num_partitions, head_dim), dtype=np.float64)
    _check(lib.oracle_partition_stats(
        _ptr(q, ctypes.c_uint16), DTYPE_CODES[dtype], num_seqs, num_q_heads,
        _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16), nb, hkv, bs, d,
        _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(sl, ctypes.c_int32), float(scale),
        int(partition_size), int(num_partitions),
        _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double), _ptr(acc, ctypes.c_double)),
        "partition_stats")
    return m, l, acc


def merge_partitions(m, l, acc):
    """Eq. (4) merge of partition statistics: [..., NP] -> [..., d]."""
    lib = _load()
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    num_partitions, head_dim = acc.shape[-2], acc.shape[-1]
    rows = int(np.prod(m.shape[:-1]))
    out = np.zeros(m.shape[:-1] + (head_dim,), dtype=np.float64)
    _check(lib.oracle_merge_partitions(
        _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double), _ptr(acc, ctypes.c_double),
        rows, num_partitions, head_dim, _ptr(out, ctypes.c_double)), "merge_partitions")
    return out


def kv_write(k, v, slot_mapping, k_cache, v_cache):
    """Scatter k, v [T, H_kv, d] into copies of the caches; returns the new caches."""
    lib = _load()
    k, v = _bits(k), _bits(v)
    kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    nb, hkv, bs, d = _geometry(kc)
    status = lib.oracle_kv_write(
        _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), _ptr(sm, ctypes.c_int64),
        int(sm.shape[0]), _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16), nb, hkv, bs, d)
    return kc, vc, status


def copy_blocks(k_cache, v_cache, pairs):
    """Apply (src, dst) whole-block copies in order to copies of the caches."""
    lib = _load()
    kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    nb, hkv, bs, d = _geometry(kc)
    status = lib.oracle_copy_blocks(_ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16),
                                    nb, hkv, bs, d, _ptr(pr, ctypes.c_int64), int(pr.shape[0]))
    return kc, vc, status


def prefill(q, cu_q, k_cache, v_cache, block_tables, seq_lens, scale, dtype, num_threads=1):
    """Causal fp64 attention of the last q_len tokens of each sequence.

    q: [total_q, H_q, d] 16-bit patterns, sequence s's queries at rows
    cu_q[s] .. cu_q[s+1]-1 (positions seq_len - q_len .. seq_len - 1).
    Returns float64 [total_q, H_q, d].
    """
    lib = _load()
    q = _bits(q)
    kc, vc = _bits(k_cache), _bits(v_cache)
    cu = np.ascontiguousarray(cu_q, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    total_q, num_q_heads, head_dim = q.shape
    nb, hkv, bs, d = _geometry(kc)
    num_seqs = sl.shape[0]
    assert cu.shape[0] == num_seqs + 1 and cu[-1] == total_q and d == head_dim
    out = np.zeros((total_q, num_q_heads, head_dim), dtype=np.float64)
    _check(lib.oracle_paged_prefill(
        _ptr(q, ctypes.c_uint16), _ptr(cu, ctypes.c_int32), DTYPE_CODES[dtype], num_seqs,
        num_q_heads, _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16), nb, hkv, bs, d,
        _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(sl, ctypes.c_int32), float(scale),
        _ptr(out, ctypes.c_double), int(num_threads)), "prefill")
    return out


def transfer_blocks(src_k, src_v, dst_k, dst_v, pairs):
    """Copy whole blocks from the source pools into copies of the destination pools."""
    lib = _load()
    sk, sv = _bits(src_k), _bits(src_v)
    dk, dv = _bits(dst_k).copy(), _bits(dst_v).copy()
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    snb, hkv, bs, d = _geometry(sk)
    dnb = dk.shape[0]
    assert dk.shape[1:] == sk.shape[1:]
    status = lib.oracle_transfer_blocks(_ptr(sk, ctypes.c_uint16), _ptr(sv, ctypes.c_uint16), snb,
                                        _ptr(dk, ctypes.c_uint16), _ptr(dv, ctypes.c_uint16), dnb,
                                        hkv, bs, d, _ptr(pr, ctypes.c_int64), int(pr.shape[0]))
    return dk, dv, status


__all__ = ["prefill", "transfer_blocks", "e4m3_to_f64", "e4m3_from_f32", "kv_write_fp8",
           "attention_fp8", "attention", "online_attention", "partition_stats", "merge_partitions", "kv_write",
           "copy_blocks", "f16_to_f64", "bf16_to_f64", "max_threads", "accounting", "build",
           "LIBRARY"]
