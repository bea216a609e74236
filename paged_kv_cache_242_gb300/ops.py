"""Python binding of the three kernels: argument marshalling only.

Every function takes torch CUDA tensors, checks their shapes / dtypes /
layout, and calls the matching ``pkv_*`` entry point of libpkv.so with raw
device pointers and the current CUDA stream.  All arithmetic runs in the
library's CUDA kernels; if the library is missing the call raises.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import CacheDesc, PKVError

_DTYPES = {torch.float16: _lib.PKV_FP16, torch.bfloat16: _lib.PKV_BF16,
           torch.uint8: _lib.PKV_FP8_E4M3}
if hasattr(torch, "float8_e4m3fn"):
    _DTYPES[torch.float8_e4m3fn] = _lib.PKV_FP8_E4M3
_16BIT = {torch.float16: _lib.PKV_FP16, torch.bfloat16: _lib.PKV_BF16}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    _require(k_cache.dim() == 4, "caches must be [num_blocks, num_kv_heads, block_size, head_dim]")
    _require(k_cache.dtype in _DTYPES, f"unsupported cache dtype {k_cache.dtype}")
    nb, hkv, bs, d = k_cache.shape
    return CacheDesc(int(nb), int(hkv), int(bs), int(d), _DTYPES[k_cache.dtype])


def _check_caches(k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    _require(k_cache.is_cuda and v_cache.is_cuda, "caches must be CUDA tensors")
    _require(k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype,
             "k_cache and v_cache must match in shape and dtype")
    _require(k_cache.is_contiguous() and v_cache.is_contiguous(), "caches must be contiguous")


def _err_ptr(err_flag: Optional[torch.Tensor]) -> Optional[int]:
    if err_flag is None:
        return None
    _require(err_flag.dtype == torch.int32 and err_flag.is_cuda and err_flag.numel() >= 1,
             "err_flag must be a CUDA int32 tensor")
    return err_flag.data_ptr()


def _check_kv_write(k, v, slot_mapping, k_cache, v_cache):
    _check_caches(k_cache, v_cache)
    desc = cache_desc(k_cache)
    T = int(slot_mapping.numel())
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.is_cuda and
             slot_mapping.is_contiguous(), "slot_mapping must be a contiguous CUDA int64 tensor")
    _require(k.shape == (T, desc.num_kv_heads, desc.head_dim) and v.shape == k.shape,
             "k and v must be [num_tokens, num_kv_heads, head_dim]")
    _require(k.dtype == k_cache.dtype and v.dtype == k_cache.dtype, "k/v dtype must match the cache")
    _require(k.is_contiguous() and v.is_contiguous() and k.is_cuda and v.is_cuda,
             "k and v must be contiguous CUDA tensors")
    return desc, T


def kv_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
             k_cache: torch.Tensor, v_cache: torch.Tensor,
             err_flag: Optional[torch.Tensor] = None) -> None:
    """Write k, v [T, H_kv, d] into the caches at ``slot_mapping`` (int64 [T])."""
    desc, T = _check_kv_write(k, v, slot_mapping, k_cache, v_cache)
    lib = _lib.load()
    _lib.check(lib.pkv_kv_write(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache),
                                _ptr(v_cache), desc, _err_ptr(err_flag), _stream(k_cache.device)),
               "pkv_kv_write")


def decode_partition_size(max_seq_len: int, block_size: int, partition_size: int = 0) -> int:
    return int(_lib.load().pkv_decode_partition_size(int(max_seq_len), int(block_size),
                                                      int(partition_size)))


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, max_seq_len: int, block_size: int,
                           partition_size: int = 0, head_dim: int = 128) -> int:
    return int(_lib.load().pkv_decode_workspace_bytes(int(num_seqs), int(num_q_heads),
                                                       int(head_dim), int(max_seq_len),
                                                       int(block_size), int(partition_size)))


def _check_decode(q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads):
    _check_caches(k_cache, v_cache)
    desc = cache_desc(k_cache)
    if num_kv_heads is not None:
        _require(int(num_kv_heads) == desc.num_kv_heads, "num_kv_heads disagrees with the cache")
    _require(q.dim() == 3 and q.shape[2] == desc.head_dim, "q must be [num_seqs, num_q_heads, d]")
    _require(q.dtype == k_cache.dtype and q.is_cuda and q.is_contiguous(),
             "q must be a contiguous CUDA tensor of the cache dtype")
    S, Hq = int(q.shape[0]), int(q.shape[1])
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and
             block_tables.shape[0] == S and block_tables.is_contiguous() and block_tables.is_cuda,
             "block_tables must be a contiguous CUDA int32 [num_seqs, max_blocks] tensor")
    _require(seq_lens.dtype == torch.int32 and seq_lens.numel() == S and seq_lens.is_cuda and
             seq_lens.is_contiguous(), "seq_lens must be a contiguous CUDA int32 [num_seqs] tensor")
    return desc, S, Hq


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, seq_lens: torch.Tensor,
                           num_kv_heads: Optional[int] = None, scale: Optional[float] = None,
                           out: Optional[torch.Tensor] = None, *,
                           max_seq_len: Optional[int] = None, partition_size: int = 0,
                           workspace: Optional[torch.Tensor] = None,
                           err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Attention of one query token per sequence over its paged K/V.

    q [S, H_q, d]; block_tables int32 [S, max_blocks]; seq_lens int32 [S].
    ``max_seq_len`` (a host int >= every seq_len) avoids a device read; if
    omitted it is taken from ``seq_lens`` with a synchronising ``.item()``.
    ``workspace`` (uint8 CUDA tensor, zero-filled when new) is allocated
    when needed and omitted; reuse one across calls to avoid allocations.
    """
    desc, S, Hq = _check_decode(q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads)
    if scale is None:
        scale = desc.head_dim ** -0.5
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if S > 0 else 0
    if out is None:
        out = torch.empty_like(q)
    _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous() and out.is_cuda,
             "out must match q")
    max_blocks = int(block_tables.shape[1])
    if workspace is None:
        need = decode_workspace_bytes(S, Hq, max_seq_len, desc.block_size, partition_size,
                                      desc.head_dim)
        if need > 0:
            workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = _lib.load()
    _lib.check(lib.pkv_paged_decode_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks, _ptr(seq_lens),
        int(max_seq_len), S, Hq, desc, ctypes.c_float(float(scale)), int(partition_size),
        _ptr(workspace), ws_bytes, _ptr(out), _err_ptr(err_flag), _stream(q.device)),
        "pkv_paged_decode_attention")
    return out


def paged_prefill_attention(q: torch.Tensor, cu_seqlens_q: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, block_tables: torch.Tensor,
                            seq_lens: torch.Tensor, scale: Optional[float] = None,
                            out: Optional[torch.Tensor] = None, *, max_q_len: Optional[int] = None,
                            max_seq_len: Optional[int] = None,
                            err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Causal attention of the last q_len cached tokens of each sequence.

    q [total_q, H_q, d]; cu_seqlens_q int32 [S + 1] (sequence s's queries are
    rows cu[s]..cu[s+1]-1 and sit at its last q_len positions); seq_lens int32
    [S] counts every cached token including the queries.  ``max_q_len`` and
    ``max_seq_len`` (host ints) avoid device reads when given.
    """
    _check_caches(k_cache, v_cache)
    desc = cache_desc(k_cache)
    _require(q.dim() == 3 and q.shape[2] == desc.head_dim and q.dtype == k_cache.dtype and
             q.is_cuda and q.is_contiguous(), "q must be a contiguous CUDA [total_q, H_q, d] tensor")
    S = int(seq_lens.numel())
    _require(cu_seqlens_q.dtype == torch.int32 and cu_seqlens_q.numel() == S + 1 and
             cu_seqlens_q.is_cuda and cu_seqlens_q.is_contiguous(),
             "cu_seqlens_q must be a contiguous CUDA int32 [num_seqs + 1] tensor")
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and
             block_tables.shape[0] == S and block_tables.is_contiguous() and block_tables.is_cuda,
             "block_tables must be a contiguous CUDA int32 [num_seqs, max_blocks] tensor")
    _require(seq_lens.dtype == torch.int32 and seq_lens.is_cuda and seq_lens.is_contiguous(),
             "seq_lens must be a contiguous CUDA int32 [num_seqs] tensor")
    if scale is None:
        scale = desc.head_dim ** -0.5
    if max_q_len is None:
        max_q_len = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if S > 0 else 0
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if S > 0 else 0
    if out is None:
        out = torch.empty_like(q)
    _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous() and out.is_cuda,
             "out must match q")
    lib = _lib.load()
    _lib.check(lib.pkv_paged_prefill_attention(
        _ptr(q), _ptr(cu_seqlens_q), int(max_q_len), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(seq_lens), int(max_seq_len), S,
        int(q.shape[1]), desc, ctypes.c_float(float(scale)), _ptr(out), _err_ptr(err_flag),
        _stream(q.device)), "pkv_paged_prefill_attention")
    return out


def _check_fp8_pools(k_cache: torch.Tensor, v_cache: torch.Tensor) -> CacheDesc:
    _check_caches(k_cache, v_cache)
    desc = cache_desc(k_cache)
    _require(desc.dtype == _lib.PKV_FP8_E4M3,
             "8-bit pools hold E4M3 codes as torch.uint8 (or torch.float8_e4m3fn)")
    return desc


def kv_write_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: float, v_scale: float,
                 err_flag: Optional[torch.Tensor] = None) -> None:
    """Store k, v [T, H_kv, d] (fp16 / bf16) as E4M3 codes of x / scale at ``slot_mapping``."""
    desc = _check_fp8_pools(k_cache, v_cache)
    T = int(slot_mapping.numel())
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.is_cuda and
             slot_mapping.is_contiguous(), "slot_mapping must be a contiguous CUDA int64 tensor")
    _require(k.shape == (T, desc.num_kv_heads, desc.head_dim) and v.shape == k.shape,
             "k and v must be [num_tokens, num_kv_heads, head_dim]")
    _require(k.dtype in _16BIT and v.dtype == k.dtype, "k and v must be float16 or bfloat16")
    _require(k.is_contiguous() and v.is_contiguous() and k.is_cuda and v.is_cuda,
             "k and v must be contiguous CUDA tensors")
    lib = _lib.load()
    _lib.check(lib.pkv_kv_write_fp8(_ptr(k), _ptr(v), _16BIT[k.dtype], _ptr(slot_mapping), T,
                                    _ptr(k_cache), _ptr(v_cache), desc,
                                    ctypes.c_float(float(k_scale)), ctypes.c_float(float(v_scale)),
                                    _err_ptr(err_flag), _stream(k_cache.device)),
               "pkv_kv_write_fp8")


def paged_decode_attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_tables: torch.Tensor, seq_lens: torch.Tensor,
                               k_scale: float, v_scale: float, scale: Optional[float] = None,
                               out: Optional[torch.Tensor] = None, *,
                               max_seq_len: Optional[int] = None,
                               workspace: Optional[torch.Tensor] = None,
                               err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """paged_decode_attention over E4M3 pools read back as code * scale.

    q [S, H_q, d] float16 / bfloat16 (the output's type); other arguments as
    ``paged_decode_attention`` in automatic mode.
    """
    desc = _check_fp8_pools(k_cache, v_cache)
    _require(q.dim() == 3 and q.shape[2] == desc.head_dim, "q must be [num_seqs, num_q_heads, d]")
    _require(q.dtype in _16BIT and q.is_cuda and q.is_contiguous(),
             "q must be a contiguous CUDA float16 / bfloat16 tensor")
    S, Hq = int(q.shape[0]), int(q.shape[1])
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and
             block_tables.shape[0] == S and block_tables.is_contiguous() and block_tables.is_cuda,
             "block_tables must be a contiguous CUDA int32 [num_seqs, max_blocks] tensor")
    _require(seq_lens.dtype == torch.int32 and seq_lens.numel() == S and seq_lens.is_cuda and
             seq_lens.is_contiguous(), "seq_lens must be a contiguous CUDA int32 [num_seqs] tensor")
    if scale is None:
        scale = desc.head_dim ** -0.5
    if max_seq_len is None:
        max_seq_len = int(seq_lens.max().item()) if S > 0 else 0
    if out is None:
        out = torch.empty_like(q)
    _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous() and out.is_cuda,
             "out must match q")
    if workspace is None:
        need = decode_workspace_bytes(S, Hq, max_seq_len, desc.block_size, 0, desc.head_dim)
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    lib = _lib.load()
    _lib.check(lib.pkv_paged_decode_attention_fp8(
        _ptr(q), _16BIT[q.dtype], _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        int(block_tables.shape[1]), _ptr(seq_lens), int(max_seq_len), S, Hq, desc,
        ctypes.c_float(float(scale)), ctypes.c_float(float(k_scale)),
        ctypes.c_float(float(v_scale)), _ptr(workspace), ws_bytes, _ptr(out),
        _err_ptr(err_flag), _stream(q.device)), "pkv_paged_decode_attention_fp8")
    return out


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs: torch.Tensor,
                err_flag: Optional[torch.Tensor] = None) -> None:
    """Copy whole blocks src -> dst of both caches; pairs int64 [P, 2] on the device."""
    _check_caches(k_cache, v_cache)
    desc = cache_desc(k_cache)
    _require(src_dst_pairs.dtype == torch.int64 and src_dst_pairs.is_cuda and
             src_dst_pairs.is_contiguous() and (src_dst_pairs.numel() == 0 or
                                                src_dst_pairs.shape[-1] == 2),
             "src_dst_pairs must be a contiguous CUDA int64 [num_pairs, 2] tensor")
    P = int(src_dst_pairs.numel() // 2)
    lib = _lib.load()
    _lib.check(lib.pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), desc, _ptr(src_dst_pairs), P,
                                   _err_ptr(err_flag), _stream(k_cache.device)),
               "pkv_copy_blocks")


def _pairs(src_dst_pairs: torch.Tensor) -> int:
    _require(src_dst_pairs.dtype == torch.int64 and src_dst_pairs.is_cuda and
             src_dst_pairs.is_contiguous() and (src_dst_pairs.numel() == 0 or
                                                src_dst_pairs.shape[-1] == 2),
             "src_dst_pairs must be a contiguous CUDA int64 [num_pairs, 2] tensor")
    return int(src_dst_pairs.numel() // 2)


def swap_blocks(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor,
                dst_v: torch.Tensor, src_dst_pairs: torch.Tensor,
                err_flag: Optional[torch.Tensor] = None) -> None:
    """Copy whole blocks src -> dst between two pairs of pools (preemption by swap).

    Pools are CUDA tensors or page-locked host tensors (``pin_memory()``), all
    [blocks, H_kv, B, d] of one dtype; pairs int64 [P, 2] on the device.
    """
    for t in (src_k, src_v, dst_k, dst_v):
        _require(t.dim() == 4 and t.is_contiguous(), "pools must be contiguous 4-D tensors")
        _require(t.is_cuda or t.is_pinned(), "pools must be CUDA or page-locked host tensors")
    _require(src_k.shape == src_v.shape and dst_k.shape == dst_v.shape and
             src_k.shape[1:] == dst_k.shape[1:] and
             len({src_k.dtype, src_v.dtype, dst_k.dtype, dst_v.dtype}) == 1,
             "pools must agree in heads, block size, head size and dtype")
    desc = cache_desc(src_k)
    P = _pairs(src_dst_pairs)
    lib = _lib.load()
    _lib.check(lib.pkv_swap_blocks(_ptr(src_k), _ptr(src_v), int(src_k.shape[0]), _ptr(dst_k),
                                   _ptr(dst_v), int(dst_k.shape[0]), desc, _ptr(src_dst_pairs), P,
                                   _err_ptr(err_flag), _stream(src_dst_pairs.device)),
               "pkv_swap_blocks")


def _pointer_array(tensors):
    arr = (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _check_layers(k_caches, v_caches):
    _require(1 <= len(k_caches) == len(v_caches) <= _lib.MAX_LAYERS,
             f"between 1 and {_lib.MAX_LAYERS} layers, as many V caches as K caches")
    for kc, vc in zip(k_caches, v_caches):
        _check_caches(kc, vc)
        _require(kc.shape == k_caches[0].shape and kc.dtype == k_caches[0].dtype,
                 "every layer's caches must have the same shape and dtype")
    return cache_desc(k_caches[0])


def kv_write_layers(k, v, slot_mapping: torch.Tensor, k_caches, v_caches,
                    err_flag: Optional[torch.Tensor] = None) -> None:
    """kv_write for every layer in one launch: k[l], v[l] -> k_caches[l], v_caches[l]."""
    desc = _check_layers(k_caches, v_caches)
    _require(len(k) == len(v) == len(k_caches), "one k and v per layer")
    T = int(slot_mapping.numel())
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.is_cuda and
             slot_mapping.is_contiguous(), "slot_mapping must be a contiguous CUDA int64 tensor")
    for kt, vt in zip(k, v):
        _require(kt.shape == (T, desc.num_kv_heads, desc.head_dim) and vt.shape == kt.shape and
                 kt.dtype == k_caches[0].dtype and vt.dtype == kt.dtype and kt.is_cuda and
                 vt.is_cuda and kt.is_contiguous() and vt.is_contiguous(),
                 "k[l], v[l] must be contiguous CUDA [num_tokens, num_kv_heads, head_dim]")
    kp, _ka = _pointer_array(k)
    vp, _va = _pointer_array(v)
    kcp, _kca = _pointer_array(k_caches)
    vcp, _vca = _pointer_array(v_caches)
    lib = _lib.load()
    _lib.check(lib.pkv_kv_write_layers(kp, vp, _ptr(slot_mapping), T, kcp, vcp, len(k_caches),
                                       desc, _err_ptr(err_flag), _stream(slot_mapping.device)),
               "pkv_kv_write_layers")


def copy_blocks_layers(k_caches, v_caches, src_dst_pairs: torch.Tensor,
                       err_flag: Optional[torch.Tensor] = None) -> None:
    """copy_blocks for every layer in one launch (the same pairs in each layer)."""
    desc = _check_layers(k_caches, v_caches)
    P = _pairs(src_dst_pairs)
    kcp, _kca = _pointer_array(k_caches)
    vcp, _vca = _pointer_array(v_caches)
    lib = _lib.load()
    _lib.check(lib.pkv_copy_blocks_layers(kcp, vcp, len(k_caches), desc, _ptr(src_dst_pairs), P,
                                          _err_ptr(err_flag), _stream(src_dst_pairs.device)),
               "pkv_copy_blocks_layers")


class KVWritePlan:
    """kv_write validated and marshalled once for a fixed set of tensors.

    A serving loop writes each step's new keys / values through the same
    tensors (their contents change, their storage does not); ``run()`` then
    issues the C call directly, without re-checking shapes and dtypes.  The
    tensors must stay alive and in place while the plan is used."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                 k_cache: torch.Tensor, v_cache: torch.Tensor,
                 err_flag: Optional[torch.Tensor] = None) -> None:
        desc, T = _check_kv_write(k, v, slot_mapping, k_cache, v_cache)
        self._tensors = (k, v, slot_mapping, k_cache, v_cache, err_flag)  # kept alive
        self._device = k_cache.device
        self._args = (_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache), desc,
                      _err_ptr(err_flag))
        self._fn = _lib.load().pkv_kv_write

    def run(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        s = (stream or torch.cuda.current_stream(self._device)).cuda_stream
        _lib.check(self._fn(*self._args, s), "pkv_kv_write")


class DecodeAttentionPlan:
    """paged_decode_attention validated and marshalled once for a fixed set of
    tensors (q, caches, block tables, lengths, out, workspace), as KVWritePlan.
    ``max_seq_len`` is fixed by the plan: every later seq_lens must stay at or
    below it (a longer one sets PKV_DEVERR_BAD_SEQ_LEN and is skipped)."""

    def __init__(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor, *,
                 max_seq_len: int, num_kv_heads: Optional[int] = None,
                 scale: Optional[float] = None, partition_size: int = 0,
                 workspace: Optional[torch.Tensor] = None,
                 err_flag: Optional[torch.Tensor] = None) -> None:
        desc, S, Hq = _check_decode(q, k_cache, v_cache, block_tables, seq_lens, num_kv_heads)
        _require(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous() and
                 out.is_cuda, "out must match q")
        need = decode_workspace_bytes(S, Hq, max_seq_len, desc.block_size, partition_size,
                                      desc.head_dim)
        if workspace is None:
            workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device)
        _require(workspace.numel() * workspace.element_size() >= need, "workspace too small")
        if scale is None:
            scale = desc.head_dim ** -0.5
        self._tensors = (q, k_cache, v_cache, block_tables, seq_lens, out, workspace, err_flag)
        self._device = q.device
        self._args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                      int(block_tables.shape[1]), _ptr(seq_lens), int(max_seq_len), S, Hq, desc,
                      ctypes.c_float(float(scale)), int(partition_size), _ptr(workspace),
                      workspace.numel() * workspace.element_size(), _ptr(out), _err_ptr(err_flag))
        self._fn = _lib.load().pkv_paged_decode_attention
        self.out = out

    def run(self, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        s = (stream or torch.cuda.current_stream(self._device)).cuda_stream
        _lib.check(self._fn(*self._args, s), "pkv_paged_decode_attention")
        return self.out


__all__ = ["kv_write", "paged_decode_attention", "copy_blocks", "decode_workspace_bytes",
           "decode_partition_size", "cache_desc", "PKVError", "swap_blocks", "kv_write_layers",
           "copy_blocks_layers", "paged_prefill_attention", "kv_write_fp8",
           "paged_decode_attention_fp8", "KVWritePlan", "DecodeAttentionPlan"]
