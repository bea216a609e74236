"""Run one decode step on the GPU (through the C ABI) and on the oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import paged_kv_cache_242_gb300 as pkv
from paged_kv_cache_242_gb300.workloads import DecodeStep, bits

ATOL = 2e-3  # max absolute error where |ref| < 0.2
RTOL = 1e-2  # max relative error where |ref| >= 0.2
THREADS = os.cpu_count() or 1


def to_device(step: DecodeStep, device="cuda"):
    d = {
        "q": step.q.to(device), "k_new": step.k_new.to(device), "v_new": step.v_new.to(device),
        "slot_mapping": step.slot_mapping.to(device), "block_tables": step.block_tables.to(device),
        "seq_lens": step.seq_lens.to(device), "cow_pairs": step.cow_pairs.to(device),
    }
    if step.k_cache is not None:
        d["k_cache"] = step.k_cache.to(device)
        d["v_cache"] = step.v_cache.to(device)
    return d


def gpu_step(step: DecodeStep, dev: dict, partition_size: int = 0, err=None,
             max_seq_len=None) -> torch.Tensor:
    """copy_blocks (if any) -> kv_write -> paged_decode_attention on the GPU."""
    if step.cow_pairs.numel():
        pkv.copy_blocks(dev["k_cache"], dev["v_cache"], dev["cow_pairs"], err_flag=err)
    pkv.kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"], dev["v_cache"],
                 err_flag=err)
    return pkv.paged_decode_attention(
        dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["seq_lens"],
        step.num_kv_heads, step.scale,
        max_seq_len=step.max_seq_len if max_seq_len is None else max_seq_len,
        partition_size=partition_size, err_flag=err)


def oracle_step(step: DecodeStep, kc: np.ndarray, vc: np.ndarray, attend: bool = True):
    """The same step on host bit patterns; returns (out fp64 | None, kc, vc)."""
    if step.cow_pairs.numel():
        kc, vc, status = oracle.copy_blocks(kc, vc, step.cow_pairs.numpy())
        assert status == 0
    kc, vc, status = oracle.kv_write(bits(step.k_new), bits(step.v_new), step.slot_mapping.numpy(),
                                     kc, vc)
    assert status == 0
    out = None
    if attend:
        out = oracle.attention(bits(step.q), kc, vc, step.block_tables.numpy(),
                               step.seq_lens.numpy(), step.scale, step.dtype, num_threads=THREADS)
    return out, kc, vc


def attention_errors(gpu_out: torch.Tensor, ref: np.ndarray):
    got = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    big = np.abs(ref) >= 0.2
    max_abs = float(err.max()) if err.size else 0.0
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    ok = err <= np.maximum(ATOL, RTOL * np.abs(ref))
    return ok, max_abs, max_rel, got


def assert_attention_close(gpu_out: torch.Tensor, ref: np.ndarray, what: str = ""):
    ok, max_abs, max_rel, got = attention_errors(gpu_out, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU output"
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        detail = [(tuple(int(x) for x in b), float(got[tuple(b)]), float(ref[tuple(b)])) for b in bad]
        raise AssertionError(f"{what}: {int((~ok).sum())} elements out of tolerance; "
                             f"max_abs={max_abs:.3e} max_rel={max_rel:.3e}; first {detail}")
    return max_abs, max_rel


def cache_bits(t: torch.Tensor) -> np.ndarray:
    return bits(t)
