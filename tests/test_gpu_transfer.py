"""Block transfers: swap to and from page-locked host pools, multi-layer ops.

Bit-exact against the oracle's block transfer / slot write / block copy.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_242_gb300 as pkv
from paged_kv_cache_242_gb300 import _lib
from paged_kv_cache_242_gb300 import workloads as W
from paged_kv_cache_242_gb300.workloads import bits

from gpu_helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib.load()


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def test_swap_out_and_back_in():
    """Preempt two sequences: their blocks go to a host pool and come back elsewhere."""
    step = W.build_decode_step("swap", [300, 1200, 40, 2000, 777], 32, 8, 16, "bfloat16", seed=90,
                               pool_factor=2.0)
    dev = to_device(step)
    pkv.kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"], dev["v_cache"])
    before = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                        dev["block_tables"], dev["seq_lens"], 8, step.scale,
                                        max_seq_len=step.max_seq_len).clone()
    victims = [1, 3]
    nblocks = [(int(step.seq_lens[s]) + 15) // 16 for s in victims]
    src = torch.cat([step.block_tables[s, :n] for s, n in zip(victims, nblocks)]).to(torch.int64)
    host_k = torch.zeros((int(src.numel()) + 3,) + tuple(step.k_cache.shape[1:]),
                         dtype=step.k_cache.dtype).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    out_pairs = torch.stack([src, torch.arange(src.numel(), dtype=torch.int64)], dim=1)
    err = _err()
    pkv.swap_blocks(dev["k_cache"], dev["v_cache"], host_k, host_v, out_pairs.cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kc_dev, vc_dev = bits(dev["k_cache"].cpu()), bits(dev["v_cache"].cpu())
    ref_k, ref_v, status = oracle.transfer_blocks(kc_dev, vc_dev, bits(torch.zeros_like(host_k)),
                                                  bits(torch.zeros_like(host_v)), out_pairs.numpy())
    assert status == 0
    assert np.array_equal(bits(host_k), ref_k) and np.array_equal(bits(host_v), ref_v)

    # the victims' device blocks are freed and overwritten; swap in to other free blocks
    used = set(step.block_tables[:, :].flatten().tolist())
    free = [b for b in range(step.k_cache.shape[0]) if b not in used]
    assert len(free) >= src.numel()
    dev["k_cache"][src.cuda()] = 0
    dev["v_cache"][src.cuda()] = 0
    new_ids = torch.tensor(free[: src.numel()], dtype=torch.int64)
    in_pairs = torch.stack([torch.arange(src.numel(), dtype=torch.int64), new_ids], dim=1)
    pkv.swap_blocks(host_k, host_v, dev["k_cache"], dev["v_cache"], in_pairs.cuda(), err_flag=err)
    bt = step.block_tables.clone()
    pos = 0
    for s, n in zip(victims, nblocks):
        bt[s, :n] = new_ids[pos:pos + n].to(torch.int32)
        pos += n
    after = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], bt.cuda(),
                                       dev["seq_lens"], 8, step.scale,
                                       max_seq_len=step.max_seq_len)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(before, after)


def test_transfer_between_device_pools():
    a = W.build_decode_step("a", [500, 60], 8, 8, 32, "float16", seed=91)
    k_src, v_src = a.k_cache.cuda(), a.v_cache.cuda()
    k_dst = torch.full((7,) + tuple(a.k_cache.shape[1:]), 3.0, dtype=torch.float16, device="cuda")
    v_dst = torch.full_like(k_dst, -2.0)
    pairs = np.array([[0, 6], [5, 0], [9, 3]], dtype=np.int64)
    dst_before_k, dst_before_v = bits(k_dst.cpu()), bits(v_dst.cpu())
    pkv.swap_blocks(k_src, v_src, k_dst, v_dst, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    ref_k, ref_v, status = oracle.transfer_blocks(bits(a.k_cache), bits(a.v_cache), dst_before_k,
                                                  dst_before_v, pairs)
    assert status == 0
    assert np.array_equal(bits(k_dst.cpu()), ref_k) and np.array_equal(bits(v_dst.cpu()), ref_v)


def test_swap_rejects_pageable_host_memory_and_flags_bad_pairs():
    a = W.build_decode_step("a", [100], 8, 8, 16, "bfloat16", seed=92)
    k_dev, v_dev = a.k_cache.cuda(), a.v_cache.cuda()
    pageable = np.zeros(a.k_cache.numel(), dtype=np.uint16)
    lib = _lib.load()
    pairs = torch.tensor([[0, 0]], dtype=torch.int64, device="cuda")
    status = lib.pkv_swap_blocks(k_dev.data_ptr(), v_dev.data_ptr(), k_dev.shape[0],
                                 pageable.ctypes.data, pageable.ctypes.data, k_dev.shape[0],
                                 pkv.cache_desc(k_dev), pairs.data_ptr(), 1, None,
                                 torch.cuda.current_stream().cuda_stream)
    assert status == 1  # PKV_ERR_INVALID_ARG, nothing enqueued
    host_k = torch.zeros_like(a.k_cache).pin_memory()
    host_v = torch.zeros_like(a.v_cache).pin_memory()
    err = _err()
    bad = torch.tensor([[0, a.k_cache.shape[0]], [1, 1]], dtype=torch.int64, device="cuda")
    pkv.swap_blocks(k_dev, v_dev, host_k, host_v, bad, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == _lib.DEVERR_BAD_PAIR
    assert torch.equal(host_k[1], a.k_cache[1]) and not host_k[0].any()


@pytest.mark.parametrize("layers", [1, 3, 32])
def test_kv_write_and_copy_blocks_for_all_layers(layers):
    base = W.build_decode_step("layers", [50, 17, 300], 16, 4, 16, "bfloat16", seed=93)
    g = torch.Generator().manual_seed(94)
    kc = [torch.randn(base.k_cache.shape, generator=g).to(torch.bfloat16) for _ in range(layers)]
    vc = [torch.randn(base.k_cache.shape, generator=g).to(torch.bfloat16) for _ in range(layers)]
    kn = [torch.randn(base.k_new.shape, generator=g).to(torch.bfloat16) for _ in range(layers)]
    vn = [torch.randn(base.k_new.shape, generator=g).to(torch.bfloat16) for _ in range(layers)]
    kc_d = [t.cuda() for t in kc]
    vc_d = [t.cuda() for t in vc]
    slots = torch.cat([base.slot_mapping, torch.tensor([-1])]).cuda()  # one padding token
    kn_d = [torch.cat([t, t[:1]]).cuda() for t in kn]
    vn_d = [torch.cat([t, t[:1]]).cuda() for t in vn]
    err = _err()
    pkv.kv_write_layers(kn_d, vn_d, slots, kc_d, vc_d, err_flag=err)
    used = set(base.block_tables.flatten().tolist())
    spare = [b for b in range(base.k_cache.shape[0]) if b not in used][:2]
    pairs = np.array([[int(base.block_tables[0, 0]), spare[0]],
                      [int(base.block_tables[2, 1]), spare[1]]], dtype=np.int64)
    pkv.copy_blocks_layers(kc_d, vc_d, torch.from_numpy(pairs).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    slots_np = slots.cpu().numpy()
    for l in range(layers):
        rk, rv, st = oracle.kv_write(bits(kn_d[l].cpu()), bits(vn_d[l].cpu()), slots_np,
                                     bits(kc[l]), bits(vc[l]))
        assert st == 0
        rk, rv, st = oracle.copy_blocks(rk, rv, pairs)
        assert st == 0
        assert np.array_equal(bits(kc_d[l].cpu()), rk), f"layer {l} keys"
        assert np.array_equal(bits(vc_d[l].cpu()), rv), f"layer {l} values"
