"""Parity of the 8-bit (E4M3) pool path with the fp64 oracle, through the C ABI.

Codes written by kv_write_fp8 must match the oracle's bit for bit over the
whole pools; attention over the codes must match the oracle's attention over
code * scale within max(2e-3, 1e-2 * |ref|) per element.  The pools are made
by quantising the seeded 16-bit pools of the decode workloads slot by slot
(each side with its own quantiser), then one decode step writes each
sequence's new token and attends.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_242_gb300 as pkv
from paged_kv_cache_242_gb300 import _lib
from paged_kv_cache_242_gb300 import workloads as W
from paged_kv_cache_242_gb300.workloads import bits

from gpu_helpers import THREADS, assert_attention_close

pytestmark = pytest.mark.gpu

# Pool scales: N(0, 1) values map onto about [-4.8, 4.8] x 448 codes, so the
# rare larger magnitudes exercise saturation.
K_SCALE, V_SCALE = 0.0107, 0.0089


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib.load()


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def slot_rows(pool: torch.Tensor) -> torch.Tensor:
    """[NB, H, B, d] pool -> [NB * B, H, d] rows in slot order (slot = block * B + offset)."""
    nb, h, b, d = pool.shape
    return pool.permute(0, 2, 1, 3).reshape(nb * b, h, d).contiguous()


def quantised_pools(step, k_scale=K_SCALE, v_scale=V_SCALE):
    """Both sides' 8-bit pools of a step's 16-bit pools: (device kc, vc), (host kc, vc)."""
    shape = tuple(step.k_cache.shape)
    nslots = shape[0] * shape[2]
    slots = torch.arange(nslots, dtype=torch.int64)
    kd = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    vd = torch.zeros_like(kd)
    err = _err()
    pkv.kv_write_fp8(slot_rows(step.k_cache).cuda(), slot_rows(step.v_cache).cuda(), slots.cuda(),
                     kd, vd, k_scale, v_scale, err_flag=err)
    kh, vh, status = oracle.kv_write_fp8(bits(slot_rows(step.k_cache)), bits(slot_rows(step.v_cache)),
                                         step.dtype, slots.numpy(), np.zeros(shape, np.uint8),
                                         np.zeros(shape, np.uint8), k_scale, v_scale)
    torch.cuda.synchronize()
    assert status == 0 and int(err.item()) == 0
    assert np.array_equal(kd.cpu().numpy(), kh), "quantised key pool differs from the oracle"
    assert np.array_equal(vd.cpu().numpy(), vh), "quantised value pool differs from the oracle"
    return (kd, vd), (kh, vh)


def fp8_step_parity(step, k_scale=K_SCALE, v_scale=V_SCALE, q=None, tail_code=None, what=""):
    """kv_write_fp8 of the new tokens, then attention, on both sides."""
    (kd, vd), (kh, vh) = quantised_pools(step, k_scale, v_scale)
    q = step.q if q is None else q
    if tail_code is not None:  # unfilled slots of each sequence's last block
        B = step.block_size
        for s, n in enumerate(step.seq_lens.tolist()):
            if n % B:
                blk = int(step.block_tables[s, (n - 1) // B])
                kh[blk, :, n % B:] = tail_code
                vh[blk, :, n % B:] = tail_code
        kd.copy_(torch.from_numpy(kh))
        vd.copy_(torch.from_numpy(vh))
    err = _err()
    pkv.kv_write_fp8(step.k_new.cuda(), step.v_new.cuda(), step.slot_mapping.cuda(), kd, vd,
                     k_scale, v_scale, err_flag=err)
    out = pkv.paged_decode_attention_fp8(q.cuda(), kd, vd, step.block_tables.cuda(),
                                         step.seq_lens.cuda(), k_scale, v_scale, step.scale,
                                         max_seq_len=step.max_seq_len, err_flag=err)
    kh, vh, status = oracle.kv_write_fp8(bits(step.k_new), bits(step.v_new), step.dtype,
                                         step.slot_mapping.numpy(), kh, vh, k_scale, v_scale)
    assert status == 0
    ref = oracle.attention_fp8(bits(q), kh, vh, step.block_tables.numpy(), step.seq_lens.numpy(),
                               step.scale, k_scale, v_scale, step.dtype, num_threads=THREADS)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(kd.cpu().numpy(), kh) and np.array_equal(vd.cpu().numpy(), vh)
    return assert_attention_close(out, ref, what or step.name)


def _custom(lengths, hq, hkv, B, dtype, seed, **kw):
    return W.build_decode_step("custom", lengths, hq, hkv, B, dtype, seed, **kw)


# ---------------------------------------------------------------------------
# kv_write_fp8
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
def test_kv_write_fp8_codes_bitwise(dtype):
    """Random slots with padding, values spanning saturation and the subnormal codes."""
    g = torch.Generator().manual_seed(61)
    H, d, B, nb, T = 4, 128, 16, 40, 300
    scale = torch.exp(torch.empty(T, H, d).uniform_(-12.0, 7.0, generator=g))
    k = (torch.randn(T, H, d, generator=g) * scale).to(W.TORCH_DTYPES[dtype])
    v = (torch.randn(T, H, d, generator=g) * scale).to(W.TORCH_DTYPES[dtype])
    slots = torch.randperm(nb * B, generator=g)[:T].to(torch.int64)
    slots[::7] = -1  # padding tokens
    init = torch.randint(0, 256, (nb, H, B, d), generator=g, dtype=torch.int32).to(torch.uint8)
    kd, vd = init.clone().cuda(), init.clone().cuda()
    err = _err()
    pkv.kv_write_fp8(k.cuda(), v.cuda(), slots.cuda(), kd, vd, 0.37, 1.9, err_flag=err)
    kh, vh, status = oracle.kv_write_fp8(bits(k), bits(v), dtype, slots.numpy(), init.numpy(),
                                         init.numpy(), 0.37, 1.9)
    torch.cuda.synchronize()
    assert status == 0 and int(err.item()) == 0
    assert np.array_equal(kd.cpu().numpy(), kh) and np.array_equal(vd.cpu().numpy(), vh)
    codes = kh.reshape(-1)
    assert (codes & 0x7F == 0x7E).any() and ((codes & 0x78) == 0).any()  # saturated, subnormal


def test_kv_write_fp8_bad_slot_sets_flag_and_is_skipped():
    step = _custom([20, 33], 8, 2, 16, "bfloat16", seed=62)
    (kd, vd), (kh, vh) = quantised_pools(step)
    slots = step.slot_mapping.clone()
    slots[1] = kd.shape[0] * kd.shape[2]  # one past the pool
    err = _err()
    pkv.kv_write_fp8(step.k_new.cuda(), step.v_new.cuda(), slots.cuda(), kd, vd, K_SCALE, V_SCALE,
                     err_flag=err)
    kh, vh, status = oracle.kv_write_fp8(bits(step.k_new), bits(step.v_new), "bfloat16",
                                         slots.numpy(), kh, vh, K_SCALE, V_SCALE)
    torch.cuda.synchronize()
    assert status != 0 and int(err.item()) == _lib.DEVERR_BAD_SLOT
    assert np.array_equal(kd.cpu().numpy(), kh) and np.array_equal(vd.cpu().numpy(), vh)


# ---------------------------------------------------------------------------
# attention over 8-bit pools
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
def test_tiny_lengths_all_block_sizes(B, dtype):
    step = _custom(W.TINY_LENGTHS, 8, 8, B, dtype, seed=63)
    fp8_step_parity(step, what=f"tiny B={B} {dtype}")


def test_gqa_batch_full_size():
    fp8_step_parity(W.gqa_batch(), what="gqa batch fp8")


def test_long_sequences_cut_across_warps():
    """Two long sequences: every segment is split over many warps and merged."""
    step = _custom([20000, 9000], 32, 8, 16, "bfloat16", seed=64)
    fp8_step_parity(step, what="long fp8")


def test_long_sequences_with_empty_ones_cut_across_warps():
    """Few long segments over many warps, with an empty and a one-token sequence."""
    step = _custom([15000, 0, 1, 7000], 16, 2, 16, "float16", seed=74)
    step.seq_lens[1] = 0  # nothing attended for sequence 1
    fp8_step_parity(step, what="long and empty")


@pytest.mark.parametrize("hq,hkv", [(16, 1), (16, 16), (32, 16), (64, 8), (48, 6)])
def test_group_sizes(hq, hkv):
    step = _custom([1, 15, 16, 17, 300, 1000], hq, hkv, 16, "bfloat16", seed=65 + hq + hkv)
    fp8_step_parity(step, what=f"Hq={hq} Hkv={hkv}")


def test_nan_codes_in_unfilled_tail_slots():
    step = _custom([3, 17, 40, 201], 8, 2, 16, "bfloat16", seed=66, unfilled=float("nan"))
    fp8_step_parity(step, tail_code=0x7F, what="NaN tail")


def test_empty_sequences_and_single_tokens():
    step = _custom([0, 0, 5, 40], 8, 8, 16, "float16", seed=67)
    step.seq_lens[0] = 0  # nothing attended at all for sequence 0
    fp8_step_parity(step, what="empty")


@pytest.mark.parametrize("factor", [1e4, 3e-7, 2e5])
def test_bfloat16_query_magnitudes(factor):
    """Huge, tiny and beyond-binary16 query rows: the power-of-two row scaling."""
    step = _custom([50, 300, 700], 32, 8, 16, "bfloat16", seed=68)
    q = (step.q.float() * factor).to(torch.bfloat16)
    q[1, 3] = 0  # an all-zero row
    fp8_step_parity(step, q=q, what=f"q x {factor}")


def test_fp16_query_extreme_logits():
    step = _custom([50, 300], 8, 8, 16, "float16", seed=69)
    q = (step.q.float() * 300).to(torch.float16)  # scores of order 1e3: near one-hot
    fp8_step_parity(step, q=q, what="fp16 extreme")


@pytest.mark.parametrize("scales", [(1.0, 1.0), (0.25, 4.0), (3.3e-3, 0.0371)])
def test_pool_scales(scales):
    step = _custom([33, 129, 500], 16, 4, 32, "bfloat16", seed=70)
    fp8_step_parity(step, k_scale=scales[0], v_scale=scales[1], what=f"scales {scales}")


def test_beyond_streaming_limits_is_unsupported():
    step = _custom([10, 20], 8 * 17, 8, 16, "bfloat16", seed=71)
    (kd, vd), _ = quantised_pools(step)
    with pytest.raises(pkv.PKVError) as exc:
        pkv.paged_decode_attention_fp8(step.q.cuda(), kd, vd, step.block_tables.cuda(),
                                       step.seq_lens.cuda(), K_SCALE, V_SCALE,
                                       max_seq_len=step.max_seq_len)
    assert exc.value.status == 2


# ---------------------------------------------------------------------------
# block copies on 8-bit pools
# ---------------------------------------------------------------------------
def test_copy_and_swap_blocks_on_fp8_pools():
    g = torch.Generator().manual_seed(72)
    nb, H, B, d = 24, 4, 16, 128
    kc = torch.randint(0, 256, (nb, H, B, d), generator=g, dtype=torch.int32).to(torch.uint8)
    vc = torch.randint(0, 256, (nb, H, B, d), generator=g, dtype=torch.int32).to(torch.uint8)
    pairs = torch.tensor([[3, 10], [5, 0], [7, 23]], dtype=torch.int64)
    kd, vd = kc.cuda(), vc.cuda()
    pkv.copy_blocks(kd, vd, pairs.cuda())
    u16 = lambda t: t.numpy().view(np.uint16)  # byte copies: view pairs of codes as 16-bit words
    kh, vh, status = oracle.copy_blocks(u16(kc), u16(vc), pairs.numpy())
    torch.cuda.synchronize()
    assert status == 0
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), kh)
    assert np.array_equal(vd.cpu().numpy().view(np.uint16), vh)
    # swap out to page-locked host pools and back
    hk = torch.zeros((8, H, B, d), dtype=torch.uint8).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = torch.tensor([[10, 0], [23, 7]], dtype=torch.int64).cuda()
    pkv.swap_blocks(kd, vd, hk, hv, out_pairs)
    torch.cuda.synchronize()
    assert torch.equal(hk[0], kd[10].cpu()) and torch.equal(hv[7], vd[23].cpu())
    back = torch.tensor([[7, 1]], dtype=torch.int64).cuda()
    pkv.swap_blocks(hk, hv, kd, vd, back)
    torch.cuda.synchronize()
    assert torch.equal(kd[1].cpu(), kd[23].cpu()) and torch.equal(vd[1].cpu(), vd[23].cpu())
