"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Cache writes and block copies must match bit for bit; attention must match
within max(2e-3, 1e-2 * |ref|) per element.  Every input is seeded and
synthetic (paged_kv_cache_242_gb300.workloads).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_242_gb300 as pkv
from paged_kv_cache_242_gb300 import _lib
from paged_kv_cache_242_gb300 import workloads as W
from paged_kv_cache_242_gb300.workloads import bits

from gpu_helpers import (assert_attention_close, gpu_step, oracle_step, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib.load()  # fail loudly if the library is missing


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _full_step_parity(step, partition_sizes=(0,)):
    kc0, vc0 = bits(step.k_cache), bits(step.v_cache)
    ref, kc_ref, vc_ref = oracle_step(step, kc0, vc0)
    results = []
    for part in partition_sizes:
        dev = to_device(step)
        err = _err()
        out = gpu_step(step, dev, partition_size=part, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        # cache writes: bit-exact over the whole pools
        assert np.array_equal(bits(dev["k_cache"].cpu()), kc_ref), "k_cache differs from oracle"
        assert np.array_equal(bits(dev["v_cache"].cpu()), vc_ref), "v_cache differs from oracle"
        results.append(assert_attention_close(out, ref, f"{step.name} P={part}"))
    return results


@pytest.mark.parametrize("block_size", [16, 32])
def test_tiny(block_size):
    step = W.tiny(block_size)
    assert step.seq_lens.tolist() == list(W.TINY_LENGTHS)
    _full_step_parity(step, partition_sizes=(0, block_size, 2 * block_size, 64, 128, 512))


def test_gqa_batch_full_size():
    _full_step_parity(W.gqa_batch(), partition_sizes=(0, 4112))


def test_opt13b_like_full_size():
    _full_step_parity(W.opt13b_like(), partition_sizes=(0,))


def test_long_context_full_size():
    _full_step_parity(W.long_context(), partition_sizes=(0, 1024))


@pytest.mark.parametrize("prompt_len", [1024, 1040])
def test_prefix_sharing_decode(prompt_len):
    """Parallel samples over shared prompts, 256 decode steps.

    Every step: copy-on-write copies, kv_write, attention.  The caches are
    compared with the oracle's replay bit for bit after every step; the
    attention output is compared at sampled steps.
    """
    sc = W.PrefixSharingScenario(prompt_len=prompt_len)
    kc, vc = bits(sc.k_cache), bits(sc.v_cache)
    k_dev, v_dev = sc.k_cache.cuda(), sc.v_cache.cuda()
    err = _err()
    checked = 0
    copies = 0
    for t in range(sc.decode_steps):
        step = sc.next_step()
        copies += step.cow_pairs.shape[0]
        dev = to_device(step)
        dev["k_cache"], dev["v_cache"] = k_dev, v_dev
        out = gpu_step(step, dev, err=err)
        attend = t in (0, 1, 31, 32, 129, sc.decode_steps - 1)
        ref, kc, vc = oracle_step(step, kc, vc, attend=attend)
        if attend:
            assert_attention_close(out, ref, f"prefix sharing step {t}")
            checked += 1
        if t in (0, 1, 32, sc.decode_steps - 1):
            torch.cuda.synchronize()
            assert np.array_equal(bits(k_dev.cpu()), kc) and np.array_equal(bits(v_dev.cpu()), vc)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and checked == 6
    expected_copies = 16 * 7 if prompt_len % 32 else 0
    assert copies == expected_copies


# --------------------------------------------------------------------------
# Edge cases
# --------------------------------------------------------------------------
def _custom(context, H_q, H_kv, B, dtype, seed, **kw):
    return W.build_decode_step("custom", context, H_q, H_kv, B, dtype, seed, **kw)


@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
def test_ragged_lengths_and_block_boundaries(B, dtype):
    # attended lengths 1, B-1, B, B+1, 2B, 3B-1, 513, 1000 (context = attended - 1)
    attended = [1, B - 1, B, B + 1, 2 * B, 3 * B - 1, 513, 1000]
    step = _custom([n - 1 for n in attended], 8, 2, B, dtype, seed=11)
    _full_step_parity(step, partition_sizes=(0, B, 3 * B, 512, 1024))


@pytest.mark.parametrize("B", [8, 16, 32, 64, 128])
def test_block_size_sweep(B):
    """Every supported block size, lengths around block and 16-token tile edges."""
    attended = [1, 7, 8, 9, 15, 16, 17, 31, 33, 127, 128, 129, 500, 3000]
    step = _custom([n - 1 for n in attended], 32, 8, B, "bfloat16", seed=60 + B)
    _full_step_parity(step, partition_sizes=(0,))
    if B in (8, 64):
        half = _custom([n - 1 for n in attended], 8, 8, B, "float16", seed=70 + B)
        _full_step_parity(half, partition_sizes=(0,))


def test_block_size_without_partition_kernel_is_unsupported():
    step = _custom([100, 200], 32, 8, 64, "bfloat16", seed=80)
    dev = to_device(step)
    with pytest.raises(pkv.PKVError) as e:
        pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["seq_lens"], 8, step.scale, max_seq_len=201,
                                   partition_size=128)
    assert e.value.status == 2


@pytest.mark.parametrize("B", [8, 16, 32])
def test_beam_search_decode(B):
    """Beams fork and fall out each step; copies, writes and attention match every step."""
    sc = W.BeamSearchScenario(block_size=B)
    kc, vc = bits(sc.k_cache), bits(sc.v_cache)
    k_dev, v_dev = sc.k_cache.cuda(), sc.v_cache.cuda()
    err = _err()
    for t in range(sc.decode_steps):
        step = sc.next_step()
        dev = to_device(step)
        dev["k_cache"], dev["v_cache"] = k_dev, v_dev
        out = gpu_step(step, dev, err=err)
        ref, kc, vc = oracle_step(step, kc, vc)
        assert_attention_close(out, ref, f"beam search step {t}")
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and sc.total_copies > 0
    assert np.array_equal(bits(k_dev.cpu()), kc) and np.array_equal(bits(v_dev.cpu()), vc)


@pytest.mark.parametrize("group", [1, 2, 4, 8, 16, 32, 64])
def test_group_sizes(group):
    H_kv = 2 if group <= 16 else 1
    step = _custom([100, 600, 33], group * H_kv, H_kv, 16, "bfloat16", seed=100 + group)
    _full_step_parity(step, partition_sizes=(0, 64))


def test_mqa_forty_heads():
    step = _custom([300, 1500], 40, 1, 16, "float16", seed=5)
    _full_step_parity(step, partition_sizes=(0, 256))


def test_single_token_is_value_row_exactly():
    """n = 1: p = 1 and l = 1, so the output is V_0 bit for bit."""
    step = _custom([0] * 6, 16, 4, 16, "bfloat16", seed=12)
    dev = to_device(step)
    out = gpu_step(step, dev)
    torch.cuda.synchronize()
    expect = step.v_new.repeat_interleave(4, dim=1)
    assert torch.equal(out.cpu(), expect)


def test_empty_sequences_give_zero():
    step = _custom([5, 40], 8, 8, 16, "float16", seed=13)
    step.seq_lens[0] = 0
    dev = to_device(step)
    out = gpu_step(step, dev)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[0]).item() == 0
    kc, vc = bits(step.k_cache), bits(step.v_cache)
    ref, _, _ = oracle_step(step, kc, vc)
    assert_attention_close(out, ref, "empty")


def test_unfilled_slots_hold_nan():
    """NaN in every slot no sequence owns must not reach any output."""
    step = _custom([3, 17, 40, 200], 8, 2, 16, "bfloat16", seed=14, unfilled=float("nan"))
    for part in (0, 32):
        _full_step_parity(step, partition_sizes=(part,))


def test_extreme_logits():
    """Scores near +-1e4: the running max keeps the softmax finite and one-hot."""
    step = _custom([63, 100], 4, 1, 16, "bfloat16", seed=15)
    step.q.zero_()
    step.q[:, :, 0] = 256.0
    step.k_cache.zero_()
    hot = []
    for s in range(2):
        t = 7 + 13 * s  # hot token
        hot.append(t)
        phys = int(step.block_tables[s, t // 16])
        step.k_cache[phys, 0, t % 16, 0] = 40.0
    kc, vc = bits(step.k_cache), bits(step.v_cache)
    ref, _, _ = oracle_step(step, kc, vc)
    dev = to_device(step)
    out = gpu_step(step, dev)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert_attention_close(out, ref, "extreme logits")
    for s, t in enumerate(hot):
        phys = int(step.block_tables[s, t // 16])
        assert torch.equal(out[s, 0].cpu(), step.v_cache[phys, 0, t % 16])


def test_paging_invariance_bitwise():
    """Moving blocks to other physical ids changes nothing, bit for bit."""
    step = _custom([100, 700, 1500], 32, 8, 16, "bfloat16", seed=16)
    dev = to_device(step)
    out_a = gpu_step(step, dev).clone()
    # permute the physical blocks and the tables consistently
    nb = step.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    dev["k_cache"] = dev["k_cache"][perm].contiguous()  # new block i = old block perm[i]
    dev["v_cache"] = dev["v_cache"][perm].contiguous()
    dev["block_tables"] = inv.to(torch.int32).cuda()[dev["block_tables"].long()].contiguous()
    out_b = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                       dev["block_tables"], dev["seq_lens"], 8, step.scale,
                                       max_seq_len=step.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)


def test_shared_prefix_equals_private_copy_bitwise():
    """Same bytes reached through shared blocks or private copies: same output."""
    step = _custom([600, 600], 32, 8, 16, "bfloat16", seed=17)
    dev = to_device(step)
    pkv.kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"], dev["v_cache"])
    bt = dev["block_tables"]
    q = dev["q"].clone()
    q[1] = q[0]
    # private copy: sequence 1's first 20 blocks get sequence 0's contents
    pairs = torch.stack([bt[0, :20], bt[1, :20]], dim=1).to(torch.int64).contiguous()
    pkv.copy_blocks(dev["k_cache"], dev["v_cache"], pairs)
    out_private = pkv.paged_decode_attention(q, dev["k_cache"], dev["v_cache"], bt,
                                             dev["seq_lens"], 8, step.scale, max_seq_len=601)
    # shared: sequence 1's first 20 logical blocks map onto sequence 0's blocks
    bt_shared = bt.clone()
    bt_shared[1, :20] = bt[0, :20]
    out_shared = pkv.paged_decode_attention(q, dev["k_cache"], dev["v_cache"], bt_shared,
                                            dev["seq_lens"], 8, step.scale, max_seq_len=601)
    torch.cuda.synchronize()
    assert torch.equal(out_private, out_shared)


@pytest.mark.parametrize("B", [16, 32])
def test_stream_many_short_and_empty_sequences(B):
    """Streaming split over many segments: warp ranges cut segments anywhere."""
    g = torch.Generator().manual_seed(30 + B)
    context = torch.randint(0, 300, (300,), generator=g).tolist()
    step = _custom(context, 16, 4, B, "bfloat16", seed=31)
    # a third of the sequences are empty (attended length 0)
    for s in range(0, 300, 3):
        step.seq_lens[s] = 0
    _full_step_parity(step, partition_sizes=(0, 64))


def test_stream_limit_and_partition_fallback():
    """4096 sequences stream; 4097 fall back to partitions; both match."""
    for S in (4096, 4097):
        g = torch.Generator().manual_seed(S)
        context = torch.randint(0, 40, (S,), generator=g).tolist()
        step = _custom(context, 8, 2, 16, "float16", seed=S)
        _full_step_parity(step, partition_sizes=(0,))


def test_stream_single_long_sequence_many_partials():
    """One 64k-token sequence over every warp: the merge combines ~1000 partials."""
    step = _custom([65535], 8, 1, 32, "bfloat16", seed=33, pool_factor=1.0)
    _full_step_parity(step, partition_sizes=(0,))


@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
def test_stream_wide_merge_with_empty_and_short_sequences(dtype):
    """Few long segments over many warps (one CTA merges each segment and query
    head), mixed with empty, one-token and one-tile sequences."""
    context = [20000, 0, 4, 0, 12000, 299, 15]
    step = _custom(context, 8, 2, 16, dtype, seed=34)
    step.seq_lens[3] = 0  # an empty sequence between two long ones
    _full_step_parity(step, partition_sizes=(0,))


def test_stream_workspace_reuse_with_leftover_contents():
    """A workspace full of unrelated bytes, reused across shapes, gives correct outputs."""
    a = _custom([3000, 900, 4000, 17], 32, 8, 16, "bfloat16", seed=40)
    b = _custom([100] * 40, 16, 4, 32, "float16", seed=41)
    need = max(pkv.decode_workspace_bytes(s.num_seqs, s.num_q_heads, s.max_seq_len, s.block_size)
               for s in (a, b))
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8,
                       generator=torch.Generator().manual_seed(5)).cuda()
    for step in (a, b, a, b):
        kc, vc = bits(step.k_cache), bits(step.v_cache)
        ref, _, _ = oracle_step(step, kc, vc)
        dev = to_device(step)
        pkv.kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                     dev["v_cache"])
        out = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                         dev["block_tables"], dev["seq_lens"], step.num_kv_heads,
                                         step.scale, max_seq_len=step.max_seq_len, workspace=ws)
        assert_attention_close(out, ref, "reused workspace")


def test_four_byte_aligned_q_and_out():
    """The 16-bit entry point accepts q and out aligned to only 4 bytes: views 4 bytes into
    larger buffers give the same bits as aligned tensors (cut segments included)."""
    step = _custom([2500, 3000, 700, 0, 1], 32, 8, 16, "bfloat16", seed=45)
    dev = to_device(step)
    pkv.kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"], dev["v_cache"])
    want = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                      dev["block_tables"], dev["seq_lens"], step.num_kv_heads,
                                      step.scale, max_seq_len=step.max_seq_len)
    n = dev["q"].numel()
    qbuf = torch.empty(n + 2, dtype=dev["q"].dtype, device="cuda")
    obuf = torch.full((n + 2,), float("nan"), dtype=dev["q"].dtype, device="cuda")
    q4 = qbuf[2:].view(dev["q"].shape)  # 4 bytes past a 256-byte boundary
    out4 = obuf[2:].view(dev["q"].shape)
    assert q4.data_ptr() % 8 == 4 and out4.data_ptr() % 8 == 4
    q4.copy_(dev["q"])
    pkv.paged_decode_attention(q4, dev["k_cache"], dev["v_cache"], dev["block_tables"],
                               dev["seq_lens"], step.num_kv_heads, step.scale, out4,
                               max_seq_len=step.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(out4, want)


def test_plans_match_the_calls():
    """KVWritePlan / DecodeAttentionPlan, validated once and run repeatedly on the same tensors
    whose contents change, give the same bits as the plain calls."""
    step = _custom([2500, 3000, 700, 1], 32, 8, 16, "bfloat16", seed=44)
    kc, vc = bits(step.k_cache), bits(step.v_cache)
    ref, _, _ = oracle_step(step, kc, vc)
    dev = to_device(step)
    plain = {k: v.clone() for k, v in dev.items()}
    pkv.kv_write(plain["k_new"], plain["v_new"], plain["slot_mapping"], plain["k_cache"],
                 plain["v_cache"])
    want = pkv.paged_decode_attention(plain["q"], plain["k_cache"], plain["v_cache"],
                                      plain["block_tables"], plain["seq_lens"], step.num_kv_heads,
                                      step.scale, max_seq_len=step.max_seq_len)
    out = torch.empty_like(dev["q"])
    write = pkv.KVWritePlan(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"],
                            dev["v_cache"])
    attend = pkv.DecodeAttentionPlan(dev["q"], dev["k_cache"], dev["v_cache"],
                                     dev["block_tables"], dev["seq_lens"], out,
                                     max_seq_len=step.max_seq_len, num_kv_heads=step.num_kv_heads,
                                     scale=step.scale)
    side = torch.cuda.Stream()
    for stream in (None, side):
        out.zero_()
        torch.cuda.synchronize()
        write.run(stream)
        got = attend.run(stream)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
        assert_attention_close(got, ref, "plan")
    # new contents in the same tensors: the plan sees them
    q2 = torch.randn(dev["q"].shape, generator=torch.Generator().manual_seed(3)).to(dev["q"].dtype)
    dev["q"].copy_(q2.cuda())
    want2 = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                       dev["block_tables"], dev["seq_lens"], step.num_kv_heads,
                                       step.scale, max_seq_len=step.max_seq_len)
    got2 = attend.run()
    torch.cuda.synchronize()
    assert torch.equal(got2, want2)


def test_cuda_graph_replay():
    """A captured attention call replays correctly."""
    step = _custom([2500, 3000, 700], 32, 8, 16, "bfloat16", seed=42)
    kc, vc = bits(step.k_cache), bits(step.v_cache)
    ref, _, _ = oracle_step(step, kc, vc)
    dev = to_device(step)
    pkv.kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"], dev["v_cache"])
    need = pkv.decode_workspace_bytes(step.num_seqs, step.num_q_heads, step.max_seq_len,
                                      step.block_size)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(dev["q"])

    def call():
        pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["seq_lens"], step.num_kv_heads, step.scale, out,
                                   max_seq_len=step.max_seq_len, workspace=ws)

    call()  # first call on this device before capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert_attention_close(out, ref, "graph replay")


def test_split_size_invariance():
    step = _custom([3000, 4000, 2500], 32, 8, 16, "bfloat16", seed=18)
    kc, vc = bits(step.k_cache), bits(step.v_cache)
    ref, _, _ = oracle_step(step, kc, vc)
    outs = []
    for part in (0, 16, 128, 512, 2048, 8192):
        dev = to_device(step)
        outs.append(gpu_step(step, dev, partition_size=part))
        assert_attention_close(outs[-1], ref, f"P={part}")


# --------------------------------------------------------------------------
# Device-side data errors: reported in the flag, never a fault
# --------------------------------------------------------------------------
def test_bad_block_id_sets_flag_and_is_skipped():
    step = _custom([40, 40], 8, 8, 16, "float16", seed=19)
    dev = to_device(step)
    bt = dev["block_tables"].clone()
    bt[1, 1] = step.k_cache.shape[0] + 5  # outside the pool
    err = _err()
    out = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], bt, dev["seq_lens"],
                                     8, step.scale, max_seq_len=41, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & _lib.DEVERR_BAD_BLOCK_ID
    assert torch.isfinite(out.float()).all()


def test_bad_slot_and_pair_set_flags():
    step = _custom([10, 10], 8, 8, 16, "float16", seed=20)
    dev = to_device(step)
    before = dev["k_cache"].clone()
    err = _err()
    bad = torch.tensor([step.k_cache.shape[0] * 16, -1], dtype=torch.int64, device="cuda")
    pkv.kv_write(dev["k_new"], dev["v_new"], bad, dev["k_cache"], dev["v_cache"], err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == _lib.DEVERR_BAD_SLOT
    assert torch.equal(before, dev["k_cache"])
    err.zero_()
    pairs = torch.tensor([[0, step.k_cache.shape[0]]], dtype=torch.int64, device="cuda")
    pkv.copy_blocks(dev["k_cache"], dev["v_cache"], pairs, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == _lib.DEVERR_BAD_PAIR
    assert torch.equal(before, dev["k_cache"])


def test_seq_len_beyond_max_sets_flag():
    step = _custom([100, 100], 8, 8, 16, "float16", seed=21)
    dev = to_device(step)
    err = _err()
    pkv.kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"], dev["v_cache"])
    out = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                     dev["seq_lens"], 8, step.scale, max_seq_len=64, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & _lib.DEVERR_BAD_SEQ_LEN
    assert torch.isfinite(out.float()).all()


def test_host_validation_statuses():
    step = _custom([10], 8, 8, 16, "bfloat16", seed=22)
    dev = to_device(step)
    with pytest.raises(pkv.PKVError) as e:
        pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["seq_lens"], 8, step.scale, max_seq_len=11,
                                   partition_size=24)  # not a multiple of the block size
    assert e.value.status == 1
    with pytest.raises(pkv.PKVError) as e:
        pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["seq_lens"], 8, step.scale, max_seq_len=10_000)
    assert e.value.status == 1  # beyond the block table's capacity
    kc64 = torch.zeros((4, 8, 16, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PKVError) as e:
        pkv.paged_decode_attention(torch.zeros((1, 8, 64), dtype=torch.bfloat16, device="cuda"),
                                   kc64, kc64, dev["block_tables"], dev["seq_lens"], 8, 0.1,
                                   max_seq_len=11)
    assert e.value.status == 2  # head_dim 64 is not implemented
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    long = _custom([2000], 8, 8, 16, "bfloat16", seed=24)
    dl = to_device(long)
    with pytest.raises(pkv.PKVError) as e:
        pkv.paged_decode_attention(dl["q"], dl["k_cache"], dl["v_cache"], dl["block_tables"],
                                   dl["seq_lens"], 8, long.scale, max_seq_len=2001,
                                   workspace=ws)
    assert e.value.status == 3
