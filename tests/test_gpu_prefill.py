"""Paged prefill attention on the GPU against the fp64 oracle."""
import pytest
import torch

import oracle
import paged_kv_cache_242_gb300 as pkv
from paged_kv_cache_242_gb300 import _lib
from paged_kv_cache_242_gb300 import workloads as W
from paged_kv_cache_242_gb300.workloads import bits

from gpu_helpers import THREADS, assert_attention_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _lib.load()


def _run(step, err=None):
    dev = {k: getattr(step, k).cuda() for k in
           ("q", "cu_q", "k_new", "v_new", "slot_mapping", "block_tables", "seq_lens",
            "k_cache", "v_cache")}
    pkv.kv_write(dev["k_new"], dev["v_new"], dev["slot_mapping"], dev["k_cache"], dev["v_cache"],
                 err_flag=err)
    out = pkv.paged_prefill_attention(dev["q"], dev["cu_q"], dev["k_cache"], dev["v_cache"],
                                      dev["block_tables"], dev["seq_lens"], step.scale,
                                      max_q_len=step.max_q_len, max_seq_len=step.max_seq_len,
                                      err_flag=err)
    return out, dev


def _reference(step):
    kc, vc, status = oracle.kv_write(bits(step.k_new), bits(step.v_new), step.slot_mapping.numpy(),
                                     bits(step.k_cache), bits(step.v_cache))
    assert status == 0
    return oracle.prefill(bits(step.q), step.cu_q.numpy(), kc, vc, step.block_tables.numpy(),
                          step.seq_lens.numpy(), step.scale, step.dtype, num_threads=THREADS)


@pytest.mark.parametrize("B", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("heads", [(8, 8), (32, 8), (16, 2), (24, 8), (20, 4)])
def test_prefill_ragged(B, heads):
    """Contexts and prompt lengths around 16-token sub-tiles and 64- / 128-key tiles; groups of
    1, 4 and 8 query heads run on the tensor-core kernel, groups of 3 and 5 on the warp-MMA one."""
    H_q, H_kv = heads
    ctx = [0, 5, 16, 100, 0, 37]
    ql = [1, 7, 16, 65, 200, 64]
    step = W.build_prefill_step("ragged", ctx, ql, H_q, H_kv, B, "bfloat16", seed=100 + B + H_q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = _run(step, err)
    ref = _reference(step)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, ref, f"prefill B={B} heads={heads}")


def test_prefill_many_items_per_cta():
    """More (256-row item, KV head, sequence) work items than CTAs: the grid is persistent, so
    each CTA carries its pipeline across many items.  The second Q tile of a sequence's last
    item is empty, partly filled or full; some sequences have no queries or nothing at all."""
    g = torch.Generator().manual_seed(12)
    S = 180
    ctx = torch.randint(0, 120, (S,), generator=g).tolist()
    ql = torch.randint(0, 81, (S,), generator=g).tolist()
    ctx[3], ql[3] = 0, 0  # an empty sequence
    ql[4] = 0  # cached context, no queries
    ql[5], ql[6], ql[7], ql[8] = 32, 33, 64, 65  # 128 / 132 / 256 / 260 rows at 4 heads a group
    step = W.build_prefill_step("many", ctx, ql, 32, 8, 16, "bfloat16", seed=12)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = _run(step, err)
    ref = _reference(step)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, ref, "prefill many items")


@pytest.mark.parametrize("B", [16, 128])
def test_prefill_fp16_ragged(B):
    """fp16 inputs: the tensor-core kernel keeps P as one binary16 value (no low part)."""
    step = W.build_prefill_step("ragged16", [0, 5, 16, 100, 0, 37, 600], [1, 7, 16, 65, 200, 64, 700],
                                32, 8, B, "float16", seed=200 + B)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = _run(step, err)
    ref = _reference(step)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, ref, f"prefill fp16 B={B}")


def test_prefill_mixed_new_tokens_and_prompts():
    """One call mixing 250 sequences that add one token after a cached context with three long
    prompts: most of the persistent grid's work list is empty items, skipped from the
    per-sequence cache in shared memory."""
    g = torch.Generator().manual_seed(13)
    S = 253
    ctx = torch.randint(100, 600, (S,), generator=g).tolist()
    ql = [1] * S
    for i, x in ((7, 1500), (100, 700), (200, 1100)):
        ctx[i], ql[i] = 0, x
    step = W.build_prefill_step("mixed", ctx, ql, 32, 8, 16, "bfloat16", seed=13)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = _run(step, err)
    ref = _reference(step)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, ref, "prefill mixed")


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
def test_prefill_growing_scores(dtype):
    """Keys whose norms grow along the prompt, so later key tiles score far above earlier ones
    (log2 score ranges of ~100): the running max must move, O and the sums must be rescaled,
    and no weight may overflow the 16-bit type."""
    step = W.build_prefill_step("grow", [0, 0, 300], [700, 130, 400], 32, 8, 16, dtype, seed=14)
    T = step.k_new.shape[0]
    growth = (1.0 + torch.arange(T, dtype=torch.float32) / 8.0).view(T, 1, 1)
    step.k_new.copy_((step.k_new.float() * growth).to(step.k_new.dtype))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = _run(step, err)
    ref = _reference(step)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(out.float()).all()
    assert_attention_close(out, ref, f"prefill growing scores {dtype}")


@pytest.mark.parametrize("heads", [(64, 1), (128, 2)])
def test_prefill_large_groups(heads):
    """Groups of 64 query heads per KV head, the largest supported: a 128-row Q tile is two
    tokens.  A group of 128 is refused with PKV_ERR_UNSUPPORTED."""
    H_q, H_kv = heads
    too_big = W.build_prefill_step("g128", [0], [3], 128, 1, 16, "bfloat16", seed=15)
    with pytest.raises(pkv.PKVError) as e:
        _run(too_big)
    assert e.value.status == 2
    step = W.build_prefill_step("groups", [0, 37, 200], [41, 9, 30], H_q, H_kv, 16, "bfloat16",
                                seed=15 + H_q + H_kv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = _run(step, err)
    ref = _reference(step)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attention_close(out, ref, f"prefill heads={heads}")


def test_prefill_fp16_and_mqa():
    step = W.build_prefill_step("fp16", [300, 0], [129, 255], 8, 1, 16, "float16", seed=7)
    out, _ = _run(step)
    assert_attention_close(out, _reference(step), "prefill fp16 MQA")


def test_prefill_larger_batch():
    step = W.build_prefill_step("larger", [512, 0, 1000, 64], [512, 700, 300, 1024], 32, 8, 16,
                                "bfloat16", seed=8)
    out, _ = _run(step)
    assert_attention_close(out, _reference(step), "prefill larger")


def test_prefill_single_query_equals_decode():
    """One query per sequence: prefill and decode attention agree with the oracle."""
    step = W.build_prefill_step("one", [10, 400, 3000], [1, 1, 1], 32, 8, 16, "bfloat16", seed=9)
    out, dev = _run(step)
    dec = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                     dev["seq_lens"], 8, step.scale, max_seq_len=step.max_seq_len)
    torch.cuda.synchronize()
    ref = _reference(step)
    assert_attention_close(out, ref, "prefill q_len 1")
    assert_attention_close(dec, ref, "decode")


def test_prefill_bad_lengths_set_flag():
    step = W.build_prefill_step("bad", [10, 10], [5, 5], 8, 8, 16, "bfloat16", seed=10)
    dev = {k: getattr(step, k).cuda() for k in
           ("q", "cu_q", "block_tables", "seq_lens", "k_cache", "v_cache")}
    dev["seq_lens"][1] = 3  # fewer cached tokens than queries
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(dev["q"])
    pkv.paged_prefill_attention(dev["q"], dev["cu_q"], dev["k_cache"], dev["v_cache"],
                                dev["block_tables"], dev["seq_lens"], step.scale, out,
                                max_q_len=5, max_seq_len=15, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & _lib.DEVERR_BAD_SEQ_LEN
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("B", [16, 128])
def test_prefill_nan_in_unfilled_slots(B):
    """NaN in every slot no sequence fills must not reach any output (the last key tile
    of a sequence reaches past its end)."""
    step = W.build_prefill_step("nan", [3, 0, 130], [40, 77, 5], 32, 8, B, "bfloat16", seed=11)
    filled = torch.zeros(step.k_cache.shape[0] * B, dtype=torch.bool)
    for s, n in enumerate(step.seq_lens.tolist()):
        for t in range(n):
            filled[int(step.block_tables[s, t // B]) * B + t % B] = True
    nb, hkv, _, d = step.k_cache.shape
    for pool in (step.k_cache, step.v_cache):
        rows = pool.permute(0, 2, 1, 3).reshape(nb * B, hkv, d)
        rows[~filled] = float("nan")
        pool.copy_(rows.reshape(nb, B, hkv, d).permute(0, 2, 1, 3))
    out, _ = _run(step)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert_attention_close(out, _reference(step), f"prefill NaN-filled B={B}")
