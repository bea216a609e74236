"""The fixed-scratch attention entry point agrees with the workspace one.

pkv_paged_decode_attention_fixed_scratch serves callers that may not
allocate device memory themselves: their host application owns every GPU
allocation (a server handing plugins pre-registered buffers, a runtime with
its own pool and budget), and an extra cudaMalloc could fail under that
budget, fragment the pool or synchronise the device mid-schedule.  Instead
of a caller workspace it uses a fixed array inside the library.

The test calls it through the C ABI twice in a row, on two different
split-mode batches (so the second call runs over scratch the first one
left behind), and compares each output with pkv_paged_decode_attention on
its own workspace, within the tolerance of the parity tests.  It also
checks that a request larger than the fixed scratch is refused.  The file
is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_242_gb300 as pkv
from paged_kv_cache_242_gb300 import _lib
from paged_kv_cache_242_gb300 import workloads as W

pytestmark = pytest.mark.gpu

FIXED_SCRATCH_BYTES = 16 << 20  # PKV_FIXED_SCRATCH_BYTES in include/pkv.h


def _entry_point():
    lib = _lib.load()
    fn = lib.pkv_paged_decode_attention_fixed_scratch
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, _lib.CacheDesc, ctypes.c_float, i32,
                   vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _call_fixed(fn, step, dev, out, err, partition_size=0, max_seq_len=None):
    desc = pkv.cache_desc(dev["k_cache"])
    return fn(dev["q"].data_ptr(), dev["k_cache"].data_ptr(), dev["v_cache"].data_ptr(),
              dev["block_tables"].data_ptr(), int(dev["block_tables"].shape[1]),
              dev["seq_lens"].data_ptr(),
              step.max_seq_len if max_seq_len is None else max_seq_len, step.num_seqs,
              step.num_q_heads, desc, ctypes.c_float(step.scale), partition_size,
              out.data_ptr(), err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _device(step):
    return {"q": step.q.cuda(), "k_cache": step.k_cache.cuda(), "v_cache": step.v_cache.cuda(),
            "block_tables": step.block_tables.cuda(), "seq_lens": step.seq_lens.cuda()}


def _assert_close(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g))
    assert np.all(np.abs(g - r) <= np.maximum(2e-3, 1e-2 * np.abs(r)))


def test_fixed_scratch_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fn = _entry_point()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    batches = [W.gqa_batch(), W.long_context()]
    for step in batches:
        need = pkv.decode_workspace_bytes(step.num_seqs, step.num_q_heads, step.max_seq_len,
                                          step.block_size)
        assert 0 < need <= FIXED_SCRATCH_BYTES  # both calls run in split mode
    for step in batches:  # two calls in a row
        dev = _device(step)
        ref = pkv.paged_decode_attention(dev["q"], dev["k_cache"], dev["v_cache"],
                                         dev["block_tables"], dev["seq_lens"], step.num_kv_heads,
                                         step.scale, max_seq_len=step.max_seq_len)
        out = torch.full_like(dev["q"], float("nan"))
        status = _call_fixed(fn, step, dev, out, err)
        torch.cuda.synchronize()
        assert status == 0, _lib.STATUS_NAMES.get(status)
        assert int(err.item()) == 0
        _assert_close(out, ref)
        del dev


def test_fixed_scratch_refuses_oversized_requests():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fn = _entry_point()
    S, Hq, max_len, B = 4096, 32, 65536, 16
    assert pkv.decode_workspace_bytes(S, Hq, max_len, B) > FIXED_SCRATCH_BYTES
    # every buffer is sized for the claimed request (all lengths zero), so the
    # call stays in bounds even if it were enqueued
    q = torch.zeros((S, Hq, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    cache = torch.zeros((4, 8, B, 128), dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros((S, max_len // B), dtype=torch.int32, device="cuda")
    lens = torch.zeros(S, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = fn(q.data_ptr(), cache.data_ptr(), cache.data_ptr(), tables.data_ptr(),
                max_len // B, lens.data_ptr(), max_len, S, Hq, pkv.cache_desc(cache),
                ctypes.c_float(0.1), 0, out.data_ptr(), err.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert status == 3  # PKV_ERR_WORKSPACE_TOO_SMALL
    assert int(err.item()) == 0
