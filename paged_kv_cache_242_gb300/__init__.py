"""GB300-native paged KV-cache decode path.

The KV cache lives in fixed-size, non-contiguous physical blocks reached
through per-sequence block tables.  Three hand-written sm_103a CUDA kernels,
behind the C ABI of ``libpkv.so`` (``include/pkv.h``), do the work:

* ``kv_write``               scatter new keys / values into block slots;
* ``paged_decode_attention`` exact one-query-token attention over the blocks
                             (MHA, GQA, MQA; split over long sequences with a
                             log-sum-exp merge);
* ``copy_blocks``            whole-block copies for copy-on-write;
* ``paged_prefill_attention`` causal attention of many query tokens per
                             sequence (the prompt phase) over the blocks;
* ``swap_blocks``            block copies between device and page-locked host
                             pools (preemption by swap);
* ``kv_write_layers`` / ``copy_blocks_layers``  the same for every layer of a
                             model in one launch;
* ``kv_write_fp8`` / ``paged_decode_attention_fp8``  the slot write and the
                             decode attention over 8-bit pools (E4M3 codes
                             with one scale per pool).

``block_manager`` is the host-side block table / refcount manager that
produces the kernels' inputs; ``workloads`` generates seeded synthetic
decode batches.
"""
from ._lib import PKVError  # noqa: F401
from .ops import (DecodeAttentionPlan, KVWritePlan, cache_desc,  # noqa: F401
                  copy_blocks, copy_blocks_layers,
                  decode_partition_size, decode_workspace_bytes, kv_write, kv_write_layers,
                  kv_write_fp8, paged_decode_attention, paged_decode_attention_fp8,
                  paged_prefill_attention, swap_blocks)

__all__ = ["kv_write", "paged_decode_attention", "copy_blocks", "decode_workspace_bytes",
           "decode_partition_size", "cache_desc", "PKVError", "swap_blocks", "kv_write_layers",
           "copy_blocks_layers", "paged_prefill_attention", "kv_write_fp8",
           "paged_decode_attention_fp8", "KVWritePlan", "DecodeAttentionPlan"]
