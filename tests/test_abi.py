"""The C ABI library loads and exports every symbol include/pkv.h declares.

No compute runs here: only host-side queries and argument validation, which
return before any CUDA call.
"""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_242_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for expected in ("pkv_kv_write", "pkv_paged_decode_attention", "pkv_copy_blocks",
                     "pkv_decode_workspace_bytes", "pkv_status_string"):
        assert expected in names


def test_every_declared_symbol_is_exported(lib):
    exported = subprocess.run(["nm", "-D", "--defined-only", build.LIBRARY], capture_output=True,
                              text=True, check=True).stdout
    symbols = {line.split()[-1] for line in exported.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in symbols, f"{name} declared in pkv.h but not exported"
        assert hasattr(lib, name)
    # nothing but the pkv_ API leaks out of the library
    assert all(s.startswith("pkv_") for s in symbols), sorted(s for s in symbols if not s.startswith("pkv_"))


def test_status_strings(lib):
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(3) == b"PKV_ERR_WORKSPACE_TOO_SMALL"
    assert lib.pkv_abi_version() == 101


def test_partition_and_workspace_queries(lib):
    assert lib.pkv_decode_partition_size(4097, 16, 0) == 512
    assert lib.pkv_decode_partition_size(300, 16, 0) == 304  # single pass, rounded to blocks
    assert lib.pkv_decode_partition_size(300, 16, 64) == 64
    assert lib.pkv_decode_partition_size(300, 16, 24) == -1  # not a multiple of the block size
    assert lib.pkv_decode_partition_size(32768, 16, 1 << 20) == 32768
    # explicit partitions: 64 seqs x 32 heads x ceil(4097/512)=9 partitions x (128 + 2) floats
    assert lib.pkv_decode_workspace_bytes(64, 32, 128, 4097, 16, 512) == 64 * 32 * 9 * 130 * 4
    assert lib.pkv_decode_workspace_bytes(5, 8, 128, 511, 16, 512) == 0  # single pass
    # automatic mode: covers the partition layout and at least one statistics
    # row of 130 floats per (sequence, query head) for the streaming layout
    auto = lib.pkv_decode_workspace_bytes(64, 32, 128, 4097, 16, 0)
    assert auto >= 64 * 32 * 9 * 130 * 4
    assert auto >= 64 * 32 * 130 * 4 + 65 * 4
    assert lib.pkv_decode_workspace_bytes(5, 8, 128, 511, 16, 0) > 0
    # beyond 4096 sequences automatic mode falls back to partitions
    assert lib.pkv_decode_workspace_bytes(5000, 8, 128, 511, 16, 0) == 0


def _desc(**kw):
    d = dict(num_blocks=64, num_kv_heads=8, block_size=16, head_dim=128, dtype=1)
    d.update(kw)
    return _lib.CacheDesc(**d)


def test_host_validation_without_launch(lib):
    """Invalid arguments are rejected before any CUDA call."""
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    null = None
    # kv_write: null pointers with tokens present
    assert lib.pkv_kv_write(null, fake, fake, 4, fake, fake, _desc(), null, null) == 1
    # kv_write: zero tokens is a no-op that succeeds without touching anything
    assert lib.pkv_kv_write(null, null, null, 0, null, null, _desc(), null, null) == 0
    # bad cache geometry
    assert lib.pkv_kv_write(fake, fake, fake, 1, fake, fake, _desc(num_blocks=0), null, null) == 1
    assert lib.pkv_kv_write(fake, fake, fake, 1, fake, fake, _desc(dtype=7), null, null) == 1
    assert lib.pkv_kv_write(fake, fake, fake, 1, fake, fake, _desc(head_dim=12), null, null) == 2
    # attention: heads not divisible, unsupported head dim / block size, capacity
    args = lambda **kw: dict(dict(q=fake, kc=fake, vc=fake, bt=fake, mb=4, sl=fake, msl=64, S=2,
                                  Hq=32, desc=_desc(), scale=0.1, part=0, ws=null, wsb=0,
                                  out=fake), **kw)

    def attn(**kw):
        a = args(**kw)
        return lib.pkv_paged_decode_attention(a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["sl"],
                                              a["msl"], a["S"], a["Hq"], a["desc"],
                                              ctypes.c_float(a["scale"]), a["part"], a["ws"],
                                              a["wsb"], a["out"], null, null)

    assert attn(Hq=30) == 1
    assert attn(desc=_desc(head_dim=64)) == 2
    assert attn(desc=_desc(block_size=24), msl=48) == 2  # not a supported block size
    assert attn(desc=_desc(block_size=64), mb=1, part=64) == 2  # partitions need 16 or 32
    assert attn(desc=_desc(block_size=8), mb=8) == 3  # streaming takes 8: needs a workspace
    assert attn(msl=65) == 1  # beyond 4 blocks x 16 slots
    assert attn(part=24) == 1
    assert attn(q=null) == 1
    assert attn(S=0) == 0
    assert attn(scale=float("nan")) == 1
    assert attn(Hq=8 * 65) == 2  # group of 65 query heads per KV head
    # split mode without a workspace
    assert attn(mb=300, msl=4097) == 3
    # swap_blocks and the layer variants: argument checks come before any CUDA call
    assert lib.pkv_swap_blocks(null, fake, 4, fake, fake, 4, _desc(), fake, 1, null, null) == 1
    assert lib.pkv_swap_blocks(fake, fake, 0, fake, fake, 4, _desc(), fake, 1, null, null) == 1
    assert lib.pkv_swap_blocks(fake, fake, 4, fake, fake, 4, _desc(), fake, 0, null, null) == 0
    arr = (ctypes.c_void_p * 2)(0x10000, 0x20000)
    parr = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    assert lib.pkv_kv_write_layers(parr, parr, fake, 1, parr, parr, 0, _desc(), null, null) == 1
    assert lib.pkv_kv_write_layers(parr, parr, fake, 1, parr, parr, 129, _desc(), null, null) == 1
    assert lib.pkv_kv_write_layers(parr, parr, fake, 0, parr, parr, 2, _desc(), null, null) == 0
    assert lib.pkv_copy_blocks_layers(parr, parr, 2, _desc(), null, 3, null, null) == 1
    assert lib.pkv_copy_blocks_layers(parr, parr, 2, _desc(), fake, 0, null, null) == 0
    # prefill
    def prefill(**kw):
        a = dict(q=fake, cu=fake, mq=4, kc=fake, vc=fake, bt=fake, mb=4, sl=fake, msl=64, S=2,
                 Hq=32, desc=_desc(), scale=0.1, out=fake)
        a.update(kw)
        return lib.pkv_paged_prefill_attention(a["q"], a["cu"], a["mq"], a["kc"], a["vc"], a["bt"],
                                               a["mb"], a["sl"], a["msl"], a["S"], a["Hq"],
                                               a["desc"], ctypes.c_float(a["scale"]), a["out"],
                                               null, null)
    assert prefill(cu=null) == 1
    assert prefill(Hq=30) == 1
    assert prefill(mq=-1) == 1
    assert prefill(msl=65) == 1
    assert prefill(desc=_desc(head_dim=64)) == 2
    assert prefill(desc=_desc(block_size=24), msl=48) == 2
    assert prefill(S=0) == 0 and prefill(mq=0) == 0
    # q and out rows move as 16-byte vectors: 4-byte aligned is refused
    assert prefill(q=ctypes.c_void_p(0x10004)) == 1
    assert prefill(out=ctypes.c_void_p(0x10008)) == 1
    # copy_blocks
    assert lib.pkv_copy_blocks(fake, fake, _desc(), null, 3, null, null) == 1
    assert lib.pkv_copy_blocks(null, null, _desc(), null, 0, null, null) == 0
    assert lib.pkv_copy_blocks(fake, fake, _desc(), fake, -1, null, null) == 1


def test_fp8_validation_without_launch(lib):
    """The 8-bit pool calls, and 8-bit pools in the 16-bit calls, fail validation first."""
    fake = ctypes.c_void_p(0x10000)
    null = None
    d8 = _desc(dtype=_lib.PKV_FP8_E4M3)
    # the 16-bit calls take 16-bit pools only
    assert lib.pkv_kv_write(fake, fake, fake, 1, fake, fake, d8, null, null) == 1
    assert lib.pkv_paged_decode_attention(fake, fake, fake, fake, 4, fake, 64, 2, 32, d8,
                                          ctypes.c_float(0.1), 0, null, 0, fake, null, null) == 1
    assert lib.pkv_paged_prefill_attention(fake, fake, 4, fake, fake, fake, 4, fake, 64, 2, 32,
                                           d8, ctypes.c_float(0.1), fake, null, null) == 1

    def kw8(**kw):
        a = dict(k=fake, v=fake, kvd=_lib.PKV_BF16, sm=fake, T=4, kc=fake, vc=fake, desc=d8,
                 ks=0.5, vs=0.5)
        a.update(kw)
        return lib.pkv_kv_write_fp8(a["k"], a["v"], a["kvd"], a["sm"], a["T"], a["kc"], a["vc"],
                                    a["desc"], ctypes.c_float(a["ks"]), ctypes.c_float(a["vs"]),
                                    null, null)

    assert kw8(T=0) == 0
    assert kw8(k=null) == 1
    assert kw8(kvd=_lib.PKV_FP8_E4M3) == 1  # new keys / values are 16-bit
    assert kw8(desc=_desc()) == 1           # the pools must be 8-bit
    assert kw8(ks=0.0) == 1 and kw8(vs=float("inf")) == 1 and kw8(ks=-1.0) == 1
    assert kw8(desc=_desc(dtype=2, head_dim=8)) == 2  # 8-byte rows

    def at8(**kw):
        a = dict(q=fake, qd=_lib.PKV_BF16, kc=fake, vc=fake, bt=fake, mb=4, sl=fake, msl=64, S=2,
                 Hq=32, desc=d8, scale=0.1, ks=0.5, vs=0.5, ws=null, wsb=0, out=fake)
        a.update(kw)
        return lib.pkv_paged_decode_attention_fp8(
            a["q"], a["qd"], a["kc"], a["vc"], a["bt"], a["mb"], a["sl"], a["msl"], a["S"],
            a["Hq"], a["desc"], ctypes.c_float(a["scale"]), ctypes.c_float(a["ks"]),
            ctypes.c_float(a["vs"]), a["ws"], a["wsb"], a["out"], null, null)

    assert at8(S=0) == 0
    assert at8() == 3  # the streaming kernel needs its workspace
    assert at8(desc=_desc()) == 1
    assert at8(qd=_lib.PKV_FP8_E4M3) == 1
    assert at8(ks=0.0) == 1 and at8(vs=float("nan")) == 1
    assert at8(scale=1e30, ks=1e30) == 1  # the combined score factor overflows
    assert at8(Hq=30) == 1
    assert at8(msl=65) == 1
    assert at8(Hq=8 * 17) == 2  # group of 17 query heads per KV head
    assert at8(desc=_desc(dtype=2, head_dim=64)) == 2
    assert at8(desc=_desc(dtype=2, block_size=24), msl=48) == 2
    assert at8(S=5000, mb=4) == 2  # more sequences than the streaming kernel takes
    assert at8(q=null, ws=fake, wsb=1 << 30) == 1
    # block copies take 8-bit pools as they are
    assert lib.pkv_copy_blocks(null, null, d8, null, 0, null, null) == 0
    assert lib.pkv_copy_blocks(fake, fake, d8, null, 3, null, null) == 1
    assert lib.pkv_swap_blocks(fake, fake, 4, fake, fake, 4, d8, fake, 0, null, null) == 0


def test_workspace_query_covers_the_fp8_call(lib):
    from paged_kv_cache_242_gb300 import ops  # noqa: F401  (binding loads)
    for S, Hq, msl in ((1, 8, 1), (64, 32, 4096), (4096, 64, 100)):
        assert lib.pkv_decode_workspace_bytes(S, Hq, 128, msl, 16, 0) > 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIBRARY", str(tmp_path / "absent.so"))
    with pytest.raises(_lib.PKVError):
        _lib.load()


def test_build_flags_decide_whether_the_library_is_current(monkeypatch, tmp_path):
    """A library built with other nvcc options than the current ones is rebuilt."""
    lib_path = tmp_path / "libpkv.so"
    monkeypatch.setattr(build, "BUILD_DIR", str(tmp_path))
    monkeypatch.setattr(build, "LIBRARY", str(lib_path))
    monkeypatch.delenv("PKV_NVCC_EXTRA_FLAGS", raising=False)
    assert not build.up_to_date()  # no library
    lib_path.write_bytes(b"")
    future = max(os.path.getmtime(p) for p in build._inputs()) + 10
    os.utime(lib_path, (future, future))
    assert not build.up_to_date()  # no record of its flags
    (tmp_path / "flags.txt").write_text(" ".join(build._flags()))
    assert build.up_to_date()
    monkeypatch.setenv("PKV_NVCC_EXTRA_FLAGS", "-DPKV_MERGE_WIDE_PIECES=16")
    assert not build.up_to_date()  # other definitions
    (tmp_path / "flags.txt").write_text(" ".join(build._flags()))
    assert build.up_to_date()
