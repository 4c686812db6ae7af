"""The C ABI without a GPU: the library loads, exports every symbol include/pa.h
declares, and rejects invalid arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_119_gb300 import _native as N
from paged_kv_cache_119_gb300 import build as B

HEADERS = [os.path.join(B.ROOT, "include", h) for h in ("pa.h", "pa_block_manager.h")]


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_and_binding_agree():
    assert declared_functions() == sorted(N.SIGNATURES)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.pa_version()
    for st in (N.PA_OK, N.PA_ERR_INVALID, N.PA_ERR_UNSUPPORTED, N.PA_ERR_WORKSPACE,
               N.PA_ERR_CUDA, 12345):
        assert lib.pa_status_string(st)


def test_workspace_bytes(lib):
    # 8 seqs x 64 heads x 64 partitions x (128 + 2) fp32 values, o rows 256-aligned
    ws = lib.pa_decode_workspace_bytes(8, 64, 128, 32768, 16, 512)
    assert ws == 8 * 64 * 64 * 128 * 4 + 8 * 64 * 64 * 2 * 4
    assert lib.pa_decode_workspace_bytes(8, 64, 128, 512, 16, 512) == 0      # never splits
    assert lib.pa_decode_workspace_bytes(8, 64, 128, 4096, 16, 0) > 0         # auto upper bound
    assert lib.pa_decode_workspace_bytes(-1, 64, 128, 4096, 16, 0) == 0
    # automatic calls that cannot split still get room for the dispatch order:
    # 8 bytes per sequence, rounded up to 256
    assert lib.pa_decode_workspace_bytes(8, 64, 128, 512, 16, 0) == 256
    assert lib.pa_decode_workspace_bytes(33, 64, 128, 512, 16, 0) == 512
    assert lib.pa_decode_workspace_bytes(8, 64, 128, 512, 16, -1) == 0


FAKE = 1 << 20        # a 16-byte-aligned non-null address; never dereferenced here


def decode_args(**kw):
    a = dict(out=FAKE, out_dtype=N.PA_BF16, q=FAKE * 2, k=FAKE * 3, v=FAKE * 4,
             kv_dtype=N.PA_BF16, num_blocks=10, bt=FAKE * 5, bt_stride=8, cl=FAKE * 6,
             max_ctx=64, S=2, Hq=4, Hkv=2, D=128, B=16, scale=0.1, part=0, ws=0, ws_bytes=0,
             stream=0)
    a.update(kw)
    return list(a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(kv_dtype=7), N.PA_ERR_INVALID),
    (dict(out_dtype=N.PA_F16), N.PA_ERR_INVALID),                 # out neither f32 nor kv dtype
    (dict(Hq=5), N.PA_ERR_INVALID),                               # Hq % Hkv != 0
    (dict(D=96), N.PA_ERR_UNSUPPORTED),
    (dict(B=8), N.PA_ERR_UNSUPPORTED),
    (dict(max_ctx=8 * 16 + 1), N.PA_ERR_INVALID),                 # beyond the table row
    (dict(num_blocks=0), N.PA_ERR_INVALID),
    (dict(num_blocks=1 << 31), N.PA_ERR_INVALID),
    (dict(scale=float("nan")), N.PA_ERR_INVALID),
    (dict(part=24), N.PA_ERR_INVALID),                            # not a multiple of B
    (dict(q=0), N.PA_ERR_INVALID),
    (dict(k=FAKE + 8), N.PA_ERR_INVALID),                         # misaligned cache
    (dict(out=FAKE * 2), N.PA_ERR_INVALID),                       # out aliases q
    (dict(S=70000), N.PA_ERR_INVALID),
])
def test_decode_rejects(lib, kw, status):
    assert lib.pa_decode(*decode_args(**kw)) == status


def test_decode_split_needs_workspace(lib):
    # an explicit split with no workspace is rejected before any launch
    assert lib.pa_decode(*decode_args(part=16, max_ctx=64)) == N.PA_ERR_WORKSPACE


def test_decode_workspace_must_not_overlap_inputs(lib):
    # the split writes partial rows into the workspace while it reads the inputs
    need = lib.pa_decode_workspace_bytes(2, 4, 128, 64, 16, 16)
    assert need > 0
    for name, base in (("out", FAKE), ("q", FAKE * 2), ("k_cache", FAKE * 3),
                       ("block_tables", FAKE * 5), ("context_lens", FAKE * 6)):
        args = decode_args(part=16, max_ctx=64, ws=base, ws_bytes=need)
        assert lib.pa_decode(*args) == N.PA_ERR_INVALID, name


def test_decode_empty_batch_is_a_no_op(lib):
    assert lib.pa_decode(*decode_args(S=0)) == N.PA_OK


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=9), N.PA_ERR_INVALID),
    (dict(D=4, dtype=N.PA_F16), N.PA_ERR_UNSUPPORTED),            # row not a multiple of 16 B
    (dict(k=FAKE + 4), N.PA_ERR_INVALID),
    (dict(T=-1), N.PA_ERR_INVALID),
    (dict(kc=FAKE * 8, vc=FAKE * 8), N.PA_ERR_INVALID),          # K and V pools overlap
])
def test_reshape_rejects(lib, kw, status):
    a = dict(k=FAKE, v=FAKE * 2, kc=FAKE * 8, vc=FAKE * 64, slots=FAKE * 4, T=3, Hkv=2, D=64,
             B=16, N=4, dtype=N.PA_BF16, stream=0)
    a.update(kw)
    assert lib.pa_reshape_and_cache(*a.values()) == status


def test_reshape_zero_tokens_is_a_no_op(lib):
    assert lib.pa_reshape_and_cache(0, 0, 0, 0, 0, 0, 2, 64, 16, 4, N.PA_BF16, 0) == N.PA_OK


def _copy(lib, pairs, num_blocks=8, block_bytes=64, layers=1):
    ptrs = (ctypes.c_void_p * layers)(*[FAKE * (i + 1) for i in range(layers)])
    flat = [x for p in pairs for x in p]
    arr = (ctypes.c_int64 * max(1, len(flat)))(*flat)
    return lib.pa_copy_blocks(ptrs, ptrs, layers, arr, len(pairs), block_bytes, num_blocks, None)


@pytest.mark.parametrize("pairs", [
    [(0, 8)],               # dst out of range
    [(-1, 2)],              # src out of range
    [(0, 2), (1, 2)],       # two pairs write one block
    [(0, 2), (2, 3)],       # a destination is also a source
])
def test_copy_blocks_rejects(lib, pairs):
    assert _copy(lib, pairs) == N.PA_ERR_INVALID


def test_copy_blocks_rejects_bad_sizes(lib):
    assert _copy(lib, [(0, 1)], block_bytes=24) == N.PA_ERR_INVALID
    assert _copy(lib, [], block_bytes=64) == N.PA_OK


def test_get_device_error_needs_a_pointer(lib):
    assert lib.pa_get_device_error(None, None) == N.PA_ERR_INVALID


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import paged_kv_cache_119_gb300 as P
    x = torch.zeros(2, 4, 64)
    with pytest.raises(ValueError, match="CUDA"):
        P.pa_decode(x, x, torch.zeros(1, 4, 16, 64), torch.zeros(1, 4, 16, 64),
                    torch.zeros(2, 1, dtype=torch.int32), torch.zeros(2, dtype=torch.int32),
                    0.125, 4, 16)


def test_noalloc_rejects_oversized_and_unsplit_requests(lib):
    # the size and partition checks happen before any CUDA call
    args = decode_args(max_ctx=32768, S=64, Hq=64, Hkv=8, bt_stride=2048, part=512)
    del args[18:20]                           # pa_decode_noalloc has no workspace arguments
    assert lib.pa_decode_noalloc(*args) == N.PA_ERR_WORKSPACE
    args = decode_args(part=-1)
    del args[18:20]
    assert lib.pa_decode_noalloc(*args) == N.PA_ERR_INVALID


def chunk_args(**kw):
    a = dict(out=FAKE, out_dtype=N.PA_F32, q=FAKE * 16, k=FAKE * 48, v=FAKE * 96,
             kv_dtype=N.PA_BF16, num_blocks=10, bt=FAKE * 130, bt_stride=8, cl=FAKE * 131,
             qs=FAKE * 132, R=12, max_q=6, max_ctx=64, S=3, Hq=8, Hkv=2, D=128, B=16,
             scale=0.1, part=-1, ws=0, ws_bytes=0, stream=0)
    a.update(kw)
    return [a[k] for k in ("out", "out_dtype", "q", "k", "v", "kv_dtype", "num_blocks", "bt",
                           "bt_stride", "cl", "qs", "R", "max_q", "max_ctx", "S", "Hq", "Hkv",
                           "D", "B", "scale", "part", "ws", "ws_bytes", "stream")]


@pytest.mark.parametrize("kw,status", [
    (dict(kv_dtype=N.PA_F32), N.PA_ERR_UNSUPPORTED),                # tensor-core path: 16-bit
    (dict(kv_dtype=9), N.PA_ERR_INVALID),
    (dict(out_dtype=N.PA_F16), N.PA_ERR_INVALID),                 # neither f32 nor the kv dtype
    (dict(Hq=6, Hkv=4), N.PA_ERR_INVALID),
    (dict(Hq=258, Hkv=1), N.PA_ERR_INVALID),                      # group above 128
    (dict(D=96), N.PA_ERR_UNSUPPORTED),
    (dict(B=8), N.PA_ERR_UNSUPPORTED),
    (dict(max_q=65), N.PA_ERR_INVALID),                           # chunk longer than any context
    (dict(max_ctx=8 * 16 + 1, max_q=6), N.PA_ERR_INVALID),        # beyond the table row
    (dict(R=-1), N.PA_ERR_INVALID),
    (dict(part=96), N.PA_ERR_INVALID),                            # not a multiple of 64
    (dict(qs=0), N.PA_ERR_INVALID),
    (dict(k=FAKE * 48 + 8), N.PA_ERR_INVALID),                    # misaligned cache
    (dict(out=FAKE * 16), N.PA_ERR_INVALID),                      # out aliases q
    (dict(S=70000), N.PA_ERR_INVALID),
    (dict(scale=float("inf")), N.PA_ERR_INVALID),
])
def test_chunk_attention_rejects(lib, kw, status):
    assert lib.pa_chunk_attention(*chunk_args(**kw)) == status


def test_chunk_workspace_must_not_overlap_inputs(lib):
    need = lib.pa_chunk_workspace_bytes(12, 8, 128, 256, 64)
    assert need > 0
    for name, base in (("out", FAKE), ("q", FAKE * 16), ("block_tables", FAKE * 130),
                       ("context_lens", FAKE * 131), ("query_start", FAKE * 132)):
        args = chunk_args(part=64, max_ctx=256, bt_stride=16, ws=base, ws_bytes=need)
        assert lib.pa_chunk_attention(*args) == N.PA_ERR_INVALID, name

def test_chunk_attention_empty_is_a_no_op(lib):
    assert lib.pa_chunk_attention(*chunk_args(S=0)) == N.PA_OK
    assert lib.pa_chunk_attention(*chunk_args(R=0)) == N.PA_OK
    assert lib.pa_chunk_attention(*chunk_args(max_q=0)) == N.PA_OK


def test_chunk_workspace_bytes(lib):
    # 100 query rows x 64 heads x 64 partitions x (128 + 2) fp32 values
    assert lib.pa_chunk_workspace_bytes(100, 64, 128, 32768, 512) == \
        100 * 64 * 64 * 128 * 4 + 100 * 64 * 64 * 2 * 4
    assert lib.pa_chunk_workspace_bytes(100, 64, 128, 512, 512) == 0
    assert lib.pa_chunk_workspace_bytes(100, 64, 128, 4096, 0) > 0
    assert lib.pa_chunk_workspace_bytes(-1, 64, 128, 4096, 0) == 0


def test_partition_queries_for_explicit_sizes(lib):
    """An explicit partition size needs no device query: the call splits exactly when
    the longest context exceeds it."""
    assert lib.pa_decode_partition_tokens(N.PA_BF16, N.PA_BF16, 8, 64, 8, 128, 16, 4096, 512) \
        == 512
    assert lib.pa_decode_partition_tokens(N.PA_BF16, N.PA_BF16, 8, 64, 8, 128, 16, 512, 512) == 0
    assert lib.pa_decode_partition_tokens(N.PA_BF16, N.PA_BF16, 8, 64, 8, 128, 16, 4096, -1) == 0
    assert lib.pa_decode_partition_tokens(N.PA_BF16, N.PA_BF16, 8, 64, 8, 128, 16, 4096, 24) \
        == N.PA_ERR_INVALID
    # only the automatic choice reorders sequences
    assert lib.pa_decode_orders_sequences(N.PA_BF16, N.PA_BF16, 256, 40, 40, 128, 16, 2048, 512) \
        == 0
    assert lib.pa_decode_orders_sequences(N.PA_BF16, N.PA_BF16, 256, 40, 40, 128, 16, 2048, -1) \
        == 0
    assert lib.pa_decode_orders_sequences(N.PA_BF16, N.PA_BF16, 256, 40, 40, 128, 16, 2048, 24) \
        == N.PA_ERR_INVALID
    assert lib.pa_chunk_partition_tokens(N.PA_BF16, 8, 64, 8, 128, 16, 512, 32768, 1024) == 1024
    assert lib.pa_chunk_partition_tokens(N.PA_BF16, 8, 64, 8, 128, 16, 512, 32768, 1000) \
        == N.PA_ERR_INVALID
    assert lib.pa_chunk_partition_tokens(N.PA_BF16, 8, 6, 4, 128, 16, 512, 32768, 0) \
        == N.PA_ERR_INVALID


def _swap(lib, pairs, block_bytes=64, ns=4, nd=6, caches=2):
    arr = (ctypes.c_int64 * (2 * len(pairs)))(*[x for pr in pairs for x in pr])
    src = (ctypes.c_void_p * caches)(*[FAKE * (i + 1) for i in range(caches)])
    dst = (ctypes.c_void_p * caches)(*[FAKE * (i + 8) for i in range(caches)])
    return lib.pa_swap_blocks(src, dst, caches, arr, len(pairs), block_bytes, ns, nd, None)


@pytest.mark.parametrize("pairs", [[(4, 0)], [(0, 6)], [(-1, 0)], [(0, 1), (2, 1)]])
def test_swap_blocks_rejects_bad_pairs(lib, pairs):
    assert _swap(lib, pairs) == N.PA_ERR_INVALID


def test_swap_blocks_rejects_bad_sizes_and_empty_is_a_no_op(lib):
    assert _swap(lib, [(0, 1)], block_bytes=24) == N.PA_ERR_INVALID
    assert _swap(lib, [(0, 1)], ns=0) == N.PA_ERR_INVALID
    assert _swap(lib, []) == N.PA_OK
    assert _swap(lib, [(0, 1)], caches=0) == N.PA_OK


def test_swap_blocks_rejects_host_memory_that_is_not_pinned(lib):
    """A pageable host buffer is not device-addressable: refused before any launch."""
    import numpy as np
    a = np.zeros(4 * 64, dtype=np.uint8)
    b = np.zeros(6 * 64, dtype=np.uint8)
    src = (ctypes.c_void_p * 1)(a.ctypes.data)
    dst = (ctypes.c_void_p * 1)(b.ctypes.data)
    arr = (ctypes.c_int64 * 2)(0, 1)
    assert lib.pa_swap_blocks(src, dst, 1, arr, 1, 64, 4, 6, None) == N.PA_ERR_INVALID


def test_wait_timeout_hook_validates_and_lasts_one_call(lib):
    assert lib.pa_test_arm_wait_timeout(-1, 5000) == N.PA_ERR_INVALID
    assert lib.pa_test_arm_wait_timeout(0, 0) == N.PA_ERR_INVALID
    assert lib.pa_test_arm_wait_timeout(0, 1000001) == N.PA_ERR_INVALID
    assert lib.pa_test_arm_wait_timeout(5, 5000) == N.PA_OK
    # the next decode call consumes the arm, even one rejected on the host
    assert lib.pa_decode(*decode_args(D=96)) == N.PA_ERR_UNSUPPORTED
