"""Python binding of libpa.so: argument marshalling only.

Each function takes PyTorch tensors (device memory owned by the caller), checks
shapes/dtypes/devices, and calls the C ABI function of the same name on the
current CUDA stream.  Every step of the computation runs in the library's CUDA
kernels; there is no PyTorch or CPU fallback.
"""
from __future__ import annotations

import ctypes

import torch

from . import _native as N

_DT = {torch.float32: N.PA_F32, torch.float16: N.PA_F16, torch.bfloat16: N.PA_BF16}


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}; expected float32, float16 or bfloat16")


def _cuda(name: str, t: torch.Tensor) -> None:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pa_decode_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int,
                              max_context_len: int, block_size: int,
                              partition_size: int = 0) -> int:
    """Workspace bytes pa_decode needs for a split call (0 when it never splits)."""
    return int(N.load().pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim,
                                                  max_context_len, block_size, partition_size))


def pa_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
              num_kv_heads: int, block_size: int, max_context_len: int | None = None,
              partition_size: int = 0, workspace: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """Paged decode attention: out[s, h] = softmax(scale q[s, h] . K_s^T) V_s, where
    K_s, V_s are sequence s's first context_lens[s] tokens reached through
    block_tables[s].

    out [S, Hq, D] (float32 or q's dtype), q [S, Hq, D], k_cache / v_cache
    [N, Hkv, B, D], block_tables [S, W] int32, context_lens [S] int32.
    max_context_len defaults to W * block_size (an upper bound needing no
    device-to-host read).  When no workspace is given, one of
    pa_decode_workspace_bytes(...) is allocated with torch: the split's partial
    rows, or for an automatic one-pass call the longest-first dispatch order.
    """
    for name, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda(name, t)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if q.dim() != 3 or out.shape != q.shape:
        raise ValueError(f"q and out must be [S, Hq, D] of one shape, got {tuple(q.shape)}, "
                         f"{tuple(out.shape)}")
    S, Hq, D = q.shape
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape or \
            tuple(k_cache.shape[1:]) != (num_kv_heads, block_size, D):
        raise ValueError(f"k_cache/v_cache must be [N, {num_kv_heads}, {block_size}, {D}], "
                         f"got {tuple(k_cache.shape)}, {tuple(v_cache.shape)}")
    if k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise TypeError("q, k_cache and v_cache must share a dtype")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, W] and context_lens [S]")
    W = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = W * block_size
    ws_need = pa_decode_workspace_bytes(S, Hq, D, max_context_len, block_size,
                                        max(partition_size, 0)) if partition_size >= 0 else 0
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_ptr, ws_bytes = (0, 0) if workspace is None else (workspace.data_ptr(),
                                                         workspace.numel() *
                                                         workspace.element_size())
    status = N.load().pa_decode(out.data_ptr(), _dtype(out), q.data_ptr(), k_cache.data_ptr(),
                                v_cache.data_ptr(), _dtype(q), k_cache.shape[0],
                                block_tables.data_ptr(), block_tables.stride(0),
                                context_lens.data_ptr(), int(max_context_len), S, Hq,
                                num_kv_heads, D, block_size, float(scale), int(partition_size),
                                ws_ptr, ws_bytes, _stream(stream))
    N.check("pa_decode", status)
    return out


def pa_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, num_kv_heads: int,
                      block_size: int, max_context_len: int | None = None,
                      partition_size: int = 0, stream=None) -> torch.Tensor:
    """pa_decode's split path with its scratch in the library's static device array
    (no workspace argument, nothing allocated).  For callers that cannot allocate
    device memory on the decode path.  Calls overlapping on the GPU share that one
    array and race; the first call on a device looks up its address, so make it
    before any stream capture."""
    for name, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda(name, t)
    if q.dim() != 3 or out.shape != q.shape or k_cache.dim() != 4:
        raise ValueError("q and out must be [S, Hq, D]; caches [N, Hkv, B, D]")
    S, Hq, D = q.shape
    if max_context_len is None:
        max_context_len = block_tables.shape[1] * block_size
    status = N.load().pa_decode_noalloc(out.data_ptr(), _dtype(out), q.data_ptr(),
                                        k_cache.data_ptr(), v_cache.data_ptr(), _dtype(q),
                                        k_cache.shape[0], block_tables.data_ptr(),
                                        block_tables.stride(0), context_lens.data_ptr(),
                                        int(max_context_len), S, Hq, num_kv_heads, D,
                                        block_size, float(scale), int(partition_size),
                                        _stream(stream))
    N.check("pa_decode_noalloc", status)
    return out


def pa_reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                         stream=None) -> None:
    """Write k[i], v[i] ([T, Hkv, D]) into the cache slot slot_mapping[i] (int64;
    negative = skip), bit for bit.  Caches are [N, Hkv, B, D]."""
    for name, t in (("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("slot_mapping", slot_mapping)):
        _cuda(name, t)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if k.dim() != 3 or v.shape != k.shape or k_cache.dim() != 4 or \
            v_cache.shape != k_cache.shape:
        raise ValueError("k, v must be [T, Hkv, D] and caches [N, Hkv, B, D]")
    T, Hkv, D = k.shape
    Nb, Hc, B, Dc = k_cache.shape
    if (Hc, Dc) != (Hkv, D) or slot_mapping.shape != (T,):
        raise ValueError("k/v heads and head_dim must match the caches; slot_mapping is [T]")
    if not (k.dtype == v.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("k, v and the caches must share a dtype")
    status = N.load().pa_reshape_and_cache(k.data_ptr(), v.data_ptr(), k_cache.data_ptr(),
                                           v_cache.data_ptr(), slot_mapping.data_ptr(), T, Hkv,
                                           D, B, Nb, _dtype(k), _stream(stream))
    N.check("pa_reshape_and_cache", status)


def pa_copy_blocks(k_caches, v_caches, src_dst_pairs, stream=None) -> None:
    """Copy whole blocks src -> dst in every layer's K and V pool (copy-on-write).

    k_caches, v_caches: lists of [N, ...] CUDA tensors, one per layer, all of one
    shape; src_dst_pairs: host sequence / array / CPU tensor of (src, dst) int pairs.
    """
    if isinstance(k_caches, torch.Tensor):
        k_caches, v_caches = [k_caches], [v_caches]
    if len(k_caches) != len(v_caches) or not k_caches:
        raise ValueError("k_caches and v_caches must be non-empty lists of equal length")
    shape = k_caches[0].shape
    for t in list(k_caches) + list(v_caches):
        _cuda("cache", t)
        if t.shape != shape or t.dtype != k_caches[0].dtype:
            raise ValueError("every cache must have the same shape and dtype")
    pairs = torch.as_tensor(src_dst_pairs, dtype=torch.int64).reshape(-1, 2).contiguous()
    if pairs.device.type != "cpu":
        raise ValueError("src_dst_pairs must live in host memory")
    n_blocks = shape[0]
    block_bytes = k_caches[0].numel() * k_caches[0].element_size() // n_blocks
    L = len(k_caches)
    kp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_caches])
    vp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_caches])
    pp = ctypes.cast(pairs.data_ptr(), ctypes.POINTER(ctypes.c_int64))
    status = N.load().pa_copy_blocks(kp, vp, L, pp, pairs.shape[0], block_bytes, n_blocks,
                                     _stream(stream))
    N.check("pa_copy_blocks", status)


def pa_swap_blocks(src_caches, dst_caches, src_dst_pairs, stream=None) -> None:
    """Move whole blocks between two pools per cache: dst_caches[c][d] = src_caches[c][s]
    for every (s, d) pair -- swapping a preempted sequence group out to a pinned host
    pool (src on the GPU, dst pinned CPU tensors) or back in (the reverse).

    src_caches, dst_caches: equal-length lists of contiguous tensors whose first dim is
    the block id, each a CUDA tensor or a pinned CPU tensor (``pin_memory()``); every
    block has the same byte size.  src_dst_pairs: host (s, d) int pairs.
    """
    if isinstance(src_caches, torch.Tensor):
        src_caches, dst_caches = [src_caches], [dst_caches]
    if len(src_caches) != len(dst_caches) or not src_caches:
        raise ValueError("src_caches and dst_caches must be non-empty lists of equal length")

    def block_bytes(t):
        if not isinstance(t, torch.Tensor) or not t.is_contiguous():
            raise ValueError("caches must be contiguous tensors")
        if t.device.type == "cpu" and not t.is_pinned():
            raise ValueError("a host pool must be pinned (tensor.pin_memory())")
        if t.device.type not in ("cpu", "cuda"):
            raise ValueError("caches must be CUDA or pinned CPU tensors")
        return t.numel() * t.element_size() // t.shape[0]

    bb = block_bytes(src_caches[0])
    for t in list(src_caches) + list(dst_caches):
        if block_bytes(t) != bb:
            raise ValueError("every pool must have the same block size in bytes")
    ns, nd = src_caches[0].shape[0], dst_caches[0].shape[0]
    if any(t.shape[0] != ns for t in src_caches) or any(t.shape[0] != nd for t in dst_caches):
        raise ValueError("the source pools (and the destination pools) must have one size")
    pairs = torch.as_tensor(src_dst_pairs, dtype=torch.int64).reshape(-1, 2).contiguous()
    if pairs.device.type != "cpu":
        raise ValueError("src_dst_pairs must live in host memory")
    C = len(src_caches)
    sp = (ctypes.c_void_p * C)(*[t.data_ptr() for t in src_caches])
    dp = (ctypes.c_void_p * C)(*[t.data_ptr() for t in dst_caches])
    pp = ctypes.cast(pairs.data_ptr(), ctypes.POINTER(ctypes.c_int64))
    status = N.load().pa_swap_blocks(sp, dp, C, pp, pairs.shape[0], bb, ns, nd, _stream(stream))
    N.check("pa_swap_blocks", status)


def _fp8_cache(name: str, t: torch.Tensor) -> None:
    _cuda(name, t)
    if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError(f"{name} must hold E4M3 codes (torch.float8_e4m3fn or uint8)")


def _scales(k_scale, v_scale, num_kv_heads):
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        _cuda(name, t)
        if t.dtype != torch.float32 or t.shape != (num_kv_heads,):
            raise ValueError(f"{name} must be float32 [num_kv_heads]")


def pa_reshape_and_cache_fp8(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                             v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                             k_scale: torch.Tensor, v_scale: torch.Tensor, stream=None) -> None:
    """Quantising cache write: k_cache[slot / B][h][slot % B] = e4m3(fp32(k[i][h]) / k_scale[h])
    (round to nearest even, saturating at +-448), likewise v.  k, v [T, Hkv, D] in fp32 /
    fp16 / bf16; caches [N, Hkv, B, D] of E4M3 codes; scales float32 [Hkv]."""
    for name, t in (("k", k), ("v", v), ("slot_mapping", slot_mapping)):
        _cuda(name, t)
    _fp8_cache("k_cache", k_cache)
    _fp8_cache("v_cache", v_cache)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    T, Hkv, D = k.shape
    if v.shape != k.shape or v.dtype != k.dtype or k_cache.shape != v_cache.shape or \
            k_cache.dim() != 4 or (k_cache.shape[1], k_cache.shape[3]) != (Hkv, D):
        raise ValueError("k, v must be [T, Hkv, D] and caches [N, Hkv, B, D]")
    _scales(k_scale, v_scale, Hkv)
    status = N.load().pa_reshape_and_cache_fp8(
        k.data_ptr(), v.data_ptr(), _dtype(k), k_cache.data_ptr(), v_cache.data_ptr(),
        k_scale.data_ptr(), v_scale.data_ptr(), slot_mapping.data_ptr(), T, Hkv, D,
        k_cache.shape[2], k_cache.shape[0], _stream(stream))
    N.check("pa_reshape_and_cache_fp8", status)


def pa_decode_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                  block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                  num_kv_heads: int, block_size: int, max_context_len: int | None = None,
                  partition_size: int = 0, workspace: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """pa_decode over E4M3 caches with per-kv-head scales (value = code * scale[h]).
    q [S, Hq, D] fp16 / bf16; out fp32 or q's dtype."""
    for name, t in (("out", out), ("q", q), ("block_tables", block_tables),
                    ("context_lens", context_lens)):
        _cuda(name, t)
    _fp8_cache("k_cache", k_cache)
    _fp8_cache("v_cache", v_cache)
    _scales(k_scale, v_scale, num_kv_heads)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if q.dim() != 3 or out.shape != q.shape:
        raise ValueError("q and out must be [S, Hq, D] of one shape")
    S, Hq, D = q.shape
    if k_cache.shape != v_cache.shape or tuple(k_cache.shape[1:]) != (num_kv_heads, block_size, D):
        raise ValueError("caches must be [N, Hkv, B, D]")
    if max_context_len is None:
        max_context_len = block_tables.shape[1] * block_size
    ws_need = pa_decode_workspace_bytes(S, Hq, D, max_context_len, block_size,
                                        max(partition_size, 0)) if partition_size >= 0 else 0
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_ptr, ws_bytes = (0, 0) if workspace is None else (workspace.data_ptr(),
                                                         workspace.numel() *
                                                         workspace.element_size())
    status = N.load().pa_decode_fp8(
        out.data_ptr(), _dtype(out), q.data_ptr(), _dtype(q), k_cache.data_ptr(),
        v_cache.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr(), k_cache.shape[0],
        block_tables.data_ptr(), block_tables.stride(0), context_lens.data_ptr(),
        int(max_context_len), S, Hq, num_kv_heads, D, block_size, float(scale),
        int(partition_size), ws_ptr, ws_bytes, _stream(stream))
    N.check("pa_decode_fp8", status)
    return out


def pa_chunk_workspace_bytes(num_query_tokens: int, num_q_heads: int, head_dim: int,
                             max_context_len: int, partition_size: int = 0) -> int:
    """Workspace bytes pa_chunk_attention needs for a split call (0 when it never splits)."""
    return int(N.load().pa_chunk_workspace_bytes(num_query_tokens, num_q_heads, head_dim,
                                                 max_context_len, partition_size))


def pa_chunk_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, block_tables: torch.Tensor,
                       context_lens: torch.Tensor, query_start: torch.Tensor, scale: float,
                       num_kv_heads: int, block_size: int, max_query_len: int,
                       max_context_len: int | None = None, partition_size: int = 0,
                       workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Causal attention of each sequence's chunk of new query tokens (chunked prefill,
    speculative verification) over the paged cache.

    q, out [R, Hq, D] (out float32 or q's dtype; q float16 or bfloat16, the caches'
    dtype); sequence s owns rows query_start[s] .. query_start[s+1]-1 (query_start
    [S+1] int32), the last n_s of its context_lens[s] cached tokens, and chunk token j
    attends to cached tokens 0 .. L_s - n_s + j.  max_query_len bounds every n_s;
    max_context_len defaults to W * block_size.  A workspace is allocated with torch
    if the call splits and none is given.
    """
    for name, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_tables", block_tables), ("context_lens", context_lens),
                    ("query_start", query_start)):
        _cuda(name, t)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or \
            query_start.dtype != torch.int32:
        raise TypeError("block_tables, context_lens and query_start must be int32")
    if q.dim() != 3 or out.shape != q.shape:
        raise ValueError(f"q and out must be [R, Hq, D] of one shape, got {tuple(q.shape)}, "
                         f"{tuple(out.shape)}")
    R, Hq, D = q.shape
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape or \
            tuple(k_cache.shape[1:]) != (num_kv_heads, block_size, D):
        raise ValueError(f"k_cache/v_cache must be [N, {num_kv_heads}, {block_size}, {D}], "
                         f"got {tuple(k_cache.shape)}, {tuple(v_cache.shape)}")
    if k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise TypeError("q, k_cache and v_cache must share a dtype")
    S = context_lens.shape[0]
    if block_tables.dim() != 2 or block_tables.shape[0] != S or query_start.shape != (S + 1,):
        raise ValueError("block_tables must be [S, W], context_lens [S], query_start [S + 1]")
    if max_context_len is None:
        max_context_len = block_tables.shape[1] * block_size
    ws_need = pa_chunk_workspace_bytes(R, Hq, D, max_context_len, max(partition_size, 0)) \
        if partition_size >= 0 else 0
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_ptr, ws_bytes = (0, 0) if workspace is None else (workspace.data_ptr(),
                                                         workspace.numel() *
                                                         workspace.element_size())
    status = N.load().pa_chunk_attention(
        out.data_ptr(), _dtype(out), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        _dtype(q), k_cache.shape[0], block_tables.data_ptr(), block_tables.stride(0),
        context_lens.data_ptr(), query_start.data_ptr(), R, int(max_query_len),
        int(max_context_len), S, Hq, num_kv_heads, D, block_size, float(scale),
        int(partition_size), ws_ptr, ws_bytes, _stream(stream))
    N.check("pa_chunk_attention", status)
    return out


def pa_chunk_attention_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                           query_start: torch.Tensor, scale: float, num_kv_heads: int,
                           block_size: int, max_query_len: int,
                           max_context_len: int | None = None, partition_size: int = 0,
                           workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """pa_chunk_attention over E4M3 caches (torch.float8_e4m3fn or uint8 codes) with
    per-kv-head scales k_scale, v_scale (float32 CUDA [Hkv]); q float16 or bfloat16."""
    for name, t in (("out", out), ("q", q), ("block_tables", block_tables),
                    ("context_lens", context_lens), ("query_start", query_start)):
        _cuda(name, t)
    _fp8_cache("k_cache", k_cache)
    _fp8_cache("v_cache", v_cache)
    if q.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("q must be float16 or bfloat16 for an E4M3 cache")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or \
            query_start.dtype != torch.int32:
        raise TypeError("block_tables, context_lens and query_start must be int32")
    if q.dim() != 3 or out.shape != q.shape:
        raise ValueError("q and out must be [R, Hq, D] of one shape")
    R, Hq, D = q.shape
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape or \
            tuple(k_cache.shape[1:]) != (num_kv_heads, block_size, D):
        raise ValueError(f"k_cache/v_cache must be [N, {num_kv_heads}, {block_size}, {D}]")
    _scales(k_scale, v_scale, num_kv_heads)
    S = context_lens.shape[0]
    if block_tables.dim() != 2 or block_tables.shape[0] != S or query_start.shape != (S + 1,):
        raise ValueError("block_tables must be [S, W], context_lens [S], query_start [S + 1]")
    if max_context_len is None:
        max_context_len = block_tables.shape[1] * block_size
    ws_need = pa_chunk_workspace_bytes(R, Hq, D, max_context_len, max(partition_size, 0)) \
        if partition_size >= 0 else 0
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_ptr, ws_bytes = (0, 0) if workspace is None else (workspace.data_ptr(),
                                                         workspace.numel() *
                                                         workspace.element_size())
    status = N.load().pa_chunk_attention_fp8(
        out.data_ptr(), _dtype(out), q.data_ptr(), _dtype(q), k_cache.data_ptr(),
        v_cache.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr(), k_cache.shape[0],
        block_tables.data_ptr(), block_tables.stride(0), context_lens.data_ptr(),
        query_start.data_ptr(), R, int(max_query_len), int(max_context_len), S, Hq,
        num_kv_heads, D, block_size, float(scale), int(partition_size), ws_ptr, ws_bytes,
        _stream(stream))
    N.check("pa_chunk_attention_fp8", status)
    return out


def pa_decode_partition_tokens(q_dtype: torch.dtype, kv_dtype: torch.dtype, num_seqs: int,
                               num_q_heads: int, num_kv_heads: int, head_dim: int,
                               block_size: int, max_context_len: int,
                               partition_size: int = 0) -> int:
    """The partition length pa_decode / pa_decode_fp8 would split contexts into
    (0: one pass, no merge launch)."""
    kv = N.PA_FP8_E4M3 if kv_dtype == torch.float8_e4m3fn else _DT[kv_dtype]
    r = int(N.load().pa_decode_partition_tokens(_DT[q_dtype], kv, num_seqs, num_q_heads,
                                                num_kv_heads, head_dim, block_size,
                                                max_context_len, partition_size))
    if r < 0:
        N.check("pa_decode_partition_tokens", r)
    return r


def pa_decode_orders_sequences(q_dtype: torch.dtype, kv_dtype: torch.dtype, num_seqs: int,
                               num_q_heads: int, num_kv_heads: int, head_dim: int,
                               block_size: int, max_context_len: int,
                               partition_size: int = 0) -> bool:
    """Whether pa_decode / pa_decode_fp8 (given its workspace) first builds the
    longest-first dispatch order of the sequences (one more launch)."""
    kv = N.PA_FP8_E4M3 if kv_dtype == torch.float8_e4m3fn else _DT[kv_dtype]
    r = int(N.load().pa_decode_orders_sequences(_DT[q_dtype], kv, num_seqs, num_q_heads,
                                                num_kv_heads, head_dim, block_size,
                                                max_context_len, partition_size))
    if r < 0:
        N.check("pa_decode_orders_sequences", r)
    return r == 1


def pa_chunk_partition_tokens(kv_dtype: torch.dtype, num_seqs: int, num_q_heads: int,
                              num_kv_heads: int, head_dim: int, block_size: int,
                              max_query_len: int, max_context_len: int,
                              partition_size: int = 0) -> int:
    """The partition length pa_chunk_attention (or, for an E4M3 kv_dtype,
    pa_chunk_attention_fp8) would split contexts into (0: one pass)."""
    kv = N.PA_FP8_E4M3 if kv_dtype in (torch.float8_e4m3fn, torch.uint8) else _DT[kv_dtype]
    r = int(N.load().pa_chunk_partition_tokens(kv, num_seqs, num_q_heads,
                                               num_kv_heads, head_dim, block_size,
                                               max_query_len, max_context_len, partition_size))
    if r < 0:
        N.check("pa_chunk_partition_tokens", r)
    return r


def _kv_code(kv_dtype: torch.dtype) -> int:
    return N.PA_FP8_E4M3 if kv_dtype in (torch.float8_e4m3fn, torch.uint8) else _DT[kv_dtype]


def pa_decode_kernel_name(kv_dtype: torch.dtype, num_q_heads: int, num_kv_heads: int,
                          head_dim: int) -> str:
    """The attention kernel pa_decode (or, for an E4M3 kv_dtype, pa_decode_fp8) runs for
    these shapes, as the library routes it."""
    r = N.load().pa_decode_kernel_name(_kv_code(kv_dtype), num_q_heads, num_kv_heads, head_dim)
    if r is None:
        raise ValueError("pa_decode_kernel_name: arguments the decode calls reject")
    return r.decode()


def pa_chunk_kernel_name(kv_dtype: torch.dtype, num_q_heads: int, num_kv_heads: int,
                         head_dim: int, max_query_len: int) -> str:
    """The attention kernel pa_chunk_attention (or pa_chunk_attention_fp8) runs for these
    shapes, as the library routes it."""
    r = N.load().pa_chunk_kernel_name(_kv_code(kv_dtype), num_q_heads, num_kv_heads, head_dim,
                                      max_query_len)
    if r is None:
        raise ValueError("pa_chunk_kernel_name: arguments the chunk calls reject")
    return r.decode()


def pa_stream_read(buf: torch.Tensor, sink: torch.Tensor, stream=None) -> None:
    """Measurement helper: stream every byte of buf once (the read-only bandwidth
    ceiling); a checksum is XORed into sink (a one-element int32 CUDA tensor)."""
    _cuda("buf", buf)
    _cuda("sink", sink)
    if sink.dtype != torch.int32 or sink.numel() < 1:
        raise TypeError("sink must be an int32 CUDA tensor")
    N.check("pa_stream_read", N.load().pa_stream_read(buf.data_ptr(),
                                                       buf.numel() * buf.element_size(),
                                                       sink.data_ptr(), _stream(stream)))


def pa_stream_read_runs(buf: torch.Tensor, run_bytes: int, order: torch.Tensor,
                        sink: torch.Tensor, stream=None) -> None:
    """Measurement helper: read run order[i] (run_bytes each) of buf for every i, CTAs
    taking consecutive entries (a block-table walk); sink (int32 CUDA, two elements)
    gets a checksum in [0] and the count of out-of-range entries in [1]."""
    for name, t in (("buf", buf), ("order", order), ("sink", sink)):
        _cuda(name, t)
    if order.dtype != torch.int32 or not order.is_contiguous():
        raise TypeError("order must be a contiguous int32 CUDA tensor")
    if sink.dtype != torch.int32 or sink.numel() < 2:
        raise TypeError("sink must be an int32 CUDA tensor of two elements")
    N.check("pa_stream_read_runs",
            N.load().pa_stream_read_runs(buf.data_ptr(), buf.numel() * buf.element_size(),
                                         int(run_bytes), order.data_ptr(), order.numel(),
                                         sink.data_ptr(), _stream(stream)))


def pa_get_device_error(stream=None) -> int:
    """Read and clear the device error word (PA_DEVERR_* bits).  Synchronises."""
    flags = ctypes.c_uint32(0)
    N.check("pa_get_device_error", N.load().pa_get_device_error(ctypes.byref(flags),
                                                                 _stream(stream)))
    return int(flags.value)


def pa_version() -> str:
    return N.load().pa_version().decode()
