"""CPU oracle for paged decode attention, reshape_and_cache and copy_blocks.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
baseline leg of ``bench.py`` may import this package.  The product path (the
``paged_kv_cache_119_gb300`` package and its CUDA library) never imports,
links or calls it, and it imports nothing from the product path.

The arithmetic lives in ``pa_oracle.c`` (fp64, plain loops, one function per
operation, each citing the page section it restates).  This module only
compiles that file with gcc and marshals numpy / torch CPU buffers into it.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
that do not come from the oracle itself: the pages' worked examples (Figures
6 and 8 of the PagedAttention write-up, the zero-based block-table table), a
hand-computed 3-token case, closed forms, PyTorch's float64
``scaled_dot_product_attention`` on the unpaged (dense) arrays, and IEEE
decoding of every fp16/bf16 bit pattern.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpa_oracle.so")

F32, F16, BF16, E4M3 = 0, 1, 2, 3
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc (OpenMP when available).  Returns the .so path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-Wall", *extra_flags, src,
            "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:-4] + ["-fopenmp"] + base[-4:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(out + ".tmp", out)
    return out


def _declare(lib):
    c_i64, c_i32, c_vp, c_dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
    lib.orc_paged_attention.restype = ctypes.c_int
    lib.orc_paged_attention.argtypes = [c_vp, c_vp, c_i32, c_vp, c_vp, c_i32, c_vp, c_vp, c_i64,
                                        c_vp, c_i64, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32,
                                        c_dbl, c_i32]
    lib.orc_chunk_attention.restype = ctypes.c_int
    lib.orc_chunk_attention.argtypes = [c_vp, c_vp, c_i32, c_vp, c_vp, c_i32, c_vp, c_vp, c_i64,
                                        c_vp, c_i64, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32,
                                        c_i32, c_dbl, c_i32]
    lib.orc_reshape_and_cache_e4m3.restype = ctypes.c_int
    lib.orc_reshape_and_cache_e4m3.argtypes = [c_vp, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp,
                                               c_i64, c_i32, c_i32, c_i32, c_i64]
    lib.orc_e4m3_to_f64.restype = c_dbl
    lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
    lib.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
    lib.orc_reshape_and_cache.restype = ctypes.c_int
    lib.orc_reshape_and_cache.argtypes = [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i32, c_i32,
                                          c_i32, c_i64, c_i32]
    lib.orc_swap_blocks.restype = ctypes.c_int
    lib.orc_swap_blocks.argtypes = [c_vp, c_vp, c_i32, c_vp, c_i64, c_i64, c_i64, c_i64]
    lib.orc_copy_blocks.restype = ctypes.c_int
    lib.orc_copy_blocks.argtypes = [c_vp, c_i32, c_vp, c_i64, c_i64, c_i64]
    lib.orc_f16_to_f64.restype = c_dbl
    lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_f64.restype = c_dbl
    lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.orc_max_threads.restype = ctypes.c_int
    lib.orc_max_threads.argtypes = []
    return lib


def load_library(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


# --------------------------------------------------------------------------- marshalling

def _dtype_code(x) -> int:
    name = str(x.dtype)
    if name in ("torch.float8_e4m3fn", "torch.uint8", "uint8"):
        return E4M3
    if name in ("torch.float32", "float32"):
        return F32
    if name in ("torch.float16", "float16"):
        return F16
    if name == "torch.bfloat16":
        return BF16
    raise TypeError(f"oracle: unsupported dtype {name}")


def _raw(x, inplace: bool = False) -> np.ndarray:
    """A C-contiguous numpy view of the raw element bits of a CPU tensor or array.
    With ``inplace`` the view must share memory with ``x`` (no hidden copy)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.device.type != "cpu":
                raise ValueError("oracle inputs must live in host memory")
            if inplace and not x.is_contiguous():
                raise ValueError("oracle: in-place operand must be contiguous")
            x = x.contiguous()
            if x.dtype in (torch.float16, torch.bfloat16):
                return x.view(torch.int16).numpy()
            if x.dtype == torch.float8_e4m3fn:
                return x.view(torch.uint8).numpy()
            return x.numpy()
    except ImportError:
        pass
    if inplace and not x.flags.c_contiguous:
        raise ValueError("oracle: in-place operand must be C-contiguous")
    return np.ascontiguousarray(x)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def max_threads() -> int:
    return load_library().orc_max_threads()


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                    num_kv_heads: int, block_size: int, num_threads: int = 1,
                    lib=None, k_scale=None, v_scale=None) -> np.ndarray:
    """Decode attention through block tables, fp64.  Returns out[S][Hq][D] as float64.

    q: [S, Hq, D]; k_cache, v_cache: [N, Hkv, B, D]; block_tables: [S, W] int32;
    context_lens: [S] int32 (current token included).  An E4M3 cache (torch
    float8_e4m3fn or uint8 codes) needs k_scale, v_scale: [Hkv] per-head scales.
    """
    lib = lib or load_library()
    ks = vs = None
    if k_scale is not None:
        ks = np.ascontiguousarray(_raw(k_scale), dtype=np.float32)
        vs = np.ascontiguousarray(_raw(v_scale), dtype=np.float32)
        assert ks.shape == (num_kv_heads,) and vs.shape == (num_kv_heads,)
    qa, ka, va = _raw(q), _raw(k_cache), _raw(v_cache)
    bt = np.ascontiguousarray(_raw(block_tables), dtype=np.int32)
    cl = np.ascontiguousarray(_raw(context_lens), dtype=np.int32)
    S, Hq, D = qa.shape
    N = ka.shape[0]
    assert ka.shape == (N, num_kv_heads, block_size, D), ka.shape
    assert bt.ndim == 2 and bt.shape[0] == S and cl.shape == (S,)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    if _dtype_code(k_cache) == E4M3 and ks is None:
        raise ValueError("an E4M3 cache needs k_scale and v_scale")
    rc = lib.orc_paged_attention(_ptr(out), _ptr(qa), _dtype_code(q), _ptr(ka), _ptr(va),
                                 _dtype_code(k_cache), None if ks is None else _ptr(ks),
                                 None if vs is None else _ptr(vs), N, _ptr(bt), bt.shape[1],
                                 _ptr(cl), S, Hq, num_kv_heads, D, block_size, float(scale),
                                 int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle paged_attention rejected its inputs (status {rc})")
    return out


def chunk_attention(q, k_cache, v_cache, block_tables, context_lens, query_start,
                    scale: float, num_kv_heads: int, block_size: int, num_threads: int = 1,
                    lib=None, k_scale=None, v_scale=None) -> np.ndarray:
    """Causal attention of each sequence's chunk of new query tokens, fp64.

    q: [R, Hq, D] query rows, sequence s owning rows query_start[s] ..
    query_start[s+1]-1 (query_start: [S+1] int32, starting at 0); the chunk is the
    last n_s of the context_lens[s] cached tokens and its token j attends to cached
    tokens 0 .. L_s - n_s + j.  Returns out[R][Hq][D] as float64.
    """
    lib = lib or load_library()
    ks = vs = None
    if k_scale is not None:
        ks = np.ascontiguousarray(_raw(k_scale), dtype=np.float32)
        vs = np.ascontiguousarray(_raw(v_scale), dtype=np.float32)
        assert ks.shape == (num_kv_heads,) and vs.shape == (num_kv_heads,)
    qa, ka, va = _raw(q), _raw(k_cache), _raw(v_cache)
    bt = np.ascontiguousarray(_raw(block_tables), dtype=np.int32)
    cl = np.ascontiguousarray(_raw(context_lens), dtype=np.int32)
    qs = np.ascontiguousarray(_raw(query_start), dtype=np.int32)
    R, Hq, D = qa.shape
    S = cl.shape[0]
    N = ka.shape[0]
    assert ka.shape == (N, num_kv_heads, block_size, D), ka.shape
    assert bt.ndim == 2 and bt.shape[0] == S and qs.shape == (S + 1,)
    assert int(qs[-1]) == R, "query_start[-1] must equal the number of query rows"
    if _dtype_code(k_cache) == E4M3 and ks is None:
        raise ValueError("an E4M3 cache needs k_scale and v_scale")
    out = np.zeros((R, Hq, D), dtype=np.float64)
    rc = lib.orc_chunk_attention(_ptr(out), _ptr(qa), _dtype_code(q), _ptr(ka), _ptr(va),
                                 _dtype_code(k_cache), None if ks is None else _ptr(ks),
                                 None if vs is None else _ptr(vs), N, _ptr(bt), bt.shape[1],
                                 _ptr(cl), _ptr(qs), S, Hq, num_kv_heads, D, block_size,
                                 float(scale), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle chunk_attention rejected its inputs (status {rc})")
    return out


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, block_size: int, lib=None) -> None:
    """Scatter new tokens' K/V rows into the caches (in place; CPU tensors or arrays)."""
    lib = lib or load_library()
    ka, va = _raw(k), _raw(v)
    kc, vc = _raw(k_cache, inplace=True), _raw(v_cache, inplace=True)
    if not (kc.flags.writeable and vc.flags.writeable):
        raise ValueError("caches must be writable")
    sm = np.ascontiguousarray(_raw(slot_mapping), dtype=np.int64)
    T, Hkv, D = ka.shape
    rc = lib.orc_reshape_and_cache(_ptr(ka), _ptr(va), _ptr(kc), _ptr(vc), _ptr(sm), T, Hkv, D,
                                   block_size, kc.shape[0], _dtype_code(k))
    if rc != 0:
        raise ValueError(f"oracle reshape_and_cache rejected its inputs (status {rc})")


def reshape_and_cache_e4m3(k, v, k_cache, v_cache, slot_mapping, block_size: int, k_scale,
                           v_scale, lib=None) -> None:
    """Quantising cache write: codes e4m3(fp32(k) / k_scale[h]) into E4M3 caches
    (torch float8_e4m3fn or uint8, in place)."""
    lib = lib or load_library()
    ka, va = _raw(k), _raw(v)
    kc, vc = _raw(k_cache, inplace=True), _raw(v_cache, inplace=True)
    sm = np.ascontiguousarray(_raw(slot_mapping), dtype=np.int64)
    ks = np.ascontiguousarray(_raw(k_scale), dtype=np.float32)
    vs = np.ascontiguousarray(_raw(v_scale), dtype=np.float32)
    T, Hkv, D = ka.shape
    assert ks.shape == (Hkv,) and vs.shape == (Hkv,)
    rc = lib.orc_reshape_and_cache_e4m3(_ptr(ka), _ptr(va), _dtype_code(k), _ptr(kc), _ptr(vc),
                                        _ptr(ks), _ptr(vs), _ptr(sm), T, Hkv, D, block_size,
                                        kc.shape[0])
    if rc != 0:
        raise ValueError(f"oracle reshape_and_cache_e4m3 rejected its inputs (status {rc})")


def e4m3_to_f64(code: int) -> float:
    return load_library().orc_e4m3_to_f64(code)


def f32_to_e4m3(x: float) -> int:
    return int(load_library().orc_f32_to_e4m3(x))


def copy_blocks(caches, pairs, lib=None) -> None:
    """Copy whole blocks src -> dst in every pool of ``caches`` (in place), from the
    pre-copy state.  ``caches`` are CPU tensors/arrays whose first dim is the block id."""
    lib = lib or load_library()
    arrs = [_raw(c, inplace=True) for c in caches]
    n_blocks = arrs[0].shape[0]
    block_bytes = arrs[0].nbytes // n_blocks
    for a in arrs:
        assert a.shape[0] == n_blocks and a.nbytes // n_blocks == block_bytes
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    ptrs = (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])
    rc = lib.orc_copy_blocks(ptrs, len(arrs), _ptr(pr), pr.shape[0], block_bytes, n_blocks)
    if rc != 0:
        raise ValueError(f"oracle copy_blocks rejected its inputs (status {rc})")


def swap_blocks(src_caches, dst_caches, pairs, lib=None) -> None:
    """Move whole blocks src -> dst between two pools per cache (in place on dst):
    dst_caches[c][d] = src_caches[c][s] for every (s, d) pair.  CPU tensors/arrays whose
    first dim is the block id; the src and dst pools of a cache may differ in size."""
    lib = lib or load_library()
    srcs = [_raw(c) for c in src_caches]
    dsts = [_raw(c, inplace=True) for c in dst_caches]
    assert len(srcs) == len(dsts)
    ns, nd = srcs[0].shape[0], dsts[0].shape[0]
    bb = srcs[0].nbytes // ns
    for a in srcs:
        assert a.shape[0] == ns and a.nbytes // ns == bb
    for a in dsts:
        assert a.shape[0] == nd and a.nbytes // nd == bb
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    sp = (ctypes.c_void_p * len(srcs))(*[_ptr(a) for a in srcs])
    dp = (ctypes.c_void_p * len(dsts))(*[_ptr(a) for a in dsts])
    rc = lib.orc_swap_blocks(dp, sp, len(srcs), _ptr(pr), pr.shape[0], bb, ns, nd)
    if rc != 0:
        raise ValueError(f"oracle swap_blocks rejected its inputs (status {rc})")


def f16_bits_to_f64(bits: int) -> float:
    return load_library().orc_f16_to_f64(bits)


def bf16_bits_to_f64(bits: int) -> float:
    return load_library().orc_bf16_to_f64(bits)
