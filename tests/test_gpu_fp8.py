"""FP8 (E4M3) KV caches on the GPU against the CPU oracle: the quantising cache write
is bit-exact over whole pools, and decode over the quantised caches (value = code x
per-kv-head scale) is within the attention tolerance, for MHA (CUDA-core kernel) and
GQA (tensor-core kernel), block sizes 16 and 32, head dims 64 and 128, split and not."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_119_gb300 as P
from paged_kv_cache_119_gb300 import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ATOL = 2e-3
NATIVE_EPS = 5e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_119_gb300 import build
    build.build()


@pytest.fixture(autouse=True)
def clear_error_word(built):
    P.pa_get_device_error()
    yield


def u8(t):
    return t.view(torch.uint8)


def step_and_compare(w, out_dtype=torch.float32, partition_size=0):
    ks, vs = w.meta["k_scale"], w.meta["v_scale"]
    snap = {n: getattr(w, n).cpu() for n in ("q", "k_cache", "v_cache", "k_new", "v_new",
                                             "slot_mapping", "block_tables", "context_lens")}
    if w.copy_pairs is not None:
        P.pa_copy_blocks([w.k_cache], [w.v_cache], w.copy_pairs)
    P.pa_reshape_and_cache_fp8(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, ks, vs)
    out = torch.empty(w.num_seqs, w.num_q_heads, w.head_dim, dtype=out_dtype, device="cuda")
    P.pa_decode_fp8(out, w.q, w.k_cache, w.v_cache, ks, vs, w.block_tables, w.context_lens,
                    w.scale, w.num_kv_heads, w.block_size, max_context_len=w.max_context_len,
                    partition_size=partition_size)
    torch.cuda.synchronize()
    kc, vc = u8(snap["k_cache"]).clone(), u8(snap["v_cache"]).clone()
    if w.copy_pairs is not None:
        oracle.copy_blocks([kc, vc], w.copy_pairs)
    oracle.reshape_and_cache_e4m3(snap["k_new"], snap["v_new"], kc, vc, snap["slot_mapping"],
                                  w.block_size, ks.cpu(), vs.cpu())
    assert torch.equal(u8(w.k_cache.cpu()), kc), "k_cache codes differ from the oracle"
    assert torch.equal(u8(w.v_cache.cpu()), vc), "v_cache codes differ from the oracle"
    ref = oracle.paged_attention(snap["q"], kc, vc, snap["block_tables"], snap["context_lens"],
                                 w.scale, w.num_kv_heads, w.block_size,
                                 num_threads=oracle.max_threads(), k_scale=ks.cpu(),
                                 v_scale=vs.cpu())
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    if out_dtype == torch.float32:
        err = np.abs(got - ref).max()
        assert err <= ATOL, f"max abs error {err:.3e}"
    else:
        lo = torch.from_numpy((ref - NATIVE_EPS).astype(np.float32)).to(out_dtype).double().numpy()
        hi = torch.from_numpy((ref + NATIVE_EPS).astype(np.float32)).to(out_dtype).double().numpy()
        assert not ((got < lo) | (got > hi)).any()
    assert P.pa_get_device_error() == 0


CASES = {
    "llama13b": dict(num_seqs=10),                                   # MHA, CUDA cores
    "opt13b": dict(num_seqs=6, max_len=900),                          # MHA, fp16 queries
    "prefix": dict(num_groups=2, group_size=4, prefix_blocks=8, max_suffix=60),   # GQA 4
    "long16": dict(num_seqs=2, context=3000),                         # GQA 8, B 16
    "long32": dict(num_seqs=2, context=3000),                         # GQA 8, B 32
}


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("part", [0, -1, 512])
def test_fp8_configs(name, part):
    w = workloads.to_fp8(workloads.make(name, device="cuda", **CASES[name]))
    step_and_compare(w, partition_size=part)


@pytest.mark.parametrize("name", ["llama13b", "long16"])
def test_fp8_native_output(name):
    w = workloads.to_fp8(workloads.make(name, device="cuda", **CASES[name]))
    step_and_compare(w, out_dtype=w.dtype)


@pytest.mark.parametrize("Hq,Hkv,D,B", [(8, 8, 64, 16), (8, 4, 64, 32), (16, 2, 64, 16),
                                         (12, 4, 128, 32), (64, 8, 128, 32)])
def test_fp8_head_groupings(Hq, Hkv, D, B):
    rng = np.random.default_rng(Hq + 7 * Hkv + D + B)
    lens = [int(x) for x in rng.integers(1, 400, size=5)]
    w = workloads._assemble("groups", rng, "cuda", lens=lens, Hq=Hq, Hkv=Hkv, D=D, B=B,
                            dtype=torch.float16, std=1.0)
    step_and_compare(workloads.to_fp8(w))


@pytest.mark.parametrize("src", [torch.float32, torch.float16, torch.bfloat16])
def test_fp8_cache_write_rounds_and_saturates(src):
    """Values at code midpoints, beyond +-448 x scale, and NaN, through the kernel."""
    Hkv, D, B, N = 2, 64, 16, 4
    ks = torch.tensor([0.5, 2.0], device="cuda")
    vs = torch.tensor([1.0, 0.25], device="cuda")
    codes = torch.arange(0, 127, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    vals = codes.float()
    mids = (vals[1:] + vals[:-1]) / 2
    pool = torch.cat([vals, mids, torch.tensor([500.0, 1e6, float("inf"), float("nan")])])
    pool = torch.cat([pool, -pool])
    T = 5
    x = pool[torch.randint(0, pool.numel(), (T, Hkv, D), generator=torch.Generator().manual_seed(3))]
    k = (x * ks.cpu()[None, :, None]).to(src)
    v = (x * vs.cpu()[None, :, None]).to(src)
    kc = torch.zeros(N, Hkv, B, D, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    slots = torch.tensor([0, 17, 33, -1, 63], device="cuda")
    P.pa_reshape_and_cache_fp8(k.cuda(), v.cuda(), kc, vc, slots, ks, vs)
    ko, vo = torch.zeros(N, Hkv, B, D, dtype=torch.uint8), torch.zeros(N, Hkv, B, D, dtype=torch.uint8)
    oracle.reshape_and_cache_e4m3(k, v, ko, vo, slots.cpu(), B, ks.cpu(), vs.cpu())
    got_k, got_v = kc.cpu(), vc.cpu()
    nan_k = (ko & 0x7F) == 0x7F
    assert torch.equal(nan_k, (got_k & 0x7F) == 0x7F)          # NaN codes where the oracle has NaN
    assert torch.equal(got_k[~nan_k], ko[~nan_k])
    nan_v = (vo & 0x7F) == 0x7F
    assert torch.equal(nan_v, (got_v & 0x7F) == 0x7F)
    assert torch.equal(got_v[~nan_v], vo[~nan_v])


@pytest.mark.parametrize("name", ["llama13b", "opt13b", "prefix", "long16", "long32"])
def test_fp8_config_full_size(name):
    """The full workloads over E4M3 caches at the launch configuration the benchmark
    times (automatic split), every output against the oracle."""
    w = workloads.to_fp8(workloads.make(name, device="cuda"))
    step_and_compare(w)


@pytest.mark.parametrize("part", [-1, 64])
def test_fp8_bad_block_inside_a_two_block_tile(part):
    """GQA 8 at head_dim 128 and block size 16 reads two cache blocks per tile.  An
    invalid id in either block of a tile (the second block of tile 1 of sequence 1, the
    first block of tile 2 of sequence 2) sets the block-id bit and makes exactly that
    sequence's rows NaN, in one pass and split into 64-token partitions; sequence 0,
    whose tiles are valid (its last tile holds one block), still matches the oracle."""
    rng = np.random.default_rng(71)
    lens = [37, 100, 250]                      # 3, 7 and 16 blocks of 16
    w = workloads.to_fp8(workloads._assemble("bad_ids", rng, "cuda", lens=lens, Hq=64, Hkv=8,
                                             D=128, B=16, dtype=torch.bfloat16, std=1.0))
    ks, vs = w.meta["k_scale"], w.meta["v_scale"]
    assert P.pa_decode_kernel_name(w.k_cache.dtype, 64, 8, 128) == "decode_mma_kernel"
    # the step's new tokens first (their slots hold the pool's NaN fill until written)
    P.pa_reshape_and_cache_fp8(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping, ks, vs)
    torch.cuda.synchronize()
    ref = oracle.paged_attention(w.q[:1].cpu(), u8(w.k_cache.cpu()), u8(w.v_cache.cpu()),
                                 w.block_tables[:1].cpu(), w.context_lens[:1].cpu(), w.scale,
                                 w.num_kv_heads, w.block_size, num_threads=oracle.max_threads(),
                                 k_scale=ks.cpu(), v_scale=vs.cpu())
    w.block_tables[1, 3] = w.k_cache.shape[0] + 5      # outside the pool
    w.block_tables[2, 4] = -7
    out = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    P.pa_decode_fp8(out, w.q, w.k_cache, w.v_cache, ks, vs, w.block_tables, w.context_lens,
                    w.scale, w.num_kv_heads, w.block_size, max_context_len=w.max_context_len,
                    partition_size=part)
    torch.cuda.synchronize()
    assert P.pa_get_device_error() == 1
    got = out.cpu()
    assert torch.isnan(got[1]).all() and torch.isnan(got[2]).all()
    err = np.abs(got[:1].double().numpy() - ref).max()
    assert err <= ATOL, f"max abs error {err:.3e}"
