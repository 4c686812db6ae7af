"""The E4M3 tensor-core decode (head_dim 128, up to four query rows per kv head and CTA)
against the CPU oracle: context lengths on and around its 128-token tiles, partitions
that cut tiles, query rows whose magnitude needs the per-row power-of-two scaling of
the E4M3 query terms, negative and zero scales, NaN queries, empty contexts, invalid
block ids, and bitwise invariance under block relabelling.  Unused slots of every
pool hold NaN codes (the workload assembler fills them so)."""
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

# lengths on, before and after multiples of the 128-token tile
EDGE_LENS = [1, 2, 16, 127, 128, 129, 255, 256, 257, 383, 640, 1000, 2049]


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_119_gb300 import build
    build.build()


@pytest.fixture(autouse=True)
def clear_error_word(built):
    P.pa_get_device_error()
    yield


def make(lens, Hq, Hkv, B, qdtype, seed, std=1.0):
    """An E4M3 workload whose step tokens are already written (quantising cache write)."""
    rng = np.random.default_rng(seed)
    w = workloads.to_fp8(workloads._assemble("tc8", rng, "cuda", lens=lens, Hq=Hq, Hkv=Hkv,
                                             D=128, B=B, dtype=qdtype, std=std))
    if w.slot_mapping.numel():
        P.pa_reshape_and_cache_fp8(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping,
                                   w.meta["k_scale"], w.meta["v_scale"])
    return w


def decode(w, out_dtype=torch.float32, partition_size=0, q=None, scale=None):
    out = torch.empty(w.num_seqs, w.num_q_heads, 128, dtype=out_dtype, device="cuda")
    P.pa_decode_fp8(out, w.q if q is None else q, w.k_cache, w.v_cache, w.meta["k_scale"],
                    w.meta["v_scale"], w.block_tables, w.context_lens,
                    w.scale if scale is None else scale, w.num_kv_heads, w.block_size,
                    max_context_len=w.max_context_len, partition_size=partition_size)
    torch.cuda.synchronize()
    return out


def reference(w, q=None, scale=None):
    return oracle.paged_attention((w.q if q is None else q).cpu(), w.k_cache.view(torch.uint8).cpu(),
                                  w.v_cache.view(torch.uint8).cpu(), w.block_tables.cpu(),
                                  w.context_lens.cpu(), w.scale if scale is None else scale,
                                  w.num_kv_heads, w.block_size, num_threads=oracle.max_threads(),
                                  k_scale=w.meta["k_scale"].cpu(), v_scale=w.meta["v_scale"].cpu())


def assert_close(got, ref):
    got = got.double().cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "NaN pattern differs from the oracle"
    m = ~np.isnan(ref)
    err = np.abs(got[m] - ref[m]).max() if m.any() else 0.0
    assert err <= ATOL, f"max abs error {err:.3e}"


@pytest.mark.parametrize("group", [1, 2, 4])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("qdtype", [torch.bfloat16, torch.float16])
def test_tile_edges(group, B, qdtype):
    w = make(EDGE_LENS, 4 * group, 4, B, qdtype, seed=group * 10 + B)
    assert_close(decode(w), reference(w))
    assert P.pa_get_device_error() == 0


@pytest.mark.parametrize("part", [-1, 16, 48, 128, 384, 512])
def test_partitions_cut_tiles(part):
    """Partitions of 16 / 48 tokens start and end inside 128-token tiles."""
    w = make(EDGE_LENS, 8, 4, 16, torch.bfloat16, seed=part + 1000)
    assert_close(decode(w, partition_size=part), reference(w))
    assert P.pa_get_device_error() == 0


def test_split_matches_one_pass_closely():
    w = make([4096, 3000, 129], 8, 2, 32, torch.bfloat16, seed=7)
    a = decode(w, partition_size=-1).double().cpu().numpy()
    b = decode(w, partition_size=256).double().cpu().numpy()
    assert np.abs(a - b).max() <= 1e-4
    assert_close(torch.from_numpy(b), reference(w))


@pytest.mark.parametrize("out_dtype", [torch.bfloat16])
def test_native_output_rounds_the_fp32_result(out_dtype):
    w = make(EDGE_LENS, 4, 4, 16, torch.bfloat16, seed=5)
    got = decode(w, out_dtype=out_dtype).double().cpu().numpy()
    ref = reference(w)
    eps = 5e-5
    lo = torch.from_numpy((ref - eps).astype(np.float32)).to(out_dtype).double().numpy()
    hi = torch.from_numpy((ref + eps).astype(np.float32)).to(out_dtype).double().numpy()
    assert not ((got < lo) | (got > hi)).any()


@pytest.mark.parametrize("mag", [1e4, 1e-4, 2.0 ** -125, 1e30])
def test_query_magnitudes(mag):
    """Rows far from unit scale: the E4M3 query terms are taken after a power-of-two
    scaling per row, so tiny and huge rows keep their relative precision."""
    w = make([300, 700, 128], 8, 4, 16, torch.bfloat16, seed=11)
    q = w.q.float().clone()
    q[0, :4] *= mag                       # four query heads of sequence 0
    q = q.to(w.q.dtype)
    if not torch.isfinite(q).all():
        pytest.skip("magnitude not representable in the query type")
    scale = w.scale if mag < 1e3 else w.scale / float(mag)   # keep the scores finite
    assert_close(decode(w, q=q, scale=scale), reference(w, q=q, scale=scale))


@pytest.mark.parametrize("scale", [-0.09, 0.0, 1.5])
def test_negative_zero_and_large_scale(scale):
    w = make([1, 200, 640], 4, 4, 32, torch.float16, seed=13, std=0.5)
    assert_close(decode(w, scale=scale), reference(w, scale=scale))


def test_nan_query_row_gives_nan_row_only():
    w = make([200, 300, 400], 8, 4, 16, torch.bfloat16, seed=17)
    q = w.q.clone()
    q[1, 5, 7] = float("nan")
    got = decode(w, q=q)
    assert torch.isnan(got[1, 5]).all()
    got[1, 5] = 0.0
    assert torch.isfinite(got).all()


def test_empty_context_gives_zeros():
    w = make([0, 130, 0, 1], 4, 4, 16, torch.bfloat16, seed=19)
    got = decode(w)
    assert torch.equal(got[0], torch.zeros_like(got[0])) and torch.equal(got[2], got[0])
    assert_close(got, reference(w))


def test_bad_block_id_is_flagged_and_poisons_its_sequence():
    w = make([300, 500, 200], 4, 4, 16, torch.bfloat16, seed=23)
    w.block_tables[1, 3] = w.num_blocks + 9
    got = decode(w)
    assert P.pa_get_device_error() & 1
    assert torch.isnan(got[1]).all()
    assert torch.isfinite(got[0]).all() and torch.isfinite(got[2]).all()


def test_block_relabelling_is_bitwise_invariant():
    w = make(EDGE_LENS, 8, 4, 16, torch.bfloat16, seed=29)
    out1 = decode(w)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(3)).cuda()
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt2 = torch.where(w.block_tables >= 0, perm[w.block_tables.long().clamp(min=0)].int(),
                      w.block_tables)
    out2 = torch.empty_like(out1)
    P.pa_decode_fp8(out2, w.q, k2, v2, w.meta["k_scale"], w.meta["v_scale"], bt2,
                    w.context_lens, w.scale, w.num_kv_heads, w.block_size,
                    max_context_len=w.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int32), out2.view(torch.int32))
