"""pa_decode_noalloc against pa_decode and the CPU oracle, through the C ABI, on the GPU.

pa_decode_noalloc is for callers that cannot allocate device memory on the
decode path (for example a plugin whose host runtime owns all device memory and
forbids cudaMalloc in its enqueue hook).  It runs the split-context decode with
its scratch in the library's fixed static device array.  This file sorts last
so a failure here comes after every other test has run.
"""
import numpy as np
import pytest
import torch

import oracle

import paged_kv_cache_119_gb300 as P
from paged_kv_cache_119_gb300 import _native as N
from paged_kv_cache_119_gb300 import workloads

pytestmark = pytest.mark.gpu

ATOL = 2e-3          # the attention tolerance of the other parity tests (fp32 output)

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_119_gb300 import build
    build.build()
    return N.load()


def _noalloc(lib, out, w, part):
    return lib.pa_decode_noalloc(out.data_ptr(), N.PA_F32, w.q.data_ptr(), w.k_cache.data_ptr(),
                                 w.v_cache.data_ptr(), {torch.bfloat16: N.PA_BF16,
                                                        torch.float16: N.PA_F16,
                                                        torch.float32: N.PA_F32}[w.dtype],
                                 w.num_blocks, w.block_tables.data_ptr(),
                                 w.block_tables.stride(0), w.context_lens.data_ptr(),
                                 w.max_context_len, w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                 w.head_dim, w.block_size, w.scale, part,
                                 torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,kw,part", [
    ("long16", dict(num_seqs=2, context=4000), 512),
    ("llama13b", dict(num_seqs=24), 256),
    ("opt13b", dict(num_seqs=8, max_len=1500), 0),
])
def test_noalloc_matches_pa_decode_on_two_calls(lib, name, kw, part):
    P.pa_get_device_error()
    w = workloads.make(name, device="cuda", **kw)
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    ref = torch.empty(w.num_seqs, w.num_q_heads, w.head_dim, device="cuda")
    P.pa_decode(ref, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                w.num_kv_heads, w.block_size, max_context_len=w.max_context_len,
                partition_size=part if part > 0 else 512)
    torch.cuda.synchronize()
    exact = oracle.paged_attention(w.q.cpu(), w.k_cache.cpu(), w.v_cache.cpu(),
                                   w.block_tables.cpu(), w.context_lens.cpu(), w.scale,
                                   w.num_kv_heads, w.block_size, num_threads=oracle.max_threads())
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, out, w, part) == N.PA_OK
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), f"call {call}: non-finite output"
        err = (out - ref).abs().max().item()
        assert err <= ATOL, f"call {call}: max abs difference from pa_decode {err:.3e}"
        err = float(np.abs(out.double().cpu().numpy() - exact).max())
        assert err <= ATOL, f"call {call}: max abs error vs the oracle {err:.3e}"
    assert P.pa_get_device_error() == 0


def test_noalloc_calls_allocate_nothing(lib):
    """After the first call on the device (which looks up the scratch array's address),
    further calls leave the device's free memory and torch's allocation count as they
    were."""
    w = workloads.make("long16", device="cuda", num_seqs=2, context=4000)
    out = torch.empty(w.num_seqs, w.num_q_heads, w.head_dim, device="cuda")
    assert _noalloc(lib, out, w, 512) == N.PA_OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    allocs0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    for _ in range(3):
        assert _noalloc(lib, out, w, 512) == N.PA_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs0
    assert P.pa_get_device_error() == 0


def test_noalloc_rejects_more_than_its_scratch(lib):
    w = workloads.make("tiny", device="cuda")
    out = torch.empty(w.num_seqs, w.num_q_heads, w.head_dim, device="cuda")
    # 64 seqs x 64 heads x 64 partitions of (128 + 2) fp32 values > 32 MiB
    need = lib.pa_decode_workspace_bytes(64, 64, 128, 32768, 16, 512)
    assert need > N.PA_NOALLOC_SCRATCH_BYTES
    status = lib.pa_decode_noalloc(out.data_ptr(), N.PA_F32, w.q.data_ptr(), w.k_cache.data_ptr(),
                                   w.v_cache.data_ptr(), N.PA_F32, w.num_blocks,
                                   w.block_tables.data_ptr(), 2048, w.context_lens.data_ptr(),
                                   32768, 64, 64, 8, 128, 16, 0.1, 512, None)
    assert status == N.PA_ERR_WORKSPACE
