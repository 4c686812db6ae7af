"""The bounded pipeline waits give up cleanly (GPU).

With the library's test hook armed, one CTA of a CUDA-core decode launch issues no copy
of the cache, so its consumer warps' waits run out after a few milliseconds instead of
completing.  Nothing is ever in flight for that CTA, so it returns like any other; no
fault, trap or hang is involved.  The launch must report PA_DEVERR_TIMEOUT in the
device error word, write NaN to exactly that CTA's rows, match the oracle everywhere
else, and leave the context usable: the next call on the same stream runs clean.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_119_gb300 as P
from paged_kv_cache_119_gb300 import _native as N
from paged_kv_cache_119_gb300 import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ATOL = 2e-3


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_119_gb300 import build
    build.build()
    return N.load()


def _decode(w):
    out = torch.zeros(w.q.shape, dtype=torch.float32, device="cuda")
    # one pass per (sequence, head), in index order: grid (1, heads, sequences)
    P.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                w.num_kv_heads, w.block_size, max_context_len=w.max_context_len,
                partition_size=-1)
    torch.cuda.synchronize()
    return out


def test_wait_timeout_poisons_one_cta_and_the_next_call_is_clean(lib):
    P.pa_get_device_error()
    w = workloads.make("llama13b", device="cuda", num_seqs=8)
    assert P.pa_decode_kernel_name(w.k_cache.dtype, w.num_q_heads, w.num_kv_heads,
                                   w.head_dim) == "decode_kernel"
    P.pa_reshape_and_cache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    torch.cuda.synchronize()
    ref = oracle.paged_attention(w.q.cpu(), w.k_cache.cpu(), w.v_cache.cpu(),
                                 w.block_tables.cpu(), w.context_lens.cpu(), w.scale,
                                 w.num_kv_heads, w.block_size, num_threads=oracle.max_threads())
    seq, head = 3, 7
    assert int(w.context_lens[seq]) > 0
    cta = 0 + 1 * (head + w.num_q_heads * seq)      # blockIdx (0, head, seq), grid (1, Hq, S)
    assert lib.pa_test_arm_wait_timeout(cta, 5000) == N.PA_OK       # 5 ms
    out = _decode(w)
    flags = P.pa_get_device_error()
    assert flags & N.PA_DEVERR_TIMEOUT, f"error word {flags:#x}"
    got = out.double().cpu().numpy()
    assert np.isnan(got[seq, head]).all()
    keep = np.ones(got.shape[:2], dtype=bool)
    keep[seq, head] = False
    assert np.isfinite(got[keep]).all()
    assert np.abs(got[keep] - ref[keep]).max() <= ATOL

    # the next call, not armed, on the same stream: clean and complete
    out = _decode(w)
    assert P.pa_get_device_error() == 0
    assert np.abs(out.double().cpu().numpy() - ref).max() <= ATOL
