"""The bandwidth probes read what they claim (GPU).

pa_stream_read and pa_stream_read_runs XOR every 32-bit word they load into a sink word,
so the sink must equal the XOR of exactly the words they were asked to read: all of the
buffer for the sequential probe and for a permutation of its runs, only the in-range runs
when the order holds entries past the end (those are skipped and counted).
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_119_gb300 as P

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_119_gb300 import build
    build.build()


def xor_words(a: np.ndarray) -> int:
    return int(np.bitwise_xor.reduce(a.view(np.uint32).ravel()))


def random_words(n, seed):
    return np.random.default_rng(seed).integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, (1 << 20) + 16 * 37])
def test_stream_read_checksum_is_the_xor_of_the_buffer(nbytes):
    words = random_words(nbytes // 4, nbytes)
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    P.pa_stream_read(buf, sink)
    torch.cuda.synchronize()
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == xor_words(words)


@pytest.mark.parametrize("run", [1024, 2048, 4096, 16384])
def test_run_read_reads_each_listed_run_once(run):
    nruns = 300
    words = random_words(nruns * run // 4, run)
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    order = torch.randperm(nruns, generator=torch.Generator().manual_seed(run),
                           dtype=torch.int32).cuda()
    sink = torch.zeros(2, dtype=torch.int32, device="cuda")
    P.pa_stream_read_runs(buf, run, order, sink)
    torch.cuda.synchronize()
    got = sink.cpu().numpy().view(np.uint32)
    assert int(got[0]) == xor_words(words) and int(got[1]) == 0


def test_run_read_skips_and_counts_entries_past_the_end():
    run, nruns = 2048, 64
    words = random_words(nruns * run // 4, 5)
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    listed = [3, 70, 5, 64, 9, 1000, 5]          # 5 twice (cancels), three past the end
    order = torch.tensor(listed, dtype=torch.int32, device="cuda")
    sink = torch.zeros(2, dtype=torch.int32, device="cuda")
    P.pa_stream_read_runs(buf, run, order, sink)
    torch.cuda.synchronize()
    runs = words.reshape(nruns, run // 4)
    want = 0
    for r in listed:
        if r < nruns:
            want ^= xor_words(runs[r])
    got = sink.cpu().numpy().view(np.uint32)
    assert int(got[0]) == want and int(got[1]) == 3


def test_run_read_rejects_other_run_sizes():
    buf = torch.zeros(4096, dtype=torch.int32, device="cuda")
    order = torch.zeros(4, dtype=torch.int32, device="cuda")
    sink = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(Exception):
        P.pa_stream_read_runs(buf, 3000, order, sink)
