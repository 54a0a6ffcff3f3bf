"""The failure path of the in-kernel waits (needs a GPU).

Every wait of the library's kernels (on a TMA copy, on a peer warp's
arrival) is bounded in time: when it runs out the kernel sets
PAGEDKV_DEVERR_TIMEOUT and exits instead of hanging. pagedkv_check_bounded_wait
enqueues a kernel whose wait is on a barrier that nothing ever arrives on;
the host must then read the timeout bit, and the context must stay usable.
No fault, trap or hang is involved.
"""
import time

import pytest
import torch

import paged_kv_cache_233_gb300 as pk
from paged_support import assert_close, gpu_decode, gpu_fill, oracle_decode, oracle_fill
from workloads import materialize, preset

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pk.load()
    torch.cuda.set_device(0)


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable(orc):
    pk.device_errors(reset=True)
    t0 = time.monotonic()
    pk.check_bounded_wait()
    flags = pk.device_errors(reset=True)   # synchronises
    elapsed = time.monotonic() - t0
    assert flags & pk.DEVERR_TIMEOUT
    assert 0.9 <= elapsed < 30.0, elapsed   # the limit is one second
    assert pk.device_errors() == 0          # the bit was cleared
    # the same context decodes correctly afterwards
    wl = preset("tiny")
    t = materialize(wl, "cuda")
    kc, vc, bt, _ = gpu_fill(wl, t)
    out, _ = gpu_decode(wl, t["q"], kc, vc, bt, 16)
    torch.cuda.synchronize()
    assert pk.device_errors() == 0
    okc, ovc, _ = oracle_fill(orc, wl, t)
    assert_close(out, oracle_decode(orc, wl, t["q"], okc, ovc), wl.dtype, what="after a timeout")
