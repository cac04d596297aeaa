"""The bounded-wait failure path on the GPU, without faulting or hanging it.

fa_selftest_wait_timeout() enqueues one CTA whose pipeline wait can never
complete; the wait must give up after its time limit, the CTA's second wait
must follow through the abort flag, fa_sync_status() must report
FA_ERR_TIMEOUT once and then clear, and the device must stay usable (a
normal forward afterwards still matches the oracle).
"""

import ctypes
import time

import numpy as np
import pytest
import torch

from exact_tiled_attention_12_gb300.synthetic import make_inputs

from ._helpers import to64

pytestmark = pytest.mark.gpu

FA_ERR_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def test_wait_timeout_is_reported_and_the_device_stays_usable():
    import oracle

    import exact_tiled_attention_12_gb300 as fa

    assert fa.sync_status() == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    assert fa.lib().fa_selftest_wait_timeout(stream) == 0
    assert fa.sync_status() == FA_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    # one wait limit (2 s, or the poll-count backstop if that comes first);
    # the second wait ends through the abort flag, not through its own limit
    assert 0.5 <= elapsed <= 30.0, elapsed
    assert fa.sync_status() == 0            # reported once, then cleared
    q, k, v, _ = make_inputs(1, 1, 256, 128, "bf16", "normal", 71, device="cuda")
    o, lse = fa.fwd(q, k, v)
    assert fa.sync_status() == 0
    ref_o, ref_lse = oracle.attention_forward_head(to64(q[0, 0]), to64(k[0, 0]), to64(v[0, 0]), 128 ** -0.5)
    assert np.max(np.abs(to64(o[0, 0]) - ref_o)) <= 1e-2
    assert np.max(np.abs(to64(lse[0, 0]) - ref_lse)) <= 1e-3
