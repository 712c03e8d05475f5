"""Failure detection on the GPU without faulting it.

Every wait inside the dispatch and combine pipelines is bounded (an mbarrier
try_wait with a suspend hint, a fixed number of attempts): when it runs out
the kernel sets EP_ERRBIT_TIMEOUT and returns instead of hanging.  Here a
self-test kernel waits on a barrier that nothing completes, with a limit of
a few milliseconds; the host must read the timeout bit, and the CUDA context
must still run the real path correctly afterwards.
"""
import numpy as np
import pytest
import torch

import ep_workloads as W
from oracle import ep_oracle as O
from tests import ep_harness as HN

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_topk_idx_gb300 as ep
    ep.load_library()
    return ep


def test_bounded_wait_runs_out_and_reports(ep):
    assert ep.selftest_bounded_wait(3000, signal=False) & ep.EP_ERRBIT_TIMEOUT
    assert ep.selftest_bounded_wait(3000, signal=True) == 0
    # a second timeout on a fresh stream behaves the same
    s = torch.cuda.Stream()
    assert ep.selftest_bounded_wait(1000, signal=False, stream=s) & ep.EP_ERRBIT_TIMEOUT


def test_context_usable_after_timeout(ep):
    assert ep.selftest_bounded_wait(2000, signal=False) & ep.EP_ERRBIT_TIMEOUT
    wl = W.WORKLOADS["tiny"]
    inp = W.make_inputs(wl, seed=2)
    cfg = HN.cfg_for(ep, wl)
    h = ep.ep_layout(cfg, inp["topk_idx"].cuda())
    lay = HN.oracle_layout(cfg, inp["topk_idx"].numpy())
    HN.check_layout(h, lay)
    out = ep.alloc_recv(h, with_weights=True)
    ep.ep_dispatch(h, inp["x"].cuda(), inp["topk_weights"].cuda(), **out)
    d = O.dispatch(lay, HN.bits16(inp["x"]), inp["topk_weights"].numpy(), False, False, True)
    HN.check_dispatch(h, lay, d, out, False, False)
    assert int(h.tensor("error_word").cpu()[0]) == 0      # no wait of the real path ran out
    h.free()
