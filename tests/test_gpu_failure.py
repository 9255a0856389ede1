"""Failure detection of the kernels' bounded waits, on the GPU, without a
fault: a wait that runs out makes the kernel give up, report through the
device error word, and leave the GPU usable for the next call.

The verify own pass (keys on the MMA's M side) takes a wait limit that a
test can lower (padoc_debug_set_wait_limit).  With a limit of 1 ns its
waits give up at once: every role leaves its loop, the TMA producers wait
for the copies they issued and the MMA thread for its products, and the CTA
frees tensor memory and exits.  padoc_device_status must then report
PADOC_ERR_DEVICE_TIMEOUT; with the default limit restored the same step
must again match the float64 oracle."""
import pytest

from oracle import tree_attention as ta
from tree_structured_shared_gb300 import padoc
from tree_structured_shared_gb300 import workloads as wl

from parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def harness(padoc_lib):
    from tree_structured_shared_gb300 import harness as h
    return h


def test_own_pass_wait_timeout_is_reported_and_recovered(harness):
    import torch
    w = wl.small_decode(77, n_pages=4, max_prefix=600, max_branches=6, max_own=300, Hq=4, Hkv=2)
    vals = wl.decode_values(w, 77)
    d = harness.Decode(w, vals, tree=True)
    padoc.device_status()  # nothing pending from earlier tests
    padoc.debug_set_wait_limit(1)
    try:
        d.run()
        torch.cuda.synchronize()
        with pytest.raises(padoc.PadocError) as e:
            padoc.device_status()
        assert e.value.code == padoc.ERR_DEVICE_TIMEOUT
    finally:
        padoc.debug_set_wait_limit(0)
    padoc.device_status()  # the word was cleared by the read above
    for _ in range(2):
        o, lse = d.run()
        torch.cuda.synchronize()
        padoc.device_status()
        O, L = ta.branch_decode(w, vals, tree=True)
        nq = w.n_queries
        check(o.float().cpu().numpy()[:nq], lse.cpu().numpy()[:nq], O, L, "bf16", "after a timed-out own pass")
