"""Failure detection of the kernels' bounded waits, on the GPU, without a
fault: a wait that runs out makes the kernel give up, report through the
device error word, and leave the GPU usable for the next call.

The verify own pass (keys on the MMA's M side) takes a wait limit that a
test can lower (padoc_debug_set_wait_limit).  With a limit of 1 ns its
waits give up at once: every role leaves its loop, the TMA producers wait
for the copies they issued and the MMA thread for its products, and the CTA
frees tensor memory and exits.  padoc_device_status must then report
PADOC_ERR_DEVICE_TIMEOUT; with the default limit restored the same step
must again match the float64 oracle.  (The kernel that runs the fused
verify step keeps the default limit; its own test runs the step as two
passes.)"""
import pytest

from oracle import tree_attention as ta
from tree_structured_shared_gb300 import padoc
from tree_structured_shared_gb300 import workloads as wl

from parity import check

pytestmark = pytest.mark.gpu


def test_own_pass_wait_timeout_is_reported_and_recovered(padoc_lib, tmp_path):
    """Run in a child with the verify step as two passes
    (PADOC_VERIFY_FUSED=0, read once per process), so the keys-on-M own
    pass runs: its waits give up, the device word reports the timeout, and
    the next two steps are compared with the oracle here."""
    import os
    import subprocess
    import sys
    import numpy as np
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = tmp_path / "o.npz"
    code = (
        "import sys, numpy as np, torch; sys.path.insert(0, %r)\n"
        "from tree_structured_shared_gb300 import harness, padoc, workloads as wl\n"
        "w = wl.small_decode(77, n_pages=4, max_prefix=600, max_branches=6, max_own=300, Hq=4, Hkv=2)\n"
        "d = harness.Decode(w, wl.decode_values(w, 77), tree=True)\n"
        "padoc.device_status()\n"
        "padoc.debug_set_wait_limit(1)\n"
        "code = 0\n"
        "try:\n"
        "    d.run(); torch.cuda.synchronize()\n"
        "    try:\n"
        "        padoc.device_status()\n"
        "    except padoc.PadocError as e:\n"
        "        code = e.code\n"
        "finally:\n"
        "    padoc.debug_set_wait_limit(0)\n"
        "padoc.device_status()\n"
        "res = {'code': np.int64(code)}\n"
        "for i in range(2):\n"
        "    o, l = d.run(); torch.cuda.synchronize(); padoc.device_status()\n"
        "    res['o%%d' %% i] = o.float().cpu().numpy()[:w.n_queries]\n"
        "    res['l%%d' %% i] = l.cpu().numpy()[:w.n_queries]\n"
        "np.savez(%r, **res)\n"
    ) % (root, str(out))
    env = dict(os.environ, PADOC_VERIFY_FUSED="0")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = np.load(out)
    assert int(got["code"]) == padoc.ERR_DEVICE_TIMEOUT
    w = wl.small_decode(77, n_pages=4, max_prefix=600, max_branches=6, max_own=300, Hq=4, Hkv=2)
    O, L = ta.branch_decode(w, wl.decode_values(w, 77), tree=True)
    for i in range(2):
        check(got["o%d" % i], got["l%d" % i], O, L, "bf16", "after a timed-out own pass")
