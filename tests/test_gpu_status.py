"""The scan's failure report on the GPU: a wait that runs out.

The scan kernels' only waits are on their own copies into shared memory.  The
test mode's SSM_TEST_STALL makes one block arm the barrier of a copy it never
issues (nothing is in flight for it), so that block's wait gives up after a
short limit (1 ms here) instead of 2 s, records the failure in the call's status
word and leaves.  No fault, trap or endless loop is involved: the block returns
and the context stays usable.

Checked: the stalled call's workspace reports SSM_ERR_TIMEOUT while a call
running at the same time on another stream with its own workspace reports
SSM_OK and matches the oracle; the blocks of the stalled call that did not
stall wrote their outputs; a normal call on the same workspace right after
reports SSM_OK and matches the oracle; calls without a workspace report to the
library-wide word, which ssm_status(NULL) reads and clears."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_128_b300 as ssm
import synth
from _gpu import host64, upload_scan

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _inputs():
    w = synth.scaled(synth.MAMBA_130M, batch=2, dim=96, seqlen=512, seed=61)
    x = synth.make_scan_inputs(w)
    return w, x, upload_scan(x)


def _call(g, w, flags, ws, stream):
    y = torch.full_like(g["u"], float("nan"))
    h = torch.full((w.batch, w.dim, w.dstate), float("nan"), dtype=torch.float32, device="cuda")
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())   # the fills come first
    ssm.ssm_scan_fwd_ex(g["u"], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"], g["D"],
                        g["z"], flags, y, h, None, ws, stream=stream)
    return y, h


@pytest.mark.parametrize("kernel", [ssm.SCAN_KERNEL_BLOCK, ssm.SCAN_KERNEL_PAIR])
def test_stalled_block_reports_timeout_in_its_own_workspace(kernel):
    """With either forward kernel (the block kernel and the two-warp-block kernel)."""
    w, x, g = _inputs()
    y_o, h_o = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                           x["delta_bias"])
    need = ssm.ssm_scan_workspace_bytes(w.batch, w.dim, w.seqlen, w.dstate, ssm.SSM_BF16)
    ws_a = torch.empty(need, dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(need, dtype=torch.uint8, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    ssm.ssm_set_test_mode(True, 1_000_000, scan_kernel=kernel)
    try:
        ya, ha = _call(g, w, ssm.SSM_SOFTPLUS | ssm.SSM_TEST_STALL, ws_a, sa)
        yb, hb = _call(g, w, ssm.SSM_SOFTPLUS, ws_b, sb)
        assert ssm.ssm_status(ws_a, sa) == ssm.SSM_ERR_TIMEOUT
        assert ssm.ssm_status(ws_b, sb) == ssm.SSM_OK
        yc, hc = _call(g, w, ssm.SSM_SOFTPLUS, ws_a, sa)  # the same kernel, right after
        assert ssm.ssm_status(ws_a, sa) == ssm.SSM_OK
    finally:
        ssm.ssm_set_test_mode(False)
    torch.cuda.synchronize()
    # the concurrent call is correct
    assert oracle.rel_err(host64(yb), y_o) <= TOL
    assert oracle.rel_err(host64(hb), h_o) <= TOL
    # the stalled block owns the first channels of batch row 0; every other block of the
    # stalled call finished: batch row 1 equals the normal call's
    assert torch.equal(ya[1], yb[1]) and torch.equal(ha[1], hb[1])
    # the stalled block left its final states unwritten
    assert torch.isnan(ha[0, 0]).all()
    # the context still works: a normal call on the same workspace, status OK, correct
    assert torch.equal(yc, yb) and torch.equal(hc, hb)
    assert ssm.ssm_status(None) == ssm.SSM_OK   # the library-wide word was not touched


def test_calls_without_workspace_report_to_the_library_word():
    w, x, g = _inputs()
    torch.cuda.synchronize()
    assert ssm.ssm_status(None) == ssm.SSM_OK
    ssm.ssm_set_test_mode(True, 1_000_000)
    try:
        _call(g, w, ssm.SSM_SOFTPLUS | ssm.SSM_TEST_STALL, None, None)
        assert ssm.ssm_status(None) == ssm.SSM_ERR_TIMEOUT
        assert ssm.ssm_status(None) == ssm.SSM_OK   # read and cleared
    finally:
        ssm.ssm_set_test_mode(False)
    y, h = _call(g, w, ssm.SSM_SOFTPLUS, None, None)
    assert ssm.ssm_status(None) == ssm.SSM_OK
    y_o, h_o = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                           x["delta_bias"])
    assert oracle.rel_err(host64(y), y_o) <= TOL
