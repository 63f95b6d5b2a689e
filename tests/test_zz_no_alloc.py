"""ssm_scan_fwd_noalloc: the scan for callers that cannot allocate device memory.

Such callers (a process whose device memory all belongs to its own pool, a
plug-in host that forbids allocation after start-up, a real-time loop that must
not block in the allocator) cannot hand ssm_scan_fwd_ex the workspace it uses to
split a long sequence across blocks.  The no-alloc entry point uses a fixed
scratch array compiled into the library instead.  These tests check:

* on the CPU, that sizes whose carry records need more scratch than the array
  holds are refused before anything runs (with the limit lowered by the test
  mode, since no plan of the current planner needs more than the 2 MiB array);
* on the GPU, that its results equal ssm_scan_fwd_ex's with a caller-allocated
  workspace bit for bit, on shapes whose plans split (so the array is really
  used), over calls in a row with different inputs and different sizes (the
  array keeps the previous call's contents), and that they match the fp64 oracle.

The file name sorts last so that a run stopping at the first failure has run
every other test first."""
import numpy as np
import pytest

import oracle
import selective_state_space_128_b300 as ssm
import synth

TOL_BF16 = 1e-2


def _noalloc_null(batch, dim, L, N):
    return ssm.load().ssm_scan_fwd_noalloc(None, None, None, None, None, None, None, None, 1,
                                           None, None, batch, dim, L, N, ssm.SSM_BF16, None,
                                           None)


def test_plans_beyond_the_fixed_scratch_are_refused():
    """Every split plan over a grid of shapes either fits the fixed array or is
    refused from the sizes alone (SSM_ERR_WORKSPACE, before any pointer is looked at
    or any work is queued)."""
    limit = ssm.static_scratch_bytes()
    hdr = ssm.SCAN_STATUS_BYTES
    split = 0
    for N in (16, 32, 64, 128):
        for batch in (1, 2):
            for dim in (8, 32, 96, 512, 1024, 2048, 4096):
                need = ssm.ssm_scan_workspace_bytes(batch, dim, 1 << 20, N, ssm.SSM_BF16) - hdr
                split += need > 0
                if need > limit:
                    assert _noalloc_null(batch, dim, 1 << 20, N) == ssm.SSM_ERR_WORKSPACE
    assert split > 20   # the grid does exercise the split plans


def test_refusal_with_a_lowered_limit():
    """With the test mode's lower limit, a plan whose carry records exceed it is
    refused with SSM_ERR_WORKSPACE; with the default limit the same call passes the
    size check (and, with null pointers, fails later for another reason)."""
    batch, dim, L, N = 1, 96, 1 << 16, 16
    carry = ssm.ssm_scan_workspace_bytes(batch, dim, L, N, ssm.SSM_BF16) - ssm.SCAN_STATUS_BYTES
    assert 0 < carry <= ssm.static_scratch_bytes()
    try:
        ssm.ssm_set_test_mode(True, 1_000_000, carry - 1)
        assert _noalloc_null(batch, dim, L, N) == ssm.SSM_ERR_WORKSPACE
        ssm.ssm_set_test_mode(True, 1_000_000, carry)
        assert _noalloc_null(batch, dim, L, N) != ssm.SSM_ERR_WORKSPACE
    finally:
        ssm.ssm_set_test_mode(False)
    assert _noalloc_null(batch, dim, L, N) != ssm.SSM_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_equals_workspace_entry_point_over_calls_in_a_row():
    import torch
    from _gpu import host64, upload_scan

    # two sizes whose plans split, alternated, each with fresh inputs
    shapes = [(1, 96, 8192 + 40, 41), (2, 64, 12288, 42), (1, 96, 8192 + 40, 43)]
    for k, (batch, dim, L, seed) in enumerate(shapes):
        w = synth.scaled(synth.MAMBA_130M, batch=batch, dim=dim, seqlen=L, seed=seed)
        need = ssm.ssm_scan_workspace_bytes(w.batch, w.dim, w.seqlen, w.dstate, ssm.SSM_BF16)
        carry = need - ssm.SCAN_STATUS_BYTES
        assert 0 < carry <= ssm.static_scratch_bytes()  # the plan splits and fits the array
        x = synth.make_scan_inputs(w)
        g = upload_scan(x)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        shape_h = (w.batch, w.dim, w.dstate)
        y_ref = torch.empty_like(g["u"])
        h_ref = torch.empty(shape_h, dtype=torch.float32, device="cuda")
        ssm.ssm_scan_fwd_ex(g["u"], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"], g["D"],
                            g["z"], True, y_ref, h_ref, workspace=ws)
        y = torch.full_like(g["u"], float("nan"))
        h = torch.full(shape_h, float("nan"), dtype=torch.float32, device="cuda")
        ssm.ssm_scan_fwd_noalloc(g["u"], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"],
                                 g["D"], g["z"], True, y, h)
        torch.cuda.synchronize()
        assert ssm.ssm_status(None) == ssm.SSM_OK
        # same plan, same arithmetic: bit for bit
        assert torch.equal(y, y_ref), ("y", k)
        assert torch.equal(h, h_ref), ("final_state", k)
        if k == 0:
            # and the oracle on the split shape
            y_o, h_o = oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                   x["delta_bias"])
            assert oracle.rel_err(host64(y), y_o) <= TOL_BF16
            assert oracle.rel_err(host64(h), h_o) <= TOL_BF16
