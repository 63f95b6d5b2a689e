"""ssm_scan_fwd_noalloc: the scan for callers that cannot allocate device memory.

Such callers (a process whose device memory all belongs to its own pool, a
plug-in host that forbids allocation after start-up, a real-time loop that must
not block in the allocator) cannot hand ssm_scan_fwd_ex the workspace it uses to
split a long sequence across blocks.  The no-alloc entry point uses a fixed
scratch array compiled into the library instead.  These tests check it against
ssm_scan_fwd_ex with a caller-allocated workspace on a shape whose plan does
split (so the scratch is really used), on two calls in a row with different
inputs (the array keeps the previous call's contents), and that sizes needing
more scratch than the array holds are refused before anything runs.

The file name sorts last so that a run stopping at the first failure has run
every other test first."""
import ctypes

import numpy as np
import pytest

import oracle
import selective_state_space_128_b300 as ssm
import synth

TOL_BF16 = 1e-2


def test_plans_beyond_the_fixed_scratch_are_refused():
    """Over a grid of shapes whose plans split the sequence, every plan either fits
    the fixed array or is refused from the sizes alone (SSM_ERR_WORKSPACE, before any
    pointer is looked at or any work is queued).  With at most 8 states per lane no
    plan needs more than about 1.2 MB, so today every split plan fits."""
    limit = ssm.static_scratch_bytes()
    lib = ssm.load()
    split = 0
    for N in (16, 32, 64, 128):
        for batch in (1, 2):
            for dim in (8, 32, 96, 512, 1024, 2048, 4096):
                need = ssm.ssm_scan_workspace_bytes(batch, dim, 1 << 20, N, ssm.SSM_BF16)
                split += need > 0
                if need > limit:
                    rc = lib.ssm_scan_fwd_noalloc(None, None, None, None, None, None, None, None,
                                                  1, None, None, batch, dim, 1 << 20, N,
                                                  ssm.SSM_BF16, None, None)
                    assert rc == ssm.SSM_ERR_WORKSPACE
    assert split > 20   # the grid does exercise the split plans


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    from _gpu import host64, upload_scan

    w = synth.scaled(synth.MAMBA_130M, batch=1, dim=96, seqlen=8192 + 40, seed=41)
    need = ssm.ssm_scan_workspace_bytes(w.batch, w.dim, w.seqlen, w.dstate, ssm.SSM_BF16)
    assert 0 < need <= ssm.static_scratch_bytes()  # the plan splits and fits the array
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for call in range(2):
        x = synth.make_scan_inputs(synth.scaled(w, seed=41 + call))
        g = upload_scan(x)
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
        yn, hn, yr, hr = host64(y), host64(h), host64(y_ref), host64(h_ref)
        assert np.isfinite(yn).all() and np.isfinite(hn).all()
        assert oracle.rel_err(yn, yr) <= TOL_BF16, ("y", call)
        assert oracle.rel_err(hn, hr) <= TOL_BF16, ("final_state", call)
