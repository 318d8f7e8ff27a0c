"""mhc_pre_run_noalloc: the forward for callers that cannot allocate device
memory (it uses the library's fixed scratch array instead of a caller
workspace).  Checked through the C ABI against mhc_pre_run on the same
inputs, on two calls in a row with different inputs, within the parity
tolerances.  This file sorts last so that a run stopping at its first failure
has already run every other test; it also passes on its own in a fresh
process."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import TOL
from mhc_synth import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


def test_noalloc_matches_run_on_two_calls(cuda_device):
    import mhc_hyper_connection_gb300 as mp
    lib = mp.library()
    cases = [make_case("training", device=cuda_device, T=700, seed=11),
             make_case("training", device=cuda_device, T=300, seed=12)]
    op = mp.MhcPre(cases[0].n, cases[0].D, need_backward=True)
    for case in cases:
        ref = op.allocate(case.T, cuda_device)
        op.run(case.x, case.phi, case.alpha, case.bias, ref, gamma=case.gamma)
        got = op.allocate(case.T, cuda_device)
        args = op.make_args(case.x, case.phi, case.alpha, case.bias, got, gamma=case.gamma)
        args.workspace = None
        args.workspace_bytes = 0
        stream = torch.cuda.current_stream(cuda_device).cuda_stream
        st = lib.mhc_pre_run_noalloc(op.handle, ctypes.byref(args), ctypes.c_void_p(stream))
        assert st == mp.MHC_OK, mp.last_error()
        assert mp.mhc_pre_status(op.handle, 0, stream) == mp.MHC_OK
        torch.cuda.synchronize()
        tol = TOL[case.impl_mode]
        for k in ("h_post", "h_res", "h_pre", "inv_rms", "norm_out"):
            assert float((got[k] - ref[k]).abs().max()) <= tol, k
        y_ref = ref["y"].float()
        assert torch.all((got["y"].float() - y_ref).abs() <= 2.0 ** -7 * y_ref.abs() + 1e-3)


def test_noalloc_rejects_workspace_and_oversize(cuda_device):
    import mhc_hyper_connection_gb300 as mp
    lib = mp.library()
    case = make_case("tiny", device=cuda_device)
    op = mp.MhcPre(case.n, case.D)
    out = op.allocate(case.T, cuda_device)
    args = op.make_args(case.x, case.phi, case.alpha, case.bias, out)
    # a workspace is not accepted here
    assert lib.mhc_pre_run_noalloc(op.handle, ctypes.byref(args), None) == mp.MHC_ERR_PARAM_INVALID
    # a shape whose scratch exceeds the fixed array is refused before any launch
    big = mp.MhcPre(8, 16384)
    need = big.workspace_size(1)
    assert need > 16 << 20
    args2 = mp.MhcPreArgs()
    args2.T = 1
    for f in ("x", "phi", "alpha", "bias", "y", "h_post", "h_res"):
        setattr(args2, f, 1 << 20)
    assert lib.mhc_pre_run_noalloc(big.handle, ctypes.byref(args2), None) == mp.MHC_ERR_PARAM_INVALID
    assert "scratch" in mp.last_error()
