"""mhc_pre_run_noalloc: the forward for callers that cannot allocate device
memory (code under an allocator lock, host runtimes with no device allocator
of their own, streams that must not block on cudaMalloc).  It runs the same
kernels as mhc_pre_run with the library's fixed scratch array in place of a
caller workspace, so its outputs must equal mhc_pre_run's bit for bit; here
that is checked through the C ABI on two calls in a row with different
inputs, on the cluster kernel, the grid-wide kernel (whose inter-CTA counters
live in that array) and fp16 x, plus once against the oracle.  Also: its
device error word is visible to mhc_pre_status(h, NULL, stream), and a call
leaves the device's free memory unchanged.

This file sorts last so that a run stopping at its first failure has already
run every other test; it also passes on its own in a fresh process."""
import ctypes

import pytest
import torch

from gpu_helpers import compare, make_op, run_oracle
from mhc_synth import make_case

pytestmark = pytest.mark.gpu

OUT_KEYS = ("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix", "sum_out", "norm_out")


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


def _noalloc(op, case, out, stream):
    import mhc_hyper_connection_gb300 as mp
    args = op.make_args(case.x, case.phi, case.alpha, case.bias, out, gamma=case.gamma, pre_mix=case.pre_mix)
    args.workspace = None
    args.workspace_bytes = 0
    return mp.library().mhc_pre_run_noalloc(op.handle, ctypes.byref(args), ctypes.c_void_p(stream))


def _check_pair(cases, op, device, expect_kernel=None):
    """Each case through mhc_pre_run (own workspace) and then through
    mhc_pre_run_noalloc on the same handle: identical outputs, bit for bit."""
    import mhc_hyper_connection_gb300 as mp
    stream = torch.cuda.current_stream(device).cuda_stream
    outs = []
    for case in cases:
        ref = op.allocate(case.T, device)
        op.run(case.x, case.phi, case.alpha, case.bias, ref, gamma=case.gamma, pre_mix=case.pre_mix)
        assert op.status(ref) == mp.MHC_OK
        got = op.allocate(case.T, device)
        assert _noalloc(op, case, got, stream) == mp.MHC_OK, mp.last_error()
        assert mp.mhc_pre_status(op.handle, 0, stream) == mp.MHC_OK, mp.last_error()
        if expect_kernel:
            assert mp.mhc_pre_last_kernel(op.handle) == expect_kernel
        torch.cuda.synchronize()
        for k in OUT_KEYS:
            if ref.get(k) is not None:
                assert torch.equal(got[k], ref[k]), k
        outs.append(got)
    return outs


def test_noalloc_matches_run_bitwise_on_two_calls(cuda_device):
    cases = [make_case("training", device=cuda_device, T=700, seed=11),
             make_case("training", device=cuda_device, T=300, seed=12)]
    op = make_op(cases[0])
    outs = _check_pair(cases, op, cuda_device, "mhc_pre_tc_kernel")
    # and the second call against the oracle, at the parity tolerances
    compare(cases[1], outs[1], run_oracle(cases[1]))


def test_noalloc_grid_wide_kernel_twice(cuda_device):
    """One 64-token tile at D = 7168 runs the grid-wide kernel, whose
    exchange counters and rings sit in the scratch array; two calls in a row
    reuse them."""
    cases = [make_case("decode", device=cuda_device, seed=21),
             make_case("decode", device=cuda_device, seed=22)]
    op = make_op(cases[0])
    _check_pair(cases, op, cuda_device, "mhc_pre_gw_kernel")


def test_noalloc_fp16(cuda_device):
    cases = [make_case("tiny", device=cuda_device, T=300, D=1024, seed=31, x_dtype=torch.float16),
             make_case("tiny", device=cuda_device, T=130, D=1024, seed=32, x_dtype=torch.float16)]
    op = make_op(cases[0])
    _check_pair(cases, op, cuda_device, "mhc_pre_tc_kernel")


def test_noalloc_error_word_is_reported(cuda_device):
    """fp16 x with a phi . gamma entry beyond fp16's range raises the range
    bit of the device error word; after a no-alloc run mhc_pre_status with no
    workspace reads it from the scratch array.  A following good run on the
    same handle clears it."""
    import mhc_hyper_connection_gb300 as mp
    stream = torch.cuda.current_stream(cuda_device).cuda_stream
    case = make_case("tiny", device=cuda_device, T=64, D=256, seed=41, x_dtype=torch.float16, gamma=True)
    op = make_op(case)
    bad = make_case("tiny", device=cuda_device, T=64, D=256, seed=41, x_dtype=torch.float16, gamma=True)
    bad.gamma = bad.gamma.clone()
    bad.gamma[0, 0] = 1e9          # phi[r, 0] * gamma[0] is far beyond 65504
    out = op.allocate(case.T, cuda_device)
    assert _noalloc(op, bad, out, stream) == mp.MHC_OK
    assert mp.mhc_pre_status(op.handle, 0, stream) == mp.MHC_ERR_RUNTIME
    assert "fp16" in mp.last_error()
    assert _noalloc(op, case, out, stream) == mp.MHC_OK
    assert mp.mhc_pre_status(op.handle, 0, stream) == mp.MHC_OK, mp.last_error()


def test_noalloc_allocates_nothing(cuda_device):
    """After a first call (which may load kernels lazily), a call leaves the
    device's free memory and torch's reserved memory unchanged."""
    import mhc_hyper_connection_gb300 as mp
    stream = torch.cuda.current_stream(cuda_device).cuda_stream
    case = make_case("training", device=cuda_device, T=500, seed=51)
    op = make_op(case)
    out = op.allocate(case.T, cuda_device)
    assert _noalloc(op, case, out, stream) == mp.MHC_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(cuda_device)
    reserved0 = torch.cuda.memory_reserved(cuda_device)
    assert _noalloc(op, case, out, stream) == mp.MHC_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(cuda_device)
    assert free1 == free0 and torch.cuda.memory_reserved(cuda_device) == reserved0
    assert mp.mhc_pre_status(op.handle, 0, stream) == mp.MHC_OK


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
