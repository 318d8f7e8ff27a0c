"""The forward and backward kernels' bounded waits, made to run out on purpose and without
any fault: with mhc_pre_set_wait_test the host asks the first CTA to leave
out its last x copy (nothing is issued for it, so no copy is in flight) and
shortens the wait limit.  The waits on that copy give up, the kernel winds
down through its abort path, mhc_pre_status reports MHC_ERR_RUNTIME (the
MhcPreSinkhorn page's 361001), and the same handle's next normal run matches
the oracle -- on the cluster kernel, its resident mode and the grid-wide
kernel."""
import pytest
import torch

from gpu_helpers import compare, make_op, run_oracle
from mhc_synth import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


@pytest.mark.parametrize("path,name,T", [("cluster", "tiny", 300), ("cluster", "decode", 64),
                                         ("grid", "decode", 64), ("grid", "tiny", 700),
                                         ("resident", "tiny", 300), ("resident", "decode", 640)])
def test_wait_gives_up_then_next_run_is_clean(cuda_device, path, name, T):
    import mhc_hyper_connection_gb300 as mp
    kernel = {"cluster": mp.MHC_KERNEL_CLUSTER, "grid": mp.MHC_KERNEL_GRID, "resident": mp.MHC_KERNEL_RESIDENT}[path]
    case = make_case(name, device=cuda_device, T=T, D=1024 if name == "tiny" else None)
    op = make_op(case, kernel=kernel)
    out = op.allocate(case.T, cuda_device)

    assert mp.mhc_pre_set_wait_test(op.handle, 2000, 1) == mp.MHC_OK      # 2 ms per wait
    op.run(case.x, case.phi, case.alpha, case.bias, out)
    assert op.status(out) == mp.MHC_ERR_RUNTIME
    assert "gave up" in mp.last_error()
    word = int(out["workspace"][:4].view(torch.int32).item())
    assert word != 0 and (word & 8) == 0                # a wait bit, not the fp16 range bit
    assert mp.mhc_pre_last_kernel(op.handle) == {"cluster": "mhc_pre_tc_kernel", "grid": "mhc_pre_gw_kernel",
                                                  "resident": "mhc_pre_tc_kernel_resident"}[path]

    assert mp.mhc_pre_set_wait_test(op.handle, 0, 0) == mp.MHC_OK
    op.run(case.x, case.phi, case.alpha, case.bias, out)
    assert op.status(out) == mp.MHC_OK
    torch.cuda.synchronize()
    compare(case, out, run_oracle(case))


def test_wait_test_arguments(cuda_device):
    import mhc_hyper_connection_gb300 as mp
    op = mp.MhcPre(4, 256)
    assert mp.mhc_pre_set_wait_test(op.handle, 0, 2) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_set_wait_test(op.handle, 10_000_001, 0) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_set_wait_test(None, 0, 0) == mp.MHC_ERR_NULLPTR


def test_backward_wait_gives_up_then_next_run_is_clean(cuda_device):
    """The same for the backward: the contraction kernel's first CTA leaves
    out the copies of its last tile, its waits give up, the status reports
    MHC_ERR_RUNTIME, and the next normal run matches the oracle."""
    import mhc_hyper_connection_gb300 as mp
    from test_bwd_gpu import _check, _run_gpu, _run_oracle, _setup
    S = _setup(cuda_device, 300, 1024, seed=5)
    c = S.case
    grads = S.op.allocate_backward(c.T, cuda_device, gamma=True)
    assert mp.mhc_pre_set_wait_test(S.op.handle, 2000, 1) == mp.MHC_OK
    S.op.backward(c.x, c.phi, c.alpha, c.gamma, S.g.g_in, S.g.g_post, S.g.g_res, S.saved, grads)
    assert S.op.status(grads) == mp.MHC_ERR_RUNTIME
    assert "gave up" in mp.last_error()
    assert mp.mhc_pre_set_wait_test(S.op.handle, 0, 0) == mp.MHC_OK
    grads = _run_gpu(S, grads)
    _check(S, grads, _run_oracle(S))
