"""Both forward kernels against the oracle: the cluster kernel (the default)
and the grid-wide kernel, each selected with MHC_PRE_PATH."""
import pytest
import torch

from gpu_helpers import compare, run_cuda, run_oracle
from mhc_synth import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


def _run(case, path, monkeypatch):
    from mhc_hyper_connection_gb300 import mhc_pre_last_launch
    monkeypatch.setenv("MHC_PRE_PATH", path)
    op, out = run_cuda(case)
    torch.cuda.synchronize()
    st, launch = mhc_pre_last_launch(op.handle)
    assert st == 0
    assert (launch["cluster"] == 0) == (path == "grid"), launch
    compare(case, out, run_oracle(case))
    return out


PATHS = ["grid", "cluster"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", ["tiny", "training", "decode", "generic_a", "generic_b"])
def test_workloads(cuda_device, monkeypatch, path, name):
    _run(make_case(name, device=cuda_device), path, monkeypatch)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [1, 127, 130, 1000])
def test_ragged_tokens(cuda_device, monkeypatch, path, T):
    _run(make_case("tiny", device=cuda_device, T=T, D=1024, need_backward=True), path, monkeypatch)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("n,alpha_len", [(6, 3), (8, 2), (8, 3)])
@pytest.mark.parametrize("D", [16, 592])
def test_streams(cuda_device, monkeypatch, path, n, alpha_len, D):
    _run(make_case("tiny", device=cuda_device, T=300, n=n, D=D, alpha_len=alpha_len,
                   need_backward=True, gamma=True), path, monkeypatch)


def test_grid_path_deterministic(cuda_device, monkeypatch):
    monkeypatch.setenv("MHC_PRE_PATH", "grid")
    case = make_case("training", device=cuda_device, T=777)
    op, a = run_cuda(case)
    _, b = run_cuda(case, op=op)
    torch.cuda.synchronize()
    for k in ("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix", "sum_out", "norm_out"):
        assert torch.equal(a[k], b[k]), k
