"""The post-mapping kernel (include/mhc_post.h) against its oracle, through
the C ABI.  Tolerance: |err| <= 2^-7 |ref| + 1e-3 elementwise (fp32
accumulation, one bf16 rounding); exact where the mathematics is exact."""
import numpy as np
import pytest
import torch

import oracle
from mhc_synth import make_post_case, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check(case, out, tokens=None):
    sel = (lambda a: a) if tokens is None else (lambda a: a[torch.as_tensor(tokens, device=a.device)])
    ref = oracle.run_post(_bits(sel(case.x)), _bits(sel(case.residual)), sel(case.post).cpu().numpy(),
                          sel(case.comb).cpu().numpy())
    got = sel(out).float().cpu().numpy().astype(np.float64)
    bad = np.abs(got - ref) > 2.0 ** -7 * np.abs(ref) + 1e-3
    assert not bad.any(), f"{bad.sum()} elements outside tolerance, max err {np.abs(got - ref).max():.3g}"


def _run(case):
    from mhc_hyper_connection_gb300 import hc_post
    out = hc_post(case.x, case.residual, case.post, case.comb)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("n", [1, 4, 6, 8])
@pytest.mark.parametrize("D", [8, 24, 520])
def test_shapes(cuda_device, n, D):
    case = make_post_case(device=cuda_device, T=37, n=n, D=D, seed=n * 100 + D)
    _check(case, _run(case))


@pytest.mark.parametrize("T", [1, 3, 257])
def test_ragged_tokens(cuda_device, T):
    case = make_post_case(device=cuda_device, T=T, n=4, D=256, seed=T)
    _check(case, _run(case))


def test_identity_comb_is_exact(cuda_device):
    case = make_post_case(device=cuda_device, T=50, n=4, D=1024, seed=5)
    case.post.zero_()
    case.comb.copy_(torch.eye(4, device=cuda_device).expand(50, 4, 4))
    out = _run(case)
    assert torch.equal(out, case.residual)


def test_prefill_shape_sampled(cuda_device):
    case = make_post_case(device=cuda_device, T=32768, n=4, D=7168, seed=9)
    out = _run(case)
    tok = sample_tokens(case.T, 96, seed=3)
    _check(case, out, tok)


def test_empty(cuda_device):
    from mhc_hyper_connection_gb300 import hc_post
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=cuda_device)
    r = torch.empty((0, 4, 64), dtype=torch.bfloat16, device=cuda_device)
    out = hc_post(x, r, torch.empty((0, 4), device=cuda_device), torch.empty((0, 4, 4), device=cuda_device))
    assert out.shape == (0, 4, 64)


def test_stream_and_determinism(cuda_device):
    from mhc_hyper_connection_gb300 import hc_post
    case = make_post_case(device=cuda_device, T=300, n=6, D=2048, seed=11)
    s = torch.cuda.Stream()
    a = hc_post(case.x, case.residual, case.post, case.comb, stream=s)
    b = hc_post(case.x, case.residual, case.post, case.comb, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    _check(case, a)


@pytest.mark.parametrize("n", [4, 8])
def test_widest_rows(cuda_device, n):
    """D = 16384, the widest hidden size of the pre-mapping it follows."""
    case = make_post_case(device=cuda_device, T=9, n=n, D=16384, seed=n)
    _check(case, _run(case))
