"""CUDA path vs the oracle on the same seeded inputs, through the C ABI.

Small cases are compared element by element on every token; full-size
workloads (the bench configuration included) on sampled tokens, plus
properties that hold for every token at any size.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import compare, run_cuda, run_oracle
from mhc_synth import make_case, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


def _full(case):
    _, out = run_cuda(case)
    torch.cuda.synchronize()
    return out, compare(case, out, run_oracle(case))


# ------------------------------------------------------------ workloads

@pytest.mark.parametrize("mode", [0, 1])
def test_tiny(cuda_device, mode):
    _full(make_case("tiny", device=cuda_device, impl_mode=mode))


@pytest.mark.parametrize("iters", [1, 2, 7])
def test_tiny_iterations(cuda_device, iters):
    _full(make_case("tiny", device=cuda_device, num_iters=iters, need_backward=True))


def test_training_shaped_with_backward_outputs(cuda_device):
    out, errs = _full(make_case("training", device=cuda_device))
    assert errs["inv_rms"] <= 1e-4


@pytest.mark.parametrize("mode", [0, 1])
def test_decode_shaped_outliers(cuda_device, mode):
    """Decode workload (1% of x scaled by 20).  In tf32 mode y is held to the
    same bound as in fp32 mode, against the HF32 simulation of the oracle."""
    _full(make_case("decode", device=cuda_device, impl_mode=mode))


@pytest.mark.parametrize("mode", [0, 1])
def test_prefill_sampled(cuda_device, mode):
    case = make_case("prefill", device=cuda_device, impl_mode=mode)
    _, out = run_cuda(case)
    torch.cuda.synchronize()
    tok = sample_tokens(case.T, 160, seed=mode)
    compare(case, out, run_oracle(case, tok), tokens=tok)
    _every_token_properties(case, out)


def test_generic_n8_pre_mix(cuda_device):
    _full(make_case("generic_a", device=cuda_device))


@pytest.mark.parametrize("mode", [0, 1])
def test_generic_n8_two_gates(cuda_device, mode):
    out, _ = _full(make_case("generic_b", device=cuda_device, impl_mode=mode))
    assert torch.all(out["h_res"] == 0)


@pytest.mark.parametrize("gamma", [False, True])
def test_training_tf32(cuda_device, gamma):
    """tf32 mode on the training shape, with and without gamma, intermediates
    included, against the oracle's HF32 simulation on the folded weight."""
    _full(make_case("training", device=cuda_device, impl_mode=1, gamma=gamma))


def _every_token_properties(case, out):
    """Hold for every token: column sums of comb are S/(S+eps) ~ 1, rows near
    1, gates in range, everything finite."""
    comb = out["h_res"]
    assert torch.isfinite(comb).all() and torch.isfinite(out["y"].float()).all()
    col = comb.sum(dim=1)
    assert (col - 1).abs().max().item() < 1e-6 + 8 * 2 ** -24 * case.n
    assert (comb.sum(dim=2) - 1).abs().max().item() < 1e-3
    hp = out["h_post"]
    assert hp.min().item() >= 0 and hp.max().item() <= 2 + 1e-6


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("T", [1, 5, 127, 129, 300])
def test_ragged_token_counts(cuda_device, T):
    _full(make_case("tiny", device=cuda_device, T=T, need_backward=True))


@pytest.mark.parametrize("D", [16, 48, 80, 208, 1040])
def test_ragged_widths(cuda_device, D):
    _full(make_case("tiny", device=cuda_device, T=130, D=D))


@pytest.mark.parametrize("alpha_len", [2, 3])
@pytest.mark.parametrize("n", [4, 6, 8])
@pytest.mark.parametrize("mode", [0, 1])
def test_streams_gates_modes(cuda_device, n, alpha_len, mode):
    _full(make_case("tiny", device=cuda_device, T=200, n=n, D=320, alpha_len=alpha_len,
                    impl_mode=mode, need_backward=True, gamma=True, pre_mix=(n == 6)))


def test_tf32_mode_is_the_pages_hf32(cuda_device):
    """Without gamma the tf32 mode multiplies exactly the operands the pages'
    HF32 simulation keeps, so it meets the fp32 tolerance against that oracle."""
    case = make_case("tiny", device=cuda_device, T=256, D=1024, impl_mode=1, need_backward=True)
    _, out = run_cuda(case)
    torch.cuda.synchronize()
    compare(case, out, run_oracle(case, hf32=True), tol=1e-4)


def test_empty_input(cuda_device):
    case = make_case("tiny", device=cuda_device, T=0)
    op, out = run_cuda(case)
    assert out["y"].numel() == 0


def test_deterministic(cuda_device):
    case = make_case("training", device=cuda_device, T=1000)
    op, a = run_cuda(case)
    _, b = run_cuda(case, op=op)
    torch.cuda.synchronize()
    for k in ("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix", "sum_out", "norm_out"):
        assert torch.equal(a[k], b[k]), k


def test_stream_and_reuse(cuda_device):
    """Runs on a side stream, reusing one output set for two different inputs."""
    s = torch.cuda.Stream()
    c1 = make_case("tiny", device=cuda_device, seed=1)
    c2 = make_case("tiny", device=cuda_device, seed=2)
    op, out = run_cuda(c1, stream=s)
    torch.cuda.synchronize()
    compare(c1, out, run_oracle(c1))
    run_cuda(c2, stream=s, out=out, op=op)
    torch.cuda.synchronize()
    compare(c2, out, run_oracle(c2))


def test_phi_gamma_at_4_byte_offset(cuda_device):
    """phi and gamma need only 4-byte alignment: the plane preparation takes
    the scalar-load path then, with the same results bit for bit."""
    case = make_case("training", device=cuda_device, T=100, D=512, need_backward=True)
    _, ref = run_cuda(case)
    buf = torch.empty(case.phi.numel() + 1, device=cuda_device)
    buf[1:].copy_(case.phi.reshape(-1))
    gbuf = torch.empty(case.gamma.numel() + 1, device=cuda_device)
    gbuf[1:].copy_(case.gamma.reshape(-1))
    case.phi = buf[1:].view(case.phi.shape)
    case.gamma = gbuf[1:].view(case.gamma.shape)
    assert case.phi.data_ptr() % 16 == 4
    _, out = run_cuda(case)
    torch.cuda.synchronize()
    for k in ("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix"):
        assert torch.equal(out[k], ref[k]), k


@pytest.mark.parametrize("n", [4, 6, 8])
def test_widest_rows(cuda_device, n):
    """D = 16384, the largest width the pages allow, for every n (n*D up to
    131072): a ragged token count with the backward outputs, in full."""
    _full(make_case("tiny", device=cuda_device, T=130, n=n, D=16384, need_backward=True, gamma=True))


# ------------------------------------------------------------ degenerate inputs

def _case(name, x, phi, alpha, bias, gamma=None, impl_mode=0, need_backward=False):
    from mhc_synth import Case
    T, n, D = x.shape
    return Case(name=name, T=T, n=n, D=D, alpha_len=alpha.numel(), num_iters=20, norm_eps=1e-6, hc_eps=1e-6,
                impl_mode=impl_mode, need_backward=need_backward, x=x, phi=phi, alpha=alpha, bias=bias,
                gamma=gamma, pre_mix=None)


def _uniform_comb(n, iters, eps):
    # equal logits: softmax gives 1/n, then every normalisation maps a -> a / (n a + eps)
    a = 1.0 / n + eps
    a = a / (n * a + eps)
    for _ in range(iters - 1):
        a = a / (n * a + eps)
        a = a / (n * a + eps)
    return a


@pytest.mark.parametrize("mode", [0, 1])
def test_all_ones_example(cuda_device, mode):
    """The MhcPreV2 page's worked call (x = phi = alpha = bias = gamma = 1,
    T = 2048, n = 4, D = 2560): the gates saturate and the softmax sees equal
    logits of about 10241, so this checks the max subtraction on the GPU.
    Closed forms: hPre = 1 + eps, hPost = 2, comb = the uniform scalar map,
    y = 4 (1 + eps), which rounds to 4.0 in bf16."""
    T, n, D = 2048, 4, 2560
    R, K = n * n + 2 * n, n * D
    f32 = dict(dtype=torch.float32, device=cuda_device)
    case = _case("all_ones", torch.ones((T, n, D), dtype=torch.bfloat16, device=cuda_device),
                 torch.ones((R, K), **f32), torch.ones(3, **f32), torch.ones(R, **f32), torch.ones((n, D), **f32),
                 impl_mode=mode)
    _, out = run_cuda(case)
    torch.cuda.synchronize()
    tol = 1e-4 if mode == 0 else 3e-3
    assert torch.all(out["y"] == 4.0)
    assert (out["h_pre"] - (1 + 1e-6)).abs().max().item() <= tol
    assert (out["h_post"] - 2.0).abs().max().item() <= tol
    assert (out["h_res"] - _uniform_comb(n, 20, 1e-6)).abs().max().item() <= tol
    compare(case, out, run_oracle(case, [0, 1, 1000, 2047]), tokens=[0, 1, 1000, 2047])


def test_alpha_zero(cuda_device):
    """alpha = 0: the gates reduce to the biases (hPre = sigmoid(b) + eps,
    hPost = 2 sigmoid(b)) and comb is the Sinkhorn of the bias matrix, the
    same for every token -- independent of x, phi and the projection."""
    case = make_case("training", device=cuda_device, T=1000)
    case.alpha = torch.zeros(3, dtype=torch.float32, device=cuda_device)
    _, out = run_cuda(case)
    torch.cuda.synchronize()
    n = case.n
    b = case.bias.double()
    pre = torch.sigmoid(b[:n]) + 1e-6
    post = 2 * torch.sigmoid(b[n:2 * n])
    assert (out["h_pre"].double() - pre).abs().max().item() <= 1e-4
    assert (out["h_post"].double() - post).abs().max().item() <= 1e-4
    assert torch.equal(out["h_res"], out["h_res"][:1].expand_as(out["h_res"]))
    compare(case, out, run_oracle(case, list(range(0, 1000, 37))), tokens=list(range(0, 1000, 37)))


def test_stable_inputs(cuda_device):
    """The Sinkhorn page's stable inputs (phi = 1/sqrt(nD), alpha = 0.25,
    bias = 0): every projection row of a token is the same number, so the
    four hPre of a token agree and comb is the uniform scalar map."""
    case = make_case("tiny", device=cuda_device, T=300, D=1024)
    K = case.n * case.D
    case.phi = torch.full_like(case.phi, 1.0 / K ** 0.5)
    case.alpha = torch.full((3,), 0.25, dtype=torch.float32, device=cuda_device)
    case.bias = torch.zeros_like(case.bias)
    _, out = run_cuda(case)
    torch.cuda.synchronize()
    hp = out["h_pre"]
    assert (hp - hp[:, :1]).abs().max().item() <= 1e-6
    assert (out["h_res"] - _uniform_comb(case.n, 20, 1e-6)).abs().max().item() <= 1e-6
    compare(case, out, run_oracle(case))
