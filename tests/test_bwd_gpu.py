"""The backward (include/mhc_pre_backward.h) against the backward oracle,
through the C ABI, on the same seeded inputs.

Both sides get the same forward intermediates: the oracle forward's, rounded
to fp32 (what the forward hands on), so no input comes from the CUDA path.

Tolerances, from the arithmetic (``abs`` is the oracle's sum of |terms| of
each output; fp32 mode / tf32 mode):
  * grad_x (bf16): |err| <= 2^-8 |ref| + c abs  -- one bf16 rounding (half an
    ulp is at most 2^-8 of the value) plus the fp32 error of the terms;
    c = 2^-14 (fp32: the only rounding before the final one is fp32
    accumulation, including the 4D-term grad_h_in . x sums), 2^-9 (tf32: G
    and phi . gamma truncated to 11 significant bits);
  * grad_phi, grad_gamma, grad_alpha, grad_bias: |err| <= c abs, c = 2^-14
    (fp32 accumulation over tokens in TMEM and in per-warp partials, plus
    the fp32 G) or 2^-9 (tf32).
A run of two identical calls must agree bitwise (fixed reduction order).
"""
import numpy as np
import pytest
import torch

import oracle
from mhc_synth import make_bwd_grads, make_case, sample_tokens

pytestmark = pytest.mark.gpu

C_REL = {0: 2.0 ** -14, 1: 2.0 ** -9}


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class _Setup:
    pass


def _setup(device, T, D, *, gamma=True, sinkhorn=True, gxp=False, impl_mode=0, seed=0, name="training"):
    from mhc_hyper_connection_gb300 import MhcPre
    case = make_case(name, seed=seed, device=device, T=T, D=D, gamma=gamma, need_backward=True,
                     impl_mode=impl_mode)
    fw = oracle.run(_bits(case.x), case.phi.cpu().numpy(), case.alpha.cpu().numpy(), case.bias.cpu().numpy(),
                    None if case.gamma is None else case.gamma.cpu().numpy(), num_iters=case.num_iters,
                    norm_eps=case.norm_eps, hc_eps=case.hc_eps, backward=True)
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    saved_np = {"inv_rms": f32(fw.inv_rms), "h_mix": f32(fw.h_mix), "h_pre": f32(fw.h_pre),
                "h_post": f32(fw.h_post),
                "sum_out": f32(fw.sum_out) if sinkhorn else None,
                "norm_out": f32(fw.norm_out) if sinkhorn else None}
    g = make_bwd_grads(seed=seed, device=device, T=T, n=case.n, D=D, grad_x_post=gxp)
    S = _Setup()
    S.case, S.g, S.saved_np = case, g, saved_np
    S.saved = {k: (None if v is None else torch.from_numpy(v).to(device)) for k, v in saved_np.items()}
    S.op = MhcPre(case.n, D, num_iters=case.num_iters, hc_eps=case.hc_eps, impl_mode=impl_mode,
                  need_backward=True)
    return S


def _run_gpu(S, grads=None):
    c = S.case
    if grads is None:
        grads = S.op.allocate_backward(c.T, c.x.device, gamma=c.gamma is not None)
    S.op.backward(c.x, c.phi, c.alpha, c.gamma, S.g.g_in, S.g.g_post, S.g.g_res, S.saved, grads,
                  grad_x_post=S.g.g_x_post)
    torch.cuda.synchronize()
    assert S.op.status(grads) == 0
    return grads


def _run_oracle(S, tokens=None, columns=None):
    c = S.case
    return oracle.run_backward(
        _bits(c.x), c.phi.cpu().numpy(), c.alpha.cpu().numpy(),
        None if c.gamma is None else c.gamma.cpu().numpy(), _bits(S.g.g_in), S.g.g_post.cpu().numpy(),
        S.g.g_res.cpu().numpy(), S.saved_np["inv_rms"], S.saved_np["h_mix"], S.saved_np["h_pre"],
        S.saved_np["h_post"], S.saved_np["sum_out"], S.saved_np["norm_out"],
        None if S.g.g_x_post is None else _bits(S.g.g_x_post), num_iters=c.num_iters, hc_eps=c.hc_eps,
        tokens=tokens, columns=columns)


def _check(S, grads, ref, tokens=None, columns=None):
    cr = C_REL[S.case.impl_mode]
    errs = {}
    gx = grads["grad_x"].float().cpu().numpy().astype(np.float64)
    if tokens is not None:
        gx = gx[tokens]
    bound = 2.0 ** -8 * np.abs(ref.grad_x) + cr * ref.grad_x_abs
    bad = np.abs(gx - ref.grad_x) > bound
    errs["grad_x"] = float((np.abs(gx - ref.grad_x) / (ref.grad_x_abs + 1e-30)).max())
    assert not bad.any(), f"grad_x: {bad.sum()} elements outside tolerance, worst {np.argwhere(bad)[:3]}"

    def chk(name, got, want, scale):
        got = np.asarray(got, dtype=np.float64)
        e = np.abs(got - want)
        errs[name] = float((e / (scale + 1e-30)).max())
        assert (e <= cr * scale + 1e-30).all(), f"{name}: max err/abs {errs[name]:.3g} > {cr:.3g}"

    gphi = grads["grad_phi"].cpu().numpy()
    if columns is not None:
        gphi = gphi[:, columns]
    chk("grad_phi", gphi, ref.grad_phi, ref.grad_phi_abs)
    if S.case.gamma is not None:
        gg = grads["grad_gamma"].cpu().numpy().reshape(-1)
        if columns is not None:
            gg = gg[columns]
        chk("grad_gamma", gg, ref.grad_gamma, ref.grad_gamma_abs)
    chk("grad_alpha", grads["grad_alpha"].cpu().numpy(), ref.grad_alpha, ref.grad_alpha_abs)
    chk("grad_bias", grads["grad_bias"].cpu().numpy(), ref.grad_bias, ref.grad_bias_abs)
    return errs


@pytest.mark.parametrize("T,D", [(1, 64), (64, 256), (65, 256), (200, 512), (1000, 1024)])
@pytest.mark.parametrize("gamma", [False, True])
def test_parity_shapes(cuda_device, T, D, gamma):
    S = _setup(cuda_device, T, D, gamma=gamma, seed=T + D)
    grads = _run_gpu(S)
    print(_check(S, grads, _run_oracle(S)))


@pytest.mark.parametrize("sinkhorn", [True, False])
@pytest.mark.parametrize("gxp", [False, True])
def test_parity_forms(cuda_device, sinkhorn, gxp):
    S = _setup(cuda_device, 300, 768, sinkhorn=sinkhorn, gxp=gxp, seed=7)
    grads = _run_gpu(S)
    print(_check(S, grads, _run_oracle(S)))


@pytest.mark.parametrize("gamma", [False, True])
def test_parity_tf32(cuda_device, gamma):
    S = _setup(cuda_device, 257, 512, gamma=gamma, impl_mode=1, seed=11)
    grads = _run_gpu(S)
    print(_check(S, grads, _run_oracle(S)))


def test_runs_span_slabs(cuda_device):
    """4096 tokens x 16 slabs: each CTA's run of items crosses slab
    boundaries, so grad_phi sums several run partials per slab."""
    S = _setup(cuda_device, 4096, 1024, seed=3)
    grads = _run_gpu(S)
    cols = np.array(sorted({0, 1, 63, 64, 511, 512, 1023, 1024, 2047, 2048, 4095, 3000, 777}), dtype=np.int64)
    toks = sample_tokens(4096, 24, seed=3, tile=64)
    print(_check(S, grads, _run_oracle(S, tokens=toks, columns=cols), tokens=toks, columns=cols))


def test_deterministic(cuda_device):
    S = _setup(cuda_device, 500, 512, seed=21, gxp=True)
    a = _run_gpu(S)
    b = _run_gpu(S)
    for k in ("grad_x", "grad_phi", "grad_alpha", "grad_bias", "grad_gamma"):
        assert torch.equal(a[k], b[k]), k


def test_empty(cuda_device):
    from mhc_hyper_connection_gb300 import MhcPre
    op = MhcPre(4, 256, need_backward=True)
    g = op.allocate_backward(0, cuda_device)
    e = torch.empty((0, 4, 256), dtype=torch.bfloat16, device=cuda_device)
    f = torch.empty((0,), dtype=torch.float32, device=cuda_device)
    phi = torch.zeros((24, 1024), device=cuda_device)
    alpha = torch.ones(3, device=cuda_device)
    saved = {"inv_rms": f, "h_mix": f, "h_pre": f, "h_post": f, "sum_out": None, "norm_out": None}
    op.backward(e, phi, alpha, None, e, f, f, saved, g)
    torch.cuda.synchronize()


def test_prefill_sampled(cuda_device):
    """T = 32768, n = 4, D = 7168 (the prefill shape) in the configuration the
    benchmark times: every output checked on sampled tokens and columns."""
    S = _setup(cuda_device, 32768, 7168, gamma=False, seed=0, name="prefill")
    grads = _run_gpu(S)
    toks = sample_tokens(32768, 16, seed=1, tile=64)
    cols = np.array(sorted({0, 63, 64, 7167, 7168, 14335, 20000, 28671}), dtype=np.int64)
    print(_check(S, grads, _run_oracle(S, tokens=toks, columns=cols), tokens=toks, columns=cols))


def test_training_shape(cuda_device):
    """The training workload (T = 4096, n = 4, D = 4096, gamma, alpha U(0.5,
    1.5)): every output on sampled tokens and columns."""
    S = _setup(cuda_device, 4096, 4096, gamma=True, seed=4, name="training")
    grads = _run_gpu(S)
    toks = sample_tokens(4096, 24, seed=2, tile=64)
    cols = np.array(sorted({0, 5, 63, 64, 4095, 4096, 8191, 9000, 16383}), dtype=np.int64)
    print(_check(S, grads, _run_oracle(S, tokens=toks, columns=cols), tokens=toks, columns=cols))


@pytest.mark.parametrize("T", [16, 64])
def test_decode_sized(cuda_device, T):
    """Decode-sized batches at D = 7168: fewer token tiles than CTAs."""
    S = _setup(cuda_device, T, 7168, gamma=False, seed=T, name="decode")
    grads = _run_gpu(S)
    print(_check(S, grads, _run_oracle(S)))


def test_phi_gamma_at_4_byte_offset(cuda_device):
    S = _setup(cuda_device, 130, 256, seed=17)
    ref = _run_gpu(S)
    c = S.case
    buf = torch.empty(c.phi.numel() + 1, device=cuda_device)
    buf[1:].copy_(c.phi.reshape(-1))
    gbuf = torch.empty(c.gamma.numel() + 1, device=cuda_device)
    gbuf[1:].copy_(c.gamma.reshape(-1))
    c.phi = buf[1:].view(c.phi.shape)
    c.gamma = gbuf[1:].view(c.gamma.shape)
    out = _run_gpu(S)
    for k in ("grad_x", "grad_phi", "grad_alpha", "grad_bias", "grad_gamma"):
        assert torch.equal(out[k], ref[k]), k


def test_repeated_runs_bitwise(cuda_device):
    """Twenty runs of one backward agree bit for bit on every gradient (the
    reductions run in a fixed order, so any difference is a read of a
    buffer before its data is in, or after it is reused)."""
    S = _setup(cuda_device, 2048, 1024, seed=5, gxp=True)
    ref = _run_gpu(S)
    ref = {k: v.clone() for k, v in ref.items() if isinstance(v, torch.Tensor)}
    grads = S.op.allocate_backward(S.case.T, cuda_device, gamma=True)
    for _ in range(20):
        _run_gpu(S, grads)
        for k, v in ref.items():
            assert torch.equal(grads[k], v), k


@pytest.mark.parametrize("D", [11264, 16384])
def test_widest_rows(cuda_device, D):
    """The widest D (16384, the pages' bound with 64-element alignment) and
    the widest that still takes a two-stage row-dot ring: every output on
    sampled tokens and columns."""
    S = _setup(cuda_device, 130, D, gamma=True, seed=D)
    grads = _run_gpu(S)
    toks = np.array(sorted({0, 1, 63, 64, 65, 127, 128, 129}), dtype=np.int64)
    cols = np.array(sorted({0, 63, 64, D - 1, D, 2 * D + 5, 4 * D - 1}), dtype=np.int64)
    print(_check(S, grads, _run_oracle(S, tokens=toks, columns=cols), tokens=toks, columns=cols))


def test_zero_upstream_gradients(cuda_device):
    """Zero gradients of y, hPost and comb give zero gradients everywhere,
    and grad_x_post passes through to grad_x unchanged (one bf16 value plus
    zero)."""
    S = _setup(cuda_device, 200, 512, seed=9, gxp=True)
    S.g.g_in.zero_()
    S.g.g_post.zero_()
    S.g.g_res.zero_()
    grads = _run_gpu(S)
    assert torch.equal(grads["grad_x"], S.g.g_x_post)
    for k in ("grad_phi", "grad_alpha", "grad_bias", "grad_gamma"):
        assert torch.count_nonzero(grads[k]).item() == 0, k


def _random_bwd_configs(count=12, seed=77):
    import random
    rnd = random.Random(seed)
    return [dict(T=rnd.choice([1, 2, 63, 64, 65, 129, 300, 700]), D=64 * rnd.randint(1, 40),
                 gamma=rnd.random() < 0.5, sinkhorn=rnd.random() < 0.7, gxp=rnd.random() < 0.4,
                 impl_mode=rnd.choice([0, 0, 1]), seed=k) for k in range(count)]


@pytest.mark.parametrize("cfg", _random_bwd_configs(),
                         ids=lambda c: "T{T}_D{D}_g{gamma:d}_s{sinkhorn:d}_x{gxp:d}_m{impl_mode}".format(**c))
def test_random_shapes(cuda_device, cfg):
    """Seeded random token counts, widths and forms, each in full against the
    backward oracle."""
    S = _setup(cuda_device, cfg["T"], cfg["D"], gamma=cfg["gamma"], sinkhorn=cfg["sinkhorn"], gxp=cfg["gxp"],
               impl_mode=cfg["impl_mode"], seed=cfg["seed"] + 1000)
    grads = _run_gpu(S)
    _check(S, grads, _run_oracle(S))
