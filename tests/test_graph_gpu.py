"""mhc_pre_run under CUDA stream capture: the forward's launches (plane
preparation or the prepared weights' header copy, then the fused kernel on
each kernel path) are recorded into a CUDA graph, which is then replayed on
new inputs copied into the captured buffers.  Every replay must equal an
eager run on the same inputs, bit for bit -- the launch overhead of a small
call (decode steps) is then paid once per graph, not per call."""
import pytest
import torch

from gpu_helpers import make_op
from mhc_synth import make_case

pytestmark = pytest.mark.gpu

OUT_KEYS = ("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix", "sum_out", "norm_out")


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


@pytest.mark.parametrize("name,kw,launch,prepared", [
    ("decode", {}, {}, True),                                   # grid-wide kernel, one tile
    ("decode", {}, {}, False),
    ("training", {"T": 4096}, {}, True),                        # resident mode, backward outputs
    ("training", {"T": 700, "impl_mode": 1}, {"kernel": 1}, False),   # cluster kernel, tf32
])
def test_capture_and_replay_match_eager(cuda_device, name, kw, launch, prepared):
    import mhc_hyper_connection_gb300 as mp
    cases = [make_case(name, device=cuda_device, seed=s, **kw) for s in (7, 8, 9)]
    for c in cases[1:]:                                         # one set of weights
        c.phi, c.gamma, c.alpha, c.bias = cases[0].phi, cases[0].gamma, cases[0].alpha, cases[0].bias
    op = make_op(cases[0], **launch)
    w = op.prepare_weights(cases[0].phi, cases[0].gamma) if prepared else None
    x = cases[0].x.clone()                                      # the captured input buffer
    out = op.allocate(cases[0].T, cuda_device)
    side = torch.cuda.Stream(cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(side):                               # warm-up outside the capture
        op.run(x, cases[0].phi, cases[0].alpha, cases[0].bias, out, gamma=cases[0].gamma, weights=w)
    torch.cuda.current_stream(cuda_device).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        op.run(x, cases[0].phi, cases[0].alpha, cases[0].bias, out, gamma=cases[0].gamma, weights=w)
    kern = mp.mhc_pre_last_kernel(op.handle)
    for case in cases[1:]:
        x.copy_(case.x)
        graph.replay()
        torch.cuda.synchronize()
        assert op.status(out) == mp.MHC_OK, mp.last_error()
        ref = op.allocate(case.T, cuda_device)
        op.run(case.x, case.phi, case.alpha, case.bias, ref, gamma=case.gamma, weights=w)
        assert op.status(ref) == mp.MHC_OK
        assert mp.mhc_pre_last_kernel(op.handle) == kern
        torch.cuda.synchronize()
        for k in OUT_KEYS:
            if ref.get(k) is not None:
                assert torch.equal(out[k], ref[k]), k


@pytest.mark.parametrize("T,D,gxp", [(700, 1024, False), (4096, 7168, True)])
def test_backward_capture_and_replay_match_eager(cuda_device, T, D, gxp):
    """The backward's five launches (the later four programmatic dependents
    of the one before) recorded into a CUDA graph: every replay on new
    inputs equals an eager run, bit for bit."""
    import mhc_hyper_connection_gb300 as mp
    from mhc_synth import make_bwd_grads
    cases = [make_case("training", device=cuda_device, seed=s, T=T, D=D, gamma=True, need_backward=True)
             for s in (21, 22, 23)]
    for c in cases[1:]:
        c.phi, c.gamma, c.alpha, c.bias = cases[0].phi, cases[0].gamma, cases[0].alpha, cases[0].bias
    fwd = mp.MhcPre(4, D, alpha_len=3, num_iters=cases[0].num_iters, hc_eps=cases[0].hc_eps, need_backward=True)
    keys = ("inv_rms", "h_mix", "h_pre", "h_post", "sum_out", "norm_out")
    inputs = []
    for i, c in enumerate(cases):
        out = fwd.allocate(T, cuda_device)
        fwd.run(c.x, c.phi, c.alpha, c.bias, out, gamma=c.gamma)
        assert fwd.status(out) == mp.MHC_OK
        inputs.append((c.x, {k: out[k] for k in keys}, make_bwd_grads(seed=30 + i, device=cuda_device, T=T, D=D,
                                                                       grad_x_post=gxp)))
    torch.cuda.synchronize()
    c0 = cases[0]
    op = mp.MhcPre(4, D, alpha_len=3, num_iters=c0.num_iters, hc_eps=c0.hc_eps, need_backward=True)
    # the captured buffers
    x = inputs[0][0].clone()
    saved = {k: v.clone() for k, v in inputs[0][1].items()}
    g = inputs[0][2]
    g_in, g_post, g_res = g.g_in.clone(), g.g_post.clone(), g.g_res.clone()
    g_xp = g.g_x_post.clone() if gxp else None
    grads = op.allocate_backward(T, cuda_device, gamma=True)

    def step(gr):
        op.backward(x, c0.phi, c0.alpha, c0.gamma, g_in, g_post, g_res, saved, gr, grad_x_post=g_xp)

    side = torch.cuda.Stream(cuda_device)
    side.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(side):                               # warm-up outside the capture
        step(grads)
    torch.cuda.current_stream(cuda_device).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(grads)
    for xi, si, gi in inputs[1:]:
        x.copy_(xi)
        for k in saved:
            saved[k].copy_(si[k])
        g_in.copy_(gi.g_in)
        g_post.copy_(gi.g_post)
        g_res.copy_(gi.g_res)
        if gxp:
            g_xp.copy_(gi.g_x_post)
        graph.replay()
        torch.cuda.synchronize()
        assert op.status(grads) == mp.MHC_OK, mp.last_error()
        ref = op.allocate_backward(T, cuda_device, gamma=True)
        step(ref)
        torch.cuda.synchronize()
        assert op.status(ref) == mp.MHC_OK
        for k in ("grad_x", "grad_phi", "grad_alpha", "grad_bias", "grad_gamma"):
            assert torch.equal(grads[k], ref[k]), k
