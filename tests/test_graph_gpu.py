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
