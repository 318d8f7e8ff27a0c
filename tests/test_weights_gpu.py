"""The weights phase: phi (.) gamma prepared once with mhc_pre_prepare_weights
and handed to later runs as args->weights, which then skip their own
preparation.  A run with prepared weights must give the same outputs, bit for
bit, as a run that prepares them itself (same kernels, same planes), on every
forward path, both precision modes and both x types; the fp16 range check
travels with the prepared weights."""
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


@pytest.mark.parametrize("name,kw", [
    ("decode", {}),                                     # grid-wide kernel (one tile)
    ("decode", {"impl_mode": 1}),
    ("training", {}),                                   # resident mode, gamma, backward outputs
    ("training", {"impl_mode": 1, "T": 700}),           # cluster kernel, tf32 with gamma
    ("tiny", {"x_dtype": torch.float16, "T": 300, "gamma": True}),
    ("generic_a", {"T": 1000}),                         # n = 8, pre_mix
])
def test_prepared_weights_match_per_call_preparation(cuda_device, name, kw):
    import mhc_hyper_connection_gb300 as mp
    cases = [make_case(name, device=cuda_device, seed=s, **kw) for s in (3, 4)]
    # the same weights for both calls, different x
    cases[1].phi, cases[1].gamma = cases[0].phi, cases[0].gamma
    op = make_op(cases[0])
    w = op.prepare_weights(cases[0].phi, cases[0].gamma)
    for case in cases:
        ref = op.allocate(case.T, cuda_device)
        op.run(case.x, case.phi, case.alpha, case.bias, ref, gamma=case.gamma, pre_mix=case.pre_mix)
        assert op.status(ref) == mp.MHC_OK
        kern = mp.mhc_pre_last_kernel(op.handle)
        got = op.allocate(case.T, cuda_device)
        op.run(case.x, None, case.alpha, case.bias, got, pre_mix=case.pre_mix, weights=w)
        assert op.status(got) == mp.MHC_OK, mp.last_error()
        assert mp.mhc_pre_last_kernel(op.handle) == kern
        torch.cuda.synchronize()
        for k in OUT_KEYS:
            if ref.get(k) is not None:
                assert torch.equal(got[k], ref[k]), k
    compare(cases[1], got, run_oracle(cases[1]))


def test_prepared_weights_carry_the_fp16_range_check(cuda_device):
    import mhc_hyper_connection_gb300 as mp
    case = make_case("tiny", device=cuda_device, T=64, D=256, seed=5, x_dtype=torch.float16, gamma=True)
    op = make_op(case)
    bad_gamma = case.gamma.clone()
    bad_gamma[0, 0] = 1e9
    w_bad = op.prepare_weights(case.phi, bad_gamma)
    w_good = op.prepare_weights(case.phi, case.gamma)
    out = op.allocate(case.T, cuda_device)
    op.run(case.x, None, case.alpha, case.bias, out, weights=w_bad)
    assert op.status(out) == mp.MHC_ERR_RUNTIME and "fp16" in mp.last_error()
    op.run(case.x, None, case.alpha, case.bias, out, weights=w_good)
    assert op.status(out) == mp.MHC_OK
    torch.cuda.synchronize()
    compare(case, out, run_oracle(case))
