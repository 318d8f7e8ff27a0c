"""The composite route (include/mhc_pre_stages.h: invRms, mixes, then gates
+ Sinkhorn + y) against the oracle with the fp32-mode tolerances of
tests/gpu_helpers.py -- every output, the invRms and mixes stages included
(they come back as inv_rms / h_mix when need_backward is set)."""
import pytest
import torch

from gpu_helpers import compare, run_oracle
from mhc_synth import make_case, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


def _composite(case):
    from mhc_hyper_connection_gb300 import MhcPre, MHC_DTYPE_BF16, MHC_DTYPE_FP16
    op = MhcPre(case.n, case.D, alpha_len=case.alpha_len, num_iters=case.num_iters, need_backward=case.need_backward,
                x_dtype=MHC_DTYPE_FP16 if case.x.dtype == torch.float16 else MHC_DTYPE_BF16)
    out = op.allocate(case.T, case.x.device)
    op.run_composite(case.x, case.phi, case.alpha, case.bias, out, gamma=case.gamma, pre_mix=case.pre_mix)
    torch.cuda.synchronize()
    assert op.status(out) == 0
    return out


@pytest.mark.parametrize("name,kw", [("tiny", {"need_backward": True}), ("training", {}), ("decode", {}),
                                     ("generic_a", {"T": 300}), ("generic_b", {"T": 300}),
                                     ("tiny", {"T": 77, "D": 80, "need_backward": True}),
                                     ("training", {"T": 100, "x_dtype": torch.float16})])
def test_composite_parity(cuda_device, name, kw):
    case = make_case(name, device=cuda_device, **kw)
    compare(case, _composite(case), run_oracle(case))


def test_composite_prefill_sampled(cuda_device):
    case = make_case("prefill", device=cuda_device, need_backward=True)
    out = _composite(case)
    tok = sample_tokens(case.T, 64, seed=5)
    compare(case, out, run_oracle(case, tok), tokens=tok)
