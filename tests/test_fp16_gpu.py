"""fp16 x (the other x type of the Sinkhorn page) through the C ABI: the
forward on fp16 x, with fp16 planes of phi . gamma, against the oracle's
fp16 path, within the same tolerances as bf16 x (tests/gpu_helpers.py);
y comes back in fp16.  Full-size prefill on sampled tokens; a phi . gamma
entry outside fp16's range is reported by mhc_pre_status."""
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


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("training", {}), ("decode", {}),
                                     ("training", {"alpha_len": 2}), ("tiny", {"T": 129, "D": 1040}),
                                     ("training", {"T": 300, "D": 512, "batch_consistent": True})])
@pytest.mark.parametrize("mode", [0, 1])
def test_fp16_parity(cuda_device, name, kw, mode):
    kw = dict(kw)
    consistent = kw.pop("batch_consistent", False)
    case = make_case(name, device=cuda_device, impl_mode=mode, x_dtype=torch.float16, **kw)
    from mhc_hyper_connection_gb300 import MhcPre, MHC_DTYPE_FP16
    op = MhcPre(case.n, case.D, alpha_len=case.alpha_len, num_iters=case.num_iters, impl_mode=mode,
                need_backward=case.need_backward, batch_consistent=consistent, x_dtype=MHC_DTYPE_FP16)
    _, out = run_cuda(case, op=op)
    torch.cuda.synchronize()
    assert out["y"].dtype == torch.float16
    compare(case, out, run_oracle(case))


@pytest.mark.parametrize("mode", [0, 1])
def test_fp16_prefill_sampled(cuda_device, mode):
    case = make_case("prefill", device=cuda_device, impl_mode=mode, x_dtype=torch.float16)
    _, out = run_cuda(case)
    torch.cuda.synchronize()
    tok = sample_tokens(case.T, 160, seed=mode)
    compare(case, out, run_oracle(case, tok), tokens=tok)


def test_fp16_phi_out_of_range_is_reported(cuda_device):
    from mhc_hyper_connection_gb300 import MhcPre, MHC_DTYPE_FP16, MHC_OK
    case = make_case("tiny", device=cuda_device, x_dtype=torch.float16)
    case.phi[3, 17] = 1.0e5
    op = MhcPre(case.n, case.D, x_dtype=MHC_DTYPE_FP16)
    out = op.allocate(case.T, cuda_device)
    op.run(case.x, case.phi, case.alpha, case.bias, out)
    assert op.status(out) != MHC_OK
    case.phi[3, 17] = 0.01
    op.run(case.x, case.phi, case.alpha, case.bias, out)
    assert op.status(out) == MHC_OK


def test_fp16_rejected_where_unsupported(cuda_device):
    from mhc_hyper_connection_gb300 import MhcPre, MhcError, MHC_DTYPE_FP16
    with pytest.raises(MhcError):
        MhcPre(8, 256, x_dtype=MHC_DTYPE_FP16)
    op = MhcPre(4, 256, x_dtype=MHC_DTYPE_FP16, need_backward=True)
    with pytest.raises(MhcError):
        op.backward_workspace_size(64)
