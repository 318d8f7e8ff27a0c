"""Every forward kernel against the oracle: the 64-token cluster kernel
(forced with the handle's kernel = MHC_KERNEL_CLUSTER), its resident mode
(MHC_KERNEL_RESIDENT, n = 4: the last chunks of each CTA's range kept in
tensor memory for y), the grid-wide kernel (kernel = MHC_KERNEL_GRID), and
the automatic choice (up to 512 tokens the grid-wide kernel when the cluster
kernel would have a single tile or need more than one round of clusters; the
cluster kernel otherwise)."""
import pytest
import torch

from gpu_helpers import compare, run_cuda, run_oracle
from mhc_synth import make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mhc_hyper_connection_gb300 import build
    build.build()


KERNEL_OF = {"grid": "mhc_pre_gw_kernel", "cluster": "mhc_pre_tc_kernel", "resident": "mhc_pre_tc_kernel_resident"}


def launch_of(path):
    """Handle launch-choice fields that force a forward path."""
    from mhc_hyper_connection_gb300 import MHC_KERNEL_CLUSTER, MHC_KERNEL_GRID, MHC_KERNEL_RESIDENT
    return {"grid": {"kernel": MHC_KERNEL_GRID}, "cluster": {"kernel": MHC_KERNEL_CLUSTER},
            "resident": {"kernel": MHC_KERNEL_RESIDENT},
            "resident2": {"kernel": MHC_KERNEL_RESIDENT, "tm_buffers": 2, "cluster": 16}}.get(path, {})


def _run(case, path):
    from mhc_hyper_connection_gb300 import mhc_pre_last_kernel
    if path == "resident" and case.n != 4:
        pytest.skip("the resident mode takes n = 4")
    want = KERNEL_OF.get(path)
    if path == "auto" and case.T > 512:     # resident mode from 4096 tokens at n = 4
        want = "mhc_pre_tc_kernel_resident" if (case.T >= 4096 and case.n == 4) else "mhc_pre_tc_kernel"
    op, out = run_cuda(case, **launch_of(path))
    torch.cuda.synchronize()
    got = mhc_pre_last_kernel(op.handle)
    assert got == want if want else got in ("mhc_pre_gw_kernel", "mhc_pre_tc_kernel")
    compare(case, out, run_oracle(case))
    return out


PATHS = ["auto", "cluster", "grid", "resident"]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("name", ["tiny", "training", "decode", "generic_a", "generic_b"])
def test_workloads(cuda_device, path, name):
    _run(make_case(name, device=cuda_device), path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [1, 127, 130, 1000])
def test_ragged_tokens(cuda_device, path, T):
    _run(make_case("tiny", device=cuda_device, T=T, D=1024, need_backward=True), path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("n,alpha_len", [(6, 3), (8, 2), (8, 3)])
@pytest.mark.parametrize("D", [16, 592])
def test_streams(cuda_device, path, n, alpha_len, D):
    _run(make_case("tiny", device=cuda_device, T=300, n=n, D=D, alpha_len=alpha_len,
                   need_backward=True, gamma=True), path)


def test_grid_path_deterministic(cuda_device):
    case = make_case("training", device=cuda_device, T=777)
    op, a = run_cuda(case, **launch_of("grid"))
    _, b = run_cuda(case, op=op)
    torch.cuda.synchronize()
    for k in ("y", "h_post", "h_res", "h_pre", "inv_rms", "h_mix", "sum_out", "norm_out"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("path", ["cluster", "grid", "resident", "resident2"])
@pytest.mark.parametrize("x_dtype", [torch.bfloat16, torch.float16])
def test_repeated_runs_bitwise(cuda_device, path, x_dtype):
    """Twenty runs of one input agree bit for bit on every output: the
    reductions run in a fixed order, so any difference is a read of a
    buffer before its data is in (or after it is reused)."""
    if x_dtype == torch.float16 and path == "grid":
        pytest.skip("fp16 x runs on the cluster kernel (plain or resident) only")
    case = make_case("training", device=cuda_device, x_dtype=x_dtype)
    op, ref = run_cuda(case, **launch_of(path))
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in ref.items() if isinstance(v, torch.Tensor)}
    out = op.allocate(case.T, cuda_device)
    for _ in range(20):
        run_cuda(case, op=op, out=out)
        torch.cuda.synchronize()
        for k, v in ref.items():
            assert torch.equal(out[k], v), k


@pytest.mark.parametrize("name,kw", [("generic_a", {}), ("tiny", {"n": 6, "D": 592, "alpha_len": 3})])
def test_repeated_runs_bitwise_unpaired(cuda_device, name, kw):
    """As above for shapes that run one stream per MMA (n = 8 three-gate,
    n = 6), whose sums of squares take the single-partial hand-off."""
    case = make_case(name, device=cuda_device, **kw)
    op, ref = run_cuda(case, **launch_of("cluster"))
    torch.cuda.synchronize()
    compare(case, ref, run_oracle(case, tokens=list(range(0, case.T, max(1, case.T // 64)))),
            tokens=list(range(0, case.T, max(1, case.T // 64))))
    ref = {k: v.clone() for k, v in ref.items() if isinstance(v, torch.Tensor)}
    out = op.allocate(case.T, cuda_device)
    for _ in range(10):
        run_cuda(case, op=op, out=out)
        torch.cuda.synchronize()
        for k, v in ref.items():
            assert torch.equal(out[k], v), k


def _random_configs(count=24, seed=20261202):
    """Seeded random shapes and flags over the forward's whole scope."""
    import random
    rnd = random.Random(seed)
    out = []
    for k in range(count):
        n = rnd.choice([4, 4, 6, 8])
        out.append(dict(T=rnd.choice([1, 2, 63, 64, 65, 127, 200, 513, 700]),
                        n=n, D=16 * rnd.randint(1, 96), alpha_len=rnd.choice([2, 3]),
                        impl_mode=rnd.choice([0, 1]), gamma=rnd.random() < 0.5,
                        pre_mix=rnd.random() < 0.3, need_backward=rnd.random() < 0.5,
                        path=rnd.choice(["auto", "cluster", "grid"]), seed=k))
    return out


@pytest.mark.parametrize("cfg", _random_configs(), ids=lambda c: "T{T}_n{n}_D{D}_a{alpha_len}_m{impl_mode}_{path}".format(**c))
def test_random_shapes(cuda_device, cfg):
    """Seeded random shapes, gate forms, modes and optional inputs on every
    forward path, each compared in full with the oracle."""
    cfg = dict(cfg)
    path = cfg.pop("path")
    seed = cfg.pop("seed")
    case = make_case("tiny", device=cuda_device, seed=seed, **cfg)
    op, out = run_cuda(case, **launch_of(path))
    torch.cuda.synchronize()
    compare(case, out, run_oracle(case))


@pytest.mark.parametrize("bufs", [1, 2])
@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("mode", [0, 1])
def test_resident_cluster_sizes(cuda_device, cluster, mode, bufs):
    """Resident mode at every cluster size: 16 d-chunks per stream split over
    the cluster, so a CTA keeps 1 .. 4 (fp32 mode) or 1 .. 6 (tf32 mode)
    chunks in tensor memory (in one buffer, or half as many per tile in two
    buffers used by alternate tiles) and re-reads the rest, if any, from L2;
    ragged token count, backward outputs, gamma."""
    from mhc_hyper_connection_gb300 import mhc_pre_last_kernel, mhc_pre_last_launch
    case = make_case("tiny", device=cuda_device, T=333, D=1024, impl_mode=mode, need_backward=True, gamma=True)
    op, out = run_cuda(case, cluster=cluster, tm_buffers=bufs, **launch_of("resident"))
    torch.cuda.synchronize()
    assert mhc_pre_last_kernel(op.handle) == "mhc_pre_tc_kernel_resident"
    assert mhc_pre_last_launch(op.handle)[1]["cluster"] == cluster
    compare(case, out, run_oracle(case))


@pytest.mark.parametrize("D", [16, 80, 592, 7168])
@pytest.mark.parametrize("x_dtype", [torch.bfloat16, torch.float16])
def test_resident_widths(cuda_device, D, x_dtype):
    """Resident mode on ragged widths (the last chunk partly past D) and the
    prefill width, both x types."""
    case = make_case("tiny", device=cuda_device, T=200, D=D, x_dtype=x_dtype, need_backward=True)
    op, out = run_cuda(case, **launch_of("resident"))
    torch.cuda.synchronize()
    compare(case, out, run_oracle(case))


@pytest.mark.parametrize("cfg", _random_configs(count=12, seed=7102026), ids=lambda c: "T{T}_D{D}_a{alpha_len}_m{impl_mode}".format(**c))
def test_random_shapes_resident(cuda_device, cfg):
    """Seeded random shapes (n = 4) on the resident mode, in full."""
    cfg = dict(cfg)
    cfg.pop("path")
    seed = cfg.pop("seed")
    cfg["n"] = 4
    case = make_case("tiny", device=cuda_device, seed=seed, **cfg)
    op, out = run_cuda(case, **launch_of("resident"))
    torch.cuda.synchronize()
    compare(case, out, run_oracle(case))
