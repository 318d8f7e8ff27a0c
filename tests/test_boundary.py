"""The C ABI without a GPU: the library loads, exports every function that
include/*.h declares, and rejects bad arguments on the host, with the status
codes of the pages, before any CUDA call."""
import ctypes
import os
import re

import pytest

import mhc_hyper_connection_gb300 as mp
from mhc_hyper_connection_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h)
           for h in ("mhc_pre.h", "mhc_post.h", "mhc_pre_backward.h", "mhc_pre_stages.h")]


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return mp.library()


def declared_functions():
    names = set()
    for header in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(header).read(), flags=re.S)
        names |= set(re.findall(r"\b(mhc_(?:pre|post)_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_api():
    names = declared_functions()
    for need in ("mhc_pre_create", "mhc_pre_workspace_size", "mhc_pre_run", "mhc_pre_status",
                 "mhc_pre_destroy", "mhc_pre_config_default", "mhc_pre_status_string",
                 "mhc_pre_last_error", "mhc_post_run", "mhc_pre_backward_workspace_size",
                 "mhc_pre_backward_run"):
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_struct_layouts_match_header():
    # Field order/sizes in the binding mirror the header (x86-64 and aarch64 LP64).
    assert ctypes.sizeof(mp.MhcPreConfig) == 8 + 8 + 4 + 4 + 8 + 8 + 4 + 4 + 4 + 4 + 8 * 4
    assert ctypes.sizeof(mp.MhcPreArgs) == 8 + 15 * 8 + 8 + 8
    assert ctypes.sizeof(mp.MhcPreBwdArgs) == 8 + 20 * 8 + 8


def test_defaults(lib):
    c = mp.mhc_pre_config_default()
    assert (c.n, c.D, c.alpha_len, c.num_iters, c.impl_mode, c.need_backward) == (4, 0, 3, 20, 0, 0)
    assert (c.batch_consistent, c.x_dtype) == (0, mp.MHC_DTYPE_BF16)
    assert c.norm_eps == 1e-6 and c.hc_eps == 1e-6
    assert all(getattr(c, f) == 0 for f in mp.LAUNCH_FIELDS)
    assert c.kernel == mp.MHC_KERNEL_AUTO


@pytest.mark.parametrize("field,value", [("n", 5), ("n", 2), ("D", 0), ("D", 24), ("D", 16400),
                                         ("alpha_len", 1), ("num_iters", 0), ("impl_mode", 2),
                                         ("impl_mode", -1), ("need_backward", 2),
                                         ("batch_consistent", 2), ("batch_consistent", -1),
                                         ("x_dtype", 2), ("x_dtype", -1),
                                         ("kernel", 4), ("kernel", -1), ("cluster", 3), ("cluster", 32),
                                         ("x_stages", 1), ("x_stages", 9), ("w_stages", 1), ("w_stages", 9),
                                         ("gw_groups", 3), ("gw_groups", -1), ("gw_x_stages", 1),
                                         ("gw_x_lead", 16), ("gw_x_lead", -1), ("tm_buffers", 3),
                                         ("tm_buffers", -1)])
def test_create_rejects_bad_config(lib, field, value):
    c = mp.mhc_pre_config_default()
    c.D = 256
    setattr(c, field, value)
    st, h = mp.mhc_pre_create(c)
    assert st == mp.MHC_ERR_PARAM_INVALID and h is None
    assert mp.last_error()


def test_create_accepts_launch_choices(lib):
    for kw in ({"kernel": mp.MHC_KERNEL_CLUSTER, "cluster": 4, "x_stages": 3, "w_stages": 2},
               {"kernel": mp.MHC_KERNEL_GRID, "gw_groups": 1, "gw_x_stages": 4, "gw_x_lead": 3}):
        op = mp.MhcPre(4, 256, **kw)
        assert op.handle is not None
        op.close()
    with pytest.raises(TypeError):
        mp.MhcPre(4, 256, tile=128)
    # batch-consistent mode fixes the cluster size itself
    c = mp.mhc_pre_config_default()
    c.D, c.batch_consistent, c.cluster = 256, 1, 4
    st, h = mp.mhc_pre_create(c)
    assert st == mp.MHC_ERR_PARAM_INVALID and h is None


def test_library_reads_no_environment():
    """Launch choices are handle fields: no C source of the library reads an
    environment variable."""
    csrc = os.path.join(ROOT, "mhc_hyper_connection_gb300", "csrc")
    for name in os.listdir(csrc):
        text = open(os.path.join(csrc, name)).read()
        assert "getenv" not in text and "environ" not in text, name


def test_create_null(lib):
    h = ctypes.c_void_p()
    assert lib.mhc_pre_create(ctypes.byref(h), None) == mp.MHC_ERR_NULLPTR
    assert lib.mhc_pre_create(None, None) == mp.MHC_ERR_NULLPTR


def test_status_strings(lib):
    assert mp.status_string(0) == "success"
    assert "NULL" in mp.status_string(161001)
    assert mp.status_string(361001)


def _handle(**kw):
    c = mp.mhc_pre_config_default()
    c.D = kw.pop("D", 256)
    for k, v in kw.items():
        setattr(c, k, v)
    st, h = mp.mhc_pre_create(c)
    assert st == mp.MHC_OK
    return h


def test_workspace_size(lib):
    h = _handle()
    st, n0 = mp.mhc_pre_workspace_size(h, 0)
    assert st == 0 and n0 == 0
    st, n1 = mp.mhc_pre_workspace_size(h, 64)
    # header + swizzled plane blocks (4 chunks x 4 streams x 72 rows of 128 bytes) +
    # the grid-wide exchange rings: 8 slots x 64 tokens x 160 CTAs x 28
    # floats of partials and 2 groups x 8 x 64 x n floats of y weights
    rings = 8 * 64 * 160 * 28 * 4 + 2 * 8 * 64 * 4 * 4
    assert st == 0 and n1 == 256 + 4 * 4 * 72 * 128 + rings
    st, _ = mp.mhc_pre_workspace_size(h, -1)
    assert st == mp.MHC_ERR_PARAM_INVALID
    h2 = _handle(impl_mode=1)
    assert mp.mhc_pre_workspace_size(h2, 64)[1] == 256 + 4 * 4 * 48 * 128 + rings
    mp.mhc_pre_destroy(h)
    mp.mhc_pre_destroy(h2)


def test_weights_phase_host_checks(lib):
    h = _handle()
    st, nb = mp.mhc_pre_weights_size(h)
    assert st == 0 and nb == 256 + 4 * 4 * 72 * 128          # header + the planes (D = 256)
    assert mp.mhc_pre_weights_size(None)[0] == mp.MHC_ERR_NULLPTR
    fake = 1 << 20
    assert mp.mhc_pre_prepare_weights(h, 0, 0, fake, nb) == mp.MHC_ERR_NULLPTR        # no phi
    assert mp.mhc_pre_prepare_weights(h, fake, 0, 0, nb) == mp.MHC_ERR_NULLPTR        # no buffer
    assert mp.mhc_pre_prepare_weights(h, fake, 0, fake + 16, nb) == mp.MHC_ERR_PARAM_INVALID   # alignment
    assert mp.mhc_pre_prepare_weights(h, fake, 0, fake, nb - 1) == mp.MHC_ERR_PARAM_INVALID    # too small
    # without a GPU the checks pass and the launch fails loudly
    assert mp.mhc_pre_prepare_weights(h, fake, 0, fake, nb) == mp.MHC_ERR_RUNTIME
    # a run given weights needs no phi; misaligned weights are refused
    a = _args(phi=0)
    assert lib.mhc_pre_run(h, ctypes.byref(a), None) == mp.MHC_ERR_NULLPTR
    a = _args(phi=0, weights=fake + 16)
    assert lib.mhc_pre_run(h, ctypes.byref(a), None) == mp.MHC_ERR_PARAM_INVALID
    a = _args(phi=0, weights=fake)
    assert lib.mhc_pre_run(h, ctypes.byref(a), None) == mp.MHC_ERR_RUNTIME
    mp.mhc_pre_destroy(h)


def _args(T=64, **over):
    a = mp.MhcPreArgs()
    fake = 1 << 20          # aligned, never dereferenced: validation fails first
    a.T = T
    for k in ("x", "phi", "alpha", "bias", "y", "h_post", "h_res"):
        setattr(a, k, fake)
    a.workspace = fake
    a.workspace_bytes = 1 << 30
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field", ["x", "phi", "alpha", "bias", "y", "h_post", "h_res"])
def test_run_null_required(lib, field):
    h = _handle()
    assert mp.mhc_pre_run(h, _args(**{field: None})) == mp.MHC_ERR_NULLPTR
    mp.mhc_pre_destroy(h)


def test_run_two_gate_h_res_optional_and_no_sinkhorn_outputs(lib):
    h = _handle(alpha_len=2, need_backward=1)
    a = _args(h_res=None, h_pre=1 << 20, inv_rms=1 << 20, h_mix=1 << 20, sum_out=1 << 20)
    assert mp.mhc_pre_run(h, a) == mp.MHC_ERR_PARAM_INVALID     # sum_out has no meaning here
    mp.mhc_pre_destroy(h)


def test_run_optional_group(lib):
    h = _handle(need_backward=1)
    full = dict(h_pre=1 << 20, inv_rms=1 << 20, h_mix=1 << 20, sum_out=1 << 20, norm_out=1 << 20)
    for drop in full:
        part = dict(full)
        part[drop] = None
        assert mp.mhc_pre_run(h, _args(**part)) == mp.MHC_ERR_NULLPTR, drop
    mp.mhc_pre_destroy(h)
    h = _handle(need_backward=0)
    assert mp.mhc_pre_run(h, _args(inv_rms=1 << 20)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_run(h, _args(pre_mix=1 << 20)) == mp.MHC_ERR_NULLPTR   # needs h_pre
    mp.mhc_pre_destroy(h)


def test_run_alignment_and_workspace(lib):
    h = _handle()
    assert mp.mhc_pre_run(h, _args(x=(1 << 20) + 8)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_run(h, _args(y=(1 << 20) + 2)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_run(h, _args(phi=(1 << 20) + 2)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_run(h, _args(workspace_bytes=100)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_run(h, _args(workspace=None)) == mp.MHC_ERR_NULLPTR
    assert mp.mhc_pre_run(h, _args(workspace=(1 << 20) + 16)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_run(h, _args(T=-1)) == mp.MHC_ERR_PARAM_INVALID
    mp.mhc_pre_destroy(h)


def test_run_empty_is_ok_without_launch(lib):
    h = _handle()
    assert mp.mhc_pre_run(h, _args(T=0, workspace=None, workspace_bytes=0)) == mp.MHC_OK
    mp.mhc_pre_destroy(h)


def test_run_without_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = _handle()
    assert mp.mhc_pre_run(h, _args()) == mp.MHC_ERR_RUNTIME
    mp.mhc_pre_destroy(h)


def test_binding_raises_when_library_missing(monkeypatch, tmp_path):
    from mhc_hyper_connection_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _binding.library()


def test_post_host_validation(lib):
    A = 1 << 20          # a 16-byte aligned fake device address (never dereferenced)
    ok = dict(T=4, n=4, D=64, x=A, residual=A, post=A, comb=A, out=A)

    def call(**kw):
        a = dict(ok, **kw)
        return mp.mhc_post_run(a["T"], a["n"], a["D"], a["x"], a["residual"], a["post"], a["comb"], a["out"])

    assert call(T=0, x=0, residual=0, post=0, comb=0, out=0) == mp.MHC_OK
    assert call(n=0) == mp.MHC_ERR_PARAM_INVALID
    assert call(n=9) == mp.MHC_ERR_PARAM_INVALID
    assert call(D=12) == mp.MHC_ERR_PARAM_INVALID
    assert call(D=0) == mp.MHC_ERR_PARAM_INVALID
    assert call(T=-1) == mp.MHC_ERR_PARAM_INVALID
    assert call(comb=0) == mp.MHC_ERR_NULLPTR
    assert call(x=A + 8) == mp.MHC_ERR_PARAM_INVALID
    assert call(out=A + 2) == mp.MHC_ERR_PARAM_INVALID
    assert call(post=A + 2) == mp.MHC_ERR_PARAM_INVALID


# ------------------------------------------------------------------ backward

def _bwd_args(T=64, **over):
    a = mp.MhcPreBwdArgs()
    A = 1 << 20          # aligned fake device address, never dereferenced
    a.T = T
    for k in ("x", "phi", "alpha", "grad_h_in", "grad_h_post", "grad_h_res", "inv_rms", "h_mix", "h_pre",
              "h_post", "sum_out", "norm_out", "grad_x", "grad_phi", "grad_alpha", "grad_bias"):
        setattr(a, k, A)
    a.workspace = A
    a.workspace_bytes = 1 << 34
    for k, v in over.items():
        setattr(a, k, v)
    return a


def test_backward_workspace_size(lib):
    h = _handle(D=7168)
    st, n = mp.mhc_pre_backward_workspace_size(h, 0)
    assert st == mp.MHC_OK and n == 0
    st, n = mp.mhc_pre_backward_workspace_size(h, 100)
    up = lambda v: (v + 255) // 256 * 256
    planes = up(112 * 4 * 3 * 32 * 128)
    tiles = up(2 * (3 * 32 * 128 + 64 * 32))
    pieces = up(112 * 8 * 32 * 256 * 4)
    parts = up(1024 * 8 * 32 * 4)
    hg = up(100 * 4 * 4)
    assert st == mp.MHC_OK and n == 256 + planes + tiles + pieces + parts + hg
    assert mp.mhc_pre_backward_workspace_size(h, -1)[0] == mp.MHC_ERR_PARAM_INVALID
    mp.mhc_pre_destroy(h)
    h = _handle(D=7168, impl_mode=1)
    st, n2 = mp.mhc_pre_backward_workspace_size(h, 100)
    assert st == mp.MHC_OK and n2 < n
    mp.mhc_pre_destroy(h)


@pytest.mark.parametrize("cfg", [dict(n=6), dict(n=8), dict(alpha_len=2), dict(D=96)])
def test_backward_scope(lib, cfg):
    h = _handle(**cfg)
    assert mp.mhc_pre_backward_workspace_size(h, 64)[0] == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args()) == mp.MHC_ERR_PARAM_INVALID
    mp.mhc_pre_destroy(h)


@pytest.mark.parametrize("field", ["x", "phi", "alpha", "grad_h_in", "grad_h_post", "grad_h_res", "inv_rms",
                                   "h_mix", "h_pre", "h_post", "grad_x", "grad_phi", "grad_alpha",
                                   "grad_bias", "workspace"])
def test_backward_null_required(lib, field):
    h = _handle(D=256)
    assert mp.mhc_pre_backward_run(h, _bwd_args(**{field: None})) == mp.MHC_ERR_NULLPTR
    mp.mhc_pre_destroy(h)


def test_backward_groups_alignment_workspace(lib):
    h = _handle(D=256)
    A = 1 << 20
    assert mp.mhc_pre_backward_run(h, _bwd_args(sum_out=None)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(norm_out=None)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(gamma=A)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(grad_gamma=A)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(x=A + 8)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(grad_x=A + 2)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(grad_x_post=A + 4)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(h_mix=A + 2)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(workspace_bytes=1000)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(T=-1)) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_backward_run(h, _bwd_args(T=0, x=None, workspace=None)) == mp.MHC_OK
    mp.mhc_pre_destroy(h)


def test_backward_without_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = _handle(D=256)
    assert mp.mhc_pre_backward_run(h, _bwd_args()) == mp.MHC_ERR_RUNTIME
    mp.mhc_pre_destroy(h)


def test_binding_refuses_non_contiguous_and_bad_layouts(lib):
    import torch
    from mhc_hyper_connection_gb300._binding import _tokens
    op = mp.MhcPre(4, 64)
    x = torch.zeros((8, 64, 4), dtype=torch.bfloat16).transpose(1, 2)    # [8, 4, 64], not contiguous
    phi = torch.zeros((24, 256))
    with pytest.raises(ValueError, match="contiguous"):
        op.make_args(x, phi, torch.ones(3), torch.zeros(24), {"y": None, "h_post": None})
    assert _tokens((6,)) == 6 and _tokens((2, 3)) == 6
    with pytest.raises(ValueError):
        _tokens((2, 3, 4))
    op.close()


def test_composite_route_host_validation(lib):
    h = _handle(D=256)
    A = 1 << 20
    assert mp.mhc_pre_inv_rms_run(h, 0, 0, 0) == mp.MHC_OK
    assert mp.mhc_pre_inv_rms_run(h, 4, 0, A) == mp.MHC_ERR_NULLPTR
    assert mp.mhc_pre_inv_rms_run(h, 4, A + 8, A) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_inv_rms_run(h, -1, A, A) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_mixes_run(h, 4, A, 0, 0, A) == mp.MHC_ERR_NULLPTR
    assert mp.mhc_pre_mixes_run(h, 4, A, A + 2, 0, A) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_sinkhorn_run(h, _args(), 0, A) == mp.MHC_ERR_NULLPTR
    assert mp.mhc_pre_sinkhorn_run(h, _args(y=A + 2), A, A) == mp.MHC_ERR_PARAM_INVALID
    assert mp.mhc_pre_sinkhorn_run(h, _args(T=0), 0, 0) == mp.MHC_OK
    import torch
    if not torch.cuda.is_available():
        assert mp.mhc_pre_inv_rms_run(h, 4, A, A) == mp.MHC_ERR_RUNTIME
        assert mp.mhc_pre_sinkhorn_run(h, _args(), A, A) == mp.MHC_ERR_RUNTIME
    mp.mhc_pre_destroy(h)
