"""attn_bwd_static_workspace: the backward for callers that cannot allocate
device memory (a host framework that owns every device allocation, or a path
that must not allocate after start-up).  Called through the C ABI and compared
with attn_bwd on the same inputs, on two calls in a row with different inputs,
so that the fixed scratch array's leftover contents from the first call cannot
leak into the second: dK and dV must be bit-identical (the same kernels run),
dQ equal to the rounding of its fp32 accumulation order.  This file is
collected last on purpose."""
import ctypes
import math

import pytest
import torch

from optimal_tiling_gb300 import attn, build, inputs

pytestmark = pytest.mark.gpu

TOL_GRAD_RL2 = 2e-2   # the relative-L2 bound the other backward tests use


def _rl2(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.load()


def _call_static(lib, q, k, v, o, do, lse, scale, dq, dk, dv):
    B, H, N, d = q.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.attn_bwd_static_workspace(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(do.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(dq.data_ptr()), ctypes.c_void_p(dk.data_ptr()), ctypes.c_void_p(dv.data_ptr()),
        B, H, N, d, ctypes.c_float(scale), attn.ATTN_DTYPE_BF16, None, stream)


def _compare_twice(lib, B, H, N, d, seeds):
    """Two calls in a row on different inputs; each against attn_bwd with its own workspace.
    Both run the same kernels: dK and dV come out bit-identical, dQ (whose fp32 accumulation
    order between key tiles is not fixed) to the rounding of those additions."""
    dev = torch.device("cuda")
    s = 1.0 / math.sqrt(d)
    for seed in seeds:
        x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=seed)
        q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
        o, lse = attn.attn_fwd(q, k, v, s)
        ref = attn.attn_bwd(q, k, v, o, do, lse, s)          # the existing entry point
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        st = _call_static(lib, q, k, v, o, do, lse, s, *got)
        assert st == attn.ATTN_OK, attn.status_string(st)
        assert attn.attn_device_status() == attn.ATTN_OK
        for g in got:
            assert torch.isfinite(g).all()
        assert torch.equal(got[1], ref[1]), "dK differs from attn_bwd"
        assert torch.equal(got[2], ref[2]), "dV differs from attn_bwd"
        assert _rl2(got[0], ref[0]) <= 1e-3
        for g, r in zip(got, ref):
            assert _rl2(g, r) <= TOL_GRAD_RL2


def test_static_workspace_matches_attn_bwd_twice(lib):
    _compare_twice(lib, 1, 4, 1024, 128, (41, 42))


def test_static_workspace_at_d256(lib):
    """d = 256 runs the two-pass backward; its row terms and accumulator fit the array too."""
    _compare_twice(lib, 1, 2, 1024, 256, (43, 44))


def test_static_workspace_with_a_split_last_wave(lib):
    """A dense shape whose last wave of 128-key tiles is split into query halves: the
    fp32 partial dK and dV of the split tiles then also live in the fixed array (after
    the row terms and the dQ accumulator), and must start from zero on every call."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    r = max(t for t in range(1, sms // 4 + 1) if sms % t == 0)
    H, N, d = sms // r + 1, 128 * r, 128
    assert lib.attn_bwd_workspace_size(1, H, N, d, attn.ATTN_DTYPE_BF16) <= 64 << 20
    _compare_twice(lib, 1, H, N, d, (43, 44))


def test_static_workspace_rejects_shapes_beyond_its_size(lib):
    dev = torch.device("cuda")
    t = torch.empty(16, device=dev, dtype=torch.bfloat16)
    B, H, N, d = 64, 16, 4096, 128   # needs ~270 MB of scratch, above the 64 MiB array
    fake = ctypes.c_void_p(t.data_ptr())
    st = lib.attn_bwd_static_workspace(fake, fake, fake, fake, fake, fake, fake, fake, fake, B, H, N, d,
                                       ctypes.c_float(0.1), attn.ATTN_DTYPE_BF16, None, None)
    assert st == attn.ATTN_ERR_WORKSPACE
