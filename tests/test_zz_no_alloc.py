"""attn_bwd_static_workspace: the backward for callers that cannot allocate
device memory (a host framework that owns every device allocation, or a path
that must not allocate after start-up).  Called through the C ABI and compared
with attn_bwd on the same inputs, on two calls in a row with different inputs,
so that the fixed scratch array's leftover contents from the first call cannot
leak into the second.  This file is collected last on purpose."""
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


def test_static_workspace_matches_attn_bwd_twice(lib):
    dev = torch.device("cuda")
    B, H, N, d = 1, 4, 1024, 128
    s = 1.0 / math.sqrt(d)
    for seed in (41, 42):  # two calls in a row, different inputs
        x = inputs.make_inputs(B, H, N, d, torch.bfloat16, seed=seed)
        q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
        o, lse = attn.attn_fwd(q, k, v, s)
        ref = attn.attn_bwd(q, k, v, o, do, lse, s)          # the existing entry point
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        st = _call_static(lib, q, k, v, o, do, lse, s, *got)
        assert st == attn.ATTN_OK, attn.status_string(st)
        assert attn.attn_device_status() == attn.ATTN_OK
        for g, r in zip(got, ref):
            assert torch.isfinite(g).all()
            assert _rl2(g, r) <= TOL_GRAD_RL2


def test_static_workspace_rejects_shapes_beyond_its_size(lib):
    dev = torch.device("cuda")
    t = torch.empty(16, device=dev, dtype=torch.bfloat16)
    B, H, N, d = 64, 16, 4096, 128   # needs ~270 MB of scratch, above the 64 MiB array
    fake = ctypes.c_void_p(t.data_ptr())
    st = lib.attn_bwd_static_workspace(fake, fake, fake, fake, fake, fake, fake, fake, fake, B, H, N, d,
                                       ctypes.c_float(0.1), attn.ATTN_DTYPE_BF16, None, None)
    assert st == attn.ATTN_ERR_WORKSPACE
