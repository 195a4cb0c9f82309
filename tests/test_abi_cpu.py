"""The C-ABI library builds for sm_103a, loads without a GPU, exports every entry
point include/attn.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

from optimal_tiling_gb300 import attn, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.load()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_bwd", "attn_fwd_materialized", "attn_bwd_workspace_size",
              "attn_fwd_materialized_workspace_size", "attn_device_status", "attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(build.LIB_PATH)
    for n in declared_functions():
        assert hasattr(raw, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for code in range(6):
        assert len(attn.status_string(code)) > 0
    assert attn.status_string(99) == "unknown status"


FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: every call below fails validation
MIS = ctypes.c_void_p(0x10008)        # 8-byte aligned only


def _fwd(lib, B=1, H=1, N=256, d=64, dt=attn.ATTN_DTYPE_BF16, q=FAKE, scale=1.0):
    return lib.attn_fwd(q, FAKE, FAKE, FAKE, FAKE, B, H, N, d, scale, dt, None, None)


def test_forward_argument_checks(lib):
    assert _fwd(lib, B=0) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, N=-1) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, q=None) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, q=MIS) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, dt=7) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, d=96) == attn.ATTN_ERR_UNSUPPORTED           # bf16 d in {64,128,256}
    assert _fwd(lib, d=300, dt=attn.ATTN_DTYPE_F32) == attn.ATTN_ERR_UNSUPPORTED
    # more (b, h) pairs than a grid dimension holds: refused before any CUDA call
    assert _fwd(lib, B=300, H=300) == attn.ATTN_ERR_UNSUPPORTED
    assert _fwd(lib, B=300, H=300, dt=attn.ATTN_DTYPE_F32) == attn.ATTN_ERR_UNSUPPORTED


def test_backward_argument_checks(lib):
    def bwd(d=128, N=256, ws=FAKE, wsz=1 << 30, dt=attn.ATTN_DTYPE_BF16):
        return lib.attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, N, d, 0.1, dt,
                            None, ws, wsz, None)
    assert bwd(d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert bwd(d=512) == attn.ATTN_ERR_UNSUPPORTED
    # bf16: the row terms and dQ accumulator have N rounded up to 64 rows per head, which
    # must stay within 2^31 rows too (3 x 715827882 rows fit, 3 x 715827904 do not)
    assert lib.attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 3, 715827882, 64, 0.1,
                        attn.ATTN_DTYPE_BF16, None, FAKE, 1 << 62, None) == attn.ATTN_ERR_UNSUPPORTED
    assert bwd(ws=None) == attn.ATTN_ERR_WORKSPACE
    need = lib.attn_bwd_workspace_size(1, 2, 256, 128, attn.ATTN_DTYPE_BF16)
    assert need >= 2 * 256 * 4 + 2 * 256 * 128 * 4
    assert bwd(wsz=need - 1) == attn.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd_workspace_size(1, 2, 256, 64, attn.ATTN_DTYPE_F32) >= 2 * 256 * 4
    assert lib.attn_bwd_workspace_size(0, 2, 256, 64, attn.ATTN_DTYPE_F32) == 0


def test_bwd_workspace_holds_the_last_wave_split(lib):
    """The size query adds fp32 dK and dV for the tiles of a last wave that is split into
    query halves: when the SM count does not divide the 128-key tiles and the remainder
    is at most half the SMs (a machine without a GPU is taken to have 152)."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    up = lambda x: -(-x // 256) * 256
    for tiles in (sms - 1, sms, sms + 1, sms + sms // 2, sms + sms // 2 + 1, 2 * sms, 3 * sms + 7):
        N = 128 * tiles
        r = tiles % sms
        split = r if tiles > sms and 0 < r and 2 * r <= sms else 0
        base = up(2 * N * 4) + up(N * 128 * 4)   # D and LSE log2(e), then the fp32 dQ accumulator
        assert lib.attn_bwd_workspace_size(1, 1, N, 128, attn.ATTN_DTYPE_BF16) == base + split * 2 * 128 * 128 * 4
        assert lib.attn_bwd_workspace_size(1, 1, N, 128, attn.ATTN_DTYPE_F32) == up(N * 4)
        # d = 256 runs two passes per key tile and never splits the last wave
        assert lib.attn_bwd_workspace_size(1, 1, N, 256, attn.ATTN_DTYPE_BF16) == up(2 * N * 4) + up(N * 256 * 4)


def test_materialized_argument_checks(lib):
    need = lib.attn_fwd_materialized_workspace_size(2, 3, 256, 64, attn.ATTN_DTYPE_BF16)
    assert need >= 6 * 256 * 256 * 2
    assert lib.attn_fwd_materialized_workspace_size(2, 3, 256, 64, attn.ATTN_DTYPE_F32) == 0
    r = lib.attn_fwd_materialized(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 3, 256, 64, 0.1, attn.ATTN_DTYPE_BF16,
                                  None, FAKE, need - 16, None)
    assert r == attn.ATTN_ERR_WORKSPACE
    r = lib.attn_fwd_materialized(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 3, 256, 64, 0.1, attn.ATTN_DTYPE_F32,
                                  None, FAKE, need, None)
    assert r == attn.ATTN_ERR_UNSUPPORTED
    # the materialising schedules take whole 128-row tiles only
    r = lib.attn_fwd_materialized(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 3, 200, 64, 0.1, attn.ATTN_DTYPE_BF16,
                                  None, FAKE, 1 << 40, None)
    assert r == attn.ATTN_ERR_UNSUPPORTED
    r = lib.attn_bwd_materialized(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 3, 200, 64, 0.1,
                                  attn.ATTN_DTYPE_BF16, None, FAKE, 1 << 40, None)
    assert r == attn.ATTN_ERR_UNSUPPORTED


def test_bwd_workspace_with_partial_tiles(lib):
    """When 128 does not divide N: D and LSE log2(e), then the fp32 dQ accumulator, with N
    rounded up to 64 rows per head, and no last-wave split (N = 128 (t + 1/2) for t tiles
    around the SM count would be split if whole)."""
    up = lambda x: -(-x // 256) * 256
    for B, H, N, d in ((1, 3, 200, 128), (2, 5, 1, 64), (1, 1, 4097, 128), (1, 1, 128 * 153 + 64, 128)):
        rows = B * H * (-(-N // 64) * 64)
        assert lib.attn_bwd_workspace_size(B, H, N, d, attn.ATTN_DTYPE_BF16) == up(2 * rows * 4) + up(rows * d * 4)
        assert lib.attn_bwd_workspace_size(B, H, N, d, attn.ATTN_DTYPE_F32) == up(B * H * N * 4)


def test_selftest_rejects_bad_limits(lib):
    assert lib.attn_selftest_timeout(0, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_timeout(10000001, None) == attn.ATTN_ERR_INVALID_ARG


def test_decode_argument_checks(lib):
    def dec(Nq=1, Nk=100, d=128, dt=attn.ATTN_DTYPE_BF16, ws=FAKE, wsz=1 << 30, q=FAKE):
        return lib.attn_decode(q, FAKE, FAKE, FAKE, FAKE, 2, 3, Nq, Nk, d, 0.1, dt, ws, wsz, None)
    assert dec(Nq=0) == attn.ATTN_ERR_INVALID_ARG
    assert dec(Nq=17) == attn.ATTN_ERR_UNSUPPORTED
    assert dec(d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert dec(dt=attn.ATTN_DTYPE_F32) == attn.ATTN_ERR_UNSUPPORTED
    assert dec(q=MIS) == attn.ATTN_ERR_INVALID_ARG
    assert dec(ws=None) == attn.ATTN_ERR_WORKSPACE
    need = lib.attn_decode_workspace_size(2, 3, 4, 1000, 128, attn.ATTN_DTYPE_BF16)
    assert need >= 2 * 3 * 4 * 130 * 4
    assert dec(Nq=4, Nk=1000, wsz=need - 4) == attn.ATTN_ERR_WORKSPACE


def test_masked_entry_point_checks(lib):
    """attn_fwd_masked / attn_bwd_masked reject a block side other than 64 or 128
    and a negative head stride before anything else happens."""
    def fwd(block=64, stride=0, blocks=FAKE, mask=True):
        bm = attn.BlockMask(blocks, block, stride)
        return lib.attn_fwd_masked(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, 1.0, attn.ATTN_DTYPE_BF16,
                                   ctypes.byref(bm) if mask else None, None)

    def bwd(block=64, stride=0, d=128):
        bm = attn.BlockMask(FAKE, block, stride)
        return lib.attn_bwd_masked(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, d, 0.1,
                                   attn.ATTN_DTYPE_BF16, ctypes.byref(bm), FAKE, 1 << 30, None)
    for blk in (0, 32, 96, 256):
        assert fwd(block=blk) == attn.ATTN_ERR_INVALID_ARG
        assert bwd(block=blk) == attn.ATTN_ERR_INVALID_ARG
    assert fwd(stride=-1) == attn.ATTN_ERR_INVALID_ARG
    assert bwd(stride=-64) == attn.ATTN_ERR_INVALID_ARG
    assert bwd(d=96) == attn.ATTN_ERR_UNSUPPORTED
    bm = attn.BlockMask(FAKE, 64, 0)
    assert lib.attn_fwd_masked(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 200, 96, 1.0, attn.ATTN_DTYPE_BF16,
                               ctypes.byref(bm), None) == attn.ATTN_ERR_UNSUPPORTED


def test_negative_scale_passes_the_argument_checks(lib):
    """A negative score scale is a valid input for every forward: with a bad pointer
    the call fails on the pointer, not on the scale."""
    assert _fwd(lib, scale=-0.5, q=MIS) == attn.ATTN_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("-inf")) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_materialized(MIS, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, -1.0, attn.ATTN_DTYPE_BF16,
                                     None, FAKE, 1 << 40, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_materialized(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, -1.0, attn.ATTN_DTYPE_BF16,
                                     None, FAKE, 16, None) == attn.ATTN_ERR_WORKSPACE


def test_static_workspace_checks_arguments_before_its_size(lib):
    """attn_bwd_static_workspace returns attn_bwd's status for a bad argument whatever
    the shape's size (64 x 16 x 4096 rows need ~270 MB, above its 64 MiB array), and
    ATTN_ERR_WORKSPACE only for a valid call that does not fit; all before any CUDA call."""
    def call(q=FAKE, d=128, dt=attn.ATTN_DTYPE_BF16, N=4096, scale=0.1):
        return lib.attn_bwd_static_workspace(q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 16, N, d,
                                             ctypes.c_float(scale), dt, None, None)
    assert call(q=None) == attn.ATTN_ERR_INVALID_ARG
    assert call(q=MIS) == attn.ATTN_ERR_INVALID_ARG
    assert call(dt=7) == attn.ATTN_ERR_INVALID_ARG
    assert call(scale=float("nan")) == attn.ATTN_ERR_INVALID_ARG
    assert call(d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert call(N=4000) == attn.ATTN_ERR_WORKSPACE   # valid (a partial last tile), too large
    assert call() == attn.ATTN_ERR_WORKSPACE


def test_block_mask_marshalling_shapes():
    import torch
    m = torch.ones((4, 4), dtype=torch.uint8)
    assert attn._block_mask(m, 64, 2, 3, 256).head_stride == 0
    per_head = torch.ones((2, 3, 4, 4), dtype=torch.uint8)
    assert attn._block_mask(per_head, 64, 2, 3, 256).head_stride == 16
    assert attn._block_mask(per_head.view(6, 4, 4), 64, 2, 3, 256).head_stride == 16
    with pytest.raises(ValueError):
        attn._block_mask(torch.ones((2, 2), dtype=torch.uint8), 64, 1, 1, 256)
    with pytest.raises(ValueError):
        attn._block_mask(torch.ones((5, 4, 4), dtype=torch.uint8), 64, 2, 3, 256)
    with pytest.raises(ValueError):
        attn._block_mask(m.float(), 64, 1, 1, 256)
