"""CPU oracle for exact softmax attention (double precision).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It never imports the CUDA path and shares no code with it: the
arithmetic lives in ``attn_oracle.c`` (plain loops, one function per defining
passage), and this file only compiles it with gcc and marshals numpy arrays.

Passages followed (see the C file for the per-function citations):

* "The I/O Complexity of Attention" exposition (blog.aeilot.top,
  attention-io-complexity), "Attention as a mathematical problem":
  O = softmax(s Q K^T) V, scores are dot products, rows are normalised.
* Same page, "Softmax without storing the score matrix": the stabilised
  online update (running max m, sum l, weighted sum u; o = u / l).
* "On Fine-Grained I/O Complexity of Attention Backward Passes" summary
  (gist.science 2410.09397), "Problem Statement": the backward pass, taken as
  the plain chain rule of the forward definition.

Every function is pinned by ``tests/test_oracle_pins.py`` against closed forms,
invariants, finite differences, an independent library evaluation and the
fixtures under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, no fast-math) and return the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    lib.oracle_fwd_naive.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_double, _u8p, _dp, _dp, _dp, _dp, _dp]
    lib.oracle_fwd_rows.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, _u8p,
                                    _dp, _dp, _dp, ctypes.c_int, _ip, _ip, _dp, _dp]
    lib.oracle_fwd_stream.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_double, _u8p, ctypes.c_int, _ip,
                                      _dp, _dp, _dp, _dp, _dp]
    lib.oracle_bwd_naive.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_double, _u8p, _dp, _dp, _dp, _dp,
                                     _dp, _dp, _dp, _dp, _dp]
    lib.oracle_bwd_rows.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, _u8p,
                                    _dp, _dp, _dp, _dp, ctypes.c_int, _ip, _dp,
                                    ctypes.c_int, _ip, _dp, _dp]
    lib.oracle_fwd_rect.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                    _dp, _dp, _dp, _dp, _dp]
    lib.oracle_fwd_naive_m.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, _u8p,
                                       ctypes.c_int, ctypes.c_longlong, _dp, _dp, _dp, _dp, _dp]
    lib.oracle_bwd_naive_m.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, _u8p,
                                       ctypes.c_int, ctypes.c_longlong, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


class Oracle:
    """The oracle's functions bound to one compiled library.

    The module-level functions use the library built from ``attn_oracle.c``;
    the planted-mistake tests build a mutated copy of the source into another
    path and wrap it here, to show the pins reject it.
    """

    def __init__(self, lib_path=None):
        self._path = lib_path

    @property
    def lib(self):
        if self._path is None:
            return _load()
        if not hasattr(self, "_lib"):
            self._lib = _bind(ctypes.CDLL(self._path))
        return self._lib


def compile_source(src_path: str, out_path: str) -> str:
    """Compile an oracle source file (used for planted-mistake copies in tests)."""
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", src_path, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


SOURCE_PATH = _SRC


def _f64(a) -> np.ndarray:
    """Widen to a C-contiguous float64 array (bf16 widens exactly via float32)."""
    if hasattr(a, "detach"):  # torch tensor on the CPU
        import torch
        a = a.detach().to("cpu")
        if a.dtype == torch.bfloat16 or a.dtype == torch.float16:
            a = a.to(torch.float32)
        a = a.numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _mask_arg(mask, N: int):
    if mask is None:
        return None, None
    m = mask.detach().cpu().numpy() if hasattr(mask, "detach") else np.asarray(mask)
    m = np.ascontiguousarray(m.astype(np.uint8))
    nb = (N + 127) // 128
    if m.shape != (nb, nb):
        raise ValueError(f"block mask must be [{nb},{nb}], got {m.shape}")
    return m, m.ctypes.data_as(_u8p)


def _same_shape(*arrays):
    for a in arrays[1:]:
        if a.shape != arrays[0].shape:
            raise ValueError(f"Q, K, V (and dO) must share one [..., N, d] shape: {a.shape} vs {arrays[0].shape}")


def _heads(x: np.ndarray):
    """Split a [..., N, d] array into (number of heads, N, d)."""
    if x.ndim < 2:
        raise ValueError("expected [..., N, d]")
    N, d = x.shape[-2], x.shape[-1]
    nh = int(np.prod(x.shape[:-2])) if x.ndim > 2 else 1
    return nh, N, d


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().oracle_num_threads())


def fwd_naive(q, k, v, scale: float, mask=None, _oracle=None):
    """Full-row forward.  Returns (O, LSE) as float64 arrays shaped like q and q[..., 0]."""
    lib = _oracle.lib if _oracle is not None else _load()
    Q, K, V = _f64(q), _f64(k), _f64(v)
    _same_shape(Q, K, V)
    nh, N, d = _heads(Q)
    m, mp = _mask_arg(mask, N)
    O = np.empty_like(Q)
    LSE = np.empty(Q.shape[:-1], dtype=np.float64)
    lib.oracle_fwd_naive(nh, N, d, float(scale), mp, _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE))
    return O, LSE


def fwd_stream(q, k, v, scale: float, block_ends, mask=None, _oracle=None):
    """Online-softmax forward over key blocks ending at ``block_ends`` (last == N)."""
    lib = _oracle.lib if _oracle is not None else _load()
    Q, K, V = _f64(q), _f64(k), _f64(v)
    _same_shape(Q, K, V)
    nh, N, d = _heads(Q)
    ends = np.ascontiguousarray(np.asarray(block_ends, dtype=np.int32))
    if ends.size == 0 or ends[-1] != N or np.any(np.diff(ends) <= 0) or ends[0] <= 0:
        raise ValueError("block_ends must be strictly increasing and end at N")
    m, mp = _mask_arg(mask, N)
    O = np.empty_like(Q)
    LSE = np.empty(Q.shape[:-1], dtype=np.float64)
    lib.oracle_fwd_stream(nh, N, d, float(scale), mp, int(ends.size), ends.ctypes.data_as(_ip),
                          _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE))
    return O, LSE


def fwd_rows(q, k, v, scale: float, heads, rows, mask=None, _oracle=None):
    """Forward outputs for chosen (flattened head, query row) pairs.

    q, k, v are [..., N, d]; ``heads`` index the flattened leading dims.
    Returns (O_rows [n, d], LSE_rows [n]).
    """
    lib = _oracle.lib if _oracle is not None else _load()
    Q, K, V = _f64(q), _f64(k), _f64(v)
    _same_shape(Q, K, V)
    nh, N, d = _heads(Q)
    hs = np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    rs = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    assert hs.shape == rs.shape and (hs.size == 0 or (hs.max() < nh and rs.max() < N))
    m, mp = _mask_arg(mask, N)
    O = np.empty((hs.size, d), dtype=np.float64)
    LSE = np.empty(hs.size, dtype=np.float64)
    lib.oracle_fwd_rows(N, d, float(scale), mp, _ptr(Q), _ptr(K), _ptr(V), int(hs.size),
                        hs.ctypes.data_as(_ip), rs.ctypes.data_as(_ip), _ptr(O), _ptr(LSE))
    return O, LSE


def bwd_naive(q, k, v, do, scale: float, mask=None, _oracle=None):
    """Chain-rule backward.  Returns (dQ, dK, dV, D, LSE) in float64."""
    lib = _oracle.lib if _oracle is not None else _load()
    Q, K, V, dO = _f64(q), _f64(k), _f64(v), _f64(do)
    _same_shape(Q, K, V, dO)
    nh, N, d = _heads(Q)
    m, mp = _mask_arg(mask, N)
    dQ, dK, dV = np.empty_like(Q), np.empty_like(Q), np.empty_like(Q)
    D = np.empty(Q.shape[:-1], dtype=np.float64)
    LSE = np.empty(Q.shape[:-1], dtype=np.float64)
    lib.oracle_bwd_naive(nh, N, d, float(scale), mp, _ptr(Q), _ptr(K), _ptr(V), _ptr(dO),
                         _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(D), _ptr(LSE))
    return dQ, dK, dV, D, LSE


def bwd_rows(q, k, v, do, scale: float, qrows, krows, mask=None, _oracle=None):
    """Backward outputs of ONE head ([N, d] inputs): dQ at ``qrows``; dK, dV at ``krows``."""
    lib = _oracle.lib if _oracle is not None else _load()
    Q, K, V, dO = _f64(q), _f64(k), _f64(v), _f64(do)
    _same_shape(Q, K, V, dO)
    if Q.ndim != 2:
        raise ValueError("bwd_rows takes one head: [N, d]")
    N, d = Q.shape
    qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int32))
    kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int32))
    m, mp = _mask_arg(mask, N)
    dQ = np.empty((qr.size, d)); dK = np.empty((kr.size, d)); dV = np.empty((kr.size, d))
    lib.oracle_bwd_rows(N, d, float(scale), mp, _ptr(Q), _ptr(K), _ptr(V), _ptr(dO),
                        int(qr.size), qr.ctypes.data_as(_ip), _ptr(dQ),
                        int(kr.size), kr.ctypes.data_as(_ip), _ptr(dK), _ptr(dV))
    return dQ, dK, dV


def fwd_rect(q, k, v, scale: float, _oracle=None):
    """Rectangular forward: q [..., Nq, d] against k, v [..., Nk, d] (no mask)."""
    lib = _oracle.lib if _oracle is not None else _load()
    Q, K, V = _f64(q), _f64(k), _f64(v)
    if K.shape != V.shape or Q.shape[:-2] != K.shape[:-2] or Q.shape[-1] != K.shape[-1]:
        raise ValueError("q [..., Nq, d], k and v [..., Nk, d] with the same leading dims and d")
    nh, Nq, d = _heads(Q)
    Nk = K.shape[-2]
    O = np.empty_like(Q)
    LSE = np.empty(Q.shape[:-1], dtype=np.float64)
    lib.oracle_fwd_rect(nh, Nq, Nk, d, float(scale), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE))
    return O, LSE


def _mask_general(mask, N: int, block: int, nh: int):
    """Block mask of side `block`: [nb, nb] shared by all heads, or [nh, nb, nb] per head."""
    if mask is None:
        return None, None, 0
    m = mask.detach().cpu().numpy() if hasattr(mask, "detach") else np.asarray(mask)
    m = np.ascontiguousarray(m.astype(np.uint8))
    nb = (N + block - 1) // block
    if m.shape == (nb, nb):
        return m, m.ctypes.data_as(_u8p), 0
    if m.shape == (nh, nb, nb):
        return m, m.ctypes.data_as(_u8p), nb * nb
    raise ValueError(f"mask must be [{nb},{nb}] or [{nh},{nb},{nb}], got {m.shape}")


def fwd_naive_m(q, k, v, scale: float, mask=None, block: int = 128, _oracle=None):
    """Forward with a general block mask: side `block`; [nb, nb] or per head [heads, nb, nb]."""
    lib = _oracle.lib if _oracle is not None else _load()
    Q, K, V = _f64(q), _f64(k), _f64(v)
    _same_shape(Q, K, V)
    nh, N, d = _heads(Q)
    m, mp, stride = _mask_general(mask, N, block, nh)
    O = np.empty_like(Q)
    LSE = np.empty(Q.shape[:-1], dtype=np.float64)
    lib.oracle_fwd_naive_m(nh, N, d, float(scale), mp, int(block), int(stride), _ptr(Q), _ptr(K), _ptr(V),
                           _ptr(O), _ptr(LSE))
    return O, LSE


def bwd_naive_m(q, k, v, do, scale: float, mask=None, block: int = 128, _oracle=None):
    """Backward with a general block mask (as fwd_naive_m).  Returns (dQ, dK, dV)."""
    lib = _oracle.lib if _oracle is not None else _load()
    Q, K, V, dO = _f64(q), _f64(k), _f64(v), _f64(do)
    _same_shape(Q, K, V, dO)
    nh, N, d = _heads(Q)
    m, mp, stride = _mask_general(mask, N, block, nh)
    dQ, dK, dV = np.empty_like(Q), np.empty_like(Q), np.empty_like(Q)
    lib.oracle_bwd_naive_m(nh, N, d, float(scale), mp, int(block), int(stride), _ptr(Q), _ptr(K), _ptr(V),
                           _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV))
    return dQ, dK, dV
