"""Helpers for the GPU parity tests: comparisons with the stated tolerances and
guard-region canaries around outputs (out-of-bounds writes show up as changed
guard bytes, without any sanitizer)."""
import numpy as np
import torch

# Tolerances (the target's: fp32 max-abs 1e-4 on O and LSE; bf16 with fp32
# accumulation max-abs 1e-2 on O, 1e-3 relative on LSE, 2e-2 relative-L2 on
# dQ/dK/dV).  fp32 gradients use max-abs 1e-4 scaled by max(1, |ref|_inf).
TOL_F32_ABS = 1e-4
TOL_BF16_O_ABS = 1e-2
TOL_BF16_LSE_REL = 1e-3
TOL_BF16_GRAD_RL2 = 2e-2

GUARD = 4096  # elements of guard on each side


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)))) if np.size(a) else 0.0


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a - b))


def lse_rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    fin = np.isfinite(b)
    assert np.array_equal(np.isneginf(a), np.isneginf(b)), "LSE -inf pattern differs"
    if not fin.any():
        return 0.0
    return float(np.max(np.abs(a[fin] - b[fin]) / np.maximum(np.abs(b[fin]), 1e-30)))


class Guarded:
    """A device tensor of `shape` living inside a larger buffer whose margins hold a canary."""

    def __init__(self, shape, dtype, device):
        n = int(np.prod(shape))
        self.buf = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
        self._fill_canary()
        self.t = self.buf[GUARD:GUARD + n].view(*shape)
        assert self.t.data_ptr() % 16 == 0

    def _fill_canary(self):
        # a fixed NaN payload (bytes 0x7F / 0xFFC1...) that no kernel produces
        if self.buf.dtype == torch.float32:
            self.buf.view(torch.int32).fill_(0x7FC1DEAD)
        elif self.buf.dtype == torch.bfloat16:
            self.buf.view(torch.int16).fill_(0x7FC3)
        else:
            self.buf.fill_(0xA5)

    def intact(self) -> bool:
        raw = self.buf.view(torch.int32 if self.buf.dtype == torch.float32 else
                            (torch.int16 if self.buf.dtype == torch.bfloat16 else torch.uint8))
        head, tail = raw[:GUARD], raw[-GUARD:]
        want = {torch.float32: 0x7FC1DEAD, torch.bfloat16: 0x7FC3}.get(self.buf.dtype, 0xA5)
        return bool((head == want).all().item() and (tail == want).all().item())
