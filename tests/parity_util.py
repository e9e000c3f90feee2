"""Shared helpers of the GPU parity tests: tolerances, sampling, comparisons."""
from __future__ import annotations

import numpy as np
import torch

from workloads import to_f64

# GPU vs fp64 oracle, bf16 inputs with fp32 accumulation
MAX_ABS = 2e-2
REL_L2 = 5e-3
NEAR_TAU = 1e-4


def errors(gpu, ref):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    diff = g - r
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(gpu, ref, what, max_abs=MAX_ABS, rel_l2=REL_L2):
    ma, rl = errors(gpu, ref)
    assert np.all(np.isfinite(np.asarray(gpu, dtype=np.float64))), f"{what}: non-finite GPU values"
    assert ma <= max_abs and rl <= rel_l2, f"{what}: max-abs {ma:.3e} (<= {max_abs}), rel-L2 {rl:.3e} (<= {rel_l2})"
    return ma, rl


def host(x: torch.Tensor):
    """float64 numpy copy of a device tensor (bf16 widened exactly)."""
    if x.dtype == torch.bfloat16:
        return to_f64(x)
    return x.detach().to("cpu").double().numpy()


def heads(x: torch.Tensor, hs):
    """float64 host copy of a [B, H, S, d] tensor restricted to heads ``hs`` (B = 1)."""
    return host(x[:, list(hs)].contiguous())


def gpu_selection(sel_idx: torch.Tensor, sel_cnt: torch.Tensor):
    """Dense boolean [.., NQB, NKB] mask from the GPU's compacted lists; checks they are ascending and in range."""
    idx = sel_idx.cpu().numpy()
    cnt = sel_cnt.cpu().numpy()
    nkb = idx.shape[-1]
    mask = np.zeros(idx.shape, dtype=bool)
    flat_idx = idx.reshape(-1, nkb)
    flat_cnt = cnt.reshape(-1)
    flat_mask = mask.reshape(-1, nkb)
    for r in range(flat_cnt.size):
        c = int(flat_cnt[r])
        assert 1 <= c <= nkb, f"row {r}: sel_cnt {c}"
        lst = flat_idx[r, :c]
        assert np.all(lst >= 0) and np.all(lst < nkb), f"row {r}: index out of range"
        assert np.all(np.diff(lst) > 0), f"row {r}: list not strictly ascending"
        flat_mask[r, lst] = True
    return mask


def compare_selection(gpu_sel, oracle_rt, band=NEAR_TAU):
    """Selections must agree except where the oracle's proxy lies within `band` of tau
    (or of the row maximum, which decides the always-kept argmax block).

    Returns the number of such near-threshold flips."""
    proxy, tau = oracle_rt["proxy"], oracle_rt["tau"][..., None]
    diff = gpu_sel != oracle_rt["sel"]
    near = (np.abs(proxy - tau) < band) | (np.abs(proxy - proxy.max(-1, keepdims=True)) < band)
    bad = diff & ~near
    assert not bad.any(), f"{int(bad.sum())} selection mismatches outside the near-tau band"
    return int(diff.sum())


GUARD_BYTES = 4096
GUARD_PATTERN = 0x5A


class Guarded:
    """A device tensor placed between two guard bands of GUARD_BYTES.  The bands and the tensor
    itself are filled with GUARD_PATTERN (as fp32 or bf16 that reads 1.5e16, so an element no
    kernel wrote also shows up in a comparison); `check` asserts that both bands are unchanged,
    i.e. that no store landed just before or just past the buffer."""

    def __init__(self, shape, dtype, device="cuda"):
        self.nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((self.nbytes + 2 * GUARD_BYTES,), GUARD_PATTERN, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(shape)

    def check(self, what):
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.nbytes:]
        ok_head = bool((head == GUARD_PATTERN).all())
        ok_tail = bool((tail == GUARD_PATTERN).all())
        assert ok_head and ok_tail, f"{what}: store outside the buffer (leading band ok={ok_head}, trailing ok={ok_tail})"
