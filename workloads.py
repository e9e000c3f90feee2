"""Seeded synthetic inputs for the attention hot path.

This module holds no part of the method's arithmetic: it only draws the
q/k/v tensors that both the GPU library and the CPU oracle consume.  The
workloads follow the shapes of the LTX-2.5 pages -- video latents flattened
in raster (t, y, x) order, with audio tokens interleaved per frame for the
Stage-2 self-attention ("Accelerating LTX-2.5 with Sol Engine", section
"Stage 2 Optimization") and ~100 audio queries against a video KV for the
cross attention ("LTX-2.5 at 4K, in half the time", section "Attention
across two GPUs").  The neighbourhood-attention workload is a decoder tile of
four latent frames ("LTX-2.5 at 4K, in half the time", section "Inside the
decoder": each decoder tile holds four frames) over a 128 x 128 grid.

Recipe: a ``torch.Generator`` on the requested device, seeded per workload,
draws float32 noise for q, k, v in that order; a fixed 3D sinusoidal position
code (identical for every head) is added to q and k where the workload asks
for it; the result is rounded to bf16 (round-to-nearest-even).  The same bf16
bytes are what the GPU sees and, widened exactly to float64, what the oracle
sees.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def position_code(t: torch.Tensor, y: torch.Tensor, x: torch.Tensor, d: int, amplitude: float = 1.0,
                  spatial_mask: torch.Tensor | None = None) -> torch.Tensor:
    """3D sinusoidal code PE(t, y, x) in R^d for integer coordinates.

    F = d // 6 frequencies per axis, omega_f = 10000^(-f/F); for axis a in
    (t, y, x) and f < F: PE[2(aF+f)] = A sin(omega_f p_a), PE[2(aF+f)+1] =
    A cos(omega_f p_a); the remaining d - 6F dims are zero.  Tokens whose
    ``spatial_mask`` is True (audio) carry only the temporal part."""
    F = d // 6
    n = t.numel()
    pe = torch.zeros(n, d, dtype=torch.float32, device=t.device)
    omega = torch.pow(10000.0, -torch.arange(F, dtype=torch.float64, device=t.device) / F).to(torch.float32)
    for a, p in enumerate((t, y, x)):
        ang = p.to(torch.float32)[:, None] * omega[None, :]
        s, c = amplitude * torch.sin(ang), amplitude * torch.cos(ang)
        if a > 0 and spatial_mask is not None:
            s = torch.where(spatial_mask[:, None], torch.zeros_like(s), s)
            c = torch.where(spatial_mask[:, None], torch.zeros_like(c), c)
        idx = 2 * (a * F + torch.arange(F, device=t.device))
        pe[:, idx] = s
        pe[:, idx + 1] = c
    return pe


def token_coords(grid, audio_per_frame: int = 0, device="cpu"):
    """Coordinates of the token sequence of a (T, Y, X) latent grid.

    Video tokens come in raster order (x fastest); when ``audio_per_frame``
    is positive, that many audio tokens follow each frame's video tokens.
    Returns (t, y, x, is_audio) as 1-D tensors."""
    T, Y, X = grid
    tt = torch.arange(T, device=device)
    per_frame = Y * X + audio_per_frame
    yy = torch.arange(Y, device=device).repeat_interleave(X)
    xx = torch.arange(X, device=device).repeat(Y)
    if audio_per_frame:
        yy = torch.cat([yy, torch.zeros(audio_per_frame, dtype=yy.dtype, device=device)])
        xx = torch.cat([xx, torch.zeros(audio_per_frame, dtype=xx.dtype, device=device)])
    t = tt.repeat_interleave(per_frame)
    y = yy.repeat(T)
    x = xx.repeat(T)
    is_audio = torch.zeros(per_frame, dtype=torch.bool, device=device)
    is_audio[Y * X:] = True
    return t, y, x, is_audio.repeat(T)


@dataclass
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Skv: int
    d: int
    seed: int
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0
    grid: tuple | None = None          # (T, Y, X) of the self-attention sequence when a position code is used
    audio_per_frame: int = 0
    pe: bool = False
    block: int = 128
    beta: float = 1.0
    n_split: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


WORKLOADS = {
    # tiny block-sparse self-attention (also run at beta = -inf)
    "tiny": Workload("tiny", B=1, H=2, Sq=1024, Skv=1024, d=64, seed=0, block=64, beta=0.5),
    # dense Stage-1 self-attention, 8x32x64 latent grid
    "dense16k": Workload("dense16k", B=1, H=32, Sq=16384, Skv=16384, d=128, seed=2, grid=(8, 32, 64), pe=True),
    # audio->video cross attention: 128 audio queries vs 32768 video keys, 8 KV chunks
    "cross": Workload("cross", B=1, H=32, Sq=128, Skv=32768, d=128, seed=3, n_split=8),
    # Stage-2 block-sparse self-attention: 16x64x64 video + 8 audio tokens per frame
    "sparse64k": Workload("sparse64k", B=1, H=32, Sq=65664, Skv=65664, d=128, seed=4, q_std=0.5, k_std=0.5,
                          grid=(16, 64, 64), audio_per_frame=8, pe=True, block=128, beta=1.0),
    # beta sweep at 32x64x64 (no audio)
    "sweep128k": Workload("sweep128k", B=1, H=32, Sq=131072, Skv=131072, d=128, seed=5, q_std=0.5, k_std=0.5,
                          grid=(32, 64, 64), pe=True, block=128, beta=1.0),
    # 3D neighbourhood attention over a 4x128x128 decoder tile, window 3x7x7 (frames x rows x columns)
    "na3d": Workload("na3d", B=1, H=32, Sq=65536, Skv=65536, d=128, seed=6, grid=(4, 128, 128), pe=True,
                     extra={"kernel": (3, 7, 7)}),
}


@dataclass
class LinearWorkload:
    """A projection y = x W^T of the transformer block: x [M, K] tokens, W [N, K]."""
    name: str
    M: int
    K: int
    N: int
    seed: int


LINEAR_WORKLOADS = {
    # the attention output projection of the Stage-2 block: 65664 tokens, hidden 32 x 128 = 4096
    "fp8_proj": LinearWorkload("fp8_proj", M=65664, K=4096, N=4096, seed=8),
}


def make_linear(w: LinearWorkload, device="cpu", M: int | None = None):
    """Draw (x bf16 [M, K], W bf16 [N, K]) for a projection.

    x ~ N(0, 1) with a per-token gain exp(0.5 N(0, 1)) (activations of
    different tokens differ in magnitude, which is what per-row scales are
    for); W ~ N(0, 1/K).  ``M`` overrides the token count."""
    M = w.M if M is None else M
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    gain = torch.exp(0.5 * torch.randn((M, 1), generator=g, device=device, dtype=torch.float32))
    x = torch.randn((M, w.K), generator=g, device=device, dtype=torch.float32) * gain
    W = torch.randn((w.N, w.K), generator=g, device=device, dtype=torch.float32) / math.sqrt(w.K)
    return x.to(torch.bfloat16), W.to(torch.bfloat16)


def make_qkv(w: Workload, device="cpu", Sq: int | None = None, Skv: int | None = None, H: int | None = None):
    """Draw (q, k, v) bf16 [B, H, S, d] for workload ``w``.

    ``Sq``/``Skv``/``H`` override the sizes (for scaled-down parity cases);
    with a position code the sequence then follows the same grid's raster
    order truncated to the requested length."""
    Sq = w.Sq if Sq is None else Sq
    Skv = w.Skv if Skv is None else Skv
    H = w.H if H is None else H
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    q = torch.randn((w.B, H, Sq, w.d), generator=g, device=device, dtype=torch.float32) * w.q_std
    k = torch.randn((w.B, H, Skv, w.d), generator=g, device=device, dtype=torch.float32) * w.k_std
    v = torch.randn((w.B, H, Skv, w.d), generator=g, device=device, dtype=torch.float32) * w.v_std
    if w.pe:
        t, y, x, aud = token_coords(w.grid, w.audio_per_frame, device=device)
        n = max(Sq, Skv)
        if n > t.numel():
            raise ValueError("sequence longer than the workload grid")
        pe = position_code(t[:n], y[:n], x[:n], w.d, 1.0, aud[:n])
        q += pe[:Sq]
        k += pe[:Skv]
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def to_f64(x: torch.Tensor):
    """Exact widening of a bf16 tensor to a float64 numpy array (host)."""
    return x.detach().to("cpu", torch.float32).double().numpy()
