"""Audio->video cross attention with the video keys/values sharded over ranks.

"LTX-2.5 at 4K, in half the time", section "Attention across two GPUs": each
GPU keeps its own part of the video keys and values, answers the audio queries
against that part (a partial answer carrying its log-sum-exp), and the GPUs
exchange only those partial answers, which merge exactly.  Here every rank
runs attn_cross_splitkv_fwd over its key slice (itself split into
``n_split`` chunks), one all-gather collects every rank's partials in rank
order, and attn_lse_merge combines them.  The exchange is
world * n_split * B * H * Sq * (d + 1) fp32 values per rank, independent of
the key count.

Argument marshalling only: the partials and the merge run in the CUDA library;
``torch.distributed`` moves the partials.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_bounds(S: int, world: int, rank: int) -> tuple[int, int]:
    """Balanced, unpadded slice [lo, hi) of S keys for ``rank`` of ``world``
    (floor(r*S/world)), the same rule as the chunks inside a rank."""
    if world < 1 or not 0 <= rank < world or S < 0:
        raise ValueError("bad shard arguments")
    return (rank * S) // world, ((rank + 1) * S) // world


def _default_partials(q, k, v, n_split, scale):
    from . import attn_cross_splitkv_fwd
    return attn_cross_splitkv_fwd(q, k, v, n_split, scale=scale)


def _default_merge(o_part, lse_part):
    from . import attn_lse_merge
    return attn_lse_merge(o_part, lse_part)


def cross_attention_sharded(q, k_local, v_local, n_split: int = 1, scale=None, group=None, partials=None,
                            merge=None):
    """Exact attention of q [B, H, Sq, d] over the keys/values of every rank.

    k_local, v_local: this rank's slice [B, H, S_r, d] (any sizes, S_r >= 1).
    Returns (out [B, H, Sq, d], lse [B, H, Sq]) on every rank.  ``partials``
    and ``merge`` default to the CUDA library's attn_cross_splitkv_fwd and
    attn_lse_merge (their signatures: partials(q, k, v, n_split, scale) ->
    (o_part [n, B, H, Sq, d], lse_part [n, B, H, Sq]); merge(o_part, lse_part)
    -> (out, lse))."""
    partials = _default_partials if partials is None else partials
    merge = _default_merge if merge is None else merge
    if scale is None:
        scale = q.shape[-1] ** -0.5
    o_part, lse_part = partials(q, k_local, v_local, n_split, scale)
    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    if world > 1:
        o_all = torch.empty((world * o_part.shape[0], *o_part.shape[1:]), dtype=o_part.dtype, device=o_part.device)
        l_all = torch.empty((world * lse_part.shape[0], *lse_part.shape[1:]), dtype=lse_part.dtype,
                            device=lse_part.device)
        dist.all_gather_into_tensor(o_all, o_part.contiguous(), group=group)
        dist.all_gather_into_tensor(l_all, lse_part.contiguous(), group=group)
        o_part, lse_part = o_all, l_all
    return merge(o_part, lse_part)
