"""Expert-parallel layer: the routed expert layer with the experts sharded over
the ranks of a torch.distributed group.

"Hardware-Native Joint Sparse-Quantization for Trillion-Scale Mixture-of-
Experts", App. D.3, serves the layer with data parallelism over tokens and
expert parallelism over experts (an all-to-all dispatch of the routed tokens
to the ranks that own their experts and an all-to-all combine back).  For
decode-sized batches this module takes the equivalent gather form:

  1. every rank gathers all ranks' tokens (x, routing ids and weights);
  2. each rank runs the layer on its own experts' weights with the routing
     mapped by moe_ep_local_routes (routes of other ranks' experts become
     invalid and are skipped), which gives its experts' share of y for every
     token;
  3. the shares are summed over the ranks and each rank keeps its own
     tokens' rows.

Each route is computed by exactly one rank and contributes zero elsewhere,
so the sum is the full layer.  The collectives are torch.distributed calls
(NCCL between GPUs, gloo on CPU); every step of the layer itself runs in the
library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional

import torch
import torch.distributed as dist


@dataclass(frozen=True)
class ExpertShard:
    """Experts [e_lo, e_hi) of E, owned by `rank` of `world` (contiguous,
    balanced: rank r owns E * r // world .. E * (r + 1) // world)."""
    E: int
    world: int
    rank: int

    def __post_init__(self):
        if self.E < 1 or self.world < 1 or not (0 <= self.rank < self.world):
            raise ValueError(f"bad shard E={self.E} world={self.world} rank={self.rank}")

    @property
    def e_lo(self) -> int:
        return self.E * self.rank // self.world

    @property
    def e_hi(self) -> int:
        return self.E * (self.rank + 1) // self.world

    @property
    def n_local(self) -> int:
        return self.e_hi - self.e_lo

    def owner(self, e: int) -> int:
        """The rank that owns expert e."""
        if not (0 <= e < self.E):
            raise ValueError(f"expert {e} outside [0, {self.E})")
        r = e * self.world // self.E
        while self.E * (r + 1) // self.world <= e:
            r += 1
        while self.E * r // self.world > e:
            r -= 1
        return r


def _local_routes_library(ids: torch.Tensor, shard: ExpertShard) -> torch.Tensor:
    from top_moe_expert_gb300 import moe_ep_local_routes
    return moe_ep_local_routes(ids.contiguous(), shard.e_lo, shard.e_hi)


def _layer_library(x, ids, w, w13, w2):
    import top_moe_expert_gb300 as moe
    M, k = ids.shape
    if w13.fmt == moe.MOE_W_NVFP4S:                    # the decode path is this format's only path
        return moe.moe_ffn_decode(x, ids, w, w13, w2, out_dtype=torch.float32)
    path, b = moe.moe_ffn_select_path(M, k, w13.E, x.shape[1], w2.K, w13.fmt)
    if path == moe.MOE_PATH_DECODE:
        return moe.moe_ffn_decode(x, ids, w, w13, w2, out_dtype=torch.float32)
    sfa = moe.moe_grouped_prepare(w13, w2) if w13.fmt == moe.MOE_W_MXFP8 else (None, None)
    aligned = moe.moe_align_block_size(ids, w13.E, b)
    return moe.moe_ffn_grouped(x, ids, w, w13, w2, sfa[0], sfa[1], aligned, b, out_dtype=torch.float32)


def _gather_rows(t: torch.Tensor, world: int, group) -> torch.Tensor:
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.cat(parts, dim=0)


def ep_moe_layer(x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor, w13_local, w2_local,
                 shard: ExpertShard, group=None,
                 layer: Optional[Callable] = None, local_routes: Optional[Callable] = None) -> torch.Tensor:
    """y [M_r, d] (fp32 from the library's layer) for this rank's tokens
    x [M_r, d] (routing ids over all
    E experts, weights [M_r, k]); w13_local / w2_local hold this rank's
    experts [e_lo, e_hi) as experts 0 .. n_local - 1.  Every rank of the
    group calls this with the same M_r.  `layer(x, ids, w, w13, w2)` and
    `local_routes(ids, shard)` default to the library's kernels."""
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    if world != shard.world:
        raise ValueError(f"shard is for {shard.world} ranks; the group has {world}")
    layer = layer or _layer_library
    local_routes = local_routes or _local_routes_library
    M_r = x.shape[0]
    if world > 1:
        X = _gather_rows(x, world, group)
        IDS = _gather_rows(topk_ids, world, group)
        W = _gather_rows(topk_w, world, group)
    else:
        X, IDS, W = x, topk_ids, topk_w
    y_part = layer(X, local_routes(IDS, shard), W, w13_local, w2_local).contiguous()
    if world > 1:
        # sum of every rank's share; this rank keeps its own tokens' rows
        dist.all_reduce(y_part, op=dist.ReduceOp.SUM, group=group)
    rank = shard.rank
    return y_part[rank * M_r:(rank + 1) * M_r]
