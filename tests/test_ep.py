"""The expert-parallel layer's host logic, on CPU.

The partition of the experts over the ranks is checked directly.  The layer
itself runs as gloo ranks in separate processes: each rank holds only its
own experts' weights and its own tokens, and ep_moe_layer gathers the
tokens, runs the rank's share and sums the shares.  On CPU the per-rank layer
is the oracle (the library's kernels need a GPU) and the routing map is a
plain statement of its definition; the sum over ranks must equal the oracle's
full layer on every rank's tokens.
"""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("E", [1, 2, 7, 10, 128, 384])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_partition_covers_every_expert_once(E, world):
    sys.path.insert(0, ROOT)
    from top_moe_expert_gb300.ep import ExpertShard
    if world > E:
        pytest.skip("more ranks than experts")
    owned = []
    for r in range(world):
        sh = ExpertShard(E, world, r)
        assert sh.n_local >= E // world and sh.n_local <= E // world + 1
        owned += list(range(sh.e_lo, sh.e_hi))
        for e in range(sh.e_lo, sh.e_hi):
            assert sh.owner(e) == r and ExpertShard(E, world, 0).owner(e) == r
    assert owned == list(range(E))


def test_partition_rejects_bad_arguments():
    sys.path.insert(0, ROOT)
    from top_moe_expert_gb300.ep import ExpertShard
    for args in ((0, 1, 0), (4, 0, 0), (4, 2, 2), (4, 2, -1)):
        with pytest.raises(ValueError):
            ExpertShard(*args)
    with pytest.raises(ValueError):
        ExpertShard(4, 2, 0).owner(4)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem(E, d, I, k, M_total, seed):
    """Seeded layer on the host: weights quantized by the oracle, tokens,
    routing (every expert id valid, plus one invalid route)."""
    import oracle
    g = np.random.Generator(np.random.PCG64(seed))
    w13 = g.normal(0, 0.02, (E, 2 * I, d))
    w2 = g.normal(0, 0.02, (E, d, I))
    q13, s13 = oracle.mxfp8_quantize_3d(w13)
    q2, s2 = oracle.mxfp8_quantize_3d(w2)
    x = g.standard_normal((M_total, d))
    ids = np.stack([g.permutation(E)[:k] for _ in range(M_total)]).astype(np.int32)
    ids[0, -1] = E                                      # an invalid route: skipped on every rank
    w = g.uniform(0.05, 1.0, (M_total, k))
    return q13, s13, q2, s2, x, ids, w


def _ep_worker(rank, world, port, E, out):
    sys.path.insert(0, ROOT)
    import torch
    import oracle
    from top_moe_expert_gb300.ep import ExpertShard, ep_moe_layer
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                         world_size=world)
    try:
        d, I, k, M_r = 64, 32, 3, 3
        q13, s13, q2, s2, x, ids, w = _problem(E, d, I, k, M_r * world, seed=17)
        sh = ExpertShard(E, world, rank)
        # this rank's weights: its experts only, renumbered from 0
        w13 = {"fmt": "mxfp8", "q": q13[sh.e_lo:sh.e_hi], "s": s13[sh.e_lo:sh.e_hi]}
        w2 = {"fmt": "mxfp8", "q": q2[sh.e_lo:sh.e_hi], "s": s2[sh.e_lo:sh.e_hi]}

        def local_routes(ids_t, shard):
            # the mapping's definition: own experts shifted to 0.., others -1
            e = ids_t
            return torch.where((e >= shard.e_lo) & (e < shard.e_hi), e - shard.e_lo, torch.full_like(e, -1))

        def layer(X, IDS, W, a, b):
            y = oracle.moe_layer(X.numpy(), IDS.numpy(), W.numpy(), sh.n_local, a, b)["y"]
            return torch.from_numpy(np.ascontiguousarray(y))

        rows = slice(rank * M_r, (rank + 1) * M_r)
        y = ep_moe_layer(torch.from_numpy(x[rows]), torch.from_numpy(ids[rows]), torch.from_numpy(w[rows]),
                         w13, w2, sh, layer=layer, local_routes=local_routes)
        full = oracle.moe_layer(x[rows], ids[rows], w[rows], E, {"fmt": "mxfp8", "q": q13, "s": s13},
                                {"fmt": "mxfp8", "q": q2, "s": s2})["y"]
        out.put((rank, float(np.abs(y.numpy() - full).max()), float(np.abs(full).max())))
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world,E", [(2, 8), (3, 10)])
def test_ep_layer_sums_to_the_full_layer_over_gloo_ranks(world, E):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ep_worker, args=(r, world, port, E, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == list(range(world))
    for rank, err, scale in got:
        # binary64 shares summed in another order than the full layer's sum
        assert scale > 0 and err <= 1e-12 * scale, (rank, err, scale)
