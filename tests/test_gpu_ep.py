"""Expert-parallel sharding on one GPU: the routing map kernel, and the
shares of two shards of the experts adding up to the full layer (the shards
run one after the other in this process; no collective, no kernel waits on
another)."""
import numpy as np
import pytest
import torch

import oracle
import top_moe_expert_gb300 as moe
from tests import gpu_setup as gs
from top_moe_expert_gb300 import inputs
from top_moe_expert_gb300.ep import ExpertShard, _layer_library, ep_moe_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gs.need_gpu()


def test_local_routes_map_bit_exact():
    g = torch.Generator().manual_seed(3)
    ids = torch.randint(-2, 130, (37, 8), generator=g, dtype=torch.int32)
    dev = ids.cuda()
    for lo, hi in ((0, 64), (64, 128), (5, 6), (0, 0), (0, 128)):
        got = moe.moe_ep_local_routes(dev, lo, hi).cpu()
        want = torch.where((ids >= lo) & (ids < hi), ids - lo, torch.full_like(ids, -1))
        assert torch.equal(got, want), (lo, hi)
    # in place, and the empty case
    moe.moe_ep_local_routes(dev, 10, 20, local_ids=dev)
    assert torch.equal(dev.cpu(), torch.where((ids >= 10) & (ids < 20), ids - 10, torch.full_like(ids, -1)))
    empty = torch.empty((0, 8), dtype=torch.int32, device="cuda")
    assert moe.moe_ep_local_routes(empty, 0, 4).numel() == 0


@pytest.mark.parametrize("M", [1, 5, 64])
def test_two_shards_sum_to_the_full_layer(M):
    wl = inputs.Workload(f"ep_m{M}", M=M, d=2048, I=768, E=128, k=8, seed=11)
    f13 = torch.from_numpy(inputs.weights_fp32(wl, "w13")).cuda()
    f2 = torch.from_numpy(inputs.weights_fp32(wl, "w2")).cuda()
    q13, s13 = moe.moe_mxfp8_quantize(f13)
    q2, s2 = moe.moe_mxfp8_quantize(f2)
    x = inputs.activations(wl).cuda()
    ids_np, w_np = gs.routing(wl)
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np.astype(np.float32)).cuda()
    total = torch.zeros((M, wl.d), dtype=torch.float32, device="cuda")
    for r in range(2):
        sh = ExpertShard(wl.E, 2, r)
        w13 = moe.Weights(moe.MOE_W_MXFP8, q13[sh.e_lo:sh.e_hi].contiguous(), s13[sh.e_lo:sh.e_hi].contiguous())
        w2 = moe.Weights(moe.MOE_W_MXFP8, q2[sh.e_lo:sh.e_hi].contiguous(), s2[sh.e_lo:sh.e_hi].contiguous())
        local = moe.moe_ep_local_routes(ids, sh.e_lo, sh.e_hi)
        total += _layer_library(x, local, w, w13, w2)
    torch.cuda.synchronize()
    oq13, os13 = oracle.mxfp8_quantize_3d(inputs.weights_fp32(wl, "w13").astype(np.float64))
    oq2, os2 = oracle.mxfp8_quantize_3d(inputs.weights_fp32(wl, "w2").astype(np.float64))
    mode = oracle.MODE_EXACT if moe.moe_ffn_select_path(M, 8, 64, 2048, 768)[0] == moe.MOE_PATH_DECODE \
        else oracle.MODE_MX
    ref = oracle.moe_layer(gs.x_exact(x.cpu()), ids_np, w_np.astype(np.float64), wl.E,
                           {"fmt": "mxfp8", "q": oq13, "s": os13}, {"fmt": "mxfp8", "q": oq2, "s": os2},
                           mode=mode)["y"]
    gs.assert_layer_close(total, ref)


def test_single_rank_layer_is_the_plain_layer():
    """Without a process group (one rank owning every expert) the layer is
    the library's layer, bit for bit."""
    wl = inputs.Workload("ep_single", M=4, d=1024, I=512, E=16, k=4, seed=12)
    f13 = torch.from_numpy(inputs.weights_fp32(wl, "w13")).cuda()
    f2 = torch.from_numpy(inputs.weights_fp32(wl, "w2")).cuda()
    w13 = moe.Weights(moe.MOE_W_MXFP8, *moe.moe_mxfp8_quantize(f13))
    w2 = moe.Weights(moe.MOE_W_MXFP8, *moe.moe_mxfp8_quantize(f2))
    x = inputs.activations(wl).cuda()
    ids_np, w_np = gs.routing(wl)
    ids = torch.from_numpy(ids_np).cuda()
    w = torch.from_numpy(w_np.astype(np.float32)).cuda()
    y = ep_moe_layer(x, ids, w, w13, w2, ExpertShard(wl.E, 1, 0))
    assert torch.equal(y, _layer_library(x, ids, w, w13, w2))
