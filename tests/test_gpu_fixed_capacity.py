"""The fixed-capacity (batched) operand layout ("Hardware-Native Joint
Sparse-Quantization ...", App. D.1): its alignment bit-exact against the
oracle, and the grouped layer on it bit-identical to the layer on the
stable-construction alignment (a route's result does not depend on the rows
it shares a block with), on random routings and on the benchmark's
imbalanced token counts."""
import numpy as np
import pytest
import torch

import oracle
import top_moe_expert_gb300 as moe
from tests import gpu_setup as gs
from top_moe_expert_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gs.need_gpu()


@pytest.mark.parametrize("M,k,E,b,C", [(21, 8, 128, 8, 8), (64, 8, 128, 16, 16), (300, 4, 16, 32, 128),
                                       (5, 2, 3, 8, 8), (1000, 8, 64, 64, 64), (3000, 1, 7, 16, 512)])
def test_align_fixed_capacity_matches_oracle(M, k, E, b, C):
    rng = np.random.default_rng(M + E)
    ids = rng.integers(0, E, (M, k)).astype(np.int32)
    ids[0, 0] = -1                                       # an invalid route
    ids[M // 2, k - 1] = E
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = moe.moe_align_fixed_capacity(torch.from_numpy(ids).cuda(), E, b, C, dev_status=st)
    torch.cuda.synchronize()
    s, e, br, npp, bad = oracle.align_fixed_capacity(ids, E, b, C)
    assert np.array_equal(out[0].cpu().numpy(), s)
    assert np.array_equal(out[1].cpu().numpy(), e)
    assert np.array_equal(out[2].cpu().numpy(), br)
    assert int(out[3].item()) == npp
    assert int(st[0].item()) == bad                      # invalid plus dropped routes


def _layer_both(wl, ids, w, b):
    layer = gs.MxLayer(wl)
    sfa13, sfa2 = moe.moe_grouped_prepare(layer.w13, layer.w2)
    x = inputs.activations(wl).cuda()
    tid = torch.from_numpy(ids).cuda()
    tw = torch.from_numpy(w).cuda()
    M, k = ids.shape
    y_al = moe.moe_ffn_grouped(x, tid, tw, layer.w13, layer.w2, sfa13, sfa2,
                               moe.moe_align_block_size(tid, wl.E, b), b, out_dtype=torch.float32)
    counts = np.bincount(ids[(ids >= 0) & (ids < wl.E)].ravel(), minlength=wl.E)
    C = max(b, -(-int(counts.max()) // b) * b)
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    fixed = moe.moe_align_fixed_capacity(tid, wl.E, b, C, dev_status=st)
    ws = torch.empty(moe.moe_ffn_grouped_workspace_size(M, k, wl.d, wl.I, b, wl.E * C), dtype=torch.uint8,
                     device="cuda")
    y_fx = moe.moe_ffn_grouped(x, tid, tw, layer.w13, layer.w2, sfa13, sfa2, fixed, b, out_dtype=torch.float32,
                               ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    return layer, x, y_al, y_fx


@pytest.mark.parametrize("b", [16, 64])
def test_batched_layer_bit_identical_to_aligned(b):
    wl = inputs.Workload("fixed_m64", M=64, d=2048, I=768, E=128, k=8, seed=21)
    ids, w = gs.routing(wl)
    layer, x, y_al, y_fx = _layer_both(wl, ids, w, b)
    assert torch.equal(y_fx, y_al)
    tok = np.arange(0, 64, 7)
    w13, w2 = layer.oracle_weights(np.unique(ids[tok]))
    ref = oracle.moe_layer(gs.x_exact(x.cpu())[tok], ids[tok], w[tok].astype(np.float64), wl.E, w13, w2,
                           mode=oracle.MODE_MX)["y"]
    gs.assert_layer_close(y_fx[torch.from_numpy(tok).cuda()], ref)


@pytest.mark.parametrize("N,G", [(64, 8), (16, 16)])
def test_batched_layer_on_the_imbalanced_counts(N, G):
    ids = inputs.imbalanced_routing(N, G)
    M = ids.shape[0]
    assert np.array_equal(np.bincount(ids.ravel(), minlength=G), inputs.imbalanced_counts(N, G))
    wl = inputs.Workload(f"fixed_t8_n{N}_g{G}", M=M, d=2048, I=768, E=G, k=1, seed=22)
    w = np.ones((M, 1), dtype=np.float32)
    layer, x, y_al, y_fx = _layer_both(wl, ids, w, 16)
    assert torch.equal(y_fx, y_al)
