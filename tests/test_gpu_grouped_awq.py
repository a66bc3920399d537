"""GPU parity of the 4-bit AWQ grouped path (tcgen05 kind::f16 on weights
dequantized into tensor memory) on the packed-AWQ study's alignment shape.

The oracle takes the exact activations (bf16 or fp16, as given) and runs in
two modes: exact (the layer's mathematics) and with h rounded to fp16, the
precision of this path's second-GEMM operand (fp16 tensor-core surfaces, as
the packed-AWQ study's path uses).  Every output is checked against both at
the layer tolerance.  Checked: the alignment of fixture A (168 routes -> 400
aligned rows in 50 blocks), the layer output, bit-identical outputs across
five repeats, and bit-identical outputs under another block size (the result
does not depend on block membership: every output accumulates its K-tiles in
one fixed order, no split-K).
"""
import hashlib

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


@pytest.fixture(scope="module")
def fixture_a():
    wl = inputs.AWQ_FIXTURE
    layer = gs.AwqLayer(wl)
    x = inputs.activations(wl, dtype=torch.float16)
    ids, w = gs.routing(wl)
    ref = oracle.moe_layer(gs.x_exact(x), ids, w.astype(np.float64), wl.E, layer.host13, layer.host2,
                           mode=oracle.MODE_H16)["y"]
    exact = oracle.moe_layer(gs.x_exact(x), ids, w.astype(np.float64), wl.E, layer.host13, layer.host2)["y"]
    return wl, layer, x, ids, w, (ref, exact)


def _run(layer, x, ids, w, b, out_dtype=torch.float32):
    wl = layer.wl
    tid = torch.from_numpy(ids).cuda()
    aligned = moe.moe_align_block_size(tid, wl.E, b)
    M, k = ids.shape
    ws = torch.zeros(moe.moe_ffn_grouped_workspace_size(M, k, wl.d, wl.I, b, aligned[0].numel()),
                     dtype=torch.uint8, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    y = moe.moe_ffn_grouped(x.cuda(), tid, torch.from_numpy(w).cuda(), layer.w13, layer.w2, None, None, aligned, b,
                            out_dtype=out_dtype, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    return y, aligned


def test_awq_grouped_fixture_a(fixture_a):
    wl, layer, x, ids, w, ref = fixture_a
    y, aligned = _run(layer, x, ids, w, 8)
    assert int(aligned[2].item()) == 400
    ex = aligned[1].cpu().numpy()
    assert int((ex >= 0).sum()) == 50
    gs.assert_layer_close(y, ref[0])
    gs.assert_layer_close(y, ref[1])


def test_awq_grouped_repeats_bit_identical(fixture_a):
    wl, layer, x, ids, w, _ = fixture_a
    digests = {hashlib.sha256(_run(layer, x, ids, w, 8)[0].cpu().numpy().tobytes()).hexdigest() for _ in range(5)}
    assert len(digests) == 1


def test_awq_grouped_independent_of_block_size(fixture_a):
    """A route's result does not depend on the block size: every output
    accumulates its K-tiles in one fixed order, whatever the block holds."""
    wl, layer, x, ids, w, ref = fixture_a
    y8, _ = _run(layer, x, ids, w, 8)
    y16, _ = _run(layer, x, ids, w, 16)
    y32, _ = _run(layer, x, ids, w, 32)
    y64, _ = _run(layer, x, ids, w, 64)
    assert torch.equal(y8, y16) and torch.equal(y16, y32) and torch.equal(y32, y64)
    gs.assert_layer_close(y8, ref[0])
    gs.assert_layer_close(y8, ref[1])


@pytest.mark.parametrize("xdt,b", [(torch.float16, 16), (torch.bfloat16, 8), (torch.float16, 64)])
def test_awq_grouped_small(xdt, b):
    wl = inputs.Workload("awq_grouped_small", M=40, d=1024, I=256, E=16, k=4, fmt="awq4", seed=8)
    layer = gs.AwqLayer(wl)
    x = inputs.activations(wl, dtype=xdt)
    ids, w = gs.routing(wl)
    y, _ = _run(layer, x, ids, w, b, out_dtype=torch.bfloat16)
    for mode in (oracle.MODE_H16, oracle.MODE_EXACT):
        ref = oracle.moe_layer(gs.x_exact(x), ids, w.astype(np.float64), wl.E, layer.host13, layer.host2,
                               mode=mode)["y"]
        gs.assert_layer_close(y, ref)


@pytest.mark.parametrize("d,b", [(1024, 136), (1152, 32)])
def test_awq_grouped_limits_rejected(d, b):
    """Blocks above 128 rows, and d not a multiple of 256, are refused on the
    host with MOE_ERR_UNSUPPORTED (before anything is launched)."""
    wl = inputs.Workload("awq_grouped_limits", M=8, d=d, I=256, E=16, k=4, fmt="awq4", seed=9)
    layer = gs.AwqLayer(wl)
    x = inputs.activations(wl, dtype=torch.float16)
    ids, w = gs.routing(wl)
    tid = torch.from_numpy(ids).cuda()
    aligned = moe.moe_align_block_size(tid, wl.E, b)
    ws = torch.zeros(moe.moe_ffn_grouped_workspace_size(wl.M, wl.k, d, wl.I, b, aligned[0].numel()),
                     dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as err:
        moe.moe_ffn_grouped(x.cuda(), tid, torch.from_numpy(w).cuda(), layer.w13, layer.w2, None, None, aligned, b,
                            ws=ws)
    assert err.value.status == 2


def test_awq_grouped_workspace_reused_across_shapes():
    """One workspace serves AWQ calls of different batch and block sizes in
    turn; every output equals the one computed with a fresh workspace."""
    runs = []
    for M, b in ((40, 16), (12, 8)):
        wl = inputs.Workload(f"awq_reuse_m{M}", M=M, d=1024, I=256, E=16, k=4, fmt="awq4", seed=12)
        layer = gs.AwqLayer(wl)
        x = inputs.activations(wl, dtype=torch.float16)
        ids, w = gs.routing(wl)
        fresh, aligned = _run(layer, x, ids, w, b)
        runs.append((wl, layer, x, ids, w, b, aligned, fresh))
    size = max(moe.moe_ffn_grouped_workspace_size(r[0].M, r[0].k, r[0].d, r[0].I, r[5], r[6][0].numel()) for r in runs)
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        for wl, layer, x, ids, w, b, aligned, fresh in runs:
            st = torch.zeros(2, dtype=torch.int32, device="cuda")
            y = moe.moe_ffn_grouped(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), layer.w13,
                                    layer.w2, None, None, aligned, b, out_dtype=torch.float32, ws=ws, dev_status=st)
            torch.cuda.synchronize()
            assert st.tolist() == [0, 0]
            assert torch.equal(y, fresh)
