"""GPU parity: top-k routing, MXFP8 quantization and route alignment.

Integer / byte / index outputs are compared bit for bit with the oracle;
routing weights (FP32 on the GPU) within 2e-6 relative.
"""
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


# ---------------------------------------------------------------- top-k

@pytest.mark.parametrize("wl", [inputs.TINY, inputs.DECODE, inputs.sweep(512), inputs.sweep(64, "zipf"),
                                inputs.LARGE_M8], ids=lambda w: w.name)
def test_topk_softmax_matches_oracle(wl):
    logits = inputs.router_logits(wl)
    ids, w = moe.moe_topk_softmax(torch.from_numpy(logits).cuda(), wl.k)
    rid, rw = oracle.topk_softmax(logits, wl.k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=0)


def test_topk_ties_and_edge_shapes():
    logits = np.zeros((3, 40), dtype=np.float32)
    logits[0, [33, 7, 20]] = 2.0                      # ties -> lower id first
    logits[1, :] = np.arange(40, dtype=np.float32) % 5  # many ties
    logits[2, 39] = 1.0
    for k in (1, 4, 8, 32):
        ids, w = moe.moe_topk_softmax(torch.from_numpy(logits).cuda(), k)
        rid, rw = oracle.topk_softmax(logits, k)
        assert np.array_equal(ids.cpu().numpy(), rid)
        np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6)
    # E not a multiple of 32, k = E
    lg = np.random.default_rng(3).standard_normal((5, 7)).astype(np.float32)
    ids, w = moe.moe_topk_softmax(torch.from_numpy(lg).cuda(), 7)
    rid, rw = oracle.topk_softmax(lg, 7)
    assert np.array_equal(ids.cpu().numpy(), rid)


# ---------------------------------------------------------------- quantize

@pytest.mark.parametrize("scale", [1.0, 0.02, 3e-30, 1e30])
def test_mxfp8_quantize_fp32_bit_exact(scale):
    g = np.random.default_rng(17)
    v = (g.standard_normal((333, 256)) * scale).astype(np.float32)
    v[0, :32] = 0.0
    v[1, 5] = -1e-38 * scale
    v[2, :] *= np.exp(g.uniform(-20, 20, 256)).astype(np.float32)   # wide in-block range
    v[3, :32] = np.float32(448.0 * 1.1)                               # saturation region
    v[~np.isfinite(v)] = 1.0                                          # inputs must be finite
    q, s = moe.moe_mxfp8_quantize(torch.from_numpy(v).cuda())
    rq, rs = oracle.mxfp8_quantize(v.astype(np.float64))
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_mxfp8_quantize_bf16_and_denormals_bit_exact():
    g = np.random.default_rng(18)
    v = torch.from_numpy(g.standard_normal((64, 512)).astype(np.float32)).to(torch.bfloat16)
    q, s = moe.moe_mxfp8_quantize(v.cuda())
    rq, rs = oracle.mxfp8_quantize(v.to(torch.float64).numpy())
    assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(s.cpu().numpy(), rs)
    d = (g.standard_normal((8, 64)) * 1e-39).astype(np.float32)       # fp32 subnormals
    q, s = moe.moe_mxfp8_quantize(torch.from_numpy(d).cuda())
    rq, rs = oracle.mxfp8_quantize(d.astype(np.float64))
    assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(s.cpu().numpy(), rs)


# ---------------------------------------------------------------- alignment

def _align_both(ids, E, b, **kw):
    dev_status = torch.zeros(2, dtype=torch.int32, device="cuda")
    s, ex, npp = moe.moe_align_block_size(torch.from_numpy(ids).cuda(), E, b, dev_status=dev_status, **kw)
    rs, rex, rnpp, rinv = oracle.align(ids, E, b, cap_rows=s.numel(), cap_blocks=ex.numel())
    assert int(npp.item()) == rnpp
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(ex.cpu().numpy(), rex)
    assert dev_status.tolist() == [rinv, 0]
    return s, ex, npp


def test_align_worked_example_counts():
    ids = inputs.fixture_a_ids()
    s, ex, npp = _align_both(ids, 128, 8)
    assert int(npp.item()) == 400
    assert int((ex >= 0).sum().item()) == 50
    assert int((s[:400] != 168).sum().item()) == 168


@pytest.mark.parametrize("M,k,E,b,routing", [
    (21, 8, 128, 8, "uniform"), (1, 8, 128, 8, "uniform"), (64, 8, 128, 16, "zipf"),
    (512, 8, 128, 8, "uniform"), (512, 8, 128, 64, "zipf"), (8, 8, 384, 8, "uniform"),
    (7, 3, 50, 1, "uniform"), (300, 6, 1000, 128, "uniform"), (16384, 8, 128, 16, "uniform"),
    (2000, 8, 128, 256, "zipf"),
])
def test_align_matches_oracle(M, k, E, b, routing):
    wl = inputs.Workload("align", M=M, d=512, I=256, E=E, k=k, routing=routing, seed=9)
    ids, _ = oracle.topk_softmax(inputs.router_logits(wl), k)
    _align_both(ids, E, b)


def test_align_invalid_ids_empty_and_repeat():
    g = np.random.default_rng(4)
    ids = g.integers(-3, 131, size=(300, 8)).astype(np.int32)    # invalid ids both sides
    a = _align_both(ids, 128, 8)
    b = _align_both(ids, 128, 8)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    _align_both(np.zeros((0, 8), dtype=np.int32), 128, 8)       # M = 0
    _align_both(np.full((40, 8), 200, dtype=np.int32), 128, 8)  # all invalid
    _align_both(np.full((40, 8), 5, dtype=np.int32), 128, 8)    # one expert
    # multi-chunk path with every expert hit and invalid ids sprinkled in
    big = g.integers(0, 128, size=(4097, 8)).astype(np.int32)
    big[::37, 3] = -1
    _align_both(big, 128, 32)


def test_align_rejects_small_capacity():
    ids = torch.from_numpy(inputs.fixture_a_ids()).cuda()
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_align_block_size(ids, 128, 8, cap_rows=400, cap_blocks=50)
    assert ei.value.status == 3
