"""GPU parity of the output-centric decode path against the oracle.

Tolerance (stated for the path): max |err| <= 2e-3 * max |ref| with FP32
accumulation, cosine >= 0.999996; bf16 outputs additionally get half a bf16
ulp.  The oracle runs in exact mode (activations and h un-quantized), the
mathematics the decode path computes.
"""
import dataclasses
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


_layers = {}


def mx_layer(wl, **kw):
    key = (wl.name, tuple(sorted(kw.items())))
    if key not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        _layers[key] = gs.MxLayer(wl, **kw)
    return _layers[key]


def run_decode(layer, x, ids, w, out_dtype, **kw):
    return moe.moe_ffn_decode(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                              layer.w13, layer.w2, out_dtype=out_dtype, **kw)


def oracle_decode(layer, x, ids, w):
    w13, w2 = layer.oracle_weights(np.unique(ids))
    return oracle.moe_layer(gs.x_exact(x), ids, w.astype(np.float64), layer.wl.E, w13, w2)["y"]


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tiny_layer(out_dtype):
    wl = inputs.TINY
    layer = mx_layer(wl)
    x = inputs.activations(wl)
    ids, w = gs.routing(wl)
    y = run_decode(layer, x, ids, w, out_dtype)
    ref = oracle_decode(layer, x, ids, w)
    gs.assert_layer_close(y, ref)


def test_decode_m1_full_size_several_steps():
    wl = inputs.DECODE
    layer = mx_layer(wl)
    for step in range(3):
        x = inputs.activations(wl, step)
        ids, w = gs.routing(wl, step)
        y = run_decode(layer, x, ids, w, torch.float32)
        gs.assert_layer_close(y, oracle_decode(layer, x, ids, w))


@pytest.mark.parametrize("M,routing", [(4, "uniform"), (8, "zipf"), (64, "uniform")])
def test_decode_sweep_sizes(M, routing):
    wl = inputs.sweep(M, routing)
    layer = mx_layer(dataclasses.replace(inputs.DECODE, name="sweep_layer", seed=wl.seed))
    x = inputs.activations(wl)
    ids, w = gs.routing(wl)
    y = run_decode(layer, x, ids, w, torch.bfloat16)
    gs.assert_layer_close(y, oracle_decode(layer, x, ids, w))


def test_decode_is_bit_reproducible_and_independent_of_batch():
    wl = inputs.sweep(16)
    layer = mx_layer(dataclasses.replace(inputs.DECODE, name="sweep_layer", seed=wl.seed))
    x = inputs.activations(wl)
    ids, w = gs.routing(wl)
    ys = [run_decode(layer, x, ids, w, torch.float32) for _ in range(5)]
    digests = {hashlib.sha256(y.cpu().numpy().tobytes()).hexdigest() for y in ys}
    assert len(digests) == 1
    # tokens computed in a smaller batch give the same bits as inside the
    # batch (a single token takes the one-kernel path, checked against the
    # oracle instead)
    for t in (0, 7, 14):
        y2 = run_decode(layer, x[t:t + 2], ids[t:t + 2], w[t:t + 2], torch.float32)
        assert torch.equal(y2, ys[0][t:t + 2])
        y1 = run_decode(layer, x[t:t + 1], ids[t:t + 1], w[t:t + 1], torch.float32)
        gs.assert_layer_close(y1, oracle_decode(layer, x[t:t + 1], ids[t:t + 1], w[t:t + 1]))


def test_decode_invalid_routes_counted_and_skipped():
    wl = inputs.TINY
    layer = mx_layer(wl)
    x = inputs.activations(wl)
    ids, w = gs.routing(wl)
    ids = ids.copy()
    ids[3, 2] = -1
    ids[5, 0] = wl.E
    ids[5, 7] = 10 ** 6
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    y = run_decode(layer, x, ids, w, torch.float32, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist() == [3, 0]
    gs.assert_layer_close(y, oracle_decode(layer, x, ids, w))


def test_decode_duplicate_experts_and_empty_batch():
    wl = inputs.TINY
    layer = mx_layer(wl)
    x = inputs.activations(wl)
    ids, w = gs.routing(wl)
    ids = ids.copy()
    ids[:, 1] = ids[:, 0]                                 # same expert twice per token
    y = run_decode(layer, x, ids, w, torch.float32)
    gs.assert_layer_close(y, oracle_decode(layer, x, ids, w))
    y0 = run_decode(layer, x[:0], ids[:0], w[:0], torch.float32)
    assert y0.shape == (0, wl.d)


@pytest.mark.parametrize("xdt", [torch.float16, torch.bfloat16])
def test_awq_decode(xdt):
    wl = inputs.Workload("awq_small", M=5, d=1024, I=256, E=16, k=4, fmt="awq4", seed=7)
    layer = gs.AwqLayer(wl)
    x = inputs.activations(wl, dtype=xdt)
    ids, w = gs.routing(wl)
    y = moe.moe_ffn_decode(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                           layer.w13, layer.w2, out_dtype=torch.float32)
    ref = oracle.moe_layer(gs.x_exact(x), ids, w.astype(np.float64), wl.E, layer.host13, layer.host2)["y"]
    gs.assert_layer_close(y, ref)


def test_awq_decode_fixture_shape():
    wl = inputs.AWQ_FIXTURE
    layer = gs.AwqLayer(wl)
    x = inputs.activations(wl, dtype=torch.float16)
    ids, w = gs.routing(wl)
    y = moe.moe_ffn_decode(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                           layer.w13, layer.w2, out_dtype=torch.float32)
    ref = oracle.moe_layer(gs.x_exact(x), ids, w.astype(np.float64), wl.E, layer.host13, layer.host2)["y"]
    gs.assert_layer_close(y, ref)


# ---- one token, MXFP8 on the standard layout: the single-kernel path

@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_mx_single_token_standard_layout(out_dtype):
    wl = inputs.DECODE
    layer = mx_layer(wl)
    for step in range(2):
        x = inputs.activations(wl, step)
        ids, w = gs.routing(wl, step)
        gs.assert_layer_close(run_decode(layer, x, ids, w, out_dtype), oracle_decode(layer, x, ids, w))


def test_mx_single_token_activation_scales_routes_and_counter():
    wl = inputs.DECODE
    layer = mx_layer(wl)
    ids, w = gs.routing(wl)
    for scale in (1e-3, 3e3):
        x = (inputs.activations(wl, dtype=torch.float32) * scale).to(torch.bfloat16)
        gs.assert_layer_close(run_decode(layer, x, ids, w, torch.float32), oracle_decode(layer, x, ids, w))
    x = inputs.activations(wl)
    ids2 = ids.copy()
    ids2[0, 1] = ids2[0, 0]                                      # a duplicate
    ids2[0, 5] = -1                                              # and an invalid route
    ws = torch.zeros(moe.moe_ffn_decode_workspace_size(1, wl.k, wl.d, wl.I), dtype=torch.uint8, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    ys = [run_decode(layer, x, ids2, w, torch.float32, ws=ws, dev_status=st) for _ in range(3)]
    torch.cuda.synchronize()
    assert st.tolist() == [3, 0]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
    gs.assert_layer_close(ys[0], oracle_decode(layer, x, ids2, w))
    # the one-kernel path: each call adds one per CTA (one CTA per SM) to the
    # CTA count in ws[0..8)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ws[:8].view(torch.int64).item() == 3 * sms


def test_mx_single_token_most_routes():
    """One token with k = 13, the most routes the one-kernel plan takes at
    d = 1024, I = 512 on 152 SMs: every CTA's gate/up stages fill the ring's
    first lap, and the down stages reuse its slots."""
    wl = inputs.Workload("one_token_d1024_i512_e128_k13", M=1, d=1024, I=512, E=128, k=13, seed=12)
    layer = mx_layer(dataclasses.replace(wl, name="most_routes_layer"))
    x = inputs.activations(wl)
    ids, w = gs.routing(wl)
    ws = torch.zeros(moe.moe_ffn_decode_workspace_size(1, 13, wl.d, wl.I), dtype=torch.uint8, device="cuda")
    ys = [run_decode(layer, x, ids, w, torch.float32, ws=ws) for _ in range(3)]
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert ws[:8].view(torch.int64).item() == 3 * sms            # the one-kernel path ran
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
    gs.assert_layer_close(ys[0], oracle_decode(layer, x, ids, w))


def test_single_token_wait_runs_out_and_reports_timeout():
    """Failure detection without a GPU fault: the one-kernel path's wait for
    h is bounded.  Made to wait for a tag that no CTA writes, it gives up
    after its time limit, reports MOE_ERR_TIMEOUT in dev_status[1] and
    returns; the context stays usable and the workspace valid, so the next
    call on the same workspace matches the oracle."""
    wl = inputs.TINY
    layer = mx_layer(wl)
    x = inputs.activations(wl)[:1]
    ids, w = gs.routing(wl)
    ids, w = ids[:1], w[:1]
    ws = torch.zeros(moe.moe_ffn_decode_workspace_size(1, wl.k, wl.d, wl.I), dtype=torch.uint8, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    moe.moe_debug_exchange_stall(True)
    try:
        run_decode(layer, x, ids, w, torch.float32, ws=ws, dev_status=st)
        torch.cuda.synchronize()
    finally:
        moe.moe_debug_exchange_stall(False)
    assert st.tolist() == [0, 6]                                   # MOE_ERR_TIMEOUT
    assert ws[:8].view(torch.int64).item() == sms                  # every CTA still counted once
    st.zero_()
    y = run_decode(layer, x, ids, w, torch.float32, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0]
    gs.assert_layer_close(y, oracle_decode(layer, x, ids, w))


# ---- one token, 4-bit AWQ: the single-kernel path (gate/up, SwiGLU, down)

AWQ_M1 = inputs.Workload("awq_m1_d2048_i768_e128_k8", M=1, d=2048, I=768, E=128, k=8, fmt="awq4", seed=3)
AWQ_M1_SMALL = inputs.Workload("awq_m1_d1024_i256_e16_k4", M=1, d=1024, I=256, E=16, k=4, fmt="awq4", seed=7)
_awq_layers = {}


def awq_layer(wl):
    if wl.name not in _awq_layers:
        _awq_layers.clear()
        torch.cuda.empty_cache()
        _awq_layers[wl.name] = gs.AwqLayer(wl)
    return _awq_layers[wl.name]


def oracle_awq(layer, x, ids, w):
    return oracle.moe_layer(gs.x_exact(x), ids, np.asarray(w, dtype=np.float64), layer.wl.E, layer.host13,
                            layer.host2)["y"]


def run_awq(layer, x, ids, w, out_dtype=torch.float32, **kw):
    return moe.moe_ffn_decode(x.cuda(), torch.as_tensor(ids, dtype=torch.int32).cuda(),
                              torch.as_tensor(w, dtype=torch.float32).cuda(), layer.w13, layer.w2,
                              out_dtype=out_dtype, **kw)


@pytest.mark.parametrize("wl", [AWQ_M1_SMALL, AWQ_M1], ids=lambda w: w.name)
@pytest.mark.parametrize("xdt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_awq_single_token(wl, xdt, out_dtype):
    layer = awq_layer(wl)
    x = inputs.activations(wl, dtype=xdt)
    ids, w = gs.routing(wl)
    y = run_awq(layer, x, ids, w, out_dtype)
    gs.assert_layer_close(y, oracle_awq(layer, x, ids, w))


def test_awq_single_token_activation_scales():
    # x is staged in f16 after an exact power-of-two rescale
    wl = AWQ_M1
    layer = awq_layer(wl)
    ids, w = gs.routing(wl)
    for scale, xdt in ((1e-3, torch.float16), (3e3, torch.bfloat16)):
        x = (inputs.activations(wl, dtype=torch.float32) * scale).to(xdt)
        gs.assert_layer_close(run_awq(layer, x, ids, w), oracle_awq(layer, x, ids, w))


def test_awq_single_token_routes_repeats_and_barrier_counter():
    wl = AWQ_M1_SMALL
    layer = awq_layer(wl)
    x = inputs.activations(wl, dtype=torch.float16)
    ids = np.array([[3, 3, -1, wl.E]], dtype=np.int32)           # a duplicate and two invalid routes
    w = np.array([[0.4, 0.3, 0.2, 0.1]], dtype=np.float32)
    ws = torch.zeros(moe.moe_ffn_decode_workspace_size(1, wl.k, wl.d, wl.I), dtype=torch.uint8, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    ys = [run_awq(layer, x, ids, w, ws=ws, dev_status=st) for _ in range(3)]
    torch.cuda.synchronize()
    assert st.tolist() == [6, 0]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])                              # repeats are bit-identical
    gs.assert_layer_close(ys[0], oracle_awq(layer, x, ids, w))
    # the one-kernel path ran: one count per CTA (one CTA per SM) per call
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ws[:8].view(torch.int64).item() == 3 * sms
    # no valid route: y = 0
    y0 = run_awq(layer, x, np.array([[-1, wl.E, 99, -5]], dtype=np.int32), w, ws=ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y0).item() == 0


@pytest.mark.parametrize("wl", [inputs.LARGE_M1, inputs.LARGE_M8], ids=lambda w: w.name)
def test_large_expert_decode(wl):
    ids, w = gs.routing(wl)
    layer = mx_layer(wl, experts=tuple(np.unique(ids).tolist()))
    x = inputs.activations(wl)
    y = run_decode(layer, x, ids, w, torch.bfloat16)
    gs.assert_layer_close(y, oracle_decode(layer, x, ids, w))


# ------------------------------------------------ workspace reuse, routing in the layer call

def test_one_workspace_serves_every_batch_size():
    """One workspace, sized for the largest batch, reused by calls of other
    batch sizes in turn: every output equals the one computed with a fresh
    workspace; the CTA count in ws[0..8) holds exactly one per CTA for each
    call of the one-kernel single-token path, and its h exchange words in
    ws[256..) all carry the last such call's tag (the call's index, from 1):
    the other paths keep their data past the reserved start."""
    layer = mx_layer(dataclasses.replace(inputs.DECODE, name="ws_reuse_layer", seed=5))
    wl = dataclasses.replace(inputs.DECODE, name="ws_reuse_m8", M=8, seed=7)
    x = inputs.activations(wl)
    ids, w = gs.routing(wl)
    ws = torch.zeros(max(moe.moe_ffn_decode_workspace_size(M, wl.k, wl.d, wl.I) for M in (1, 3, 4, 8)),
                     dtype=torch.uint8, device="cuda")
    calls = [1, 3, 8, 1, 4, 1, 1]
    for M in calls:
        args = (layer, x[:M], ids[:M], w[:M], torch.float32)
        fresh = run_decode(*args)
        assert torch.equal(run_decode(*args, ws=ws), fresh), M
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n1 = calls.count(1)
    assert ws[:8].view(torch.int64).item() == n1 * sms
    words = ws[256:256 + wl.k * wl.I * 8].view(torch.int32).view(-1, 2).cpu()
    assert bool((words[:, 1] == n1).all())
    assert bool(torch.isfinite(words[:, 0].view(torch.float32)).all())


@pytest.mark.parametrize("M", [1, 3])
def test_decode_logits_equals_topk_then_decode(M):
    """moe_ffn_decode_logits is, bit for bit, moe_topk_softmax followed by
    moe_ffn_decode (one kernel that routes the token itself at M = 1, two
    calls otherwise); its routing equals the oracle's top-k and its output the
    oracle's layer."""
    layer = mx_layer(dataclasses.replace(inputs.DECODE, name="logits_layer", seed=7))
    wl = dataclasses.replace(inputs.DECODE, name=f"logits_m{M}", M=M, seed=7)
    for step in range(3):
        logits_np = inputs.router_logits(wl, step)
        logits = torch.from_numpy(logits_np).cuda()
        x = inputs.activations(wl, step).cuda()
        y1, ids1, w1 = moe.moe_ffn_decode_logits(logits, x, wl.k, layer.w13, layer.w2, out_dtype=torch.float32)
        ids2 = torch.empty((M, wl.k), dtype=torch.int32, device="cuda")
        w2_ = torch.empty((M, wl.k), dtype=torch.float32, device="cuda")
        moe.moe_topk_softmax(logits, wl.k, ids2, w2_)
        y2 = moe.moe_ffn_decode(x, ids2, w2_, layer.w13, layer.w2, out_dtype=torch.float32)
        assert torch.equal(ids1, ids2) and torch.equal(w1, w2_)
        assert torch.equal(y1, y2)
        ids_ref, w_ref = oracle.topk_softmax(logits_np, wl.k)
        assert np.array_equal(ids1.cpu().numpy(), ids_ref)
        np.testing.assert_allclose(w1.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)
        gs.assert_layer_close(y1, oracle_decode(layer, x.cpu(), ids_ref, w_ref.astype(np.float32)))


def test_decode_logits_ties_go_to_the_lower_expert():
    """The in-kernel routing ranks the logits: equal logits go to the lower
    expert id, slots in descending order -- the same as the oracle."""
    wl = inputs.DECODE
    layer = mx_layer(wl)
    logits_np = np.zeros((1, wl.E), dtype=np.float32)
    logits_np[0, [5, 77, 3, 100, 64, 2, 9, 40, 41]] = [2.0, 2.0, 1.5, 1.5, 1.5, 1.0, 1.0, 0.5, 0.5]
    x = inputs.activations(wl).cuda()
    y, ids, w = moe.moe_ffn_decode_logits(torch.from_numpy(logits_np).cuda(), x, wl.k, layer.w13, layer.w2,
                                          out_dtype=torch.float32)
    ids_ref, w_ref = oracle.topk_softmax(logits_np, wl.k)
    assert ids.cpu().numpy().tolist() == ids_ref.tolist() == [[5, 77, 3, 64, 100, 2, 9, 40]]
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)
    gs.assert_layer_close(y, oracle_decode(layer, x.cpu(), ids_ref, w_ref.astype(np.float32)))


# ------------------------------------------------ paired 4:8 sparse NVFP4

NV4 = inputs.Workload("nvfp4s_m4_d1024_i512_e16_k4", M=4, d=1024, I=512, E=16, k=4, seed=21)


def _nvfp4s_layer(wl):
    """Packed weights from the oracle's quantizer (the format is packed
    offline), on the device, and the same packing for the oracle."""
    p13 = oracle.nvfp4s_quantize_3d(inputs.weights_fp32(wl, "w13").astype(np.float64))
    p2 = oracle.nvfp4s_quantize_3d(inputs.weights_fp32(wl, "w2").astype(np.float64))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    mk = lambda p: moe.Weights(moe.MOE_W_NVFP4S, dev(p["v"]), dev(p["s"]), dev(p["m"]), dev(p["alpha"]))
    return mk(p13), mk(p2), p13, p2


@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float16])
def test_nvfp4s_decode_matches_oracle(xdt):
    w13, w2, p13, p2 = _nvfp4s_layer(NV4)
    x = inputs.activations(NV4, dtype=xdt)
    ids, w = gs.routing(NV4)
    ids = ids.copy()
    ids[1, 2] = -1                                            # an invalid route
    ref = oracle.moe_layer(gs.x_exact(x), ids, w.astype(np.float64), NV4.E, p13, p2)["y"]
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    for out_dtype in (torch.float32, torch.bfloat16):
        y = moe.moe_ffn_decode(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), w13, w2,
                               out_dtype=out_dtype, dev_status=st)
        gs.assert_layer_close(y, ref)
    torch.cuda.synchronize()
    assert st.tolist() == [2, 0]
    # a token's result does not depend on the batch's other tokens (two
    # tokens and four take the same two-kernel form; one token takes the
    # single-token kernel, checked on its own below)
    y2 = moe.moe_ffn_decode(x[:2].cuda(), torch.from_numpy(ids[:2]).cuda(), torch.from_numpy(w[:2]).cuda(), w13, w2,
                            out_dtype=torch.float32)
    assert torch.equal(y2[:2], moe.moe_ffn_decode(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                                                  w13, w2, out_dtype=torch.float32)[:2])


NV4_M1 = inputs.Workload("nvfp4s_m1_d2048_i768_e32_k8", M=1, d=2048, I=768, E=32, k=8, seed=24)
NV4_M1_SMALL = inputs.Workload("nvfp4s_m1_d1024_i512_e16_k4", M=1, d=1024, I=512, E=16, k=4, seed=25)
_NV4_CACHE = {}


def _nv4_cached(wl):
    if wl.name not in _NV4_CACHE:
        _NV4_CACHE[wl.name] = _nvfp4s_layer(wl)
    return _NV4_CACHE[wl.name]


@pytest.mark.parametrize("wl", [NV4_M1_SMALL, NV4_M1], ids=lambda w: w.name)
@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float16])
def test_nvfp4s_single_token(wl, xdt):
    """One token, paired 4:8 sparse NVFP4: the one-kernel path against the
    oracle (exact activations), and the counter of the kernel's launches
    shows that the one-kernel path ran."""
    w13, w2, p13, p2 = _nv4_cached(wl)
    x = inputs.activations(wl, dtype=xdt)
    ids, w = gs.routing(wl)
    ref = oracle.moe_layer(gs.x_exact(x), ids, w.astype(np.float64), wl.E, p13, p2)["y"]
    ws = torch.zeros(moe.moe_ffn_decode_workspace_size(1, wl.k, wl.d, wl.I), dtype=torch.uint8, device="cuda")
    for out_dtype in (torch.float32, torch.bfloat16):
        y = moe.moe_ffn_decode(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), w13, w2,
                               out_dtype=out_dtype, ws=ws)
        gs.assert_layer_close(y, ref)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ws[:8].view(torch.int64).item() == 2 * sms


def test_nvfp4s_single_token_routes_and_repeats():
    wl = NV4_M1_SMALL
    w13, w2, p13, p2 = _nv4_cached(wl)
    x = inputs.activations(wl, dtype=torch.bfloat16)
    ids = np.array([[5, 5, -1, wl.E]], dtype=np.int32)           # a duplicate and two invalid routes
    w = np.array([[0.4, 0.3, 0.2, 0.1]], dtype=np.float32)
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    ys = [moe.moe_ffn_decode(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), w13, w2,
                             out_dtype=torch.float32, dev_status=st) for _ in range(3)]
    torch.cuda.synchronize()
    assert st.tolist() == [6, 0]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
    gs.assert_layer_close(ys[0], oracle.moe_layer(gs.x_exact(x), ids, w.astype(np.float64), wl.E, p13, p2)["y"])


@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float16])
def test_nvfp4s_decode_logits_equals_topk_then_decode(xdt):
    """One token, NVFP4S: the routing inside the one kernel gives, bit for
    bit, moe_topk_softmax followed by moe_ffn_decode."""
    wl = NV4_M1
    w13, w2, p13, p2 = _nv4_cached(wl)
    x = inputs.activations(wl, dtype=xdt).cuda()
    logits = torch.from_numpy(inputs.router_logits(wl)).cuda()
    y1, ids1, w1 = moe.moe_ffn_decode_logits(logits, x, wl.k, w13, w2, out_dtype=torch.float32)
    ids2, wt2 = moe.moe_topk_softmax(logits, wl.k)
    y2 = moe.moe_ffn_decode(x, ids2, wt2, w13, w2, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(ids1, ids2) and torch.equal(w1, wt2)
    assert torch.equal(y1, y2)
    gs.assert_layer_close(y1, oracle.moe_layer(gs.x_exact(x.cpu()), ids2.cpu().numpy(),
                                               wt2.cpu().numpy().astype(np.float64), wl.E, p13, p2)["y"])


@pytest.mark.parametrize("xdt", [torch.float16, torch.bfloat16])
def test_awq_decode_logits_equals_topk_then_decode(xdt):
    """4-bit AWQ, one token: moe_ffn_decode_logits routes inside the one
    kernel and gives, bit for bit, moe_topk_softmax followed by
    moe_ffn_decode, with the same routing written out."""
    wl = AWQ_M1
    layer = awq_layer(wl)
    x = inputs.activations(wl, dtype=xdt).cuda()
    logits = torch.from_numpy(inputs.router_logits(wl)).cuda()
    y1, ids1, w1 = moe.moe_ffn_decode_logits(logits, x, wl.k, layer.w13, layer.w2, out_dtype=torch.float32)
    ids2, w2 = moe.moe_topk_softmax(logits, wl.k)
    y2 = moe.moe_ffn_decode(x, ids2, w2, layer.w13, layer.w2, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(ids1, ids2) and torch.equal(w1, w2)
    assert torch.equal(y1, y2)
    gs.assert_layer_close(y1, oracle_awq(layer, x.cpu(), ids2.cpu().numpy(), w2.cpu().numpy()))
