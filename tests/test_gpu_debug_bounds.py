"""The debug bounds-check build (libmoe_ffn_debug.so: the same sources with
MOE_DEBUG_BOUNDS): on valid inputs it gives the release build's bits; given
alignment outputs that break their contract (an expert id out of range, a row
count past the capacity, a negative route id, a block row past the end) it
skips what they would address, finishes, and reports MOE_ERR_BOUNDS in
dev_status[1].  The corrupted inputs are run on the debug build only: every
index they feed is one the debug build checks before use."""
import numpy as np
import pytest
import torch

import top_moe_expert_gb300 as moe
from tests import gpu_setup as gs
from top_moe_expert_gb300 import build, inputs

pytestmark = pytest.mark.gpu
MOE_ERR_BOUNDS = 7


@pytest.fixture(scope="module")
def debug_lib():
    gs.need_gpu()
    path = build.build(debug=True)
    yield path
    moe.use_library(build.LIB)


def _grouped(layer, sfa, x, ids, w, aligned, b, rows):
    M, k = ids.shape
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    ws = torch.zeros(moe.moe_ffn_grouped_workspace_size(M, k, layer.wl.d, layer.wl.I, b, rows), dtype=torch.uint8,
                     device="cuda")
    y = moe.moe_ffn_grouped(x, ids, w, layer.w13, layer.w2, sfa[0], sfa[1], aligned, b, out_dtype=torch.float32,
                            ws=ws, dev_status=st)
    torch.cuda.synchronize()
    return y, st.tolist()


def test_debug_build_gives_the_release_bits(debug_lib):
    wl = inputs.Workload("dbg_m64", M=64, d=1024, I=512, E=16, k=4, seed=40)
    layer = gs.MxLayer(wl)
    sfa = moe.moe_grouped_prepare(layer.w13, layer.w2)
    x = inputs.activations(wl).cuda()
    ids_np, w_np = gs.routing(wl)
    ids, w = torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda()
    b = 16
    outs = {}
    for name in ("release", "debug"):
        moe.use_library(build.LIB if name == "release" else debug_lib)
        al = moe.moe_align_block_size(ids, wl.E, b)
        y1, st1 = _grouped(layer, sfa, x, ids, w, al, b, al[0].numel())
        C = -(-int(np.bincount(ids_np.ravel(), minlength=wl.E).max()) // b) * b
        fx = moe.moe_align_fixed_capacity(ids, wl.E, b, C)
        y2, st2 = _grouped(layer, sfa, x, ids, w, fx, b, wl.E * C)
        y3 = moe.moe_ffn_decode(x[:1], ids[:1], w[:1], layer.w13, layer.w2, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert st1 == [0, 0] and st2 == [0, 0], name
        outs[name] = (y1, y2, y3)
    moe.use_library(build.LIB)
    for a, c in zip(outs["release"], outs["debug"]):
        assert torch.equal(a, c)


def test_debug_build_reports_bad_alignment_outputs(debug_lib):
    wl = inputs.Workload("dbg_bad", M=48, d=1024, I=512, E=16, k=4, seed=41)
    layer = gs.MxLayer(wl)
    sfa = moe.moe_grouped_prepare(layer.w13, layer.w2)
    x = inputs.activations(wl).cuda()
    ids_np, w_np = gs.routing(wl)
    ids, w = torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda()
    b = 16
    moe.use_library(debug_lib)
    try:
        good = moe.moe_align_block_size(ids, wl.E, b)
        rows = good[0].numel()
        cases = []
        a = [t.clone() for t in good]
        a[1][1] = wl.E + 3                                  # an expert id out of range
        cases.append(a)
        a = [t.clone() for t in good]
        a[2][0] = rows + 64 * b                             # more rows than the capacity
        cases.append(a)
        a = [t.clone() for t in good]
        a[0][5] = -7                                        # a negative route id
        cases.append(a)
        for al in cases:
            y, st = _grouped(layer, sfa, x, ids, w, tuple(al), b, rows)
            assert st[1] == MOE_ERR_BOUNDS, st
        # the fixed-capacity layout: a block row past the end
        C = -(-int(np.bincount(ids_np.ravel(), minlength=wl.E).max()) // b) * b
        fx = [t.clone() for t in moe.moe_align_fixed_capacity(ids, wl.E, b, C)]
        fx[2][0] = wl.E * C
        y, st = _grouped(layer, sfa, x, ids, w, tuple(fx), b, wl.E * C)
        assert st[1] == MOE_ERR_BOUNDS, st
        # the AWQ grouped kernel: an expert id out of range
        awl = inputs.Workload("dbg_awq", M=40, d=1024, I=256, E=16, k=4, fmt="awq4", seed=42)
        aw = gs.AwqLayer(awl)
        xa = inputs.activations(awl, dtype=torch.float16).cuda()
        aids_np, aw_np = gs.routing(awl)
        aids, awt = torch.from_numpy(aids_np).cuda(), torch.from_numpy(aw_np).cuda()
        al = [t.clone() for t in moe.moe_align_block_size(aids, awl.E, 8)]
        al[1][2] = -5
        st = torch.zeros(2, dtype=torch.int32, device="cuda")
        ws = torch.zeros(moe.moe_ffn_grouped_workspace_size(40, 4, 1024, 256, 8, al[0].numel()), dtype=torch.uint8,
                         device="cuda")
        moe.moe_ffn_grouped(xa, aids, awt, aw.w13, aw.w2, None, None, tuple(al), 8, ws=ws, dev_status=st)
        torch.cuda.synchronize()
        assert st.tolist()[1] == MOE_ERR_BOUNDS
    finally:
        moe.use_library(build.LIB)
    # the context stays usable: a valid call on the release build afterwards
    y, st = _grouped(layer, sfa, x, ids, w, good, b, rows)
    assert st == [0, 0]
