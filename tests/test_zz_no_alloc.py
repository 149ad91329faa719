"""moe_ffn_forward_noalloc: the step for callers that cannot allocate memory.

Some callers may not enter any allocator (for example code running inside another
allocator's hooks, in a real-time path, or under a memory budget already handed
out), so they cannot provide a workspace. This entry point runs the same decode
kernels on a fixed scratch array compiled into the library. These tests call it
through the C ABI on two calls in a row (the second call reuses the scratch the
first left behind) and check each call against the float64 oracle and, bit for bit,
against the workspace entry point, which runs the same kernels with the same
arithmetic.

This file is collected last on purpose: a run that stops at the first failure has
then already run every other test.
"""

import os

import numpy as np
import pytest

import expert_ffn_decode_gb300 as ffn
from expert_ffn_decode_gb300 import synth
from oracle import moe_oracle as mo
from tests.helpers import OUT_REL_L2, GpuLayer, compare, margin_tokens, oracle_cfg, rel_l2


def _built():
    if not os.path.exists(ffn.LIB_PATH):
        from expert_ffn_decode_gb300 import build
        build.build()


NOALLOC_SCRATCH_BYTES = 512 * 1024  # the fixed scratch compiled into the library


def test_noalloc_scratch_holds_the_largest_layer_and_rejects_workspace_flags():
    _built()
    # one token of the largest admitted layer: 32 picks of F = 3072 and a shared expert of
    # 3072 give 101376 f32 activations; with the control block, 1024 logits and the picks,
    # one copy of the arrays many CTAs read needs about 401 KiB, which the fixed scratch
    # holds. The workspace entry point keeps eight copies (about 3.2 MiB here); the fixed
    # scratch keeps as many as fit.
    one_copy = 512 + 1024 * 4 + 101376 * 4 + 3 * 256
    assert 400 * 1024 < one_copy <= NOALLOC_SCRATCH_BYTES
    cfg = ffn.make_cfg(hidden=3072, n_experts=1024, top_k=32, expert_ff=3072, shared_ff=3072, n_tokens=1)
    assert ffn.moe_workspace_size(cfg) > 8 * 101376 * 4
    # host staging and tracing need a workspace: rejected before anything is launched
    for flags in (ffn.MOE_HOST_IO, ffn.MOE_TRACE):
        cfg = ffn.make_cfg(hidden=256, n_experts=16, top_k=2, expert_ff=128, n_tokens=1, flags=flags)
        rc = ffn.moe_ffn_forward_noalloc(1 << 24, 1 << 28, None, 1 << 30, None, cfg, 1 << 26)
        assert rc == ffn.MOE_ERR_UNSUPPORTED
        assert "device buffers only" in ffn.moe_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("flags", [0, ffn.MOE_F32_ACT], ids=["fixed", "f32"])
@pytest.mark.parametrize("name", ["flint_decode_t1", "tiny_q4_0_t4"])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(name, flags):
    import torch
    _built()
    w = synth.WORKLOADS[name]
    layer = synth.make_layer(w)
    g = GpuLayer(layer, w)
    T = max(2, w["n_tokens"])
    cfg = ffn.make_cfg(**{**w, "n_tokens": T, "flags": flags})
    for call in range(2):
        x, _ = margin_tokens(layer, w, T, seed=w["seed"], stream=20 + call)
        ref, rid, rwt = mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                                   layer["shared_blocks"], oracle_cfg(w))
        want, ids, wts = g.run(x, flags=flags)  # moe_ffn_forward_ex with a workspace
        compare(want, ids, wts, ref, rid, rwt, f"{name} workspace call {call}")
        xd = torch.from_numpy(x).cuda()
        out = torch.full_like(xd, float("nan"))
        ffn.check(ffn.moe_ffn_forward_noalloc(xd, g.router_w, g.bias, g.experts, g.shared, cfg, out,
                                              torch.cuda.current_stream()))
        got = out.cpu().numpy()
        for t in range(T):
            assert rel_l2(got[t], ref[t]) <= OUT_REL_L2, (name, call, t)
        assert np.array_equal(got, want), (name, call)
