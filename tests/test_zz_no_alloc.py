"""moe_route_permute_static: the routing entry point for callers that cannot
allocate device memory (engines that pre-reserve all memory in their own pool,
code under allocators that must not see extra allocations, host paths that may
not call cudaMalloc mid-step).  It keeps its scratch in a fixed device array
inside the library instead of a caller workspace.

Checked through the C ABI against moe_route_permute (the workspace version) on
calls in a row with different inputs and sizes: every output is identical, so
the array's leftover contents from one call do not leak into the next.  The
sequence covers both ways the routing fills its per-chunk histograms: short
batches clear the histogram and add into it, long ones (more than four chunks
per SM's worth, here 8192 tokens) overwrite every row, and a short call right
after a long one must not see the long call's counts.
This file is collected last so that a failure here stops a `-x` run only after
every other test has run.
"""
import numpy as np
import pytest
import torch

import inputs

from gpu_util import built_lib, dev, host

pytestmark = pytest.mark.gpu


def _buffers(pipeline, spec):
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=256, E=spec["E"], top_k=spec["top_k"])
    return pipeline.MoeBuffers(s)


def _outputs(b, R):
    perm = host(b.perm_token)[:R]
    # padding rows carry zero scales and unwritten nibbles: compare the real rows' nibbles
    return dict(ids=host(b.topk_ids), w=host(b.topk_w), counts=host(b.counts), offsets=host(b.offsets),
                perm=perm, inv=host(b.inv_perm), a1_q=host(b.a1_q)[:R][perm >= 0], a1_sf=host(b.a1_sf))


def test_static_scratch_route_permute_matches_workspace_version_twice():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import pipeline

    specs = [inputs.moe_spec(T=1000, H=1024, I=256, E=64, top_k=6, seed=41, zipf=True),
             inputs.moe_spec(T=256, H=7168, I=256, E=256, top_k=8, seed=42),      # decode-sized second call
             inputs.moe_spec(T=8192, H=256, I=256, E=32, top_k=4, seed=43, zipf=True),   # histogram rows overwritten
             inputs.moe_spec(T=300, H=512, I=256, E=32, top_k=4, seed=44)]       # short again, same E as before
    for spec in specs:
        logits = dev(inputs.moe_logits(spec))
        x_t, _ = inputs.moe_x(spec)
        x = x_t.cuda()
        ref = _buffers(pipeline, spec)
        nv.moe_route_permute(logits, x, spec["top_k"], ref.topk_ids, ref.topk_w, ref.counts, ref.offsets,
                             ref.perm_token, ref.inv_perm, ref.a1_q, ref.a1_sf, ref.workspace)
        got = _buffers(pipeline, spec)
        got.a1_sf.copy_(ref.a1_sf)          # bytes past the groups are not written by either call
        nv.moe_route_permute_static(logits, x, spec["top_k"], got.topk_ids, got.topk_w, got.counts, got.offsets,
                                    got.perm_token, got.inv_perm, got.a1_q, got.a1_sf)
        nv.nvfp4_device_status()
        R = int(host(ref.offsets)[-1])
        a, b = _outputs(ref, R), _outputs(got, R)
        for key in a:
            if key == "w":
                assert np.allclose(a[key], b[key], rtol=2e-6, atol=1e-7), key
            else:
                assert np.array_equal(a[key], b[key]), key


def test_static_scratch_routing_only_then_staging():
    """Routing only (a1_q, a1_sf NULL) through the static-scratch call, then the
    staging on its own (moe_stage_activation, which allocates nothing either):
    the same bytes as the workspace version's routing with staging."""
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import pipeline

    spec = inputs.moe_spec(T=700, H=1088, I=256, E=48, top_k=5, seed=45, zipf=True)
    logits = dev(inputs.moe_logits(spec))
    x = inputs.moe_x(spec)[0].cuda()
    ref = _buffers(pipeline, spec)
    nv.moe_route_permute(logits, x, spec["top_k"], ref.topk_ids, ref.topk_w, ref.counts, ref.offsets,
                         ref.perm_token, ref.inv_perm, ref.a1_q, ref.a1_sf, ref.workspace)
    got = _buffers(pipeline, spec)
    got.a1_sf.copy_(ref.a1_sf)
    got.a1_sf[:int(host(ref.offsets)[-1]) // 128 * 512 * (spec["H"] // 64)].fill_(0xEE)   # the groups' bands
    nv.moe_route_permute_static(logits, x, spec["top_k"], got.topk_ids, got.topk_w, got.counts, got.offsets,
                                got.perm_token, got.inv_perm, None, None)
    nv.moe_stage_activation(dict(x=x, inv_perm=got.inv_perm, counts=got.counts, offsets=got.offsets,
                                 a1_q=got.a1_q, a1_sf=got.a1_sf))
    nv.nvfp4_device_status()
    R = int(host(ref.offsets)[-1])
    a, b = _outputs(ref, R), _outputs(got, R)
    for key in a:
        if key == "w":
            assert np.allclose(a[key], b[key], rtol=2e-6, atol=1e-7), key
        else:
            assert np.array_equal(a[key], b[key]), key


def test_static_scratch_rejects_problems_beyond_its_array():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    lib = nv.load()
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    # 2^20 tokens over 1024 experts need 32 MiB of chunk histograms: more than the fixed 16 MiB
    st = lib.moe_route_permute_static(p, p, 1 << 20, 7168, 1024, 8, p, p, p, p, p, p, p, p, None, None, None)
    assert st == 2
    assert b"scratch" in lib.nvfp4_last_error()
