"""Full-size oracle parity of the MoE path on every expert the batch touches.

The decode and prefill workloads run in the launch configuration the benchmark
times (the same weights, routing and calls; no debug outputs).  For every
touched expert the test picks the rows where the GEMM kernels change path:
the group's first and last real rows, a random real row, and, where the group
has an odd number of 128-row blocks, the first row of its last block (the even
CTA of a half-empty pair tile; that tile's odd CTA has no rows).  Cold experts
with a single row are covered like the hot ones.

For each picked row (token t, slot j of expert e):
  * L1 + SwiGLU + NVFP4: a few 16-blocks of the re-quantised output (the first,
    the last and random ones), computed by the oracle from x[t] and just the W1
    rows those blocks read (the oracle quantiser works row by row, so a subset
    of rows quantises exactly as inside the whole matrix).  Bound: <= 0.1% of
    nibbles and scale bytes differ, each nibble by at most one E2M1 step.
  * L2: BF16 output columns at the edges of the 256-column tiles, of each CTA's
    128-column half and of the 32-row scale groups, the matrix's ends and
    random ones, against the oracle's float64 GEMM
    of the GPU's own a2 row (dequantised by the oracle) with the W2 rows of
    those columns, rounded once to BF16.  Bound: relative Frobenius 2e-3 (the
    path's bound for fused-path GEMM outputs fed the GPU's own quantised
    intermediates) and nearly all values identical.
The dense L1 workload's rows and the end-to-end y of sampled tokens are
checked against the fully CPU-quantised oracle in test_gpu_gemm.py and
test_gpu_moe.py.  The serving pipeline at both sizes gives the plain
forward's y bit for bit.
"""
import numpy as np
import pytest
import torch

import inputs
from oracle import moe as omoe
from oracle import nvfp4 as onv

from gpu_util import built_lib, compare_requantised, dev, host, rel_frobenius

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import pipeline
    return nv, pipeline


def _picked_rows(counts, offs, rng):
    """{padded row: expert} -- the rows where the kernels change path, for every touched expert."""
    picks = {}
    for e in np.nonzero(counts)[0]:
        lo, n = int(offs[e]), int(counts[e])
        rows = {lo, lo + n - 1, lo + int(rng.integers(n))}
        blocks = -(-n // 128)
        if blocks % 2 == 1:
            rows.add(lo + 128 * (blocks - 1))
        for r in rows:
            picks[r] = int(e)
    return picks


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_every_touched_expert_at_full_size(nv, name):
    nv, pipeline = nv
    spec = dict(inputs.CONFIGS[name])
    T, H, I, E, k = spec["T"], spec["H"], spec["I"], spec["E"], spec["top_k"]
    s = pipeline.MoeShape(T=T, H=H, I=I, E=E, top_k=k)
    w = pipeline.MoeWeights(s)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    b = pipeline.MoeBuffers(s)
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    pipeline.moe_forward(x_t.cuda(), dev(logits), w, b)
    nv.nvfp4_device_status()

    counts, offs, perm = host(b.counts), host(b.offsets), host(b.perm_token)
    rng = np.random.default_rng(spec["seed"] + 101)
    picks = _picked_rows(counts, offs, rng)
    rows = np.array(sorted(picks), dtype=np.int64)
    assert len(set(picks.values())) == int((counts > 0).sum())        # every touched expert
    r_dev = torch.from_numpy(rows).cuda()
    g_q = b.a2_q[r_dev].cpu().numpy()
    g_sf = onv.unswizzle_sf(host(b.a2_sf), b.rows_max, I // 16)[rows]
    g_out = b.rows_out[r_dev].float().cpu().numpy()
    tokens = perm[rows]
    assert np.all(tokens >= 0)
    xq, xsf = onv.quantize_rows(x[tokens])
    a1 = onv.dequantize_rows(xq, xsf)

    n_blk = I // 16
    # L2 output columns: edges of the 256-column tiles, of each CTA's 128-column
    # half and of 32-row scale groups, the matrix's ends, random ones
    edges = [0, 31, 32, 127, 128, 255, 256, 383, 384, H // 2 - 1, H // 2, H - 257, H - 256, H - 129, H - 128,
             H - 1]
    l1 = ([], [], [], [])          # GPU q, GPU sf, oracle q, oracle sf
    l2_got, l2_ref = [], []
    for e in sorted(set(picks.values())):
        sel = np.nonzero([picks[r] == e for r in rows])[0]
        blocks = np.unique(np.concatenate([[0, n_blk - 1], rng.choice(n_blk, 2, replace=False)]))
        # W1 rows 32b .. 32b+31 hold the interleaved gate/up columns of h block b
        w1_rows = (32 * blocks[:, None] + np.arange(32)[None, :]).ravel()
        wq, wsf = onv.quantize_rows(inputs.moe_w1_rows(spec, e, w1_rows))
        g = a1[sel] @ onv.dequantize_rows(wq, wsf).T
        oq, osf, _ = omoe.l1_swiglu_requant(g)
        byte_cols = (8 * blocks[:, None] + np.arange(8)[None, :]).ravel()
        # one 16-block per line (8 nibble bytes, 1 scale), so experts with different block counts stack
        l1[0].append(g_q[sel][:, byte_cols].reshape(-1, 8))
        l1[1].append(g_sf[sel][:, blocks].reshape(-1, 1))
        l1[2].append(oq.reshape(-1, 8))
        l1[3].append(osf.reshape(-1, 1))
        cols = np.unique(np.concatenate([edges, rng.choice(H, 14, replace=False)]))
        vq, vsf = onv.quantize_rows(inputs.moe_w2_rows(spec, e, cols))
        a2 = onv.dequantize_rows(g_q[sel], g_sf[sel])
        l2_ref.append(omoe.round_to_bf16(a2 @ onv.dequantize_rows(vq, vsf).T))
        l2_got.append(g_out[sel][:, cols])
    res = compare_requantised(*(np.concatenate(part) for part in l1))
    assert res["ok"], res
    got, ref = np.concatenate([a.ravel() for a in l2_got]), np.concatenate([a.ravel() for a in l2_ref])
    assert rel_frobenius(got, ref) <= 2e-3
    assert np.mean(got == ref) > 0.97


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_serving_pipeline_equals_plain_forward_at_full_size(nv, name):
    """The serving pipeline over two full-size batches (batch 1's staging inside
    batch 0's L2 GEMM, batch 0's combine inside batch 1's L1 GEMM; on the
    prefill batch both run on the CTA-pair kernels' side warps, on the decode
    batch as their own launches) gives each batch the plain forward's y, bit
    for bit."""
    nv, pipeline = nv
    spec = dict(inputs.CONFIGS[name])
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    w = pipeline.MoeWeights(s)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    del pool
    x_t, _ = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    xs = [x_t.cuda(), x_t.flip(0).contiguous().cuda()]
    lgs = [dev(logits), dev(np.ascontiguousarray(logits[::-1]))]
    plain = pipeline.MoeBuffers(s)
    ys = [pipeline.moe_forward(xs[i], lgs[i], w, plain).clone() for i in range(2)]
    del plain
    bufs = [pipeline.MoeBuffers(s), pipeline.MoeBuffers(s)]
    pipeline.moe_forward_deferred(xs[0], lgs[0], w, bufs[0])
    pipeline.moe_forward_deferred(xs[1], lgs[1], w, bufs[1], prev=bufs[0])
    y1 = pipeline.moe_finish_deferred(w, bufs[1])
    nv.nvfp4_device_status()
    assert torch.equal(bufs[0].y, ys[0])
    assert torch.equal(y1, ys[1])
