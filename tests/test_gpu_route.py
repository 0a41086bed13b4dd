"""GPU parity: moe_route_permute (routing ids, offsets, counts, permutation and
the staged NVFP4 activation are bit-exact; routing weights within fp32
rounding) and moe_combine (within BF16 rounding of the float64 sum)."""
import numpy as np
import pytest
import torch

import inputs
from oracle import moe as omoe
from oracle import nvfp4 as onv

from gpu_util import built_lib, dev, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import pipeline
    return nv, pipeline


def _route(nv, pipeline, x_t, logits, top_k, H):
    T, E = logits.shape
    s = pipeline.MoeShape(T=T, H=H, I=256, E=E, top_k=top_k)
    b = pipeline.MoeBuffers(s)
    b.perm_token.fill_(-7)
    b.a1_q.fill_(0x5A)
    b.a1_sf.fill_(0x5A)
    nv.moe_route_permute(dev(logits), x_t.cuda(), top_k, b.topk_ids, b.topk_w, b.counts, b.offsets,
                         b.perm_token, b.inv_perm, b.a1_q, b.a1_sf, b.workspace)
    nv.nvfp4_device_status()
    return b


@pytest.mark.parametrize("T,H,E,k,zipf", [(128, 512, 8, 2, False), (300, 256, 8, 2, False),
                                          (1000, 128, 64, 6, True), (77, 64, 256, 8, False),
                                          (5, 128, 3, 3, False), (513, 1024, 130, 4, True),
                                          (260, 128, 1024, 16, True), (200, 64, 500, 32, False),
                                          (5000, 64, 256, 8, True),    # >= 38 chunks: one top-k block per chunk
                                          # short batches (split top-k), E = 1024, k = 32
                                          (256, 7168, 256, 8, False), (1, 64, 1024, 8, False),
                                          (256, 64, 1024, 32, True), (255, 128, 64, 6, True),
                                          # 258 chunks: a long chunk walk in the offsets kernel
                                          (33000, 64, 256, 4, True)])
def test_route_permute_matches_oracle(nv, T, H, E, k, zipf):
    nv, pipeline = nv
    spec = inputs.moe_spec(T=T, H=H, I=256, E=E, top_k=k, seed=T + E, zipf=zipf)
    logits = inputs.moe_logits(spec)
    if T > 4:
        logits[3, :] = 0.25                              # a fully tied token
        logits[4, 1] = logits[4, 2] = logits[4].max() + 1
    x_t, x = inputs.moe_x(spec)
    b = _route(nv, pipeline, x_t, logits, k, H)
    ids, w = omoe.route_topk(logits, k)
    p = omoe.permute(ids, E)
    assert np.array_equal(host(b.topk_ids), ids)
    assert np.allclose(host(b.topk_w), w, rtol=2e-6, atol=1e-7)
    assert np.array_equal(host(b.counts), p["counts"])
    assert np.array_equal(host(b.offsets), p["offsets"])
    R = int(p["offsets"][-1])
    assert np.array_equal(host(b.perm_token)[:R], p["perm_token"])
    assert np.all(host(b.perm_token)[R:] == -7)                    # untouched past the groups
    assert np.array_equal(host(b.inv_perm), p["inv_perm"])
    a_q, a_sf = omoe.stage_activation(x, p["perm_token"])
    real = p["perm_token"] >= 0
    got_q = host(b.a1_q)[:R]
    assert np.array_equal(got_q[real], a_q[real])
    # padding rows: scales zero (below), nibbles not written (a zero scale makes them zero whatever they hold)
    assert np.all(got_q[~real] == 0x5A)
    gsf = onv.unswizzle_sf(host(b.a1_sf), R, H // 16)
    assert np.array_equal(gsf, a_sf)
    # every SF byte of the groups' 128-row bands is written (padding rows zero)
    assert np.array_equal(host(b.a1_sf)[:onv.sf_padded_bytes(R, H)], onv.swizzle_sf_fast(a_sf))


def test_route_permute_zero_tokens(nv):
    nv, pipeline = nv
    s = pipeline.MoeShape(T=0, H=64, I=256, E=4, top_k=2)
    b = pipeline.MoeBuffers(s)
    b.offsets.fill_(9)
    b.counts.fill_(9)
    logits = torch.empty((0, 4), dtype=torch.float32, device="cuda")
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    nv.moe_route_permute(logits, x, 2, b.topk_ids, b.topk_w, b.counts, b.offsets, b.perm_token, b.inv_perm,
                         b.a1_q, b.a1_sf, b.workspace)
    nv.nvfp4_device_status()
    assert host(b.offsets).tolist() == [0] * 5 and host(b.counts).tolist() == [0] * 4


@pytest.mark.parametrize("T,H,k", [(1, 8, 1), (64, 512, 2), (33, 7168, 8),
                                   (4100, 256, 4)])              # >= 4096 tokens: one block per token
def test_combine_matches_oracle(nv, T, H, k):
    nv, _ = nv
    rng = np.random.default_rng(T * H + k)
    n_rows = T * k + 5
    rows = omoe.round_to_bf16(rng.standard_normal((n_rows, H)))
    inv = rng.permutation(n_rows)[:T * k].reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    nv.moe_combine(dev(rows.astype(np.float32), torch.bfloat16), dev(inv), dev(w), y)
    nv.nvfp4_device_status()
    ref = omoe.combine(rows, inv, w.astype(np.float64))
    got = y.float().cpu().numpy()
    # fp32 accumulation then one BF16 rounding: within one BF16 ulp of the float64
    # result, plus the fp32 accumulation error on the magnitudes summed
    mag = omoe.combine(np.abs(rows), inv, w.astype(np.float64))
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 4e-7 * mag + 1e-30)
    assert np.mean(got != ref) < 0.01
