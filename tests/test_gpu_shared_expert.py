"""GPU parity of the shared expert: a dense NVFP4 FFN of every token (staging,
L1 + SwiGLU + re-quantisation, L2 on the dense GEMM path) whose rows the combine
adds after the routed slots, against the oracle (``moe.shared_expert_rows``,
``moe.moe_ffn(shared=...)``, ``moe.moe_ffn_tokens(shared=...)``).

Bit-exact: the shared weights' and the staged x's codes.  Within bounds: the
shared expert's re-quantised codes (0.1% / one step), its BF16 rows (relative
Frobenius 2e-3) and y (2e-2); the combine with a shared row within the fp32
accumulation bound of the routed-only combine.
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


@pytest.mark.parametrize("T,H,k", [(1, 8, 1), (64, 512, 2), (33, 7168, 8)])
def test_combine_with_shared_rows(nv, T, H, k):
    nv, _ = nv
    rng = np.random.default_rng(T * H + k + 7)
    n_rows = T * k + 5
    rows = omoe.round_to_bf16(rng.standard_normal((n_rows, H)))
    shared = omoe.round_to_bf16(rng.standard_normal((T, H)) * 3)
    inv = rng.permutation(n_rows)[:T * k].reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    nv.moe_combine(dev(rows.astype(np.float32), torch.bfloat16), dev(inv), dev(w), y,
                   shared=dev(shared.astype(np.float32), torch.bfloat16))
    nv.nvfp4_device_status()
    ref = omoe.combine(rows, inv, w.astype(np.float64), shared)
    got = y.float().cpu().numpy()
    mag = omoe.combine(np.abs(rows), inv, w.astype(np.float64), np.abs(shared))
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 4e-7 * mag + 1e-30)
    assert np.mean(got != ref) < 0.01


def _setup(pipeline, spec, i_shared):
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    w = pipeline.MoeWeights(s)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    sh = pipeline.SharedExpert(s, i_shared)
    w1s, w2s = inputs.moe_shared_weights(spec, i_shared)
    sh.set_weights(torch.from_numpy(w1s).cuda(), torch.from_numpy(w2s).cuda())
    return s, w, pipeline.MoeBuffers(s), sh, (w1s, w2s)


@pytest.mark.parametrize("spec", [dict(inputs.CONFIGS["tiny"]),
                                  inputs.moe_spec(T=300, H=512, I=256, E=8, top_k=2, seed=81, zipf=True)],
                         ids=["tiny", "zipf300"])
def test_moe_with_shared_expert_small(nv, spec):
    nv, pipeline = nv
    s, w, b, sh, (w1s, w2s) = _setup(pipeline, spec, spec["I"])
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    y = pipeline.moe_forward(x_t.cuda(), dev(logits), w, b, shared=sh)
    nv.nvfp4_device_status()
    w1, w2 = inputs.moe_all_weights(spec)
    o = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"], shared=(w1s, w2s))
    so = o["shared"]
    T, H, Is = spec["T"], spec["H"], spec["I"]
    assert np.array_equal(host(sh.w1_q)[0], so["w1_q"]) and np.array_equal(host(sh.w2_q)[0], so["w2_q"])
    assert np.array_equal(onv.unswizzle_sf(host(sh.w1_sf)[0], 2 * Is, H // 16), so["w1_sf"])
    assert np.array_equal(host(sh.x_q)[:T], so["x_q"])
    assert np.array_equal(onv.unswizzle_sf(host(sh.x_sf), sh.rows, H // 16)[:T], so["x_sf"])
    a2_sf = onv.unswizzle_sf(host(sh.a2_sf), sh.rows, Is // 16)[:T]
    res = compare_requantised(host(sh.a2_q)[:T], a2_sf, so["a2_q"], so["a2_sf"])
    assert res["ok"], res
    rows = sh.out.float().cpu().numpy()[:T]
    assert rel_frobenius(rows, so["rows"]) <= 2e-3
    assert rel_frobenius(y.float().cpu().numpy(), o["y"]) <= 2e-2


def test_moe_with_shared_expert_full_size_sampled_tokens(nv):
    nv, pipeline = nv
    spec = dict(inputs.CONFIGS["prefill"])
    s, w, b, sh, (w1s, w2s) = _setup(pipeline, spec, spec["I"])
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    y = pipeline.moe_forward(x_t.cuda(), dev(logits), w, b, shared=sh)
    nv.nvfp4_device_status()
    pick = np.random.default_rng(82).choice(spec["T"], size=4, replace=False)
    tok = omoe.moe_ffn_tokens(x[pick], logits[pick], lambda e: inputs.moe_w1(spec, e),
                              lambda e: inputs.moe_w2(spec, e), spec["top_k"], shared=(w1s, w2s))
    so = omoe.shared_expert_rows(x[pick], w1s, w2s)
    assert rel_frobenius(sh.out.float().cpu().numpy()[pick], so["rows"]) <= 2e-3
    assert rel_frobenius(y.float().cpu().numpy()[pick], tok["y"]) <= 2e-2
