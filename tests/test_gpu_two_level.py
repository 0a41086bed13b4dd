"""GPU parity of the two-level NVFP4 scale (per-tensor encode scale g next to the
per-16 E4M3 scales): nvfp4_global_scale, the quantiser and the routing stage
under g, the GEMMs' per-group alpha and scaled re-quantisation, and the whole
FFN with every tensor's scale, against the oracle (``oracle.nvfp4.global_scale``,
``quantize_rows(x, g)``, ``moe.moe_ffn(a2_gscale=...)``).

Integer results (g, codes, scale bytes, weights, staged activations) are
compared bit for bit; h, BF16 rows and y within the path's bounds.  g of x and
of the weights is computed on each side from the same fp32 values; the L1
output's scale is an input (a calibration constant) and comes from the oracle.
"""
import contextlib

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
    return nv


def _scalar(v):
    return torch.tensor([v], dtype=torch.float32, device="cuda")


def _gpu_g(nv, t):
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    nv.nvfp4_global_scale(t, g)
    nv.nvfp4_device_status()
    return np.float32(host(g)[0])


@pytest.mark.parametrize("case", ["normal", "bf16", "strided", "zeros", "tiny", "huge"])
def test_global_scale_bit_exact(nv, case):
    rng = np.random.default_rng(60)
    x = (rng.standard_t(3, size=(333, 264)) * 0.3).astype(np.float32)
    if case == "zeros":
        x[:] = 0.0
    if case == "tiny":
        x = (x * np.float32(1e-40)).astype(np.float32)       # amax subnormal: 2688 / amax overflows
    if case == "huge":
        x[17, 5] = np.float32(3.0e38)
    t = torch.from_numpy(x).cuda()
    if case == "bf16":
        t = t.to(torch.bfloat16)
        x = t.float().cpu().numpy()
    if case == "strided":
        big = torch.zeros((333, 400), dtype=torch.float32, device="cuda")
        big[:, :264] = t
        big[:, 300:] = 1e6                                   # outside the columns: must be ignored
        g = torch.empty(1, dtype=torch.float32, device="cuda")
        nv.nvfp4_global_scale(big, g, cols=264)
        nv.nvfp4_device_status()
        assert np.float32(host(g)[0]) == onv.global_scale(x)
        return
    assert _gpu_g(nv, t) == onv.global_scale(x)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_quantize_plain_two_level_bit_exact(nv, dtype):
    x = inputs.plain_input_with_ties(61, 256, 512, dtype)
    t = torch.from_numpy(x).cuda()
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    g_dev = torch.empty(1, dtype=torch.float32, device="cuda")
    nv.nvfp4_global_scale(t, g_dev)
    q = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty(nv.sf_bytes(256, 512), dtype=torch.uint8, device="cuda")
    nv.nvfp4_quantize(t, 512, nv.MODE_PLAIN, q, sf, global_scale=g_dev)
    nv.nvfp4_device_status()
    g = onv.global_scale(x)
    assert np.float32(host(g_dev)[0]) == g
    oq, osf = onv.quantize_rows(x, g)
    assert np.array_equal(host(q), oq)
    assert np.array_equal(onv.unswizzle_sf(host(sf), 256, 32), osf)


def test_quantize_swiglu_two_level_bit_exact_on_its_h(nv):
    rows, cols = 300, 1024
    gu_t, _ = inputs.quantizer_input(dict(seed=62), rows=rows, cols=cols)
    g = np.float32(53.25)
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty(nv.sf_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    h = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    nv.nvfp4_quantize(gu_t.cuda(), cols, nv.MODE_SWIGLU_GU8, q, sf, h_debug=h, global_scale=_scalar(g))
    h1 = torch.empty_like(h)
    nv.nvfp4_quantize(gu_t.cuda(), cols, nv.MODE_SWIGLU_GU8, torch.empty_like(q), torch.empty_like(sf), h_debug=h1)
    nv.nvfp4_device_status()
    assert torch.equal(h, h1)                          # h_debug reports h before the scale
    oq, osf = onv.quantize_rows(host(h), g)
    assert np.array_equal(host(q), oq)
    assert np.array_equal(onv.unswizzle_sf(host(sf), rows, cols // 16), osf)


@contextlib.contextmanager
def _tiles(nv, mode):
    nv.nvfp4_set_gemm_tiles(mode)
    try:
        yield
    finally:
        nv.nvfp4_set_gemm_tiles(nv.GEMM_TILES_AUTO)


def test_grouped_gemm_two_level_both_kernels(nv):
    sizes, counts, N, K = [512, 128, 384], [500, 128, 300], 512, 768
    rows_max = sum(sizes)
    G = len(sizes)
    a_q, a_sf = inputs.random_nvfp4_operand(63, 0, rows_max, K)
    b = [inputs.random_nvfp4_operand(63, 1 + g, N, K) for g in range(G)]

    def swz(sf_lin):
        r, k = sf_lin.shape
        out = torch.empty(nv.sf_bytes(r, 16 * k), dtype=torch.uint8, device="cuda")
        nv.nvfp4_sf_swizzle(dev(sf_lin), r, k, k, 1, out)
        return out

    a_q_d, a_sf_d = dev(a_q), swz(a_sf)
    b_q_d = dev(np.stack([x[0] for x in b]))
    b_sf_d = torch.stack([swz(x[1]) for x in b])
    offs_np = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    offs, cnt = dev(offs_np), dev(np.array(counts, np.int32))
    ga, gb, gout = np.float32(3.7), np.array([0.9, 12.5, 0.031], np.float32), np.float32(41.0)
    alpha = 1.25
    outs = {}
    for mode in ("single", "pair"):
        out = torch.zeros((rows_max, N), dtype=torch.bfloat16, device="cuda")
        oq = torch.full((rows_max, N // 4), 0x77, dtype=torch.uint8, device="cuda")
        osf = torch.zeros(nv.sf_bytes(rows_max, N // 2), dtype=torch.uint8, device="cuda")
        h = torch.zeros((rows_max, N // 2), dtype=torch.float32, device="cuda")
        with _tiles(nv, {"single": nv.GEMM_TILES_SINGLE, "pair": nv.GEMM_TILES_PAIR}[mode]):
            kw = dict(a_global_scale=_scalar(ga), b_global_scale=dev(gb))
            nv.nvfp4_grouped_gemm(a_q_d, a_sf_d, rows_max, offs, cnt, G, N, K, b_q_d, b_sf_d, alpha, nv.EPI_BF16,
                                  out_bf16=out, **kw)
            nv.nvfp4_grouped_gemm(a_q_d, a_sf_d, rows_max, offs, cnt, G, N, K, b_q_d, b_sf_d, alpha,
                                  nv.EPI_SWIGLU_NVFP4, out_q=oq, out_sf=osf, h_debug=h,
                                  out_global_scale=_scalar(gout), **kw)
        nv.nvfp4_device_status()
        outs[mode] = (out.float().cpu().numpy(), host(oq), host(osf), host(h))
    for x, y in zip(outs["single"], outs["pair"]):
        assert np.array_equal(x, y)
    got, gq, gsf_sw, gh = outs["single"]
    valid = np.concatenate([np.arange(offs_np[g], offs_np[g] + counts[g]) for g in range(G)])
    a_deq = onv.dequantize_rows(a_q, a_sf)
    b_deq = np.stack([onv.dequantize_rows(*x) for x in b])
    acc = omoe.grouped_gemm(a_deq, offs_np, b_deq, alpha, ga, gb)
    ref = omoe.round_to_bf16(acc)
    assert rel_frobenius(got[valid].astype(np.float64), ref[valid]) <= 2e-3
    assert np.mean(got[valid] == ref[valid]) > 0.97
    oq_o, osf_o, oh = omoe.l1_swiglu_requant(acc, gout)
    assert rel_frobenius(gh[valid], oh[valid]) <= 2e-3
    gsf = onv.unswizzle_sf(gsf_sw, rows_max, N // 32)
    res = compare_requantised(gq[valid], gsf[valid], oq_o[valid], osf_o[valid])
    assert res["ok"], res
    hq, hsf = onv.quantize_rows(gh[valid], gout)
    assert np.array_equal(hq, gq[valid]) and np.array_equal(hsf, gsf[valid])


def _setup(pipeline, spec, two_level=True):
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    w = pipeline.MoeWeights(s, two_level=two_level)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    return s, w, pipeline.MoeBuffers(s)


@pytest.mark.parametrize("spec", [dict(inputs.CONFIGS["tiny"]),
                                  inputs.moe_spec(T=200, H=256, I=512, E=5, top_k=3, seed=64, zipf=True)],
                         ids=["tiny", "zipf200"])
def test_moe_two_level_end_to_end_small(nv, spec):
    from nvfp4_block_scaled_moe_gb300 import pipeline
    s, w, b = _setup(pipeline, spec)
    b.enable_h_debug()
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    w1, w2 = inputs.moe_all_weights(spec)
    # the L1 output's encode scale: calibrated by the oracle on its own h
    ga2 = onv.global_scale(omoe.moe_ffn(x, logits, w1, w2, spec["top_k"], a2_gscale=np.float32(1.0))["h"])
    b.a2_gs = _scalar(ga2)
    y = pipeline.moe_forward(x_t.cuda(), dev(logits), w, b, two_level=True)
    nv.nvfp4_device_status()
    o = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"], a2_gscale=ga2)
    E, H, I = spec["E"], spec["H"], spec["I"]
    assert np.float32(host(b.x_gs)[0]) == o["gscales"]["x"]
    assert np.array_equal(host(w.w1_gs), o["gscales"]["w1"]) and np.array_equal(host(w.w2_gs), o["gscales"]["w2"])
    assert np.array_equal(host(w.w1_q), o["w1_q"]) and np.array_equal(host(w.w2_q), o["w2_q"])
    w1_sf = np.stack([onv.unswizzle_sf(host(w.w1_sf)[e], 2 * I, H // 16) for e in range(E)])
    assert np.array_equal(w1_sf, o["w1_sf"])
    R = int(o["offsets"][-1])
    assert np.array_equal(host(b.offsets), o["offsets"])
    real = o["perm_token"] >= 0
    assert np.array_equal(host(b.a1_q)[:R][real], o["a1_q"][real])     # padding rows: zero scales only
    assert np.array_equal(onv.unswizzle_sf(host(b.a1_sf), b.rows_max, H // 16)[:R], o["a1_sf"])
    assert rel_frobenius(host(b.h_debug)[:R][real], o["h"][real]) <= 2e-3
    a2_sf = onv.unswizzle_sf(host(b.a2_sf), b.rows_max, I // 16)[:R]
    res = compare_requantised(host(b.a2_q)[:R][real], a2_sf[real], o["a2_q"][real], o["a2_sf"][real])
    assert res["ok"], res
    assert rel_frobenius(y.float().cpu().numpy(), o["y"]) <= 2e-2
    # the calibration pass: 2688 / amax of the h the kernels produce
    g_cal = pipeline.calibrate_a2_scale(x_t.cuda(), dev(logits), w, b)
    nv.nvfp4_device_status()
    b.enable_h_debug()
    b.a2_gs = None
    pipeline.moe_forward(x_t.cuda(), dev(logits), w, b, two_level=True)
    nv.nvfp4_device_status()
    assert np.float32(host(g_cal)[0]) == onv.global_scale(host(b.h_debug))


def test_moe_two_level_full_size_sampled_tokens(nv):
    from nvfp4_block_scaled_moe_gb300 import pipeline
    spec = dict(inputs.CONFIGS["prefill"])
    s, w, b = _setup(pipeline, spec)
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    ga2 = np.float32(84.0)
    b.a2_gs = _scalar(ga2)
    y = pipeline.moe_forward(x_t.cuda(), dev(logits), w, b, two_level=True)
    nv.nvfp4_device_status()
    gx = onv.global_scale(x)
    assert np.float32(host(b.x_gs)[0]) == gx
    T, k = spec["T"], spec["top_k"]
    pick = np.random.default_rng(65).choice(T, size=4, replace=False)
    tok = omoe.moe_ffn_tokens(x[pick], logits[pick], lambda e: inputs.moe_w1(spec, e),
                              lambda e: inputs.moe_w2(spec, e), k, two_level=dict(x=gx, a2=ga2))
    ids = host(b.topk_ids)
    assert np.array_equal(ids[pick], tok["ids"])
    for e in np.unique(tok["ids"]):
        assert host(w.w1_gs)[e] == onv.global_scale(inputs.moe_w1(spec, int(e)))
        assert host(w.w2_gs)[e] == onv.global_scale(inputs.moe_w2(spec, int(e)))
    rows = host(b.inv_perm)[pick].ravel()
    a2_sf = onv.unswizzle_sf(host(b.a2_sf), b.rows_max, spec["I"] // 16)[rows]
    res = compare_requantised(host(b.a2_q)[rows], a2_sf, tok["a2_q"].reshape(len(rows), -1),
                              tok["a2_sf"].reshape(len(rows), -1))
    assert res["ok"], res
    assert rel_frobenius(y.float().cpu().numpy()[pick], tok["y"]) <= 2e-2


def test_serving_pipeline_two_level_equals_plain(nv):
    """The serving pipeline with two-level scales (each batch's x scale computed
    in its own step; the staging, with x's scale, inside the previous batch's L2
    GEMM; the combine inside the next batch's L1 GEMM) gives every batch the
    plain two-level forward's y bit for bit, over three batches on two buffer
    sets sharing one calibrated L1-output scale."""
    from nvfp4_block_scaled_moe_gb300 import pipeline
    spec = inputs.moe_spec(T=600, H=1024, I=512, E=16, top_k=4, seed=66, zipf=True)
    s, w, b0 = _setup(pipeline, spec)
    x_t, _ = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    xs = [x_t.cuda(), (x_t.flip(0) * 3).contiguous().cuda(), (x_t.roll(5, 0) * 0.25).contiguous().cuda()]
    lgs = [dev(logits), dev(np.ascontiguousarray(logits[::-1])), dev(np.ascontiguousarray(np.roll(logits, 5, 0)))]
    a2_gs = pipeline.calibrate_a2_scale(xs[0], lgs[0], w, b0).clone()
    b0.h_debug = None
    plain = []
    for i in range(3):
        bp = pipeline.MoeBuffers(s)
        bp.a2_gs = a2_gs
        plain.append(pipeline.moe_forward(xs[i], lgs[i], w, bp, two_level=True).clone())
    bufs = [pipeline.MoeBuffers(s), pipeline.MoeBuffers(s)]
    for bb in bufs:
        bb.a2_gs = a2_gs
    ys = []
    for i in range(3):
        pipeline.moe_forward_deferred(xs[i], lgs[i], w, bufs[i & 1], prev=bufs[(i - 1) & 1] if i else None,
                                      two_level=True)
        if i:
            ys.append(bufs[(i - 1) & 1].y.clone())
    ys.append(pipeline.moe_finish_deferred(w, bufs[0], two_level=True).clone())
    nv.nvfp4_device_status()
    for i in range(3):
        assert torch.equal(ys[i], plain[i]), i
