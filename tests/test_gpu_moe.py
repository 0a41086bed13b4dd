"""GPU parity of the whole path (route_permute -> L1 + SwiGLU + requant -> L2 ->
combine) against the fully CPU-quantised oracle.

Small workloads (the tiny configuration and ragged variants) are compared on
every output; the full-size decode and prefill workloads, run in the launch
configuration the benchmark times, are compared on sampled tokens that the
oracle computes one by one, plus invariants that hold at any size.
Bounds (from the path's specification): weights, routing, permutation and the
staged activation bit-exact; fused-epilogue h within relative Frobenius 2e-3;
re-quantised nibbles <= 0.1% different by <= one E2M1 step; y within relative
Frobenius 2e-2.
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


def _gpu_setup(pipeline, spec):
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    w = pipeline.MoeWeights(s)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    b = pipeline.MoeBuffers(s)
    return s, w, b


SMALL = [dict(inputs.CONFIGS["tiny"]),
         inputs.moe_spec(T=300, H=512, I=256, E=8, top_k=2, seed=21),
         inputs.moe_spec(T=200, H=256, I=512, E=5, top_k=3, seed=22, zipf=True),
         # more experts than the CTA-pair kernel takes groups: the GEMMs use the single-CTA kernel
         inputs.moe_spec(T=400, H=256, I=256, E=600, top_k=4, seed=23),
         # one expert, every token on it (one group of ceil(T/128) blocks)
         inputs.moe_spec(T=300, H=256, I=256, E=1, top_k=1, seed=27),
         # every token on every expert (k = E)
         inputs.moe_spec(T=150, H=256, I=256, E=4, top_k=4, seed=28),
         # 512 groups, the most the CTA-pair kernel takes, with top-32
         inputs.moe_spec(T=2100, H=256, I=256, E=512, top_k=32, seed=29, zipf=True),
         # a single token
         inputs.moe_spec(T=1, H=512, I=256, E=16, top_k=8, seed=30)]


@pytest.mark.parametrize("spec", SMALL, ids=["tiny", "ragged300", "zipf200", "e600", "e1", "k_eq_e", "e512k32",
                                             "t1"])
def test_moe_end_to_end_small(nv, spec):
    nv, pipeline = nv
    s, w, b = _gpu_setup(pipeline, spec)
    b.enable_h_debug()
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    y = pipeline.moe_forward(x_t.cuda(), dev(logits), w, b)
    nv.nvfp4_device_status()
    w1, w2 = inputs.moe_all_weights(spec)
    o = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"])
    E, H, I = spec["E"], spec["H"], spec["I"]
    # weights quantised on the GPU: bit-exact
    assert np.array_equal(host(w.w1_q), o["w1_q"]) and np.array_equal(host(w.w2_q), o["w2_q"])
    for e in range(E):
        assert np.array_equal(onv.unswizzle_sf(host(w.w1_sf[e]), 2 * I, H // 16), o["w1_sf"][e])
        assert np.array_equal(onv.unswizzle_sf(host(w.w2_sf[e]), H, I // 16), o["w2_sf"][e])
    # routing, permutation, staged activation: bit-exact
    assert np.array_equal(host(b.topk_ids), o["ids"])
    assert np.array_equal(host(b.offsets), o["offsets"])
    R = int(o["offsets"][-1])
    assert np.array_equal(host(b.perm_token)[:R], o["perm_token"])
    assert np.array_equal(host(b.inv_perm), o["inv_perm"])
    real = o["perm_token"] >= 0
    assert np.array_equal(host(b.a1_q)[:R][real], o["a1_q"][real])     # padding rows: zero scales only
    # fused L1 epilogue
    gh = host(b.h_debug)[:R]
    assert rel_frobenius(gh[real], o["h"][real]) <= 2e-3
    gsf = onv.unswizzle_sf(host(b.a2_sf), R, I // 16)
    res = compare_requantised(host(b.a2_q)[:R][real], gsf[real], o["a2_q"][real], o["a2_sf"][real])
    assert res["ok"], res
    # L2 rows and the combined output
    rows = b.rows_out.float().cpu().numpy()[:R]
    assert rel_frobenius(rows[real], o["rows"][real]) <= 2e-2
    assert rel_frobenius(y.float().cpu().numpy(), o["y"]) <= 2e-2


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_moe_full_size_sampled_tokens(nv, name):
    nv, pipeline = nv
    spec = dict(inputs.CONFIGS[name])
    s, w, b = _gpu_setup(pipeline, spec)
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    y = pipeline.moe_forward(x_t.cuda(), dev(logits), w, b)
    nv.nvfp4_device_status()
    T, k, E = spec["T"], spec["top_k"], spec["E"]
    # invariants at full size
    counts, offs = host(b.counts), host(b.offsets)
    inv, perm = host(b.inv_perm), host(b.perm_token)
    ids = host(b.topk_ids)
    assert counts.sum() == T * k and np.all(offs % 128 == 0)
    assert np.all(np.diff(offs) == -(-counts // 128) * 128)
    assert np.array_equal(perm[inv.ravel()], np.repeat(np.arange(T), k))
    e_of_row = np.searchsorted(offs, inv, side="right") - 1
    assert np.array_equal(e_of_row, ids)
    # sampled tokens, computed one by one by the oracle (prefill tokens mostly share
    # the hot experts, so more of them cost little; decode tokens touch 8 new experts each)
    pick = np.random.default_rng(spec["seed"]).choice(T, size=16 if name == "prefill" else 6, replace=False)
    tok = omoe.moe_ffn_tokens(x[pick], logits[pick], lambda e: inputs.moe_w1(spec, e),
                              lambda e: inputs.moe_w2(spec, e), k)
    assert np.array_equal(ids[pick], tok["ids"])
    assert np.allclose(host(b.topk_w)[pick], tok["w"], rtol=2e-6, atol=1e-7)
    rows = inv[pick].ravel()
    a2_sf = onv.unswizzle_sf(host(b.a2_sf), b.rows_max, spec["I"] // 16)[rows]
    res = compare_requantised(host(b.a2_q)[rows], a2_sf, tok["a2_q"].reshape(len(rows), -1),
                              tok["a2_sf"].reshape(len(rows), -1))
    assert res["ok"], res
    got = y.float().cpu().numpy()[pick]
    assert rel_frobenius(got, tok["y"]) <= 2e-2


def test_forward_from_host_buffers(nv):
    """nvfp4_moe_forward_host: host x and logits in, host y out, one C-ABI call.
    Its y equals the device-pointer forward's bit for bit (the same kernels on
    the same inputs) and is within the oracle bound; two calls in a row on
    alternating buffer sets and streams give the same bytes."""
    nv, pipeline = nv
    spec = inputs.moe_spec(T=300, H=512, I=256, E=8, top_k=2, seed=24, zipf=True)
    s, w, b = _gpu_setup(pipeline, spec)
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    y_dev = pipeline.moe_forward(x_t.cuda(), dev(logits), w, b).cpu()
    x_h, logits_h = x_t.pin_memory(), torch.from_numpy(logits).pin_memory()
    sets = [pipeline.MoeBuffers(s).enable_host_io(), pipeline.MoeBuffers(s).enable_host_io()]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.zeros((spec["T"], spec["H"]), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    for j in range(2):
        nv.nvfp4_moe_forward_host(x_h, logits_h, outs[j], spec["top_k"], w, sets[j], stream=streams[j])
    torch.cuda.synchronize()
    nv.nvfp4_device_status()
    assert torch.equal(outs[0], y_dev) and torch.equal(outs[1], y_dev)
    w1, w2 = inputs.moe_all_weights(spec)
    ref = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"])["y"]
    assert rel_frobenius(outs[0].float().numpy(), ref) <= 2e-2


def test_serving_loop_from_host_buffers(nv):
    """nvfp4_moe_step_host / nvfp4_moe_finish_host over three different batches on
    two buffer sets and two streams: each step routes its batch, runs the
    previous batch's L2 (staging this batch alongside) and its own L1 (running
    the previous batch's combine alongside), and copies the previous batch's y
    out.  Every y equals the plain forward's bit for bit."""
    nv, pipeline = nv
    spec = inputs.moe_spec(T=300, H=512, I=256, E=8, top_k=2, seed=25, zipf=True)
    s, w, _ = _gpu_setup(pipeline, spec)
    x_t, _ = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    xs = [x_t, x_t.flip(0).contiguous(), x_t.roll(7, 0).contiguous()]
    lgs = [logits, np.ascontiguousarray(logits[::-1]), np.ascontiguousarray(np.roll(logits, 7, 0))]
    plain = [pipeline.moe_forward(xs[i].cuda(), dev(lgs[i]), w, pipeline.MoeBuffers(s)).cpu() for i in range(3)]
    x_h = [x.pin_memory() for x in xs]
    l_h = [torch.from_numpy(l).pin_memory() for l in lgs]
    sets = [pipeline.MoeBuffers(s).enable_host_io(), pipeline.MoeBuffers(s).enable_host_io()]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    for ev, st in zip(done, streams):
        ev.record(st)
    y_h = [torch.zeros((spec["T"], spec["H"]), dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    for i in range(3):
        j = i & 1
        nv.nvfp4_moe_step_host(x_h[i], l_h[i], spec["top_k"], w, sets[j], prev=sets[1 - j] if i else None,
                               prev_y_host=y_h[i - 1] if i else None, compute_after=done[1 - j] if i else None,
                               compute_done=done[j], stream=streams[j])
    nv.nvfp4_moe_finish_host(w, sets[0], spec["top_k"], y_h[2], stream=streams[0])
    torch.cuda.synchronize()
    nv.nvfp4_device_status()
    for i in range(3):
        assert torch.equal(y_h[i], plain[i]), i


def test_serving_loop_with_batches_of_different_sizes(nv):
    """The serving loop over batches of 300, 37, 1 and 200 tokens through buffer
    sets sized for 300: each batch's y equals the plain forward of that batch
    alone, bit for bit.  (Buffers this small send the GEMMs to the single-CTA
    kernel, so the side jobs run as their own launches before each GEMM;
    test_gpu_side_jobs.py covers them inside the CTA-pair kernels.)"""
    nv, pipeline = nv
    spec = inputs.moe_spec(T=300, H=512, I=256, E=8, top_k=2, seed=26, zipf=True)
    s, w, _ = _gpu_setup(pipeline, spec)
    x_t, _ = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    sizes = [300, 37, 1, 200]
    starts = [0, 11, 299, 50]
    xs = [x_t[a:a + n].contiguous() for a, n in zip(starts, sizes)]
    lgs = [np.ascontiguousarray(logits[a:a + n]) for a, n in zip(starts, sizes)]
    plain = []
    for x, lg in zip(xs, lgs):
        si = pipeline.MoeShape(T=x.shape[0], H=s.H, I=s.I, E=s.E, top_k=s.top_k)
        plain.append(pipeline.moe_forward(x.cuda(), dev(lg), w, pipeline.MoeBuffers(si)).cpu())
    x_h = [x.pin_memory() for x in xs]
    l_h = [torch.from_numpy(l).pin_memory() for l in lgs]
    sets = [pipeline.MoeBuffers(s).enable_host_io() for _ in range(3)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    done = [torch.cuda.Event() for _ in range(3)]
    for ev, st in zip(done, streams):
        ev.record(st)
    y_h = [torch.zeros((n, spec["H"]), dtype=torch.bfloat16).pin_memory() for n in sizes]
    for i in range(len(sizes)):
        j, p = i % 3, (i - 1) % 3
        nv.nvfp4_moe_step_host(x_h[i], l_h[i], spec["top_k"], w, sets[j], prev=sets[p] if i else None,
                               prev_y_host=y_h[i - 1] if i else None, compute_after=done[p] if i else None,
                               compute_done=done[j], stream=streams[j])
    last = (len(sizes) - 1) % 3
    nv.nvfp4_moe_finish_host(w, sets[last], spec["top_k"], y_h[-1], stream=streams[last])
    torch.cuda.synchronize()
    nv.nvfp4_device_status()
    for i in range(len(sizes)):
        assert torch.equal(y_h[i], plain[i]), i
