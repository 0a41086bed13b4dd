"""GPU checks of the side jobs the CTA-pair GEMMs run on two extra warps per CTA
(or, with any other kernel, as their own launch before the GEMM):

* the combine of an earlier batch inside the SwiGLU (L1) GEMM: y equals
  moe_combine's bit for bit (the same fp32 slot-order sum and one rounding);
* the activation staging of a later batch inside the BF16 (L2) GEMM: the
  bytes equal the oracle's staging and moe_route_permute's (every real row's
  nibbles, every scale byte of the groups' 128-row bands), padding nibbles
  are left untouched, with and without the two-level scale;
* either way the GEMM's own outputs are the bytes it writes without the side
  job, on both tile kernels (a GEMM with tiles for fewer than half the SMs
  runs the job as its own launch, like the single-CTA kernel), for short and
  long batches and top-k up to 32;
* the serving pipeline (route(i); L2(i-1) staging batch i; L1(i) combining
  batch i-1; the last batch's L2 and combine at the end) gives every batch the
  y of the plain forward, bit for bit.
"""
import contextlib

import numpy as np
import pytest
import torch

import inputs
from oracle import moe as omoe
from oracle import nvfp4 as onv

from gpu_util import built_lib, dev, host, rel_frobenius

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    built_lib()
    import nvfp4_block_scaled_moe_gb300 as nv
    from nvfp4_block_scaled_moe_gb300 import pipeline
    return nv, pipeline


@contextlib.contextmanager
def _tiles(nv, mode):
    nv.nvfp4_set_gemm_tiles(mode)
    try:
        yield
    finally:
        nv.nvfp4_set_gemm_tiles(nv.GEMM_TILES_AUTO)


def _swizzled(nv, sf_lin):
    rows, k_sf = sf_lin.shape
    out = torch.empty(nv.sf_bytes(rows, 16 * k_sf), dtype=torch.uint8, device="cuda")
    nv.nvfp4_sf_swizzle(dev(sf_lin), rows, k_sf, k_sf, 1, out)
    return out


@pytest.mark.parametrize("T,H,k", [(300, 1024, 8), (4100, 512, 4), (33, 7168, 32), (1, 64, 1)])
def test_side_combine_equals_combine(nv, T, H, k):
    nv, _ = nv
    # N = 2048: enough tiles (64) that the pair kernel hosts the job on its own warps
    sizes, counts, N, K = [512, 384, 256], [500, 300, 256], 2048, 768
    rows_max, G = sum(sizes), len(sizes)
    a_q, a_sf = inputs.random_nvfp4_operand(61, 0, rows_max, K)
    b = [inputs.random_nvfp4_operand(61, 1 + g, N, K) for g in range(G)]
    a_q_d, a_sf_d = dev(a_q), _swizzled(nv, a_sf)
    b_q_d, b_sf_d = dev(np.stack([x[0] for x in b])), torch.stack([_swizzled(nv, x[1]) for x in b])
    offs = dev(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32))
    cnt = dev(np.array(counts, np.int32))
    # the earlier batch: random BF16 rows, a permutation, weights
    rng = np.random.default_rng(T * H + k)
    n_rows = T * k + 5
    rows = dev(omoe.round_to_bf16(rng.standard_normal((n_rows, H))).astype(np.float32), torch.bfloat16)
    inv = dev(rng.permutation(n_rows)[:T * k].reshape(T, k).astype(np.int32))
    w = dev(rng.random((T, k)).astype(np.float32))
    y_ref = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    nv.moe_combine(rows, inv, w, y_ref)

    def gemm(side):
        oq = torch.full((rows_max, N // 4), 0x77, dtype=torch.uint8, device="cuda")
        osf = torch.zeros(nv.sf_bytes(rows_max, N // 2), dtype=torch.uint8, device="cuda")
        y = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
        nv.nvfp4_grouped_gemm(a_q_d, a_sf_d, rows_max, offs, cnt, G, N, K, b_q_d, b_sf_d, 1.0, nv.EPI_SWIGLU_NVFP4,
                              out_q=oq, out_sf=osf, side_combine=(rows, inv, w, y) if side else None)
        nv.nvfp4_device_status()
        return host(oq), host(osf), y

    plain_q, plain_sf, _ = gemm(False)
    for mode in (nv.GEMM_TILES_PAIR, nv.GEMM_TILES_SINGLE):
        with _tiles(nv, mode):
            q, sf, y = gemm(True)
        assert np.array_equal(q, plain_q) and np.array_equal(sf, plain_sf)
        assert torch.equal(y, y_ref), mode


@pytest.mark.parametrize("T,H,E,k,zipf,two_level", [
    (300, 1088, 8, 2, True, False),       # two 1024-column segments, the second two lanes wide
    (77, 64, 256, 8, False, False),       # one segment of two lanes; mostly cold experts
    (1000, 512, 64, 6, True, True),       # two-level: x quantised as fp32(x * g)
    (5, 128, 3, 3, False, False),
    (4100, 256, 130, 4, True, False),     # many segments per side warp
    (256, 64, 1024, 32, True, False)])    # top-32 of 1024 experts
def test_side_stage_equals_route_staging(nv, T, H, E, k, zipf, two_level):
    nv, pipeline = nv
    spec = inputs.moe_spec(T=T, H=H, I=256, E=E, top_k=k, seed=T + 7 * E, zipf=zipf)
    logits = inputs.moe_logits(spec)
    x_t, x = inputs.moe_x(spec)
    s = pipeline.MoeShape(T=T, H=H, I=256, E=E, top_k=k)
    x_d, lg = x_t.cuda(), dev(logits)
    gs = torch.ones(1, dtype=torch.float32, device="cuda")
    if two_level:
        nv.nvfp4_global_scale(x_d, gs)
    gsa = gs if two_level else None

    ref = pipeline.MoeBuffers(s)
    ref.a1_q.fill_(0x5A)
    nv.moe_route_permute(lg, x_d, k, ref.topk_ids, ref.topk_w, ref.counts, ref.offsets, ref.perm_token,
                         ref.inv_perm, ref.a1_q, ref.a1_sf, ref.workspace, x_global_scale=gsa)
    b = pipeline.MoeBuffers(s)
    nv.moe_route_permute(lg, x_d, k, b.topk_ids, b.topk_w, b.counts, b.offsets, b.perm_token, b.inv_perm,
                         None, None, b.workspace)
    nv.nvfp4_device_status()
    R = int(host(ref.offsets)[-1])
    for name in ("topk_ids", "counts", "offsets", "inv_perm"):
        assert torch.equal(getattr(b, name), getattr(ref, name)), name
    assert torch.equal(b.perm_token[:R], ref.perm_token[:R])       # rows past the groups are not written
    perm = host(ref.perm_token)[:R]
    real = perm >= 0
    n_sf = nv.sf_bytes(R, H)
    # the oracle's staging of the same rows
    o_q, o_sf = omoe.stage_activation(x, perm, gscale=float(host(gs)[0]) if two_level else None)
    assert np.array_equal(host(ref.a1_q)[:R][real], o_q[real])
    assert np.array_equal(host(ref.a1_sf)[:n_sf], onv.swizzle_sf_fast(o_sf))
    job = dict(x=x_d, inv_perm=b.inv_perm, counts=b.counts, offsets=b.offsets, a1_q=b.a1_q, a1_sf=b.a1_sf,
               x_global_scale=gsa)

    # a BF16 grouped GEMM to host the job (N % 256 == 0: CTA pairs; 64 tiles, so
    # the pair kernel runs it on its own warps)
    sizes, N, K = [512, 384, 256], 2048, 768
    rows_max, G = sum(sizes), len(sizes)
    a_q, a_sf = inputs.random_nvfp4_operand(63, 0, rows_max, K)
    bw = [inputs.random_nvfp4_operand(63, 1 + g, N, K) for g in range(G)]
    a_q_d, a_sf_d = dev(a_q), _swizzled(nv, a_sf)
    b_q_d, b_sf_d = dev(np.stack([q for q, _ in bw])), torch.stack([_swizzled(nv, sf) for _, sf in bw])
    offs = dev(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32))
    cnt = dev(np.array([500, 300, 256], np.int32))

    def gemm(side):
        out = torch.full((rows_max, N), 3.0, dtype=torch.bfloat16, device="cuda")
        nv.nvfp4_grouped_gemm(a_q_d, a_sf_d, rows_max, offs, cnt, G, N, K, b_q_d, b_sf_d, 1.0, nv.EPI_BF16,
                              out_bf16=out, side_stage=job if side else None)
        return out

    plain_out = gemm(False)
    runs = [("own call", lambda: nv.moe_stage_activation(job))]
    runs += [(f"side job, tiles {m}", (lambda m=m: _with_tiles(nv, m, lambda: gemm(True))))
             for m in (nv.GEMM_TILES_PAIR, nv.GEMM_TILES_SINGLE)]
    for what, run in runs:
        b.a1_q.fill_(0x5A)
        b.a1_sf.fill_(0xA5)
        out = run()
        nv.nvfp4_device_status()
        got_q = host(b.a1_q)[:R]
        assert np.array_equal(got_q[real], o_q[real]), what
        assert np.all(got_q[~real] == 0x5A), what                    # padding nibbles are not written
        assert torch.equal(b.a1_sf[:n_sf], ref.a1_sf[:n_sf]), what
        if out is not None:
            assert torch.equal(out, plain_out), what


def _with_tiles(nv, mode, fn):
    with _tiles(nv, mode):
        return fn()


def test_pipelined_forward_equals_plain(nv):
    """The serving pipeline over three batches on two buffer sets: batch i's
    staging runs inside batch i-1's L2 GEMM, batch i-1's combine inside batch
    i's L1 GEMM; the last batch's L2 and combine close it.  Every y equals the
    plain forward's bit for bit, and is within the oracle bound."""
    nv, pipeline = nv
    spec = inputs.moe_spec(T=600, H=1024, I=512, E=16, top_k=4, seed=62, zipf=True)
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    w = pipeline.MoeWeights(s)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    xs = [x_t.cuda(), x_t.flip(0).contiguous().cuda(), x_t.roll(11, 0).contiguous().cuda()]   # three batches
    lgs = [dev(logits), dev(np.ascontiguousarray(logits[::-1])), dev(np.ascontiguousarray(np.roll(logits, 11, 0)))]
    plain = [pipeline.moe_forward(xs[i], lgs[i], w, pipeline.MoeBuffers(s)).clone() for i in range(3)]
    bufs = [pipeline.MoeBuffers(s), pipeline.MoeBuffers(s)]
    ys = []
    for i in range(3):
        pipeline.moe_forward_deferred(xs[i], lgs[i], w, bufs[i & 1], prev=bufs[(i - 1) & 1] if i else None)
        if i:
            ys.append(bufs[(i - 1) & 1].y.clone())                  # batch i-1 is complete
    ys.append(pipeline.moe_finish_deferred(w, bufs[0]).clone())
    nv.nvfp4_device_status()
    for i in range(3):
        assert torch.equal(ys[i], plain[i]), i
    w1, w2 = inputs.moe_all_weights(spec)
    ref = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"])["y"]
    assert rel_frobenius(ys[0].float().cpu().numpy(), ref) <= 2e-2


def test_side_jobs_check_their_row_indices(nv):
    """A staging job whose rows_max is below the routed rows writes nothing past
    it and reports a device index error; so does a side combine whose row count
    is below an inv_perm entry (those slots add nothing).  The buffers behind
    both jobs are full size, so the checks, not the memory, are what is tested."""
    nv, pipeline = nv
    spec = inputs.moe_spec(T=300, H=512, I=256, E=8, top_k=2, seed=64, zipf=True)
    s = pipeline.MoeShape(T=300, H=512, I=256, E=8, top_k=2)
    x_d, lg = inputs.moe_x(spec)[0].cuda(), dev(inputs.moe_logits(spec))
    ref, b = pipeline.MoeBuffers(s), pipeline.MoeBuffers(s)
    nv.moe_route_permute(lg, x_d, 2, ref.topk_ids, ref.topk_w, ref.counts, ref.offsets, ref.perm_token,
                         ref.inv_perm, ref.a1_q, ref.a1_sf, ref.workspace)
    nv.moe_route_permute(lg, x_d, 2, b.topk_ids, b.topk_w, b.counts, b.offsets, b.perm_token, b.inv_perm,
                         None, None, b.workspace)
    nv.nvfp4_device_status()
    R = int(host(ref.offsets)[-1])
    assert R > 256
    b.a1_q.fill_(0x5A)
    nv.moe_stage_activation(dict(x=x_d, inv_perm=b.inv_perm, counts=b.counts, offsets=b.offsets, a1_q=b.a1_q,
                                 a1_sf=b.a1_sf, rows_max=256))
    with pytest.raises(nv.Nvfp4Error) as ei:
        nv.nvfp4_device_status()
    assert ei.value.status == 6                                    # NVFP4_ERR_DEVICE
    perm = host(ref.perm_token)[:R]
    real = perm >= 0
    got = host(b.a1_q)
    lo = real & (np.arange(R) < 256)
    assert np.array_equal(got[:R][lo], host(ref.a1_q)[:R][lo])    # rows below rows_max staged
    assert np.all(got[256:] == 0x5A)                               # nothing past it
    nv.nvfp4_device_status()                                       # the word was cleared

    # a side combine told rows_bf16 has fewer rows (a view of the full rows) than
    # some tokens' slots reach: inside the CTA-pair SwiGLU GEMM (64 tiles) and as
    # its own launch (single CTAs)
    rows = torch.randn((R, 512), device="cuda").to(torch.bfloat16)
    y_full = torch.empty((300, 512), dtype=torch.bfloat16, device="cuda")
    nv.moe_combine(rows, ref.inv_perm, ref.topk_w, y_full)
    a_q, a_sf = inputs.random_nvfp4_operand(65, 0, 2048, 256)
    bq, bsf = inputs.random_nvfp4_operand(65, 1, 2048, 256)
    a_q_d, a_sf_d, bq_d, bsf_d = dev(a_q), _swizzled(nv, a_sf), dev(bq), _swizzled(nv, bsf)
    inv = host(ref.inv_perm)
    n_rows = int(np.median(inv.max(axis=1)))
    ok = torch.from_numpy(inv.max(axis=1) < n_rows).cuda()
    assert ok.any() and not ok.all()
    for mode in (nv.GEMM_TILES_PAIR, nv.GEMM_TILES_SINGLE):
        y = torch.zeros_like(y_full)
        oq = torch.empty((2048, 512), dtype=torch.uint8, device="cuda")
        osf = torch.empty(nv.sf_bytes(2048, 1024), dtype=torch.uint8, device="cuda")
        with _tiles(nv, mode):
            nv.nvfp4_grouped_gemm(a_q_d, a_sf_d, 2048, None, None, 1, 2048, 256, bq_d, bsf_d, 1.0,
                                  nv.EPI_SWIGLU_NVFP4, out_q=oq, out_sf=osf,
                                  side_combine=(rows[:n_rows], ref.inv_perm, ref.topk_w, y))
        with pytest.raises(nv.Nvfp4Error) as ei:
            nv.nvfp4_device_status()
        assert ei.value.status == 6, mode
        assert torch.equal(y[ok], y_full[ok]), mode
