"""GPU parity of the gathering L1 (x quantised once in token order; the L1 GEMM
loads its A rows through perm_token with TMA tile::gather4, so the permuted
copy of the activations is never written).

* the token-order rows are bit-exact against the oracle's quantisation of x,
  and the permuted scales equal those of the materialising call;
* a grouped GEMM on gathered rows gives the same bytes as on the materialised
  permuted rows, on both tile kernels, with padding entries (-1) in the index
  (gathering is the L1 GEMM's, so its SwiGLU + NVFP4 epilogue; any other
  epilogue with an index is refused as unsupported), and its codes are within
  the re-quantisation bound of the oracle's float64 GEMM on the rows the index
  selects;
* an index past the end sets the device error word and copies nothing from
  outside the matrix;
* whole forwards with and without gathering give the same bytes (small and
  the full-size prefill batch), and a gathered forward matches the fully
  CPU-quantised oracle (routing bit-exact, re-quantised codes within the bound,
  y within relative Frobenius 2e-2).
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
    from nvfp4_block_scaled_moe_gb300 import pipeline
    return nv, pipeline


@contextlib.contextmanager
def _tiles(nv, mode):
    nv.nvfp4_set_gemm_tiles(mode)
    try:
        yield
    finally:
        nv.nvfp4_set_gemm_tiles(nv.GEMM_TILES_AUTO)


def test_route_token_order_rows(nv):
    nv, pipeline = nv
    spec = inputs.moe_spec(T=300, H=512, I=256, E=8, top_k=2, seed=95, zipf=True)
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    x_t, x = inputs.moe_x(spec)
    logits = dev(inputs.moe_logits(spec))
    mat, gat = pipeline.MoeBuffers(s), pipeline.MoeBuffers(s, gather=True)
    gat.a1_sf.copy_(torch.zeros_like(gat.a1_sf))
    mat.a1_sf.copy_(torch.zeros_like(mat.a1_sf))
    for b in (mat, gat):
        nv.moe_route_permute(logits, x_t.cuda(), s.top_k, b.topk_ids, b.topk_w, b.counts, b.offsets, b.perm_token,
                             b.inv_perm, b.a1_q, b.a1_sf, b.workspace, x_q=b.x_q)
    nv.nvfp4_device_status()
    oq, _ = onv.quantize_rows(x)
    assert np.array_equal(host(gat.x_q), oq)
    R = int(host(mat.offsets)[-1])        # perm_token past the last group is not written
    assert torch.equal(mat.a1_sf, gat.a1_sf) and torch.equal(mat.perm_token[:R], gat.perm_token[:R])
    perm = host(mat.perm_token)[:R]
    assert np.array_equal(host(mat.a1_q)[:R][perm >= 0], oq[perm[perm >= 0]])


def _gathered_case(seed, sizes, counts, K):
    """Token rows, a padded permutation index (-1 on padding) and the
    materialised permuted rows and scales it stands for."""
    rng = np.random.default_rng(seed)
    T = sum(counts) + 7
    x_q, x_sf = inputs.random_nvfp4_operand(seed, 0, T, K)
    index = np.full(sum(sizes), -1, np.int32)
    a_q = np.zeros((sum(sizes), K // 2), np.uint8)
    a_sf = np.zeros((sum(sizes), K // 16), np.uint8)
    r0 = 0
    for size, c in zip(sizes, counts):
        rows = rng.choice(T, size=c, replace=False)
        index[r0:r0 + c] = rows
        a_q[r0:r0 + c] = x_q[rows]
        a_sf[r0:r0 + c] = x_sf[rows]
        r0 += size
    return x_q, index, a_q, a_sf


def test_gathered_gemm_equals_materialised(nv):
    nv, _ = nv
    sizes, counts, N, K = [512, 128, 0, 384], [500, 128, 0, 300], 512, 768
    G, rows_max = len(sizes), sum(sizes)
    x_q, index, a_q, a_sf = _gathered_case(96, sizes, counts, K)
    b = [inputs.random_nvfp4_operand(96, 1 + g, N, K) for g in range(G)]

    def swz(sf_lin):
        r, k = sf_lin.shape
        out = torch.empty(nv.sf_bytes(r, 16 * k), dtype=torch.uint8, device="cuda")
        nv.nvfp4_sf_swizzle(dev(sf_lin), r, k, k, 1, out)
        return out

    a_sf_d, b_q_d = swz(a_sf), dev(np.stack([x[0] for x in b]))
    b_sf_d = torch.stack([swz(x[1]) for x in b])
    offs = dev(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32))
    cnt = dev(np.array(counts, np.int32))
    results = []
    for mode in (nv.GEMM_TILES_SINGLE, nv.GEMM_TILES_PAIR):
        for gathered in (False, True):
            out = torch.zeros((rows_max, N), dtype=torch.bfloat16, device="cuda")
            oq = torch.zeros((rows_max, N // 4), dtype=torch.uint8, device="cuda")
            osf = torch.zeros(nv.sf_bytes(rows_max, N // 2), dtype=torch.uint8, device="cuda")
            src = dict(a_gather=dev(index), a_gather_rows=x_q.shape[0]) if gathered else {}
            a_src = dev(x_q) if gathered else dev(a_q)
            with _tiles(nv, mode):
                if gathered:
                    with pytest.raises(nv.Nvfp4Error) as ei:
                        nv.nvfp4_grouped_gemm(a_src, a_sf_d, rows_max, offs, cnt, G, N, K, b_q_d, b_sf_d, 1.0,
                                              nv.EPI_BF16, out_bf16=out, **src)
                    assert ei.value.status == 2            # NVFP4_ERR_UNSUPPORTED
                else:
                    nv.nvfp4_grouped_gemm(a_src, a_sf_d, rows_max, offs, cnt, G, N, K, b_q_d, b_sf_d, 1.0,
                                          nv.EPI_BF16, out_bf16=out)
                nv.nvfp4_grouped_gemm(a_src, a_sf_d, rows_max, offs, cnt, G, N, K, b_q_d, b_sf_d, 1.0,
                                      nv.EPI_SWIGLU_NVFP4, out_q=oq, out_sf=osf, **src)
            nv.nvfp4_device_status()
            results.append((host(oq), host(osf)))
    for r in results[1:]:
        for a, b_ in zip(results[0], r):
            assert np.array_equal(a, b_)
    # the oracle: the rows the index selects (zero rows for -1), float64 GEMM, SwiGLU, requantisation
    offs_np = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    a_deq = onv.dequantize_rows(a_q, a_sf)
    b_deq = np.stack([onv.dequantize_rows(*x) for x in b])
    oq, osf, _ = omoe.l1_swiglu_requant(omoe.grouped_gemm(a_deq, offs_np, b_deq, 1.0))
    valid = np.concatenate([np.arange(offs_np[g], offs_np[g] + counts[g]) for g in range(G)])
    gq, gsf_sw = results[1]                                # gathered, single CTAs (equal to every other form)
    gsf = onv.unswizzle_sf(gsf_sw, rows_max, N // 32)
    res = compare_requantised(gq[valid], gsf[valid], oq[valid], osf[valid])
    assert res["ok"], res


def test_gathered_forward_matches_oracle(nv):
    nv, pipeline = nv
    spec = inputs.moe_spec(T=300, H=512, I=256, E=8, top_k=2, seed=99, zipf=True)
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    w = pipeline.MoeWeights(s)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    b = pipeline.MoeBuffers(s, gather=True)
    x_t, x = inputs.moe_x(spec)
    logits = inputs.moe_logits(spec)
    y = pipeline.moe_forward(x_t.cuda(), dev(logits), w, b)
    nv.nvfp4_device_status()
    w1, w2 = inputs.moe_all_weights(spec)
    o = omoe.moe_ffn(x, logits, w1, w2, spec["top_k"])
    assert np.array_equal(host(b.topk_ids), o["ids"]) and np.array_equal(host(b.offsets), o["offsets"])
    R = int(o["offsets"][-1])
    assert np.array_equal(host(b.perm_token)[:R], o["perm_token"])
    oq, _ = onv.quantize_rows(x)
    assert np.array_equal(host(b.x_q), oq)                 # the token-order rows the L1 gathers
    real = o["perm_token"] >= 0
    gsf = onv.unswizzle_sf(host(b.a2_sf), R, spec["I"] // 16)
    res = compare_requantised(host(b.a2_q)[:R][real], gsf[real], o["a2_q"][real], o["a2_sf"][real])
    assert res["ok"], res
    assert rel_frobenius(y.float().cpu().numpy(), o["y"]) <= 2e-2


def test_gather_index_past_the_end_is_flagged(nv):
    nv, _ = nv
    K, N = 256, 256
    x_q, x_sf = inputs.random_nvfp4_operand(97, 0, 64, K)
    b_q, b_sf = inputs.random_nvfp4_operand(97, 1, N, K)
    index = np.zeros(128, np.int32)
    index[5] = 64                                       # one past the last row
    sf = torch.empty(nv.sf_bytes(128, K), dtype=torch.uint8, device="cuda")
    nv.nvfp4_sf_swizzle(dev(np.zeros((128, K // 16), np.uint8)), 128, K // 16, K // 16, 1, sf)
    bsf = torch.empty(nv.sf_bytes(N, K), dtype=torch.uint8, device="cuda")
    nv.nvfp4_sf_swizzle(dev(b_sf), N, K // 16, K // 16, 1, bsf)
    oq = torch.empty((128, N // 4), dtype=torch.uint8, device="cuda")
    osf = torch.empty(nv.sf_bytes(128, N // 2), dtype=torch.uint8, device="cuda")
    nv.nvfp4_grouped_gemm(dev(x_q), sf, 128, None, None, 1, N, K, dev(b_q)[None], bsf[None], 1.0,
                          nv.EPI_SWIGLU_NVFP4, out_q=oq, out_sf=osf, a_gather=dev(index), a_gather_rows=64)
    with pytest.raises(nv.Nvfp4Error) as ei:
        nv.nvfp4_device_status()
    assert ei.value.status == 6                         # NVFP4_ERR_DEVICE
    nv.nvfp4_device_status()                            # the word was cleared; the context works


@pytest.mark.parametrize("name", ["small", "prefill"])
def test_forward_with_and_without_gathering(nv, name):
    nv, pipeline = nv
    spec = (inputs.moe_spec(T=300, H=512, I=256, E=8, top_k=2, seed=98, zipf=True) if name == "small"
            else dict(inputs.CONFIGS["prefill"]))
    s = pipeline.MoeShape(T=spec["T"], H=spec["H"], I=spec["I"], E=spec["E"], top_k=spec["top_k"])
    w = pipeline.MoeWeights(s)
    pool, o1, o2 = inputs.moe_weight_pool(spec)
    w.set_from_pool(torch.from_numpy(pool).cuda(), o1, o2, float(inputs.WEIGHT_STD))
    x_t, _ = inputs.moe_x(spec)
    x, logits = x_t.cuda(), dev(inputs.moe_logits(spec))
    ys, a2s = [], []
    for gather in (False, True):
        b = pipeline.MoeBuffers(s, gather=gather)
        ys.append(pipeline.moe_forward(x, logits, w, b).clone())
        R = int(host(b.offsets)[-1])
        real = host(b.perm_token)[:R] >= 0               # a2 is written for real rows only
        a2s.append(host(b.a2_q)[:R][real])
        nv.nvfp4_device_status()
        del b
    assert torch.equal(ys[0], ys[1])
    assert np.array_equal(a2s[0], a2s[1])
