"""MoE expert-FFN oracle: routing, padded permutation, block-scaled GEMMs,
fused SwiGLU + NVFP4 re-quantisation, and the routing-weighted combine.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pipeline follows the "NVFP4 MegaMoE Debug Log", section "NVFP4 MoE
Pipeline": stage the activation to NVFP4, L1 GEMM into interleaved gate/up
columns, SiLU(gate) * up, re-stage to NVFP4, L2 GEMM, scatter with routing
weights.  The padded per-expert grouping is the "padded_dst" / "padded
activated fp4" layout of "NVFP4-1.1 Approach, Part 2".

Readings where the pages are silent:
* routing: the k largest logits, ties to the lower expert index, slots in
  descending-logit order; weights = softmax over the k selected logits;
* grouping: rows of expert e in ascending token order, each group padded to a
  multiple of 128 rows (the SF atom's M extent and the MMA's M); padding rows
  hold zero nibbles and zero scales and are marked -1 in ``perm_token``;
* GEMMs accumulate exactly (float64 on dequantised operands) and apply the fp32
  ``alpha`` scalar (global scale 1 by default);
* two-level scale (optional): per-tensor encode scales g (``nvfp4.global_scale``)
  for x and for each expert's W1 and W2, and a given encode scale for the L1
  output; each GEMM then applies fp32(alpha / fp32(g_A * g_B[e])) to the
  product of the one-level dequantised operands ("alpha = igs * global_sf");
* the L1 output is quantised from fp32 h (never from a BF16-rounded h);
* L2 rows and the combined output are BF16 (round-to-nearest-even); the
  combine sums the k slots in slot order.
* shared expert (optional): a dense FFN of every token through the same NVFP4
  steps (stage x per 16, L1 + SwiGLU + re-quantisation, L2 -> BF16 rows S); its
  row is added after the k routed slots, before the one rounding:
  y = bf16(sum_j w_j * O_j + S).  The pages' checkpoint notes list a shared
  expert beside the routed ones and print nothing about its combination.
"""
from __future__ import annotations

import numpy as np

from . import nvfp4

ROW_ALIGN = 128


# ------------------------------------------------------------ BF16 rounding --
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest BF16 value (8 significant bits, ties
    to even), returned as float64.  Values stay in BF16's normal range here."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0) / 256.0            # 8 significant bits, half-even
    return np.ldexp(r, e)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 BF16 encodings of values that are already BF16-representable."""
    f = np.asarray(x, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(b: np.ndarray) -> np.ndarray:
    """float32 values of uint16 BF16 encodings."""
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ routing --
def route_topk(logits: np.ndarray, k: int) -> tuple:
    """(ids int32 [T,k], w float64 [T,k]): top-k experts and softmax over them."""
    logits = np.asarray(logits, dtype=np.float32)
    t_count, e_count = logits.shape
    if not 0 < k <= e_count:
        raise ValueError("need 0 < k <= E")
    # a stable sort of -logit keeps equal logits in ascending expert order
    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    z = np.exp(sel - sel[:, :1])
    w = z / z.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w


def permute(ids: np.ndarray, n_experts: int, align: int = ROW_ALIGN) -> dict:
    """Group the (token, slot) pairs by expert, each group padded to ``align`` rows.

    Returns counts [E], offsets [E+1] (padded, exclusive), perm_token [R_pad]
    (token of each row, -1 on padding) and inv_perm [T,k] (row of each pair).
    """
    ids = np.asarray(ids, dtype=np.int64)
    t_count, k = ids.shape
    counts = np.zeros(n_experts, dtype=np.int64)
    for e in ids.ravel():
        counts[e] += 1
    padded = -(-counts // align) * align
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    perm_token = np.full(int(offsets[-1]), -1, dtype=np.int64)
    inv_perm = np.zeros((t_count, k), dtype=np.int64)
    fill = offsets[:-1].copy()
    for t in range(t_count):
        for j in range(k):
            e = ids[t, j]
            r = fill[e]
            fill[e] += 1
            perm_token[r] = t
            inv_perm[t, j] = r
    return dict(counts=counts.astype(np.int32), offsets=offsets.astype(np.int32),
                perm_token=perm_token.astype(np.int32), inv_perm=inv_perm.astype(np.int32))


def stage_activation(x: np.ndarray, perm_token: np.ndarray, gscale=None) -> tuple:
    """Quantise x (fp32 view of the BF16 activations, [T,H]) into the permuted,
    padded rows: (a1_q [R_pad, H/2], a1_sf row-major [R_pad, H/16]).  Padding
    rows are zero.  ``gscale``: the two-level encode scale of x, if any."""
    x = np.asarray(x, dtype=np.float32)
    xq, xsf = nvfp4.quantize_rows(x, gscale)
    r_pad = len(perm_token)
    a_q = np.zeros((r_pad, xq.shape[1]), dtype=np.uint8)
    a_sf = np.zeros((r_pad, xsf.shape[1]), dtype=np.uint8)
    real = perm_token >= 0
    a_q[real] = xq[perm_token[real]]
    a_sf[real] = xsf[perm_token[real]]
    return a_q, a_sf


# -------------------------------------------------------------------- GEMMs --
def expert_of_rows(offsets: np.ndarray) -> np.ndarray:
    """Expert index of every padded row."""
    offsets = np.asarray(offsets, dtype=np.int64)
    return np.repeat(np.arange(len(offsets) - 1), np.diff(offsets))


def two_level_alpha(alpha: float, ga, gb) -> np.float32:
    """fp32(alpha / fp32(ga * gb)): a GEMM's alpha under encode scales ga, gb."""
    return np.float32(np.float32(alpha) / np.float32(np.float32(ga) * np.float32(gb)))


def grouped_gemm(a_deq: np.ndarray, offsets: np.ndarray, b_deq: np.ndarray,
                 alpha: float = 1.0, a_gscale=None, b_gscale=None) -> np.ndarray:
    """out[r, n] = alpha_e * sum_k a[r, k] * b_e[n, k] for the expert e owning row r
    (float64; ``b_deq`` is [E, N, K]), the operands dequantised at one level.
    alpha_e = alpha, or two_level_alpha(alpha, a_gscale, b_gscale[e]) when either
    encode scale is given."""
    offsets = np.asarray(offsets, dtype=np.int64)
    out = np.zeros((a_deq.shape[0], b_deq.shape[1]), dtype=np.float64)
    for e in range(len(offsets) - 1):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            if a_gscale is None and b_gscale is None:
                alpha_e = np.float32(alpha)
            else:
                alpha_e = two_level_alpha(alpha, 1.0 if a_gscale is None else a_gscale,
                                          1.0 if b_gscale is None else b_gscale[e])
            out[lo:hi] = np.float64(alpha_e) * (a_deq[lo:hi] @ b_deq[e].T)
    return out


def l1_swiglu_requant(g_full: np.ndarray, out_gscale=None) -> tuple:
    """Fused L1 epilogue on the interleaved gate/up accumulator rows
    (float64 [rows, 2I]): h = silu(g) * u -> fp32, then NVFP4 per 16 (of
    fp32(h * out_gscale) under a two-level encode scale).
    Returns (a2_q [rows, I/2], a2_sf row-major [rows, I/16], h fp32 [rows, I])."""
    g, u = nvfp4.deinterleave_gu8(g_full)
    h = nvfp4.swiglu_h(g, u)
    q, sf = nvfp4.quantize_rows(h, out_gscale)
    return q, sf, h


def l1_swiglu_bf16(g_full: np.ndarray) -> np.ndarray:
    """The compact BF16 L1 output (the pages' "compact SwiGLU output" plan): h =
    silu(g) * u from the interleaved accumulator rows, fp32, then rounded to BF16
    [rows, I] (no re-quantisation)."""
    g, u = nvfp4.deinterleave_gu8(g_full)
    return round_to_bf16(nvfp4.swiglu_h(g, u))


def combine(rows_bf16: np.ndarray, inv_perm: np.ndarray, w: np.ndarray,
            shared_bf16: np.ndarray | None = None) -> np.ndarray:
    """y[t] = sum_j w[t,j] * rows[inv_perm[t,j]] (+ shared[t]) (float64, slot order,
    the shared row last) -> BF16 values."""
    rows = np.asarray(rows_bf16, dtype=np.float64)
    t_count, k = inv_perm.shape
    acc = np.zeros((t_count, rows.shape[1]), dtype=np.float64)
    for j in range(k):
        acc += np.asarray(w[:, j], dtype=np.float64)[:, None] * rows[inv_perm[:, j]]
    if shared_bf16 is not None:
        acc += np.asarray(shared_bf16, dtype=np.float64)
    return round_to_bf16(acc)


def shared_expert_rows(x: np.ndarray, w1s: np.ndarray, w2s: np.ndarray,
                       alpha1: float = 1.0, alpha2: float = 1.0) -> dict:
    """The shared expert on every token row of x (fp32 [T,H]): NVFP4 staging of x,
    L1 + SwiGLU + re-quantisation, L2 -> BF16 rows S [T,H].  The same steps as one
    routed expert holding all T rows."""
    xq, xsf = nvfp4.quantize_rows(np.asarray(x, dtype=np.float32))
    w1q, w1sf = nvfp4.quantize_rows(w1s)
    w2q, w2sf = nvfp4.quantize_rows(w2s)
    g_full = np.float64(np.float32(alpha1)) * (nvfp4.dequantize_rows(xq, xsf) @ nvfp4.dequantize_rows(w1q, w1sf).T)
    a2q, a2sf, h = l1_swiglu_requant(g_full)
    o = np.float64(np.float32(alpha2)) * (nvfp4.dequantize_rows(a2q, a2sf) @ nvfp4.dequantize_rows(w2q, w2sf).T)
    return dict(x_q=xq, x_sf=xsf, w1_q=w1q, w1_sf=w1sf, w2_q=w2q, w2_sf=w2sf, h=h, a2_q=a2q, a2_sf=a2sf,
                rows=round_to_bf16(o))


# ---------------------------------------------------------- whole FFN path --
def dequant_weights(w_q: np.ndarray, w_sf_rows: np.ndarray) -> np.ndarray:
    """[E, N, K/2] nibbles + [E, N, K/16] row-major SF -> float64 [E, N, K]."""
    e_count = w_q.shape[0]
    return np.stack([nvfp4.dequantize_rows(w_q[e], w_sf_rows[e]) for e in range(e_count)])


def quantize_weights(w: np.ndarray, gscales=None) -> tuple:
    """fp32 [E, N, K] -> ([E, N, K/2] nibbles, [E, N, K/16] row-major SF), each
    expert under its own encode scale gscales[e] if given."""
    qs, sfs = zip(*(nvfp4.quantize_rows(w[e], None if gscales is None else gscales[e])
                    for e in range(w.shape[0])))
    return np.stack(qs), np.stack(sfs)


def two_level_scales(x: np.ndarray, w1: np.ndarray, w2: np.ndarray) -> dict:
    """Encode scales of the two-level scheme: x's and every expert's W1 and W2."""
    return dict(x=nvfp4.global_scale(x),
                w1=np.array([nvfp4.global_scale(w1[e]) for e in range(w1.shape[0])], dtype=np.float32),
                w2=np.array([nvfp4.global_scale(w2[e]) for e in range(w2.shape[0])], dtype=np.float32))


def moe_ffn(x: np.ndarray, logits: np.ndarray, w1: np.ndarray, w2: np.ndarray, top_k: int,
            alpha1: float = 1.0, alpha2: float = 1.0, a2_gscale=None, shared=None) -> dict:
    """The whole path on CPU.  x: fp32 values of the BF16 activations [T,H];
    logits fp32 [T,E]; w1 fp32 [E, 2I, H] (rows interleaved 8|8); w2 fp32 [E, H, I].
    With ``a2_gscale`` (the L1 output's encode scale, given as a calibrated
    constant) the path runs the two-level scheme: x, W1 and W2 get their own
    encode scales (two_level_scales) and every GEMM's alpha follows.
    ``shared``: None or (w1s, w2s), a shared expert added to every token's output.
    Returns every intermediate (all computed here, none supplied from outside)."""
    e_count = w1.shape[0]
    ids, w = route_topk(logits, top_k)
    p = permute(ids, e_count)
    gs = two_level_scales(x, w1, w2) if a2_gscale is not None else dict(x=None, w1=None, w2=None)
    a1_q, a1_sf = stage_activation(x, p["perm_token"], gs["x"])
    w1_q, w1_sf = quantize_weights(w1, gs["w1"])
    w2_q, w2_sf = quantize_weights(w2, gs["w2"])
    g_full = grouped_gemm(nvfp4.dequantize_rows(a1_q, a1_sf), p["offsets"],
                          dequant_weights(w1_q, w1_sf), alpha1, gs["x"], gs["w1"])
    a2_q, a2_sf, h = l1_swiglu_requant(g_full, a2_gscale)
    o = grouped_gemm(nvfp4.dequantize_rows(a2_q, a2_sf), p["offsets"],
                     dequant_weights(w2_q, w2_sf), alpha2, a2_gscale, gs["w2"])
    rows = round_to_bf16(o)
    sh = None if shared is None else shared_expert_rows(x, shared[0], shared[1], alpha1, alpha2)
    y = combine(rows, p["inv_perm"], w, None if sh is None else sh["rows"])
    return dict(ids=ids, w=w, a1_q=a1_q, a1_sf=a1_sf, w1_q=w1_q, w1_sf=w1_sf, w2_q=w2_q,
                w2_sf=w2_sf, g_full=g_full, h=h, a2_q=a2_q, a2_sf=a2_sf, rows=rows, y=y, gscales=gs,
                shared=sh, **p)


def moe_ffn_tokens(x_rows: np.ndarray, logits_rows: np.ndarray, w1_of, w2_of, top_k: int,
                   alpha1: float = 1.0, alpha2: float = 1.0, cache: dict | None = None,
                   two_level: dict | None = None, shared=None) -> dict:
    """The same path for a few sampled tokens, one at a time (every step is
    row-independent: a token's output depends only on its own row, its routing
    and its experts' weights).  ``w1_of(e)`` / ``w2_of(e)`` return expert e's fp32
    weights; their quantised, dequantised forms are cached in ``cache``.
    Returns ids, w, a2 rows (q, row-major sf) per (token, slot), and y (BF16 values).
    ``two_level``: dict(x=g_x of the whole batch, a2=the L1 output's encode scale);
    each expert's weight encode scales are computed from its weights.
    ``shared``: None or (w1s, w2s), a shared expert added to every token's output."""
    cache = {} if cache is None else cache

    def deq(kind, e, fn):
        key = (kind, e, two_level is not None)
        if key not in cache:
            wt = fn(e)
            g = nvfp4.global_scale(wt) if two_level is not None else None
            q, sf = nvfp4.quantize_rows(wt, g)
            cache[key] = (nvfp4.dequantize_rows(q, sf), np.float32(1.0) if g is None else g)
        return cache[key]

    def alpha_of(alpha, ga, gb):
        return np.float32(alpha) if two_level is None else two_level_alpha(alpha, ga, gb)

    gx = None if two_level is None else two_level["x"]
    ga2 = None if two_level is None else two_level["a2"]
    ids, w = route_topk(logits_rows, top_k)
    xq, xsf = nvfp4.quantize_rows(np.asarray(x_rows, dtype=np.float32), gx)
    a1 = nvfp4.dequantize_rows(xq, xsf)
    n_tok = len(x_rows)
    y, a2_q, a2_sf, h_all = [], [], [], []
    for t in range(n_tok):
        acc = None
        for j in range(top_k):
            e = int(ids[t, j])
            w1d, g1 = deq("w1", e, w1_of)
            w2d, g2 = deq("w2", e, w2_of)
            g_full = np.float64(alpha_of(alpha1, gx, g1)) * (a1[t:t + 1] @ w1d.T)
            q, sf, h = l1_swiglu_requant(g_full, ga2)
            o = np.float64(alpha_of(alpha2, ga2, g2)) * (nvfp4.dequantize_rows(q, sf) @ w2d.T)
            row = round_to_bf16(o)[0]
            acc = w[t, j] * row if acc is None else acc + w[t, j] * row
            a2_q.append(q[0])
            a2_sf.append(sf[0])
            h_all.append(h[0])
        if shared is not None:
            acc = acc + shared_expert_rows(x_rows[t:t + 1], shared[0], shared[1], alpha1, alpha2)["rows"][0]
        y.append(round_to_bf16(acc))
    return dict(ids=ids, w=w, a2_q=np.array(a2_q).reshape(n_tok, top_k, -1),
                a2_sf=np.array(a2_sf).reshape(n_tok, top_k, -1), h=np.array(h_all).reshape(n_tok, top_k, -1),
                y=np.array(y))
