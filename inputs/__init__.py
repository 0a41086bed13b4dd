"""Seeded synthetic inputs for the NVFP4 MoE expert FFN.

This module is shared by the tests, ``bench.py`` and ``__graft_entry__``: it
feeds the same bytes to the CUDA library and to the CPU oracle.  It holds none
of the method's arithmetic -- no quantisation, routing, GEMM or SwiGLU -- only
random draws, dtype conversion (fp32 -> BF16 via PyTorch) and the placement of
planted edge-case values.

Every tensor is drawn from its own numpy PCG64 stream keyed by
(seed, stream id, index), so a single expert's weights can be regenerated on
its own (the oracle re-draws only the experts a sampled token touches).

Workloads (the five seeded configurations of the path):

=========  ==================================================================
tiny       T=128 tokens, H=512, I=256, E=8 experts, top-2, seed 0
quantizer  standalone SwiGLU + NVFP4 quantiser, BF16 gate/up (32768, 2x2048),
           Student-t(3) x 0.5; 1% of 16-blocks x1e-3, 1% x3000, 1% planted
           exact midpoint blocks; seed 1
dense      single-expert L1: A 8192 x 7168 N(0,1), B 4096 x 7168 N(0,0.02); seed 2
decode     T=256, H=7168, I=2048, E=256, top-8, logits N(0,1); seed 3
prefill    T=16384, rest as decode, logits N(0,1) + 1.5 ln(Zipf(1.2) rank
           weight) with rank = expert index + 1; seed 4
=========  ==================================================================

Activations are N(0,1) rounded to BF16, weights N(0,0.02) fp32 (the weights
are quantised to NVFP4 by each side's own quantiser), router logits fp32.
Expert weights come from one seeded pool (``moe_weight_pool``).
"""
from __future__ import annotations

import numpy as np

try:                                    # torch is only needed for BF16 tensors
    import torch
except ImportError:                     # pragma: no cover
    torch = None

# stream ids
_LOGITS, _X, _W1, _W2, _PLANT, _GU, _DENSE_A, _DENSE_B, _RAND_OP, _SHARED = range(10)

CONFIGS = {
    "tiny": dict(kind="moe", T=128, H=512, I=256, E=8, top_k=2, seed=0, zipf=False),
    "quantizer": dict(kind="quant", rows=32768, cols=2048, seed=1),
    "dense": dict(kind="dense", M=8192, N=4096, K=7168, seed=2),
    # the prefill batch's L2 GEMM as one dense group: 16384 rows x H=7168 x I=2048, BF16 out
    "dense_l2": dict(kind="dense", M=16384, N=7168, K=2048, seed=5, epilogue="bf16"),
    "decode": dict(kind="moe", T=256, H=7168, I=2048, E=256, top_k=8, seed=3, zipf=False),
    "prefill": dict(kind="moe", T=16384, H=7168, I=2048, E=256, top_k=8, seed=4, zipf=True),
}

# scaled magnitudes that sit exactly on a rounding tie of the two-stage E2M1
# rule: half-step ties (x.25 / x.75) and E2M1-grid ties (2.5, 3.5, 5.0)
MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.25, 2.75, 3.25, 3.75, 4.25, 4.75, 5.25, 5.75,
             2.5, 3.5, 5.0)


def moe_spec(T, H, I, E, top_k, seed, zipf=False) -> dict:
    """A custom MoE workload (used for small parity cases with ragged shapes)."""
    return dict(kind="moe", T=T, H=H, I=I, E=E, top_k=top_k, seed=seed, zipf=zipf)


def _rng(seed: int, stream: int, index: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, index])))


def to_bf16(a: np.ndarray):
    """fp32 numpy -> (torch BF16 tensor, fp32 numpy of the BF16 values)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t, t.float().numpy()


# ------------------------------------------------------------------- MoE --
def moe_logits(spec: dict) -> np.ndarray:
    T, E = spec["T"], spec["E"]
    z = _rng(spec["seed"], _LOGITS).standard_normal((T, E))
    if spec.get("zipf"):
        r = np.arange(1, E + 1, dtype=np.float64)
        wr = r ** -1.2
        wr /= wr.sum()
        z = z + 1.5 * np.log(wr)[None, :]
    return z.astype(np.float32)


def moe_x(spec: dict):
    """Activations: (torch BF16 [T,H], fp32 numpy of the same values)."""
    a = _rng(spec["seed"], _X).standard_normal((spec["T"], spec["H"]), dtype=np.float32)
    return to_bf16(a)


POOL_MAX = 1 << 26          # values in the shared weight pool of the large workloads


def moe_weight_pool(spec: dict):
    """Expert weights are windows of one seeded N(0,1) fp32 pool.

    Returns (pool, w1_off [E], w2_off [E]); expert e's W1 is
    pool[w1_off[e] : w1_off[e] + 2I*H] * 0.02 viewed as [2I, H], W2 likewise
    [H, I].  When all experts fit in POOL_MAX values the windows are disjoint
    (every weight an independent draw); above that (the 256-expert workloads,
    11.3 G weights) the windows sit at seeded offsets in a 2^26-value pool and
    overlap, which keeps each window N(0, 0.02) while making the draw cheap.
    The pool carries one window's worth of wrap-around so every window is a
    contiguous slice.
    """
    key = (spec["seed"], spec["E"], spec["H"], spec["I"])
    hit = _POOL_CACHE.get(key)
    if hit is not None:
        return hit
    E, H, I = spec["E"], spec["H"], spec["I"]
    n1, n2 = 2 * I * H, H * I
    total = E * (n1 + n2)
    if total <= POOL_MAX:
        pool = _rng(spec["seed"], _W1).standard_normal(total, dtype=np.float32)
        w1_off = np.arange(E, dtype=np.int64) * n1
        w2_off = E * n1 + np.arange(E, dtype=np.int64) * n2
    else:
        base = _rng(spec["seed"], _W1).standard_normal(POOL_MAX, dtype=np.float32)
        pool = np.concatenate([base, base[:max(n1, n2)]])
        orng = _rng(spec["seed"], _W2)
        w1_off = orng.integers(0, POOL_MAX, size=E, dtype=np.int64)
        w2_off = orng.integers(0, POOL_MAX, size=E, dtype=np.int64)
    _POOL_CACHE.clear()
    _POOL_CACHE[key] = (pool, w1_off, w2_off)
    return _POOL_CACHE[key]


_POOL_CACHE: dict = {}
WEIGHT_STD = np.float32(0.02)


def moe_w1(spec: dict, e: int) -> np.ndarray:
    """fp32 [2I, H] for expert e; rows are already interleaved 8|8 (rows 16g..16g+7
    are gate rows 8g..8g+7, rows 16g+8..16g+15 the matching up rows)."""
    pool, w1_off, _ = moe_weight_pool(spec)
    n = 2 * spec["I"] * spec["H"]
    return (pool[w1_off[e]:w1_off[e] + n] * WEIGHT_STD).reshape(2 * spec["I"], spec["H"])


def moe_w2(spec: dict, e: int) -> np.ndarray:
    """fp32 [H, I] for expert e."""
    pool, _, w2_off = moe_weight_pool(spec)
    n = spec["H"] * spec["I"]
    return (pool[w2_off[e]:w2_off[e] + n] * WEIGHT_STD).reshape(spec["H"], spec["I"])


def moe_w1_rows(spec: dict, e: int, rows) -> np.ndarray:
    """fp32 [len(rows), H]: the given rows of expert e's W1 (``moe_w1(spec, e)[rows]``
    without materialising the whole matrix)."""
    pool, w1_off, _ = moe_weight_pool(spec)
    H = spec["H"]
    idx = w1_off[e] + np.asarray(rows, dtype=np.int64)[:, None] * H + np.arange(H)[None, :]
    return pool[idx] * WEIGHT_STD


def moe_w2_rows(spec: dict, e: int, rows) -> np.ndarray:
    """fp32 [len(rows), I]: the given rows of expert e's W2 (``moe_w2(spec, e)[rows]``)."""
    pool, _, w2_off = moe_weight_pool(spec)
    I = spec["I"]
    idx = w2_off[e] + np.asarray(rows, dtype=np.int64)[:, None] * I + np.arange(I)[None, :]
    return pool[idx] * WEIGHT_STD


def moe_shared_weights(spec: dict, i_shared: int | None = None):
    """A shared expert's fp32 weights (W1 [2*Is, H] interleaved 8|8 like the routed
    experts, W2 [H, Is]), N(0, 0.02) on their own stream; Is defaults to I."""
    i_s = spec["I"] if i_shared is None else i_shared
    rng = _rng(spec["seed"], _SHARED)
    w1 = rng.standard_normal((2 * i_s, spec["H"]), dtype=np.float32) * WEIGHT_STD
    w2 = rng.standard_normal((spec["H"], i_s), dtype=np.float32) * WEIGHT_STD
    return w1, w2


def moe_all_weights(spec: dict):
    """(w1 [E,2I,H], w2 [E,H,I]) fp32 -- only for small workloads."""
    w1 = np.stack([moe_w1(spec, e) for e in range(spec["E"])])
    w2 = np.stack([moe_w2(spec, e) for e in range(spec["E"])])
    return w1, w2


# ------------------------------------------------------------- quantiser --
def quantizer_input(spec: dict, rows: int | None = None, cols: int | None = None):
    """BF16 gate/up pairs interleaved 8|8, shape [rows, 2*cols], as a torch BF16
    tensor plus a dict of the planted 16-blocks.  Output block b of a row reads
    interleaved columns [32b, 32b+32): g0(8) u0(8) g1(8) u1(8)."""
    rows = spec["rows"] if rows is None else rows
    cols = spec["cols"] if cols is None else cols
    seed = spec["seed"]
    gu = (_rng(seed, _GU).standard_t(3, size=(rows, 2 * cols)) * 0.5).astype(np.float32)
    nblk = rows * (cols // 16)
    prng = _rng(seed, _PLANT)
    perm = prng.permutation(nblk)
    n1 = max(1, nblk // 100)
    tiny_blk, sat_blk, mid_blk = perm[:n1], perm[n1:2 * n1], perm[2 * n1:3 * n1]
    v = gu.reshape(rows, cols // 16, 2, 2, 8)          # [row, block, half, g/u, 8]
    for blks, factor in ((tiny_blk, 1e-3), (sat_blk, 3000.0)):
        r, b = np.divmod(blks, cols // 16)
        v[r, b, :, 1, :] *= np.float32(factor)
    # planted blocks: g = 64 makes silu(g) == 64 exactly in fp32 on both sides,
    # one u at 6 * 2^(q-6) fixes the block scale at 2^q, the other fifteen sit on
    # rounding ties m * 2^q with m in MIDPOINTS.
    r, b = np.divmod(mid_blk, cols // 16)
    q = prng.integers(-9, 9, size=len(mid_blk))
    m = np.asarray(MIDPOINTS)[prng.integers(0, len(MIDPOINTS), size=(len(mid_blk), 16))]
    sgn = np.where(prng.random((len(mid_blk), 16)) < 0.5, -1.0, 1.0)
    pos_max = prng.integers(0, 16, size=len(mid_blk))
    m[np.arange(len(mid_blk)), pos_max] = 6.0
    u = (sgn * m * np.exp2(q - 6.0)[:, None]).astype(np.float32).reshape(-1, 2, 8)
    v[r, b, :, 0, :] = np.float32(64.0)
    v[r, b, :, 1, :] = u
    t, _ = to_bf16(gu)
    return t, dict(tiny=tiny_blk, saturate=sat_blk, midpoint=mid_blk)


def plain_input_with_ties(seed: int, rows: int, cols: int, dtype: str = "f32"):
    """Plain-mode quantiser input: N(0,1) values with 5% of the 16-blocks replaced
    by exact rounding ties (one element 6 * 2^q, the rest m * 2^q), 2% scaled into
    the E4M3 subnormal / zero scale range and 2% into saturation.  Returns fp32
    numpy (and, for dtype 'bf16', values already rounded to BF16)."""
    rng = _rng(seed, _PLANT, 7)
    a = rng.standard_normal((rows, cols)).astype(np.float32)
    v = a.reshape(rows * (cols // 16), 16)
    nb = v.shape[0]
    perm = rng.permutation(nb)
    n_tie, n_small = max(1, nb // 20), max(1, nb // 50)
    tie, small, big = perm[:n_tie], perm[n_tie:n_tie + n_small], perm[n_tie + n_small:n_tie + 2 * n_small]
    q = rng.integers(-9, 9, size=len(tie))
    m = np.asarray(MIDPOINTS)[rng.integers(0, len(MIDPOINTS), size=(len(tie), 16))]
    m[np.arange(len(tie)), rng.integers(0, 16, size=len(tie))] = 6.0
    sgn = np.where(rng.random((len(tie), 16)) < 0.5, -1.0, 1.0)
    v[tie] = (sgn * m * np.exp2(q)[:, None]).astype(np.float32)
    v[small] *= np.float32(10.0) ** rng.uniform(-5, -2, size=(len(small), 1)).astype(np.float32)
    v[big] *= np.float32(10.0) ** rng.uniform(2.5, 4.5, size=(len(big), 1)).astype(np.float32)
    if dtype == "bf16":
        _, a = to_bf16(a)
    return a


# ----------------------------------------------------------------- dense --
def dense_inputs(spec: dict):
    """(A fp32 [M,K] N(0,1), B fp32 [N,K] N(0,0.02)); B's rows interleaved 8|8."""
    a = _rng(spec["seed"], _DENSE_A).standard_normal((spec["M"], spec["K"]), dtype=np.float32)
    b = (_rng(spec["seed"], _DENSE_B).standard_normal((spec["N"], spec["K"]), dtype=np.float32)
         * np.float32(0.02))
    return a, b


# ------------------------------------------------ raw NVFP4 GEMM operands --
def random_nvfp4_operand(seed: int, index: int, rows: int, k: int,
                         sf_lo: int = 0x30, sf_hi: int = 0x44):
    """Random packed NVFP4 bytes [rows, k/2] and random row-major E4M3 scale codes
    [rows, k/16] drawn uniformly from [sf_lo, sf_hi] (non-uniform scales are
    what exposes a wrong SF layout)."""
    rng = _rng(seed, _RAND_OP, index)
    q = rng.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)
    sf = rng.integers(sf_lo, sf_hi + 1, size=(rows, k // 16), dtype=np.uint8)
    return q, sf
