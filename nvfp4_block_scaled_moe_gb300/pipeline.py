"""Device buffers and the three-call forward of the NVFP4 MoE expert FFN.

Plumbing only: PyTorch allocates device memory; every step is one call into
libnvfp4moe.so (route + permute + stage, L1/SwiGLU/requant/L2, combine), and
the serving-loop step (moe_forward_deferred) orders the same calls so that each
batch's staging runs inside the previous batch's L2 GEMM and each batch's
combine inside the next batch's L1 GEMM.

Two-level scale (optional): the pages' pipeline carries per-tensor global scales
("NVFP4 MoE Pipeline": stage_activation returns an input_global_scale; alpha =
igs * global_sf).  Here every tensor gets a device fp32 encode scale g (see
include/nvfp4moe.h): the weights one per expert, computed from their fp32 values
when they are quantised; x one per forward, computed on the device before the
routing call; the L1 output one calibrated ahead (``calibrate_a2_scale``), since
the fused epilogue quantises each tile before the tensor's amax exists.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (EPI_BF16, EPI_SWIGLU_NVFP4, MODE_PLAIN, moe_combine, moe_padded_rows_max, moe_route_permute,
               moe_route_permute_workspace, nvfp4_global_scale, nvfp4_grouped_gemm, nvfp4_moe_ffn_forward,
               nvfp4_quantize, sf_bytes)


@dataclass
class MoeShape:
    T: int
    H: int
    I: int
    E: int
    top_k: int

    @property
    def rows_max(self) -> int:
        return moe_padded_rows_max(self.T, self.E, self.top_k)


class MoeBuffers:
    """Every output and intermediate of one forward, sized for the worst case.
    gather: the routing call writes x's NVFP4 rows once in token order (x_q) and
    L1 gathers its A rows through perm_token, instead of a permuted copy a1_q."""

    def __init__(self, s: MoeShape, device="cuda", gather: bool = False):
        u8, i32, f32 = torch.uint8, torch.int32, torch.float32
        R = max(s.rows_max, 128)
        self.shape = s
        self.rows_max = R
        self.topk_ids = torch.empty((s.T, s.top_k), dtype=i32, device=device)
        self.topk_w = torch.empty((s.T, s.top_k), dtype=f32, device=device)
        self.counts = torch.empty(s.E, dtype=i32, device=device)
        self.offsets = torch.empty(s.E + 1, dtype=i32, device=device)
        self.perm_token = torch.empty(R, dtype=i32, device=device)
        self.inv_perm = torch.empty((s.T, s.top_k), dtype=i32, device=device)
        self.gather = gather
        self.a1_q = None if gather else torch.empty((R, s.H // 2), dtype=u8, device=device)
        self.x_q = torch.empty((max(s.T, 1), s.H // 2), dtype=u8, device=device) if gather else None
        self.a1_sf = torch.empty(sf_bytes(R, s.H), dtype=u8, device=device)
        self.a2_q = torch.empty((R, s.I // 2), dtype=u8, device=device)
        self.a2_sf = torch.empty(sf_bytes(R, s.I), dtype=u8, device=device)
        self.rows_out = torch.empty((R, s.H), dtype=torch.bfloat16, device=device)
        self.y = torch.empty((s.T, s.H), dtype=torch.bfloat16, device=device)
        self.workspace = torch.empty(moe_route_permute_workspace(s.T, s.H, s.E, s.top_k), dtype=u8, device=device)
        self.h_debug = None
        self.x_gs = torch.ones(1, dtype=f32, device=device)       # x's encode scale (two-level forwards)
        self.a2_gs = None                                         # L1 output's encode scale, once calibrated

    def enable_host_io(self):
        """Device x and logits for the host-buffer call (nvfp4_moe_forward_host), which
        copies the host inputs into them; y is the output row buffer above."""
        s = self.shape
        dev = self.y.device
        self.x = torch.empty((s.T, s.H), dtype=torch.bfloat16, device=dev)
        self.logits = torch.empty((s.T, s.E), dtype=torch.float32, device=dev)
        return self

    def enable_h_debug(self):
        # zeros: the GEMM writes h only for real rows
        self.h_debug = torch.zeros((self.rows_max, self.shape.I), dtype=torch.float32, device=self.a2_sf.device)


class MoeWeights:
    """Expert weights in NVFP4: W1 [E, 2I, H] (rows interleaved 8|8) and W2 [E, H, I],
    each expert's SF swizzled for its own N x K matrix."""

    def __init__(self, s: MoeShape, device="cuda", two_level: bool = False):
        u8 = torch.uint8
        self.shape = s
        self.w1_q = torch.empty((s.E, 2 * s.I, s.H // 2), dtype=u8, device=device)
        self.w1_sf = torch.empty((s.E, sf_bytes(2 * s.I, s.H)), dtype=u8, device=device)
        self.w2_q = torch.empty((s.E, s.H, s.I // 2), dtype=u8, device=device)
        self.w2_sf = torch.empty((s.E, sf_bytes(s.H, s.I)), dtype=u8, device=device)
        # per-expert encode scales of the two-level scheme (None: one level)
        self.w1_gs = torch.ones(s.E, dtype=torch.float32, device=device) if two_level else None
        self.w2_gs = torch.ones(s.E, dtype=torch.float32, device=device) if two_level else None

    def set_expert(self, e: int, w1_f32: torch.Tensor, w2_f32: torch.Tensor):
        """Quantise one expert's fp32 weights (CUDA tensors) with the library's quantiser
        (two-level: under encode scales computed from those weights on the device)."""
        s = self.shape
        g1 = g2 = None
        if self.w1_gs is not None:
            g1, g2 = self.w1_gs[e:e + 1], self.w2_gs[e:e + 1]
            nvfp4_global_scale(w1_f32, g1)
            nvfp4_global_scale(w2_f32, g2)
        nvfp4_quantize(w1_f32, s.H, MODE_PLAIN, self.w1_q[e], self.w1_sf[e], global_scale=g1)
        nvfp4_quantize(w2_f32, s.I, MODE_PLAIN, self.w2_q[e], self.w2_sf[e], global_scale=g2)

    def set_from_pool(self, pool: torch.Tensor, w1_off, w2_off, std: float):
        """Quantise every expert from windows of a device fp32 pool: expert e's W1 is
        pool[w1_off[e] : + 2I*H] * std viewed [2I, H], W2 likewise [H, I]."""
        s = self.shape
        n1, n2 = 2 * s.I * s.H, s.H * s.I
        scale = torch.tensor(std, dtype=torch.float32, device=pool.device)
        for e in range(s.E):
            o1, o2 = int(w1_off[e]), int(w2_off[e])
            w1 = (pool[o1:o1 + n1] * scale).view(2 * s.I, s.H)
            w2 = (pool[o2:o2 + n2] * scale).view(s.H, s.I)
            self.set_expert(e, w1, w2)


class SharedExpert:
    """A shared expert: one dense NVFP4 FFN (W1 [2*Is, H] interleaved 8|8, W2 [H, Is])
    applied to every token, with its buffers for T tokens (rows padded to 128)."""

    def __init__(self, s: MoeShape, i_shared: int, device="cuda"):
        u8 = torch.uint8
        self.shape, self.I = s, i_shared
        self.rows = max(128, -(-s.T // 128) * 128)
        self.w1_q = torch.empty((1, 2 * i_shared, s.H // 2), dtype=u8, device=device)
        self.w1_sf = torch.empty((1, sf_bytes(2 * i_shared, s.H)), dtype=u8, device=device)
        self.w2_q = torch.empty((1, s.H, i_shared // 2), dtype=u8, device=device)
        self.w2_sf = torch.empty((1, sf_bytes(s.H, i_shared)), dtype=u8, device=device)
        # rows past T stay zero (nibbles) / zero-scaled (SF): they compute to zero
        self.x_q = torch.zeros((self.rows, s.H // 2), dtype=u8, device=device)
        self.x_sf = torch.zeros(sf_bytes(self.rows, s.H), dtype=u8, device=device)
        self.a2_q = torch.empty((self.rows, i_shared // 2), dtype=u8, device=device)
        self.a2_sf = torch.empty(sf_bytes(self.rows, i_shared), dtype=u8, device=device)
        self.out = torch.empty((self.rows, s.H), dtype=torch.bfloat16, device=device)

    def set_weights(self, w1_f32: torch.Tensor, w2_f32: torch.Tensor):
        nvfp4_quantize(w1_f32, self.shape.H, MODE_PLAIN, self.w1_q[0], self.w1_sf[0])
        nvfp4_quantize(w2_f32, self.I, MODE_PLAIN, self.w2_q[0], self.w2_sf[0])

    def forward(self, x: torch.Tensor, alpha1: float = 1.0, alpha2: float = 1.0) -> torch.Tensor:
        """out[:T] = the shared FFN of x: NVFP4 staging, L1 + SwiGLU + requant, L2 (dense GEMMs)."""
        s = self.shape
        nvfp4_quantize(x, s.H, MODE_PLAIN, self.x_q, self.x_sf)
        nvfp4_grouped_gemm(self.x_q, self.x_sf, self.rows, None, None, 1, 2 * self.I, s.H, self.w1_q, self.w1_sf,
                           alpha1, EPI_SWIGLU_NVFP4, out_q=self.a2_q, out_sf=self.a2_sf)
        nvfp4_grouped_gemm(self.a2_q, self.a2_sf, self.rows, None, None, 1, s.H, self.I, self.w2_q, self.w2_sf,
                           alpha2, EPI_BF16, out_bf16=self.out)
        return self.out


def moe_forward(x: torch.Tensor, logits: torch.Tensor, w: MoeWeights, b: MoeBuffers,
                alpha1: float = 1.0, alpha2: float = 1.0, two_level: bool = False,
                shared: SharedExpert | None = None) -> torch.Tensor:
    """y = MoE-FFN(x): route + permute + stage, L1 + SwiGLU + requant + L2, combine.
    two_level: x's encode scale is computed here, the weights' are those of ``w``
    (built with two_level=True) and the L1 output's is ``b.a2_gs`` (None: 1).
    shared: a shared expert whose rows the combine adds to every token (one level)."""
    s = b.shape
    x_gs = None
    if two_level:
        if w.w1_gs is None:
            raise ValueError("two-level forward needs weights quantised with two_level=True")
        if s.T > 0:
            nvfp4_global_scale(x, b.x_gs)
        x_gs = b.x_gs
    moe_route_permute(logits, x, s.top_k, b.topk_ids, b.topk_w, b.counts, b.offsets, b.perm_token,
                      b.inv_perm, b.a1_q, b.a1_sf, b.workspace, x_global_scale=x_gs, x_q=b.x_q)
    if s.T > 0:
        gather = dict(a1_gather=b.perm_token, a1_gather_rows=s.T) if b.gather else {}
        nvfp4_moe_ffn_forward(b.x_q if b.gather else b.a1_q, b.a1_sf, b.offsets, b.counts, s.E, s.H, s.I,
                              b.rows_max, w.w1_q, w.w1_sf, w.w2_q, w.w2_sf, alpha1, alpha2, b.a2_q, b.a2_sf,
                              b.rows_out, b.h_debug, x_global_scale=x_gs,
                              w1_global_scale=w.w1_gs if two_level else None,
                              a2_global_scale=b.a2_gs if two_level else None,
                              w2_global_scale=w.w2_gs if two_level else None, **gather)
        shared_rows = None if shared is None else shared.forward(x, alpha1, alpha2)
        moe_combine(b.rows_out, b.inv_perm, b.topk_w, b.y, shared=shared_rows)
    return b.y


def _l1(w: MoeWeights, b: MoeBuffers, side_combine=None, two_level: bool = False) -> None:
    s = b.shape
    gs = dict(a_global_scale=b.x_gs, b_global_scale=w.w1_gs, out_global_scale=b.a2_gs) if two_level else {}
    nvfp4_grouped_gemm(b.a1_q, b.a1_sf, b.rows_max, b.offsets, b.counts, s.E, 2 * s.I, s.H, w.w1_q, w.w1_sf, 1.0,
                       EPI_SWIGLU_NVFP4, out_q=b.a2_q, out_sf=b.a2_sf, h_debug=b.h_debug, side_combine=side_combine,
                       **gs)


def _l2(w: MoeWeights, b: MoeBuffers, side_stage=None, two_level: bool = False) -> None:
    s = b.shape
    gs = dict(a_global_scale=b.a2_gs, b_global_scale=w.w2_gs) if two_level else {}
    nvfp4_grouped_gemm(b.a2_q, b.a2_sf, b.rows_max, b.offsets, b.counts, s.E, s.H, s.I, w.w2_q, w.w2_sf, 1.0,
                       EPI_BF16, out_bf16=b.rows_out, side_stage=side_stage, **gs)


def moe_forward_deferred(x: torch.Tensor, logits: torch.Tensor, w: MoeWeights, b: MoeBuffers,
                         prev: MoeBuffers | None = None, two_level: bool = False) -> None:
    """One step of a serving loop.  Without ``prev``: route + permute + stage and
    the L1 GEMM of this batch into ``b``.  With ``prev`` (an earlier batch whose
    L2 and combine are pending): routing of this batch without staging; prev's
    L2 GEMM, which stages this batch on spare warps; this batch's L1 GEMM, which
    runs prev's combine on spare warps (into prev.y).  This batch's L2 and
    combine stay pending: a later step's prev, or moe_finish_deferred.  A loop
    alternates two buffer sets.  two_level: as moe_forward's (x's encode scale
    computed here into b.x_gs, the weights' from ``w``, the L1 output's
    ``b.a2_gs``; every step of a loop must pass the same value).  Alpha 1, no
    shared expert, no gathered L1."""
    s = b.shape
    if prev is b:
        raise ValueError("prev must be another buffer set: this batch's staging runs beside prev's L2 GEMM")
    if b.gather or (prev is not None and prev.gather):
        raise ValueError("the deferred serving step stages permuted rows (no gathered L1)")
    if two_level and w.w1_gs is None:
        raise ValueError("two-level forward needs weights quantised with two_level=True")
    x_gs = None
    if two_level:
        if s.T > 0:
            nvfp4_global_scale(x, b.x_gs)
        x_gs = b.x_gs
    live_prev = prev is not None and prev.shape.T > 0
    moe_route_permute(logits, x, s.top_k, b.topk_ids, b.topk_w, b.counts, b.offsets, b.perm_token, b.inv_perm,
                      None if live_prev else b.a1_q, None if live_prev else b.a1_sf, b.workspace,
                      x_global_scale=None if live_prev else x_gs)
    job = None
    if live_prev:
        stage = (dict(x=x, inv_perm=b.inv_perm, counts=b.counts, offsets=b.offsets, a1_q=b.a1_q, a1_sf=b.a1_sf,
                      x_global_scale=x_gs) if s.T > 0 else None)
        _l2(w, prev, side_stage=stage, two_level=two_level)
        job = (prev.rows_out, prev.inv_perm, prev.topk_w, prev.y)
    if s.T > 0:
        _l1(w, b, side_combine=job, two_level=two_level)
    elif job is not None:
        moe_combine(*job)


def moe_finish_deferred(w: MoeWeights, b: MoeBuffers, two_level: bool = False) -> torch.Tensor:
    """The pending L2 GEMM and combine of the batch in ``b`` (after moe_forward_deferred)."""
    if b.shape.T > 0:
        _l2(w, b, two_level=two_level)
        moe_combine(b.rows_out, b.inv_perm, b.topk_w, b.y)
    return b.y


def calibrate_a2_scale(x: torch.Tensor, logits: torch.Tensor, w: MoeWeights, b: MoeBuffers,
                       alpha1: float = 1.0) -> torch.Tensor:
    """Set b.a2_gs = 2688 / amax of the L1 output h of this batch (two-level): one
    forward with the L1 output at scale 1 and h recorded, then a device reduction."""
    saved_h, saved_gs = b.h_debug, b.a2_gs
    b.enable_h_debug()
    b.a2_gs = None
    moe_forward(x, logits, w, b, alpha1=alpha1, two_level=True)
    gs = torch.ones(1, dtype=torch.float32, device=b.y.device) if saved_gs is None else saved_gs
    nvfp4_global_scale(b.h_debug, gs)
    b.h_debug, b.a2_gs = saved_h, gs
    return gs
