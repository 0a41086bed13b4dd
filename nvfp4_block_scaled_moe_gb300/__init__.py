"""Python binding of libnvfp4moe.so, the GB300 (sm_103a) NVFP4 MoE expert FFN.

Argument marshalling only: every function here passes device pointers, sizes
and the current CUDA stream to the C ABI declared in ``include/nvfp4moe.h``
and raises ``Nvfp4Error`` on a non-zero status.  Every step of the path runs in
the library's CUDA kernels; there is no CPU fallback, and importing a function
fails loudly when the library is not built.

PyTorch provides device memory and streams (``torch.cuda.current_stream()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "Nvfp4Error", "lib_path", "load", "sf_bytes", "moe_padded_rows_max",
    "moe_route_permute_workspace", "nvfp4_quantize", "nvfp4_sf_swizzle",
    "moe_route_permute", "moe_route_permute_static", "moe_stage_activation", "nvfp4_grouped_gemm",
    "nvfp4_moe_ffn_forward",
    "moe_combine", "nvfp4_moe_forward_host", "nvfp4_moe_step_host", "nvfp4_moe_finish_host",
    "nvfp4_device_status", "nvfp4_selftest_bounded_wait",
    "nvfp4_set_gemm_tiles", "nvfp4_global_scale", "nvfp4_mma_peak_probe",
    "MODE_PLAIN", "MODE_SWIGLU_GU8", "EPI_SWIGLU_NVFP4", "EPI_BF16",
]

MODE_PLAIN, MODE_SWIGLU_GU8, MODE_DEINTERLEAVE_GU8 = 0, 1, 2
IN_BF16, IN_F32 = 0, 1
EPI_SWIGLU_NVFP4, EPI_BF16, EPI_SWIGLU_BF16 = 0, 1, 2

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "ALIGNMENT", 4: "CUDA", 5: "TIMEOUT", 6: "DEVICE"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def lib_path() -> str:
    return os.path.join(_HERE, "libnvfp4moe.so")


_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


class _MoeWeightsC(ctypes.Structure):
    """nvfp4_moe_weights (include/nvfp4moe.h)."""
    _fields_ = [("w1_q", _vp), ("w1_sf", _vp), ("w2_q", _vp), ("w2_sf", _vp)]


class _CombineJobC(ctypes.Structure):
    """nvfp4_combine_job (include/nvfp4moe.h)."""
    _fields_ = [("rows_bf16", _vp), ("inv_perm", _vp), ("topk_w", _vp), ("T", _i32), ("top_k", _i32),
                ("H", _i32), ("y_bf16", _vp), ("rows", _i64)]


class _StageJobC(ctypes.Structure):
    """nvfp4_stage_job (include/nvfp4moe.h)."""
    _fields_ = [("x_bf16", _vp), ("x_global_scale", _vp), ("inv_perm", _vp), ("expert_counts", _vp),
                ("expert_offsets", _vp), ("a1_q", _vp), ("a1_sf", _vp), ("T", _i32), ("H", _i32), ("E", _i32),
                ("top_k", _i32), ("rows_max", _i64)]


class _MoeBuffersC(ctypes.Structure):
    """nvfp4_moe_buffers (include/nvfp4moe.h)."""
    _fields_ = [("x_bf16", _vp), ("logits", _vp), ("y_bf16", _vp), ("topk_ids", _vp), ("topk_w", _vp),
                ("expert_counts", _vp), ("expert_offsets", _vp), ("perm_token", _vp), ("inv_perm", _vp),
                ("a1_q", _vp), ("a1_sf", _vp), ("a2_q", _vp), ("a2_sf", _vp), ("rows_bf16", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz), ("rows_max", _i64)]
_SIGS = {
    "nvfp4_sf_bytes": (_sz, [_i64, _i64]),
    "moe_padded_rows_max": (_i64, [_i32, _i32, _i32]),
    "moe_route_permute_workspace": (_sz, [_i32, _i32, _i32, _i32]),
    "nvfp4_quantize": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                      _vp]),
    "nvfp4_global_scale": (ctypes.c_int, [_vp, ctypes.c_int, _i64, _i64, _i64, _vp, _vp]),
    "nvfp4_sf_swizzle": (ctypes.c_int, [_vp, _i64, _i64, _i64, _i64, _vp, ctypes.c_int, _vp]),
    "moe_route_permute": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                         _vp, _vp, _vp, _vp, _sz, _vp]),
    "nvfp4_grouped_gemm": (ctypes.c_int, [_vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _f32,
                                          _vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i64,
                                          ctypes.POINTER(_CombineJobC), ctypes.POINTER(_StageJobC), _vp]),
    "moe_stage_activation": (ctypes.c_int, [ctypes.POINTER(_StageJobC), _vp]),
    "nvfp4_moe_ffn_forward": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _vp, _vp, _vp, _vp,
                                             _f32, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                             ctypes.POINTER(_CombineJobC), _vp]),
    "moe_combine": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_route_permute_static": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                                _vp, _vp, _vp, _vp, _vp]),
    "nvfp4_moe_forward_host": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                              ctypes.POINTER(_MoeWeightsC), ctypes.POINTER(_MoeBuffersC), _vp]),
    "nvfp4_moe_step_host": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _i32, _i32, ctypes.POINTER(_MoeWeightsC),
                                           ctypes.POINTER(_MoeBuffersC), ctypes.POINTER(_MoeBuffersC), _i32, _vp,
                                           _vp, _vp, _vp]),
    "nvfp4_moe_finish_host": (ctypes.c_int, [ctypes.POINTER(_MoeWeightsC), ctypes.POINTER(_MoeBuffersC), _i32, _i32,
                                             _i32, _i32, _i32, _vp, _vp]),
    "nvfp4_last_error": (ctypes.c_char_p, []),
    "nvfp4_device_status": (ctypes.c_int, [_vp]),
    "nvfp4_selftest_bounded_wait": (ctypes.c_int, [_vp, _i64, _vp]),
    "nvfp4_set_gemm_tiles": (ctypes.c_int, [ctypes.c_int32]),
    "nvfp4_mma_peak_probe": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(ctypes.c_double),
                                            ctypes.POINTER(ctypes.c_double), _vp]),
}


def load():
    """Load the in-tree library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m nvfp4_block_scaled_moe_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _LIB = lib
    return _LIB


def _check(status: int) -> None:
    if status != 0:
        raise Nvfp4Error(status, load().nvfp4_last_error().decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


# ----------------------------------------------------------------- sizes --
def sf_bytes(rows: int, cols: int) -> int:
    return load().nvfp4_sf_bytes(rows, cols)


def moe_padded_rows_max(T: int, E: int, top_k: int) -> int:
    return load().moe_padded_rows_max(T, E, top_k)


def moe_route_permute_workspace(T: int, H: int, E: int, top_k: int) -> int:
    return load().moe_route_permute_workspace(T, H, E, top_k)


# ----------------------------------------------------------------- calls --
def nvfp4_quantize(inp, out_cols, mode, q_out, sf_out, h_debug=None, in_ld=None, stream=None, global_scale=None):
    """inp: BF16 or fp32 [rows, in_cols] CUDA tensor (rows may be strided);
    global_scale: None or a device fp32 scalar tensor (two-level encode scale)."""
    dtype = IN_BF16 if inp.dtype == torch.bfloat16 else IN_F32
    ld = inp.stride(0) if in_ld is None else in_ld
    _check(load().nvfp4_quantize(_p(inp), dtype, mode, inp.shape[0], out_cols, ld, _p(q_out), _p(sf_out),
                                 _p(global_scale), _p(h_debug), _stream(stream)))


def nvfp4_global_scale(inp, g_out, cols=None, in_ld=None, stream=None):
    """g_out (device fp32 scalar) = 2688 / amax |inp| (1 for an all-zero tensor)."""
    dtype = IN_BF16 if inp.dtype == torch.bfloat16 else IN_F32
    rows = inp.shape[0] if inp.dim() > 1 else 1
    cols = (inp.shape[-1] if inp.dim() > 1 else inp.numel()) if cols is None else cols
    ld = (inp.stride(0) if inp.dim() > 1 else cols) if in_ld is None else in_ld
    _check(load().nvfp4_global_scale(_p(inp), dtype, rows, cols, ld, _p(g_out), _stream(stream)))


def nvfp4_sf_swizzle(sf_in, mn_rows, k_sf_cols, stride_mn, stride_ksf, sf_out, inverse=False, stream=None):
    _check(load().nvfp4_sf_swizzle(_p(sf_in), mn_rows, k_sf_cols, stride_mn, stride_ksf, _p(sf_out),
                                   1 if inverse else 0, _stream(stream)))


def moe_route_permute(logits, x, top_k, topk_ids, topk_w, expert_counts, expert_offsets, perm_token, inv_perm,
                      a1_q, a1_sf, workspace, stream=None, x_global_scale=None, x_q=None):
    T, E = logits.shape
    H = x.shape[1]
    _check(load().moe_route_permute(_p(logits), _p(x), T, H, E, top_k, _p(topk_ids), _p(topk_w),
                                    _p(expert_counts), _p(expert_offsets), _p(perm_token), _p(inv_perm),
                                    _p(a1_q), _p(a1_sf), _p(x_q), _p(x_global_scale), _p(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_route_permute_static(logits, x, top_k, topk_ids, topk_w, expert_counts, expert_offsets, perm_token,
                             inv_perm, a1_q, a1_sf, stream=None, x_global_scale=None, x_q=None):
    """moe_route_permute with the library's fixed device scratch instead of a
    caller workspace, for callers that cannot allocate (see include/nvfp4moe.h)."""
    T, E = logits.shape
    H = x.shape[1]
    _check(load().moe_route_permute_static(_p(logits), _p(x), T, H, E, top_k, _p(topk_ids), _p(topk_w),
                                           _p(expert_counts), _p(expert_offsets), _p(perm_token), _p(inv_perm),
                                           _p(a1_q), _p(a1_sf), _p(x_q), _p(x_global_scale), _stream(stream)))


def _combine_job(job):
    """(rows, inv_perm, topk_w, y) tensors -> a pointer to nvfp4_combine_job (None -> NULL)."""
    if job is None:
        return None
    rows, inv, w, y = job
    return ctypes.byref(_CombineJobC(rows.data_ptr(), inv.data_ptr(), w.data_ptr(), inv.shape[0], inv.shape[1],
                                     y.shape[1], y.data_ptr(), rows.shape[0]))


def _stage_job(job):
    """dict(x, inv_perm, counts, offsets, a1_q, a1_sf[, x_global_scale, rows_max])
    of device tensors -> a pointer to nvfp4_stage_job (None -> NULL); rows_max
    defaults to a1_q's rows."""
    if job is None:
        return None
    x, inv = job["x"], job["inv_perm"]
    return ctypes.byref(_StageJobC(x.data_ptr(), _p(job.get("x_global_scale")), inv.data_ptr(),
                                   job["counts"].data_ptr(), job["offsets"].data_ptr(), job["a1_q"].data_ptr(),
                                   job["a1_sf"].data_ptr(), x.shape[0], x.shape[1], job["counts"].shape[0],
                                   inv.shape[1], job.get("rows_max", job["a1_q"].shape[0])))


def moe_stage_activation(job, stream=None):
    """The staging half of moe_route_permute for a batch routed with a1_sf None
    (``job`` as for nvfp4_grouped_gemm's side_stage)."""
    _check(load().moe_stage_activation(_stage_job(job), _stream(stream)))


def nvfp4_grouped_gemm(a_q, a_sf, rows_max, group_offsets, group_counts, G, N, K, b_q, b_sf, alpha, epilogue,
                       out_q=None, out_sf=None, out_bf16=None, h_debug=None, stream=None, a_global_scale=None,
                       b_global_scale=None, out_global_scale=None, a_gather=None, a_gather_rows=0,
                       side_combine=None, side_stage=None):
    """side_combine: None, or (rows, inv_perm, topk_w, y) of an earlier batch to
    combine alongside (run on spare warps of the CTA-pair SwiGLU kernel).
    side_stage: None, or dict(x, inv_perm, counts, offsets, a1_q, a1_sf[,
    x_global_scale]) of a later batch to stage alongside (spare warps of the
    CTA-pair BF16 kernel)."""
    _check(load().nvfp4_grouped_gemm(_p(a_q), _p(a_sf), rows_max, _p(group_offsets), _p(group_counts), G, N, K,
                                     _p(b_q), _p(b_sf), alpha, _p(a_global_scale), _p(b_global_scale),
                                     _p(out_global_scale), epilogue, _p(out_q), _p(out_sf), _p(out_bf16),
                                     _p(h_debug), _p(a_gather), a_gather_rows, _combine_job(side_combine),
                                     _stage_job(side_stage), _stream(stream)))


def nvfp4_moe_ffn_forward(a1_q, a1_sf, expert_offsets, expert_counts, E, H, I, rows_max, w1_q, w1_sf, w2_q, w2_sf,
                          alpha1, alpha2, a2_q, a2_sf, rows_out, h_debug=None, stream=None, x_global_scale=None,
                          w1_global_scale=None, a2_global_scale=None, w2_global_scale=None, a1_gather=None,
                          a1_gather_rows=0, prev_combine=None):
    """prev_combine: None, or (rows, inv_perm, topk_w, y) of an earlier batch whose
    combine the L1 GEMM runs on spare warps (y = moe_combine(rows, inv_perm, topk_w))."""
    job = _combine_job(prev_combine)
    _check(load().nvfp4_moe_ffn_forward(_p(a1_q), _p(a1_sf), _p(expert_offsets), _p(expert_counts), E, H, I,
                                        rows_max, _p(w1_q), _p(w1_sf), _p(w2_q), _p(w2_sf), alpha1, alpha2,
                                        _p(x_global_scale), _p(w1_global_scale), _p(a2_global_scale),
                                        _p(w2_global_scale), _p(a2_q), _p(a2_sf), _p(rows_out), _p(h_debug),
                                        _p(a1_gather), a1_gather_rows, job, _stream(stream)))


def _weights_c(weights):
    return _MoeWeightsC(weights.w1_q.data_ptr(), weights.w1_sf.data_ptr(), weights.w2_q.data_ptr(),
                        weights.w2_sf.data_ptr())


def _buffers_c(b):
    return _MoeBuffersC(b.x.data_ptr(), b.logits.data_ptr(), b.y.data_ptr(), b.topk_ids.data_ptr(),
                        b.topk_w.data_ptr(), b.counts.data_ptr(), b.offsets.data_ptr(), b.perm_token.data_ptr(),
                        b.inv_perm.data_ptr(), b.a1_q.data_ptr(), b.a1_sf.data_ptr(), b.a2_q.data_ptr(),
                        b.a2_sf.data_ptr(), b.rows_out.data_ptr(), b.workspace.data_ptr(),
                        b.workspace.numel() * b.workspace.element_size(), b.rows_max)


def _event(ev):
    """torch.cuda.Event (already recorded once, so that it exists) -> its handle."""
    return None if ev is None else ctypes.c_void_p(ev.cuda_event)


def nvfp4_moe_step_host(x_host, logits_host, top_k, weights, buffers, prev=None, prev_y_host=None,
                        compute_after=None, compute_done=None, stream=None, prev_T=None):
    """One step of a serving loop from host buffers: copy this batch in and route
    it; with ``prev`` (an earlier batch whose L2 and combine are pending), prev's
    L2 GEMM stages this batch alongside and this batch's L1 GEMM runs prev's
    combine alongside, then prev's y is copied out to ``prev_y_host``; without,
    route with staging and L1.  This batch's L2 and combine stay pending (a
    later step's prev, or nvfp4_moe_finish_host).  Events are torch.cuda.Event
    objects (recorded once beforehand) or None.  Batches may differ in size up
    to the buffers' T: prev_T is the earlier batch's token count (default: the
    rows of prev_y_host)."""
    T, H = x_host.shape
    E = logits_host.shape[1]
    I = 2 * buffers.a2_q.shape[1]
    prev_c = ctypes.byref(_buffers_c(prev)) if prev is not None else None
    if prev is None:
        prev_T = 0
    elif prev_T is None:
        prev_T = prev_y_host.shape[0]
    _check(load().nvfp4_moe_step_host(_p(x_host), _p(logits_host), T, H, I, E, top_k,
                                      ctypes.byref(_weights_c(weights)), ctypes.byref(_buffers_c(buffers)), prev_c,
                                      prev_T, _p(prev_y_host), _event(compute_after), _event(compute_done),
                                      _stream(stream)))


def nvfp4_moe_finish_host(weights, buffers, top_k, y_host, stream=None):
    """The pending L2 GEMM and combine of the batch in ``buffers``, then its y
    copied out to y_host."""
    T, H = y_host.shape
    E = buffers.counts.shape[0]
    I = 2 * buffers.a2_q.shape[1]
    _check(load().nvfp4_moe_finish_host(ctypes.byref(_weights_c(weights)), ctypes.byref(_buffers_c(buffers)), T, H,
                                        I, E, top_k, _p(y_host), _stream(stream)))


def nvfp4_moe_forward_host(x_host, logits_host, y_host, top_k, weights, buffers, stream=None):
    """The whole path from host x [T, H] BF16 and logits [T, E] fp32 to host y [T, H]
    BF16 in one C-ABI call (copies in, route, FFN, combine, copy out, all on
    `stream`).  Host tensors should be pinned.  ``weights`` has w1_q, w1_sf, w2_q,
    w2_sf; ``buffers`` the device tensors x, logits, y, topk_ids, topk_w, counts,
    offsets, perm_token, inv_perm, a1_q, a1_sf, a2_q, a2_sf, rows_out, workspace
    and the int rows_max (pipeline.MoeBuffers with host I/O enabled)."""
    T, H = x_host.shape
    E = logits_host.shape[1]
    I = 2 * buffers.a2_q.shape[1]
    _check(load().nvfp4_moe_forward_host(_p(x_host), _p(logits_host), _p(y_host), T, H, I, E, top_k,
                                         ctypes.byref(_weights_c(weights)), ctypes.byref(_buffers_c(buffers)),
                                         _stream(stream)))


def moe_combine(rows, inv_perm, topk_w, y, stream=None, shared=None):
    T, top_k = inv_perm.shape
    H = y.shape[1]
    _check(load().moe_combine(_p(rows), _p(inv_perm), _p(topk_w), T, H, top_k, _p(shared), _p(y),
                              _stream(stream)))


def nvfp4_device_status(stream=None):
    _check(load().nvfp4_device_status(_stream(stream)))


GEMM_TILES_AUTO, GEMM_TILES_SINGLE, GEMM_TILES_PAIR = 0, 1, 2


def nvfp4_set_gemm_tiles(mode):
    """Process-wide tile choice of nvfp4_grouped_gemm: GEMM_TILES_AUTO (by shape;
    grouped CTA-pair GEMMs split with a single-CTA launch beside them),
    GEMM_TILES_SINGLE or GEMM_TILES_PAIR (the pair kernel alone)."""
    _check(load().nvfp4_set_gemm_tiles(mode))


def nvfp4_mma_peak_probe(iters=20000, stream=None):
    """(TFLOP/s, SM MHz) of the CTA-pair GEMM's FP4 MMA stream with resident
    operands on every SM pair: the instruction ceiling. Synchronises the stream."""
    tf, mhz = ctypes.c_double(0.0), ctypes.c_double(0.0)
    _check(load().nvfp4_mma_peak_probe(iters, ctypes.byref(tf), ctypes.byref(mhz), _stream(stream)))
    return tf.value, mhz.value


def nvfp4_selftest_bounded_wait(flag, limit_ns, stream=None):
    _check(load().nvfp4_selftest_bounded_wait(_p(flag), limit_ns, _stream(stream)))
