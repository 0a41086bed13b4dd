"""CPU checks of the C ABI: the library builds for sm_103a, loads without a GPU,
exports every function include/nvfp4moe.h declares, and rejects bad arguments
on the host before any CUDA call (no compute is launched here)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4moe.h")

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z][a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_scaled_moe_gb300 import build, load
    build.build()
    return load()


def test_header_declares_the_five_path_calls():
    names = declared_functions()
    for n in ("nvfp4_quantize", "nvfp4_sf_swizzle", "moe_route_permute", "nvfp4_moe_ffn_forward", "moe_combine"):
        assert n in names


@needs_nvcc
def test_library_exports_every_declared_function(lib):
    raw = ctypes.CDLL(os.path.join(ROOT, "nvfp4_block_scaled_moe_gb300", "libnvfp4moe.so"))
    for name in declared_functions():
        assert hasattr(raw, name), name


@needs_nvcc
def test_size_helpers(lib):
    assert lib.nvfp4_sf_bytes(128, 64) == 512
    assert lib.nvfp4_sf_bytes(129, 65) == 2 * 2 * 512
    assert lib.nvfp4_sf_bytes(0, 64) == 0
    # worst case: every group padded by 127 rows, result a multiple of 128
    r = lib.moe_padded_rows_max(16384, 256, 8)
    assert r % 128 == 0 and r >= 16384 * 8 and r <= 16384 * 8 + 127 * 256
    assert lib.moe_padded_rows_max(1, 256, 8) == 1024        # 8 rows, each its own group
    # the workspace holds one int32 expert count per (128-token chunk, expert)
    assert lib.moe_route_permute_workspace(256, 7168, 256, 8) >= 2 * 256 * 4
    assert lib.moe_route_permute_workspace(16384, 7168, 256, 8) >= 128 * 256 * 4


def nvb_job(rows, inv, w, T, k, H, y, n_rows=1024):
    import nvfp4_block_scaled_moe_gb300 as nvb
    return nvb._CombineJobC(rows, inv, w, T, k, H, y, n_rows)


def nvb_stage(x, gs, inv, counts, offsets, a1_q, a1_sf, T, H, E, k, rows_max=1024):
    import nvfp4_block_scaled_moe_gb300 as nvb
    return nvb._StageJobC(x, gs, inv, counts, offsets, a1_q, a1_sf, T, H, E, k, rows_max)


@needs_nvcc
def test_host_validation_without_gpu(lib):
    import nvfp4_block_scaled_moe_gb300 as nv
    vp = ctypes.c_void_p
    buf = ctypes.create_string_buffer(4096 + 64)
    base = (ctypes.addressof(buf) + 15) & ~15
    p = vp(base)
    odd = vp(base + 1)
    # null input
    assert lib.nvfp4_quantize(None, 0, 0, 4, 16, 16, p, p, None, None, None) == 1
    # out_cols not a multiple of 16
    assert lib.nvfp4_quantize(p, 0, 0, 4, 24, 24, p, p, None, None, None) == 2
    # misaligned input
    assert lib.nvfp4_quantize(odd, 0, 0, 4, 16, 16, p, p, None, None, None) == 3
    # SwiGLU mode needs BF16
    assert lib.nvfp4_quantize(p, 1, 1, 4, 16, 32, p, p, None, None, None) == 2
    assert lib.nvfp4_quantize(p, 0, 0, 4, 16, 16, p, p, vp(base + 2), None, None) == 3    # misaligned scale
    # the nibbles of a 16-block leave as one 8-byte store: q_out must be 8-byte aligned
    assert lib.nvfp4_quantize(p, 0, 0, 4, 16, 16, vp(base + 4), p, None, None, None) == 3
    assert lib.nvfp4_quantize(p, 0, 0, 4, 16, 16, p, vp(base + 2), None, None, None) == 3   # SF words: 4 bytes
    # global scale: null input, cols not a multiple of 8, misaligned output
    assert lib.nvfp4_global_scale(None, 0, 4, 16, 16, p, None) == 1
    assert lib.nvfp4_global_scale(p, 0, 4, 12, 12, p, None) == 2
    assert lib.nvfp4_global_scale(p, 0, 4, 16, 16, vp(base + 2), None) == 3
    assert lib.nvfp4_sf_swizzle(p, 4, 4, 0, 1, p, 0, None) == 1
    # K not a multiple of 256; N not a multiple of 128 (BF16) / 256 (SwiGLU); G without offsets
    assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 1, 256, 200, p, p, 1.0, None, None, None, 1, None, None, p, None, None, 0, None, None, None) == 2
    assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 1, 192, 256, p, p, 1.0, None, None, None, 1, None, None, p, None, None, 0, None, None, None) == 2
    assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 1, 128, 256, p, p, 1.0, None, None, None, 0, p, p, None, None, None, 0, None, None, None) == 2
    assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 4, 256, 256, p, p, 1.0, None, None, None, 1, None, None, p, None, None, 0, None, None, None) == 2
    assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 1, 256, 256, p, p, 1.0, None, None, None, 7, None, None, p, None, None, 0, None, None, None) == 1
    # routing limits
    assert lib.moe_route_permute(p, p, 8, 64, 2000, 2, p, p, p, p, p, p, p, p, None, None, p, 1 << 20, None) == 2
    assert lib.moe_route_permute(p, p, 8, 64, 8, 9, p, p, p, p, p, p, p, p, None, None, p, 1 << 20, None) == 2
    assert lib.moe_route_permute(p, p, 8, 60, 8, 2, p, p, p, p, p, p, p, p, None, None, p, 1 << 20, None) == 2
    assert lib.moe_route_permute(p, p, 8, 64, 8, 2, p, p, p, p, p, p, p, p, None, None, p, 16, None) == 1
    # neither permuted rows nor token-order rows requested; misaligned token-order rows
    assert lib.moe_route_permute(p, p, 8, 64, 8, 2, p, p, p, p, p, p, None, p, None, None, p, 1 << 20, None) == 1
    assert lib.moe_route_permute(p, p, 8, 64, 8, 2, p, p, p, p, p, p, None, p, vp(base + 4), None, p, 1 << 20,
                                 None) == 3
    # gathered A: a row count is required, the index must be 16-byte aligned
    assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 1, 256, 256, p, p, 1.0, None, None, None, 1, None, None, p,
                                  None, p, 0, None, None, None) == 1
    assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 1, 256, 256, p, p, 1.0, None, None, None, 1, None, None, p,
                                  None, vp(base + 4), 64, None, None, None) == 3
    # gathered A with an epilogue other than SwiGLU + NVFP4 (the L1 GEMM's) is not built
    assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 1, 256, 256, p, p, 1.0, None, None, None, 1, None, None, p,
                                  None, p, 64, None, None, None) == 2
    assert lib.nvfp4_moe_ffn_forward(p, p, p, p, 8, 512, 200, 128, p, p, p, p, 1.0, 1.0, None, None, None, None, p, p, p, None, None, 0, None, None) == 2
    # a side combine job: its own checks, before anything is launched
    job_bad_k = nvb_job(base, base, base, 4, 40, 512, base)
    job_null = nvb_job(base, None, base, 4, 2, 512, base)
    job_odd_y = nvb_job(base, base, base, 4, 2, 512, base + 8)
    job_odd_h = nvb_job(base, base, base, 4, 2, 500, base)
    job_no_rows = nvb_job(base, base, base, 4, 2, 512, base, 0)
    for job, st in ((job_bad_k, 1), (job_null, 1), (job_odd_y, 3), (job_odd_h, 2), (job_no_rows, 1)):
        assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 1, 256, 256, p, p, 1.0, None, None, None, 0, p, p,
                                      None, None, None, 0, ctypes.byref(job), None, None) == st
    # a side staging job: its own checks, before anything is launched
    def stage(x=base, inv=base, cnt=base, off=base, q=base, sf=base, T=4, H=512, E=8, k=2, rows_max=1024):
        return nvb_stage(x, None, inv, cnt, off, q, sf, T, H, E, k, rows_max)
    for job, st in ((stage(inv=None), 1), (stage(sf=None), 1), (stage(E=2000), 2), (stage(k=9), 2),
                    (stage(k=40, E=64), 2), (stage(H=96), 2), (stage(x=base + 8), 3), (stage(q=base + 4), 3),
                    (stage(rows_max=0), 2), (stage(rows_max=200), 2)):
        assert lib.nvfp4_grouped_gemm(p, p, 128, None, None, 1, 256, 256, p, p, 1.0, None, None, None, 1, None, None,
                                      p, None, None, 0, None, ctypes.byref(job), None) == st
        assert lib.moe_stage_activation(ctypes.byref(job), None) == st
    assert lib.moe_stage_activation(None, None) == 1
    # routing only (a1_sf NULL) takes neither a1_q nor x_q
    assert lib.moe_route_permute(p, p, 8, 64, 8, 2, p, p, p, p, p, p, p, None, None, None, p, 1 << 20, None) == 1
    assert lib.moe_route_permute(p, p, 8, 64, 8, 2, p, p, p, p, p, p, None, None, p, None, p, 1 << 20, None) == 1
    assert lib.moe_route_permute_static(p, p, 8, 64, 8, 2, p, p, p, p, p, p, p, None, None, None, None) == 1
    # the forward's job must have the forward's H
    job_h = nvb_job(base, base, base, 4, 2, 768, base)
    assert lib.nvfp4_moe_ffn_forward(p, p, p, p, 8, 512, 256, 128, p, p, p, p, 1.0, 1.0, None, None, None, None, p, p,
                                     p, None, None, 0, ctypes.byref(job_h), None) == 1
    # the host-buffer forward: null pointers, no tokens, a short workspace, an unaligned buffer
    import nvfp4_block_scaled_moe_gb300 as nvb
    wts = nvb._MoeWeightsC(base, base, base, base)
    bufs = nvb._MoeBuffersC(*([base] * 15), 1 << 20, 1024)
    assert lib.nvfp4_moe_forward_host(None, p, p, 4, 512, 256, 8, 2, ctypes.byref(wts), ctypes.byref(bufs),
                                      None) == 1
    assert lib.nvfp4_moe_forward_host(p, p, p, 0, 512, 256, 8, 2, ctypes.byref(wts), ctypes.byref(bufs), None) == 1
    assert lib.nvfp4_moe_forward_host(p, p, p, 4, 500, 256, 8, 2, ctypes.byref(wts), ctypes.byref(bufs), None) == 2
    short = nvb._MoeBuffersC(*([base] * 15), 4, 1024)
    assert lib.nvfp4_moe_forward_host(p, p, p, 4, 512, 256, 8, 2, ctypes.byref(wts), ctypes.byref(short),
                                      None) == 1
    odd_buf = nvb._MoeBuffersC(*([base] * 9 + [base + 8] + [base] * 5), 1 << 20, 1024)
    assert lib.nvfp4_moe_forward_host(p, p, p, 4, 512, 256, 8, 2, ctypes.byref(wts), ctypes.byref(odd_buf),
                                      None) == 3
    # serving-loop steps: prev may not be this step's set, needs a y buffer on the host and its own checks
    assert lib.nvfp4_moe_step_host(p, p, 4, 512, 256, 8, 2, ctypes.byref(wts), ctypes.byref(bufs),
                                   ctypes.byref(bufs), 4, p, None, None, None) == 1
    other = nvb._MoeBuffersC(*([base] * 15), 1 << 20, 1024)
    assert lib.nvfp4_moe_step_host(p, p, 4, 512, 256, 8, 2, ctypes.byref(wts), ctypes.byref(bufs),
                                   ctypes.byref(other), 4, None, None, None, None) == 1
    assert lib.nvfp4_moe_step_host(p, p, 4, 512, 256, 8, 2, ctypes.byref(wts), ctypes.byref(bufs),
                                   ctypes.byref(short), 4, p, None, None, None) == 1
    assert lib.nvfp4_moe_step_host(p, p, 4, 512, 256, 8, 2, ctypes.byref(wts), ctypes.byref(bufs),
                                   ctypes.byref(other), 0, p, None, None, None) == 1
    assert lib.nvfp4_moe_finish_host(ctypes.byref(wts), ctypes.byref(bufs), 4, 512, 256, 8, 2, None, None) == 1
    assert lib.nvfp4_moe_finish_host(ctypes.byref(wts), ctypes.byref(odd_buf), 4, 512, 256, 8, 2, p, None) == 3
    assert lib.moe_combine(p, p, p, 4, 12, 2, None, p, None) == 2
    assert lib.moe_combine(p, p, p, 4, 16, 2, vp(base + 8), p, None) == 3     # misaligned shared rows
    d = ctypes.c_double(0.0)
    assert lib.nvfp4_mma_peak_probe(100, None, ctypes.byref(d), None) == 1       # null result pointer
    assert lib.nvfp4_mma_peak_probe(0, ctypes.byref(d), ctypes.byref(d), None) == 1
    assert lib.nvfp4_mma_peak_probe(1 << 21, ctypes.byref(d), ctypes.byref(d), None) == 1
    assert lib.nvfp4_selftest_bounded_wait(None, 10, None) == 1
    assert b"selftest" in lib.nvfp4_last_error()
    # tile-kernel choice: three modes, anything else refused; the default restored
    assert lib.nvfp4_set_gemm_tiles(3) == 1 and lib.nvfp4_set_gemm_tiles(-1) == 1
    for mode in (2, 1, 0):
        assert lib.nvfp4_set_gemm_tiles(mode) == 0
    with pytest.raises(nv.Nvfp4Error) as ei:
        nv._check(2)
    assert ei.value.status == 2


def test_product_package_has_no_cpu_fallback():
    """The binding refuses to run without the built library and never imports the oracle."""
    src_dir = os.path.join(ROOT, "nvfp4_block_scaled_moe_gb300")
    for dirpath, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("# oracle", ""), f
                assert "inputs" not in re.findall(r"^\s*(?:from|import)\s+(\w+)", text, flags=re.M), f
