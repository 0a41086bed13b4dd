"""Helpers for the GPU parity tests: build/load the library, move arrays, compare."""
import numpy as np
import torch

from oracle import nvfp4 as onv


def built_lib():
    from nvfp4_block_scaled_moe_gb300 import build, load
    build.build()
    return load()


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    return t.detach().cpu().numpy()


def e2m1_step_distance(a_nib, b_nib):
    """Distance in E2M1 grid steps between nibble codes (sign-aware: -x and +x
    differ by the number of steps through zero)."""
    def signed_index(n):
        n = n.astype(np.int64)
        mag = n & 7
        return np.where(n & 8, -mag, mag)
    return np.abs(signed_index(a_nib) - signed_index(b_nib))


def compare_requantised(gpu_q, gpu_sf_rows, ora_q, ora_sf_rows, max_frac=1e-3):
    """The path's bound for re-quantised NVFP4: at most 0.1% of nibbles differ,
    each by at most one E2M1 step (a nibble of a block whose scale code differs
    is compared after that block is excluded; such blocks are also <= 0.1%)."""
    gn, on = onv.unpack_nibbles(gpu_q), onv.unpack_nibbles(ora_q)
    sf_diff = gpu_sf_rows != ora_sf_rows
    same_scale = ~np.repeat(sf_diff, 16, axis=1)
    diff = (gn != on)
    frac_nib = diff.mean()
    frac_sf = sf_diff.mean()
    dist = e2m1_step_distance(gn, on)
    max_step = int(dist[same_scale].max()) if same_scale.any() else 0
    return dict(frac_nib=float(frac_nib), frac_sf=float(frac_sf), max_step=max_step,
                ok=frac_nib <= max_frac and frac_sf <= max_frac and max_step <= 1)


def rel_frobenius(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))
