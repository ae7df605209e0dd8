"""Shared helpers for the GPU parity tests (comparison arithmetic only)."""
import numpy as np
import torch


def bits16(t):
    """uint16 numpy copy of a BF16 (or int16/uint16) tensor."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def u8(t):
    return t.detach().contiguous().cpu().numpy()


def f32(t):
    return t.detach().contiguous().cpu().numpy()


def bf16_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_bf16(v):
    """Spacing of BF16 values at |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


# GEMM tolerances.  Contract (the stated accuracy): 1e-3 * sum|a b| plus half
# a BF16 ulp of the output.  Tight: what FP32 accumulation of exact FP8
# products with per-slab FP32 promotion can reach, 2^-14 * sum|a b| (each slab
# partial and each promotion step adds at most a few binary32 roundings
# relative to sum|a b|), used to catch errors the loose bound would hide.
CONTRACT_REL = 1e-3
TIGHT_REL = 2.0 ** -14


def gemm_violations(y_bits, y_ref, absref, rel):
    y = bf16_to_f64(y_bits)
    tol = rel * absref + 0.5 * np.maximum(ulp_bf16(y_ref), ulp_bf16(y))
    err = np.abs(y - y_ref)
    return err > tol, err, tol


def assert_gemm_close(y_bits, y_ref, absref, what=""):
    for rel, name in ((CONTRACT_REL, "contract"), (TIGHT_REL, "tight")):
        bad, err, tol = gemm_violations(y_bits, y_ref, absref, rel)
        if bad.any():
            idx = np.argwhere(bad)[:5]
            raise AssertionError(
                f"{what}: {int(bad.sum())} of {bad.size} outputs outside the {name} tolerance; "
                f"first {idx.tolist()}, err {err[bad][:5]}, tol {tol[bad][:5]}, "
                f"ref {np.asarray(y_ref)[bad][:5]}, gpu {bf16_to_f64(y_bits)[bad][:5]}")
