"""Comparison helpers shared by the GPU parity tests.

Tolerances (|got - ref| <= atol + rtol * |ref|, element by element, against the
fp64 oracle evaluated on the very values the GPU received):
  bf16: atol = rtol = 5e-3, plus cosine similarity > 0.999 over the whole output
        (tolerance table of the Triton-distributed precision page, section 3.4;
        the bf16 criteria of the juejin ring-attention page, section 二);
  fp32: atol = rtol = 1e-5 (same table).
"""
import numpy as np
import torch

BF16_TOL = 5e-3
F32_TOL = 1e-5


def to_np(t):
    return t.detach().float().cpu().double().numpy() if t.dtype != torch.float64 else t.cpu().numpy()


def cosine(a, b):
    a, b = np.ravel(a), np.ravel(b)
    return float((a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum()))


def assert_close(got, ref, tol, what="", cos_min=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bound = tol + tol * np.abs(ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance; "
                           f"max abs err {err.max():.3e}, worst ratio {(err / bound).max():.3f}")
    if cos_min is not None:
        c = cosine(got, ref)
        assert c > cos_min, f"{what}: cosine {c}"
    return float(err.max())


def assert_bf16_close(got, ref, what=""):
    return assert_close(got, ref, BF16_TOL, what, cos_min=0.999)


def assert_f32_close(got, ref, what=""):
    return assert_close(got, ref, F32_TOL, what)
