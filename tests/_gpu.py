"""Helpers shared by the GPU parity tests (device transfer, comparisons)."""
import numpy as np
import pytest
import torch

from sparse_moe_fine_gb300 import binding as B


def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.lib()
    return torch.device("cuda:0")


def to_dev(a, dev, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return t.to(torch.bfloat16) if bf16 else t


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def max_rel(got, ref, floor_frac=1e-4):
    """max |got - ref| / max(|ref|, floor_frac * max|ref|): relative error, with entries that
    cancel to near zero measured against a small fraction of the array's scale."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if not ref.size:
        return 0.0
    floor = max(floor_frac * float(np.max(np.abs(ref))), 1e-300)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))


def max_rel_terms(got, ref, *terms):
    """max |got - ref| / max(|ref|, |each term|): the relative error of a sum or difference
    measured against the size of its terms, so a result that cancels to near zero (an updated
    weight crossing zero) is held to the rounding of the terms that formed it."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.abs(ref)
    for t in terms:
        scale = np.maximum(scale, np.abs(np.asarray(t, np.float64)))
    return float(np.max(np.abs(got - ref) / np.maximum(scale, 1e-300))) if ref.size else 0.0
