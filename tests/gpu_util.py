"""Helpers shared by the GPU parity tests: move raw-code numpy arrays to and
from the device with the right torch dtype, and build the library once."""
import numpy as np
import pytest
import torch

_built = False


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    global _built
    if not _built:
        from paged_kv_cache_309_gb300 import build
        build.build()
        _built = True


_VIEW = {"bf16": (np.uint16, torch.int16, torch.bfloat16),
         "fp16": (np.uint16, torch.int16, torch.float16),
         "e4m3": (np.uint8, torch.uint8, torch.float8_e4m3fn),
         "fp32": (np.float32, torch.float32, torch.float32)}


def to_dev(codes: np.ndarray, kind: str) -> torch.Tensor:
    npt, raw, typ = _VIEW[kind]
    a = np.ascontiguousarray(codes).astype(npt, copy=False)
    if kind == "fp32":
        return torch.from_numpy(a).cuda()
    t = torch.from_numpy(a.view(np.int16) if npt == np.uint16 else a).cuda()
    return t.view(typ)


def to_host(t: torch.Tensor, kind: str) -> np.ndarray:
    npt, raw, typ = _VIEW[kind]
    if kind == "fp32":
        return t.cpu().numpy()
    a = t.view(raw).cpu().numpy()
    return a.view(npt)


def codes_equal(a: np.ndarray, b: np.ndarray, kind: str) -> np.ndarray:
    """Bitwise equality, with every NaN code equal to every other NaN code."""
    if kind == "fp32":
        ai, bi = a.view(np.uint32), b.view(np.uint32)
        return (ai == bi) | (np.isnan(a) & np.isnan(b))
    if kind == "e4m3":
        na, nb = (a & 0x7F) == 0x7F, (b & 0x7F) == 0x7F
    elif kind == "bf16":
        na = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
        nb = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    else:  # fp16
        na = ((a & 0x7C00) == 0x7C00) & ((a & 0x3FF) != 0)
        nb = ((b & 0x7C00) == 0x7C00) & ((b & 0x3FF) != 0)
    return (a == b) | (na & nb)


def bf16_codes_to_f64(codes: np.ndarray) -> np.ndarray:
    return (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
