"""Small conversions shared by the tests (no method arithmetic here)."""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def to_np(t: torch.Tensor) -> np.ndarray:
    """CPU tensor -> numpy; bf16 becomes its uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def from_np(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    if dtype == torch.bfloat16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a))


def bits(a: np.ndarray) -> np.ndarray:
    """Bit patterns for exact comparison (uint16 stays, float32 -> uint32)."""
    if a.dtype == np.float32:
        return a.view(np.uint32)
    return a


def dtype_of(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def exact_in(values, dtype: torch.dtype) -> torch.Tensor:
    """Hand-typed values as a tensor of `dtype`; fails unless each is exactly representable."""
    f = torch.tensor(values, dtype=torch.float64)
    t = f.to(dtype)
    assert torch.equal(t.to(torch.float64), f), f"value not exact in {dtype}: {values}"
    return t


def golden_case_tensors(case):
    """(ids int64 [n], grad [n, H], main_grad [V, H]) for one hand case, on the CPU."""
    gdt = dtype_of(case["grad_dtype"])
    mdt = dtype_of(case["main_grad_dtype"])
    V, H = case["num_embeddings"], case["hidden"]
    ids = torch.tensor(case["ids"], dtype=torch.int64)
    grad = exact_in(case["grad"], gdt)
    mg = torch.zeros(V, H, dtype=mdt)
    for k, row in case["main_grad_init"].items():
        mg[int(k)] = exact_in(row, mdt)
    return ids, grad, mg


def golden_expected(case, mg_init: torch.Tensor) -> torch.Tensor:
    out = mg_init.clone()
    for k, row in case["expected"].items():
        out[int(k)] = exact_in(row, mg_init.dtype)
    return out
