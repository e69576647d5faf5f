"""Helpers shared by the GPU tests: move seeded inputs to the device, compare with the oracle."""
import numpy as np
import torch

import oracle

TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Storage-format numpy array (fp32, or bf16 bit patterns) -> CUDA tensor."""
    if dtype == "bf16" and a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda").view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")


def from_dev(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = max(float(np.max(np.abs(ref))), 1e-30)
    return float(np.max(np.abs(got - ref))) / den


def dev_inputs(inp: dict, dtype: str) -> dict:
    out = {}
    for k in ("u", "delta", "z", "B", "C"):
        if inp.get(k) is not None:
            out[k] = to_dev(inp[k], dtype)
    for k in ("A", "D", "delta_bias"):
        if inp.get(k) is not None:
            out[k] = torch.from_numpy(np.ascontiguousarray(inp[k], np.float32)).to("cuda")
    return out


def oracle_scan_full(inp: dict, dtype: str, softplus=True, nthreads=0):
    return oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp.get("D"),
                       inp.get("z"), inp.get("delta_bias"), softplus, dtype, nthreads=nthreads)


def sample_rows(nrows: int, k: int, seed: int = 0) -> np.ndarray:
    """k channels spread over all batches and channel blocks, always including the first/last."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(nrows, size=min(k, nrows), replace=False).tolist())
    pick.update({0, nrows - 1})
    return np.array(sorted(pick), dtype=np.int64)
