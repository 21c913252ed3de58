"""Shared helpers for the GPU parity tests: moving seeded inputs to the device
and the error measures the tolerances are stated in."""
import numpy as np

TOL_LOSS = 1e-3          # |loss - oracle|
TOL_REL = 5e-3           # relative Frobenius error of dH and dW (bf16 inputs)
TOL_LSE = 1e-3           # per-row lse, diagnostic


def to_device(x, dev="cuda:0"):
    import torch
    if x.bf16:
        H = torch.from_numpy(x.H.view(np.int16)).to(dev).view(torch.bfloat16)
        W = torch.from_numpy(x.W.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        H = torch.from_numpy(x.H).to(dev)
        W = torch.from_numpy(x.W).to(dev)
    return H, W, torch.from_numpy(x.targets).to(dev)


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a - b))


def np64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)
