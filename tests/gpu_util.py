"""Helpers shared by the GPU parity tests (device transfers, error norms and
the record of each parity margin, printed at the end of the run)."""
import json
from pathlib import Path

import numpy as np

# (test, quantity, measured error, gate): printed by conftest's terminal summary
MARGINS = []


def record_margin(test: str, what: str, err: float, gate: float) -> float:
    MARGINS.append((test, what, float(err), float(gate)))
    return err


def page_constant(name: str):
    """A number the pages print (tests/golden/page_constants.json)."""
    p = Path(__file__).resolve().parent / "golden" / "page_constants.json"
    return json.loads(p.read_text())[name]


def rel_frob(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def to_dev(a, dtype=None, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def to_np(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def bf16_input(rng, shape, scale=1.0):
    """A bf16 device tensor of N(0, scale^2) values and its exact f64 copy."""
    import torch
    t = torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)
    return t.cuda(), t.to(torch.float64).numpy()


def q8_dev(w):
    """Device tensors (q, s, b) of a synth q8 weight dict."""
    import torch
    q = to_dev(w["q"])
    s = to_dev(w["s"], torch.float32)
    b = to_dev(w["b"], torch.float32) if w["b"] is not None else None
    return q, s, b
