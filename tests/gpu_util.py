"""Helpers shared by the GPU tests: moving seeded inputs to the device and
reading results back.  No method arithmetic here."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dsa_sparse_mla_prefill_gb300 import build as b
    b.build()


def bf(a, dev="cuda"):
    """uint16 bf16 bits (numpy) -> torch.bfloat16 on the device."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def i32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def f32(t):
    return t.float().cpu().numpy().astype(np.float64)


def stratified_tokens(T, n, rng, must=()):
    """A sorted sample of token ids: fixed ones, both ends, and uniform strata."""
    picks = set(int(x) for x in must if 0 <= x < T)
    picks.update([0, T - 1])
    edges = np.linspace(0, T, n + 1).astype(int)
    for a, b in zip(edges[:-1], edges[1:]):
        if b > a:
            picks.add(int(rng.integers(a, b)))
    return sorted(picks)
