"""Writes the regression fixtures in this folder.  Calls only ``oracle/`` and
the seeded generator ``synth/``; nothing here comes from the CUDA path.

    python tests/golden/make_golden.py

tiny_sparse_case.json: per-token sparse prefill on a 6-token, 20-row case
with D_QK = 24 (16 "NoPE" + 8 "RoPE") and D_V = 16, -1 anywhere in the rows
and a row wider than k (the definition of the per-token form: "[Perf][DSA]
Grouped sparse prefill with the FlashMLA head-group-mask kernel", commit
message), plus the union/mask of the same indices for G = 2 (same page, How).
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle.dsa_oracle as O  # noqa: E402
from synth import normal_bf16  # noqa: E402


def tiny_case():
    rng = np.random.default_rng(1234)
    T, N, H, d_qk, d_v, k, ld = 6, 20, 2, 24, 16, 7, 9
    q = normal_bf16(rng, (T, H, d_qk))
    kv = normal_bf16(rng, (N, d_qk))
    idx = np.full((T, ld), -1, dtype=np.int32)
    for t in range(T):
        n = int(rng.integers(0, k + 1))
        idx[t, rng.choice(k, size=n, replace=False)] = rng.choice(N, size=n, replace=False)
        idx[t, k:] = rng.integers(-1, N, size=ld - k)
    scale = 0.25
    out, lse = O.sparse_prefill(q, kv, idx, k, scale, d_qk, d_v)
    upad = O.union_pad(2, k, 4)
    u, ul, m = O.union_build(idx, k, 2, N, [0, T], upad)
    return dict(
        citation="per-token definition and union/mask: '[Perf][DSA] Grouped sparse prefill with the "
                 "FlashMLA head-group-mask kernel', commit message and How",
        T=T, N=N, H=H, d_qk=d_qk, d_v=d_v, k=k, ld=ld, scale=scale, G=2, union_block=4,
        q_bits=q.tolist(), kv_bits=kv.tolist(), idx=idx.tolist(),
        out=np.round(out, 15).tolist(), lse=[[None if not np.isfinite(x) else float(x) for x in r] for r in lse],
        union=u.tolist(), union_len=ul.tolist(), mask=m.tolist())


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_sparse_case.json"), "w") as f:
        json.dump(tiny_case(), f, indent=None, separators=(",", ":"))
    print("wrote tiny_sparse_case.json")
