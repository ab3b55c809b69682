"""Golden regression fixture of the oracle, and properties of the seeded
workload generators (shape, causality, -1 padding, union size)."""
import json
import os

import numpy as np
import pytest

import oracle.dsa_oracle as O
from synth import WORKLOADS, locality_topk, make_indices, uniform_topk, scaled_down

HERE = os.path.dirname(os.path.abspath(__file__))


def test_golden_tiny_case_reproduces():
    d = json.load(open(os.path.join(HERE, "golden", "tiny_sparse_case.json")))
    q = np.array(d["q_bits"], dtype=np.uint16)
    kv = np.array(d["kv_bits"], dtype=np.uint16)
    idx = np.array(d["idx"], dtype=np.int32)
    out, lse = O.sparse_prefill(q, kv, idx, d["k"], d["scale"], d["d_qk"], d["d_v"])
    assert np.max(np.abs(out - np.array(d["out"]))) < 1e-12
    want = np.array([[-np.inf if x is None else x for x in r] for r in d["lse"]])
    assert np.array_equal(np.isinf(lse), np.isinf(want))
    f = np.isfinite(want)
    assert np.max(np.abs(lse[f] - want[f])) < 1e-12
    u, ul, m = O.union_build(idx, d["k"], d["G"], d["N"], [0, d["T"]], O.union_pad(d["G"], d["k"], d["union_block"]))
    assert u.tolist() == d["union"] and ul.tolist() == d["union_len"] and m.tolist() == d["mask"]


def test_uniform_generator_causal_and_counts():
    rng = np.random.default_rng(0)
    pos = np.arange(300)
    idx = uniform_topk(rng, pos, 128, 130, kv_offset=5)
    for t in range(300):
        v = idx[t][idx[t] >= 0] - 5
        assert len(v) == min(t + 1, 128)
        assert len(np.unique(v)) == len(v)
        assert v.max() <= t and v.min() >= 0
        assert np.all(idx[t, len(v):] == -1)


@pytest.mark.parametrize("wide", [False, True])
def test_locality_generator_union_and_causality(wide):
    rng = np.random.default_rng(1)
    pos = np.arange(6000, 6400)
    idx = locality_topk(rng, pos, 2048, 2176, wide=wide)
    for t in range(0, 400, 37):
        v = idx[t][idx[t] >= 0]
        assert len(v) == 2048 and len(np.unique(v)) == 2048
        assert v.max() <= pos[t]
        assert np.all(idx[t, 2048:] == -1)
    us = [len(np.unique(idx[g:g + 8][idx[g:g + 8] >= 0])) for g in range(0, 400, 8)]
    if wide:
        assert np.mean(us) > 3000
    else:
        assert 2300 <= np.mean(us) <= 2400


def test_locality_dense_below_k():
    rng = np.random.default_rng(2)
    idx = locality_topk(rng, np.arange(0, 64), 32, 32)
    for t in range(64):
        v = np.sort(idx[t][idx[t] >= 0])
        if t + 1 <= 32:
            assert np.array_equal(v, np.arange(t + 1))
        else:
            assert len(v) == 32


def test_workload_table_shapes():
    w = WORKLOADS["grouped_21k_of_32k"]
    assert w.T == 21504 and w.N == 32768 and w.positions()[0][0] == 11264
    w = WORKLOADS["nope_2x8192"]
    assert w.ld == 2176 and w.d_qk == 512 and list(w.cu_seqlens_kv()) == [0, 8192, 16384]
    small = scaled_down(w, (40, 33), (40, 33), k=16, ld=20)
    idx = make_indices(small, np.random.default_rng(0))
    assert idx.shape == (73, 20)
    # second request's indices are offset into its own KV rows
    assert idx[40:][idx[40:] >= 0].min() >= 40
