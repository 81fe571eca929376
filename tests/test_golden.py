"""Fixtures of values the pages print (``tests/golden/``, each file citing its
page and section), checked on the CPU against the oracle and against the
workload definitions that the tests and the bench use."""

import os

import numpy as np
import torch

import bench
import oracle
from long_context_causal_gqa_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def _table(name):
    return {r[0]: [int(x) for x in r[1:]] for r in _lines(name)}


def test_sparse_tail_counts():
    """A row that selects only its own four-token block sees exactly the
    printed number of its tokens.  Equal scores (q = 0) make the output the
    mean of the visible V rows; V row t of the block is the unit vector e_(t -
    4 floor(p / 4)), so the output is 1 / count on the first count d and 0
    elsewhere.  The three rows after p exist in the cache (they are later
    rows' positions), so a clamp that let them through would show."""
    D, page, Hq = 16, 16, 6
    sentinel = D - 1
    for p_s, count_s in _lines("sparse_tail_counts.txt"):
        p, count = int(p_s), int(count_s)
        rows = 4
        ctx_len = p + rows                    # row 0 sits at position p
        n_pages = (ctx_len + page - 1) // page
        q = torch.zeros(rows, Hq, D, dtype=torch.float16)
        k = torch.zeros(n_pages, page, 1, D, dtype=torch.float16)
        v = torch.zeros(n_pages, page, 1, D, dtype=torch.float16)
        base = 4 * (p // 4)
        for t in range(ctx_len):
            d = t - base if base <= t < base + 4 else sentinel
            v[t // page, t % page, 0, d] = 1.0
        table = torch.arange(n_pages, dtype=torch.int32)
        sel = torch.tensor([[(p + r) // 4] for r in range(rows)], dtype=torch.int32)
        cnt = torch.ones(rows, dtype=torch.int32)
        out = oracle.sparse_blocks(q, k, v, table, sel, cnt, ctx_len, 1.0 / 16, rows=[0])
        want = np.zeros(D)
        want[:count] = 1.0 / count
        for h in range(Hq):
            assert np.allclose(out[0, h], want, rtol=0, atol=1e-15), (p, count, out[0, h])


def test_prefill_sweep_elements():
    g = {k: v[0] for k, v in _table("prefill_sweep_elements.txt").items()}
    kvs = list(range(g["kv_first"], g["kv_last"] + 1, g["kv_step"]))
    assert len(kvs) == g["shapes"]
    assert bench.KV_SWEEP == kvs
    # One D-vector per query row and query head: the output layout [Q, Hq, D].
    assert len(kvs) * g["Q"] * g["Hq"] * g["D"] == g["elements"]
    d = inputs.dense_inputs(5, 9, seed=0, D=16)
    assert oracle.dense(d.q, d.k, d.v, d.scale).shape == (5, g["Hq"], 16)


def test_paged_tail_workload():
    g = _table("paged_tail_workload.txt")
    cap, ctx, page, D = g["capacity"][0], g["ctx_len"][0], g["page"][0], g["D"][0]
    assert ctx <= cap
    assert (ctx + page - 1) // page == g["logical_pages"][0]
    assert cap // page == g["physical_pages"][0]
    assert (bench.TAIL_CAPACITY, bench.TAIL_CTX) == (cap, ctx)
    assert bench.tail_kv_bytes(ctx) == g["kv_bytes"][0] == 2 * ctx * D
    assert g["query_rows"] == list(range(1, 9))
    # The generator lays out capacity / page physical pages and maps the
    # ceil(ctx / page) logical ones into them (checked on a small instance).
    p = inputs.paged_e4m3_inputs(R=2, ctx_len=1000, capacity=2048, seed=0, page=page, D=16)
    assert p.kcache.shape[:2] == (2048 // page, page)
    assert p.block_table.numel() == (1000 + page - 1) // page
