"""Pins for the FP64 oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics
fix: a 40-digit ``decimal`` brute force written separately here from the
definition softmax(QK^T*scale + causal mask)V ("[Kernel][SM70] Default
long-prefill GQA architecture", Purpose), closed forms, invariants (rows of P
sum to one, masked keys do not matter), reductions of one variant to another,
and torch's float8_e4m3fn decoding as a library routine for the E4M3 codes.
"""

import decimal
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gqa_gb300 import inputs

decimal.getcontext().prec = 40
D_ = decimal.Decimal


def _f64(t):
    return t.to(torch.float64).numpy()


def _brute(qf, kf, vf, scale, visible_of):
    """Decimal brute force: qf [rows,Hq,D], kf/vf [N,Hkv,D] float64 arrays;
    visible_of(i) -> iterable of visible key indices of query row i."""
    rows, Hq, D = qf.shape
    Hkv = kf.shape[1]
    group = Hq // Hkv
    out = np.zeros((rows, Hq, D))
    sc = D_(repr(float(scale)))
    for i in range(rows):
        keys = sorted(set(visible_of(i)))
        for h in range(Hq):
            g = h // group
            if not keys:
                continue
            s = []
            for j in keys:
                acc = D_(0)
                for d in range(D):
                    acc += D_(float(qf[i, h, d])) * D_(float(kf[j, g, d]))
                s.append(acc * sc)
            m = max(s)
            w = [(x - m).exp() for x in s]
            den = sum(w)
            for d in range(D):
                num = sum(wj * D_(float(vf[j, g, d])) for wj, j in zip(w, keys))
                out[i, h, d] = float(num / den)
    return out


def _rand16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.float16)


# ---------------------------------------------------------------- E4M3 decode

def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


# ---------------------------------------------------------------- dense

@pytest.mark.parametrize("Q,KV,Hq,Hkv,D", [(3, 7, 6, 1, 8), (4, 9, 6, 2, 8), (2, 5, 6, 3, 4),
                                           (4, 4, 6, 1, 8), (1, 6, 6, 6, 3)])
def test_dense_matches_decimal_bruteforce(Q, KV, Hq, Hkv, D):
    q = _rand16((Q, Hq, D), 1, 2.0)
    k = _rand16((KV, Hkv, D), 2, 2.0)
    v = _rand16((KV, Hkv, D), 3)
    scale = 0.37
    got = oracle.dense(q, k, v, scale)
    ref = _brute(_f64(q), _f64(k), _f64(v), scale, lambda i: range(KV - Q + i + 1))
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_dense_row_subset_matches_full():
    q, k, v = _rand16((9, 6, 16), 4), _rand16((20, 1, 16), 5), _rand16((20, 1, 16), 6)
    full = oracle.dense(q, k, v, 0.25)
    part = oracle.dense(q, k, v, 0.25, rows=[8, 0, 3])
    assert np.array_equal(part, full[[8, 0, 3]])


def test_single_key_returns_its_value_exactly():
    q, k, v = _rand16((1, 6, 256), 7), _rand16((1, 1, 256), 8), _rand16((1, 1, 256), 9)
    got = oracle.dense(q, k, v, 1 / 16)
    assert np.array_equal(got, np.broadcast_to(_f64(v)[0:1], got.shape))


def test_one_hot_keys_closed_form():
    # k_j = e_j (basis rows), q = c * e_t: score_t = c*scale, every other score 0.
    Q, KV, D, c, scale = 5, 12, 16, 3.0, 0.5
    k = torch.zeros(KV, 1, D, dtype=torch.float16)
    for j in range(KV):
        k[j, 0, j] = 1.0
    v = _rand16((KV, 1, D), 10)
    q = torch.zeros(Q, 6, D, dtype=torch.float16)
    targets = {}
    for i in range(Q):
        for h in range(6):
            t = (3 * i + h) % KV  # some targets visible, some in the future
            q[i, h, t] = c
            targets[(i, h)] = t
    got = oracle.dense(q, k, v, scale)
    vf = _f64(v)[:, 0]
    E = math.exp(c * scale)
    for (i, h), t in targets.items():
        last = KV - Q + i
        n = last + 1
        if t <= last:
            ref = (E * vf[t] + vf[: n].sum(0) - vf[t]) / (E + n - 1)
        else:
            ref = vf[:n].mean(0)
        np.testing.assert_allclose(got[i, h], ref, rtol=1e-13, atol=1e-15)


def test_identical_keys_give_mean_of_visible_values():
    Q, KV, D = 4, 10, 32
    k = _rand16((1, 1, D), 11).repeat(KV, 1, 1)
    v = _rand16((KV, 1, D), 12)
    q = _rand16((Q, 6, D), 13, 3.0)
    got = oracle.dense(q, k, v, 1 / 16)
    vf = _f64(v)[:, 0]
    for i in range(Q):
        ref = vf[: KV - Q + i + 1].mean(0)
        for h in range(6):
            np.testing.assert_allclose(got[i, h], ref, rtol=1e-13, atol=1e-15)


def test_future_keys_do_not_change_output():
    Q, KV, D = 6, 15, 16
    q, k, v = _rand16((Q, 6, D), 14), _rand16((KV, 1, D), 15), _rand16((KV, 1, D), 16)
    base = oracle.dense(q, k, v, 0.3)
    for i in range(Q):
        last = KV - Q + i
        k2, v2 = k.clone(), v.clone()
        k2[last + 1:] = 7.0
        v2[last + 1:] = -5.0
        got = oracle.dense(q, k2, v2, 0.3, rows=[i])
        assert np.array_equal(got[0], base[i])
        # ...while the last visible key does matter.
        v3 = v.clone()
        v3[last] += 1.0
        assert not np.array_equal(oracle.dense(q, k, v3, 0.3, rows=[i])[0], base[i])


def test_probabilities_sum_to_one():
    Q, KV, D = 3, 50, 64
    q, k, v = _rand16((Q, 6, D), 17, 4.0), _rand16((KV, 1, D), 18), _rand16((KV, 1, D), 19)
    for row in range(Q):
        for head in (0, 5):
            p = oracle.dense_probs(q, k, v, 1 / 16, row, head)
            assert len(p) == KV - Q + row + 1
            assert abs(p.sum() - 1.0) < 1e-14 and (p > 0).all()


# ---------------------------------------------------------------- paged E4M3

def _decode_torch(cache):
    return cache.view(torch.float8_e4m3fn).to(torch.float64)


def _unpage(cache_f, table, ctx_len, page):
    """Logical [ctx_len, Hkv, D] view of a paged cache, via torch indexing."""
    n = (ctx_len + page - 1) // page
    return cache_f[table[:n].long()].reshape(n * page, *cache_f.shape[2:])[:ctx_len]


def test_paged_matches_decimal_bruteforce():
    inp = inputs.paged_e4m3_inputs(R=3, ctx_len=37, capacity=64, seed=3, page=16, D=8)
    got = oracle.paged_e4m3(inp.q, inp.kcache, inp.vcache, inp.kscale, inp.vscale,
                            inp.block_table, inp.ctx_len, 0.3)
    kf = _unpage(_decode_torch(inp.kcache), inp.block_table, 37, 16).numpy() * inp.kscale
    vf = _unpage(_decode_torch(inp.vcache), inp.block_table, 37, 16).numpy() * inp.vscale
    ref = _brute(_f64(inp.q), kf, vf, 0.3, lambda i: range(37 - 3 + i + 1))
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_paged_unit_scale_equals_dense_on_decoded_values():
    inp = inputs.paged_e4m3_inputs(R=8, ctx_len=300, capacity=512, seed=4, page=16, D=32)
    got = oracle.paged_e4m3(inp.q, inp.kcache, inp.vcache, 1.0, 1.0, inp.block_table,
                            inp.ctx_len, 1 / 16)
    # E4M3 values are exactly representable in fp16, so this dense input is exact.
    k16 = _unpage(_decode_torch(inp.kcache), inp.block_table, 300, 16).to(torch.float16)
    v16 = _unpage(_decode_torch(inp.vcache), inp.block_table, 300, 16).to(torch.float16)
    ref = oracle.dense(inp.q, k16, v16, 1 / 16)
    assert np.array_equal(got, ref)


def test_paged_scale_semantics_are_exact_powers_of_two():
    inp = inputs.paged_e4m3_inputs(R=2, ctx_len=100, capacity=128, seed=5, page=16, D=16)
    a = oracle.paged_e4m3(inp.q, inp.kcache, inp.vcache, inp.kscale, inp.vscale,
                          inp.block_table, 100, 1 / 16)
    b = oracle.paged_e4m3(inp.q, inp.kcache, inp.vcache, inp.kscale, 2 * inp.vscale,
                          inp.block_table, 100, 1 / 16)
    c = oracle.paged_e4m3(inp.q, inp.kcache, inp.vcache, 2 * inp.kscale, inp.vscale,
                          inp.block_table, 100, 1 / 32)
    assert np.array_equal(b, 2 * a)
    assert np.array_equal(c, a)


def test_paged_ignores_unreferenced_pages():
    inp = inputs.paged_e4m3_inputs(R=8, ctx_len=200, capacity=1024, seed=6, page=16, D=16)
    got = oracle.paged_e4m3(inp.q, inp.kcache, inp.vcache, inp.kscale, inp.vscale,
                            inp.block_table, 200, 1 / 16)
    assert np.isfinite(got).all()
    kc = inp.kcache.clone()
    used = set(inp.block_table.tolist())
    unused = [p for p in range(kc.shape[0]) if p not in used]
    kc[unused] = 0x11
    again = oracle.paged_e4m3(inp.q, kc, inp.vcache, inp.kscale, inp.vscale,
                              inp.block_table, 200, 1 / 16)
    assert np.array_equal(got, again)


# ---------------------------------------------------------------- sparse blocks

def _visible_sparse(sel, cnt, ctx_len, rows):
    def f(i):
        p = ctx_len - rows + i
        out = set()
        for b in sel[i, : cnt[i]].tolist():
            if b < 0:
                continue
            out.update(j for j in range(4 * b, 4 * b + 4) if j <= p)
        return out
    return f


def test_sparse_matches_decimal_bruteforce():
    inp = inputs.sparse_inputs(rows=5, ctx_len=41, tokens=12, seed=2, page=16, D=8)
    got = oracle.sparse_blocks(inp.q, inp.kcache, inp.vcache, inp.block_table, inp.sel_idx,
                               inp.sel_cnt, inp.ctx_len, 0.4)
    kf = _unpage(inp.kcache.to(torch.float64), inp.block_table, 41, 16).numpy()
    vf = _unpage(inp.vcache.to(torch.float64), inp.block_table, 41, 16).numpy()
    ref = _brute(_f64(inp.q), kf, vf, 0.4,
                 _visible_sparse(inp.sel_idx, inp.sel_cnt, 41, 5))
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def _all_blocks(rows, ctx_len):
    nb = (ctx_len + 3) // 4
    sel = torch.full((rows, nb), -1, dtype=torch.int32)
    cnt = torch.zeros(rows, dtype=torch.int32)
    for i in range(rows):
        p = ctx_len - rows + i
        n = p // 4 + 1
        sel[i, :n] = torch.arange(n, dtype=torch.int32)
        cnt[i] = n
    return sel, cnt


def test_sparse_with_every_block_equals_dense():
    rows, ctx_len = 7, 90
    inp = inputs.sparse_inputs(rows=rows, ctx_len=ctx_len, tokens=8, seed=7, page=16, D=16)
    sel, cnt = _all_blocks(rows, ctx_len)
    got = oracle.sparse_blocks(inp.q, inp.kcache, inp.vcache, inp.block_table, sel, cnt,
                               ctx_len, 1 / 16)
    k16 = _unpage(inp.kcache, inp.block_table, ctx_len, 16)
    v16 = _unpage(inp.vcache, inp.block_table, ctx_len, 16)
    ref = oracle.dense(inp.q, k16, v16, 1 / 16)
    assert np.array_equal(got, ref)


def test_sparse_clamps_the_rows_own_block():
    rows, ctx_len = 4, 64
    inp = inputs.sparse_inputs(rows=rows, ctx_len=ctx_len, tokens=16, seed=8, page=16, D=16)
    base = oracle.sparse_blocks(inp.q, inp.kcache, inp.vcache, inp.block_table, inp.sel_idx,
                                inp.sel_cnt, ctx_len, 1 / 16)
    # Row 0 sits at p = 60 (first token of block 15): tokens 61..63 must not count.
    kc, vc = inp.kcache.clone(), inp.vcache.clone()
    t = inp.block_table.long()
    for tok in (61, 62, 63):
        kc[t[tok // 16], tok % 16] = 9.0
        vc[t[tok // 16], tok % 16] = 9.0
    got = oracle.sparse_blocks(inp.q, kc, vc, inp.block_table, inp.sel_idx, inp.sel_cnt,
                               ctx_len, 1 / 16, rows=[0])
    assert np.array_equal(got[0], base[0])
    # Row 3 (p = 63) does see token 63.
    got3 = oracle.sparse_blocks(inp.q, kc, vc, inp.block_table, inp.sel_idx, inp.sel_cnt,
                                ctx_len, 1 / 16, rows=[3])
    assert not np.array_equal(got3[0], base[3])


def test_sparse_selection_order_and_out_of_range_ids():
    rows, ctx_len = 6, 200
    inp = inputs.sparse_inputs(rows=rows, ctx_len=ctx_len, tokens=40, seed=9, page=16, D=16)
    base = oracle.sparse_blocks(inp.q, inp.kcache, inp.vcache, inp.block_table, inp.sel_idx,
                                inp.sel_cnt, ctx_len, 1 / 16)
    g = torch.Generator().manual_seed(1)
    sel = inp.sel_idx.clone()
    for i in range(rows):
        n = int(inp.sel_cnt[i])
        sel[i, :n] = sel[i, :n][torch.randperm(n, generator=g)]
    shuffled = oracle.sparse_blocks(inp.q, inp.kcache, inp.vcache, inp.block_table, sel,
                                    inp.sel_cnt, ctx_len, 1 / 16)
    np.testing.assert_allclose(shuffled, base, rtol=1e-14, atol=1e-15)
    # Extra ids that are negative or past the row's own block select nothing.
    wide = torch.full((rows, inp.max_sel + 2), -1, dtype=torch.int32)
    wide[:, : inp.max_sel] = inp.sel_idx
    cnt = inp.sel_cnt.clone()
    for i in range(rows):
        n = int(cnt[i])
        p = ctx_len - rows + i
        wide[i, n] = p // 4 + 1
        wide[i, n + 1] = -3
        cnt[i] = n + 2
    got = oracle.sparse_blocks(inp.q, inp.kcache, inp.vcache, inp.block_table, wide, cnt,
                               ctx_len, 1 / 16)
    assert np.array_equal(got, base)


def test_sparse_ignores_nan_poisoned_pages_and_tokens():
    inp = inputs.sparse_inputs(rows=32, ctx_len=500, tokens=64, seed=10, page=16, D=16,
                               num_pages=64)
    got = oracle.sparse_blocks(inp.q, inp.kcache, inp.vcache, inp.block_table, inp.sel_idx,
                               inp.sel_cnt, inp.ctx_len, 1 / 16)
    assert np.isfinite(got).all()


# ---------------------------------------------------------------- generators

def test_sparse_selection_properties():
    rows, ctx, T = 300, 2048, 64
    sel, cnt, max_sel = inputs.sparse_selection(rows, ctx, T, seed=3)
    assert max_sel == T // 4
    for i in range(rows):
        p = ctx - rows + i
        n = int(cnt[i])
        ids = sel[i, :n].tolist()
        assert n == min(T // 4, p // 4 + 1)
        assert ids == sorted(set(ids)) and ids[-1] == p // 4 and ids[0] >= 0
        assert (sel[i, n:] == -1).all()


def test_e4m3_encoding_uses_absmax_over_448():
    x = torch.randn(1000, 1, 8, generator=torch.Generator().manual_seed(0))
    b, s = inputs.e4m3_encode(x)
    assert abs(s - float(x.abs().max()) / 448.0) <= 1e-7 * s
    dec = b.view(torch.float8_e4m3fn).to(torch.float32) * s
    assert dec.abs().max() <= 448.0 * s * (1 + 1e-6)
    assert (dec - x).abs().max() <= 0.0625 * x.abs().max()


def test_block_table_is_injective():
    t = inputs.permuted_block_table(100, 256, seed=1)
    assert len(set(t.tolist())) == 100 and int(t.min()) >= 0 and int(t.max()) < 256


# ---------------------------------------------------------------- sparse over an E4M3 cache

def test_sparse_e4m3_matches_decimal_bruteforce():
    inp = inputs.sparse_e4m3_inputs(rows=5, ctx_len=41, tokens=12, seed=2, page=16, D=8)
    got = oracle.sparse_blocks_e4m3(inp.q, inp.kcache, inp.vcache, inp.kscale, inp.vscale,
                                    inp.block_table, inp.sel_idx, inp.sel_cnt, inp.ctx_len, 0.4)
    kf = _unpage(_decode_torch(inp.kcache), inp.block_table, 41, 16).numpy() * inp.kscale
    vf = _unpage(_decode_torch(inp.vcache), inp.block_table, 41, 16).numpy() * inp.vscale
    ref = _brute(_f64(inp.q), kf, vf, 0.4, _visible_sparse(inp.sel_idx, inp.sel_cnt, 41, 5))
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_sparse_e4m3_with_every_block_equals_paged_tail():
    """Selecting every visible block turns the sparse visible set into the
    causal one, so the result is the E4M3 tail's over the same cache, bit for
    bit."""
    rows, ctx_len = 6, 300
    inp = inputs.sparse_e4m3_inputs(rows=rows, ctx_len=ctx_len, tokens=8, seed=5, page=16,
                                    D=32, num_pages=24)
    sel, cnt = _all_blocks(rows, ctx_len)
    got = oracle.sparse_blocks_e4m3(inp.q, inp.kcache, inp.vcache, inp.kscale, inp.vscale,
                                    inp.block_table, sel, cnt, ctx_len, 1 / 16)
    ref = oracle.paged_e4m3(inp.q, inp.kcache, inp.vcache, inp.kscale, inp.vscale,
                            inp.block_table, ctx_len, 1 / 16)
    assert np.array_equal(got, ref)


def test_sparse_e4m3_equals_fp16_sparse_on_decoded_values():
    """With power-of-two scales every decode(byte) * scale is exact in fp16,
    so the E4M3 sparse result equals the fp16 sparse result on the decoded
    cache, bit for bit."""
    inp = inputs.sparse_e4m3_inputs(rows=7, ctx_len=200, tokens=40, seed=6, page=16, D=16)
    ks, vs = 2.0 ** -4, 2.0 ** -3
    kd = (_decode_torch(inp.kcache) * ks).to(torch.float16)
    vd = (_decode_torch(inp.vcache) * vs).to(torch.float16)
    live = torch.isfinite(_decode_torch(inp.kcache))
    assert torch.equal(kd.to(torch.float64)[live], (_decode_torch(inp.kcache) * ks)[live])
    got = oracle.sparse_blocks_e4m3(inp.q, inp.kcache, inp.vcache, ks, vs, inp.block_table,
                                    inp.sel_idx, inp.sel_cnt, inp.ctx_len, 1 / 16)
    ref = oracle.sparse_blocks(inp.q, kd, vd, inp.block_table, inp.sel_idx, inp.sel_cnt,
                               inp.ctx_len, 1 / 16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- dense over E4M3

def test_dense_e4m3_matches_decimal_bruteforce():
    inp = inputs.dense_e4m3_inputs(Q=3, KV=11, seed=9, D=8)
    got = oracle.dense_e4m3(inp.q, inp.k, inp.v, inp.kscale, inp.vscale, 0.3)
    kf = _decode_torch(inp.k).numpy() * inp.kscale
    vf = _decode_torch(inp.v).numpy() * inp.vscale
    ref = _brute(_f64(inp.q), kf, vf, 0.3, lambda i: range(11 - 3 + i + 1))
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_dense_e4m3_unit_scales_equal_dense_on_decoded_values():
    """With scales 1 the E4M3 values are exact fp16 values: the dense fp16
    oracle on them gives bit-identical results."""
    inp = inputs.dense_e4m3_inputs(Q=40, KV=300, seed=10, Hq=6, Hkv=2, D=32)
    got = oracle.dense_e4m3(inp.q, inp.k, inp.v, 1.0, 1.0, 1 / 16)
    ref = oracle.dense(inp.q, _decode_torch(inp.k).to(torch.float16),
                       _decode_torch(inp.v).to(torch.float16), 1 / 16)
    assert np.array_equal(got, ref)


def test_dense_e4m3_equals_paged_tail_on_a_permuted_layout():
    """The same codes stored in permuted page-16 blocks and read through the
    block table give bit-identical rows (the paged tail's arithmetic)."""
    inp = inputs.dense_e4m3_inputs(Q=5, KV=77, seed=11, D=16)
    page, n_log = 16, (77 + 15) // 16
    table = inputs.permuted_block_table(n_log, n_log + 3, seed=12)
    kc = torch.full((n_log + 3, page, 1, 16), 0x7F, dtype=torch.uint8)
    vc = torch.full((n_log + 3, page, 1, 16), 0x7F, dtype=torch.uint8)
    for t in range(77):
        kc[table[t // page], t % page] = inp.k[t]
        vc[table[t // page], t % page] = inp.v[t]
    a = oracle.dense_e4m3(inp.q, inp.k, inp.v, inp.kscale, inp.vscale, 1 / 16)
    b = oracle.paged_e4m3(inp.q, kc, vc, inp.kscale, inp.vscale, table, 77, 1 / 16)
    assert np.array_equal(a, b)
