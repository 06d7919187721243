"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

Each test ties an oracle function to something other than the oracle itself:
values printed on the pages (tests/golden), closed forms, library routines,
brute force on tiny inputs, or invariants.  All run on the CPU.
"""
import math
import os
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden
import workloads as W

NEG_INF = float("-inf")


# ---------------------------------------------------------------- mask ----

def _bits_to_dense(mask_row, n):
    return np.array([(int(mask_row[v // 64]) >> (v % 64)) & 1 for v in range(n)], dtype=np.int64)


def test_mask_matches_printed_6node_example(oracle):
    g = read_golden("specinfer_mask_6node.txt")
    parent = np.array([int(x) for x in g[0][1]], np.int32)
    printed = np.array([[0.0 if x == "0" else NEG_INF for x in row] for k, row in g[1:]])
    mask, depth, status = oracle.mask_build(parent, [0, 6], 6)
    assert status.tolist() == [0]
    got = np.array([[0.0 if b else NEG_INF for b in _bits_to_dense(mask[u], 6)] for u in range(6)])
    assert np.array_equal(got, printed)
    assert depth.tolist() == [0, 1, 1, 2, 2, 2]


def test_mask_chain_is_lower_triangular(oracle):
    for n in (1, 2, 63, 64, 65, 130):
        parent = W.chain_tree(n).numpy()
        mask, depth, status = oracle.mask_build(parent, [0, n], n)
        dense = np.stack([_bits_to_dense(mask[u], n) for u in range(n)])
        assert np.array_equal(dense, np.tril(np.ones((n, n), np.int64)))
        assert depth.tolist() == list(range(n))


def _closure(parent):
    """Ancestor-or-self relation by boolean transitive closure of the parent
    adjacency (A[u][p] = 1), computed by repeated squaring."""
    n = len(parent)
    A = np.zeros((n, n), bool)
    for u in range(1, n):
        A[u, parent[u]] = True
    R = np.eye(n, dtype=bool) | A
    for _ in range(int(math.ceil(math.log2(max(n, 2)))) + 1):
        R = R | ((R.astype(np.int64) @ R.astype(np.int64)) > 0)
    return R


def test_mask_bruteforce_closure_random_trees(oracle):
    rng = np.random.default_rng(5)
    for n in (1, 5, 17, 64, 65, 200):
        gen = np.random.Generator(np.random.PCG64(n))
        parent = W.random_parent_tree(n, gen).numpy()
        tree_off = [0, n]
        mask, depth, status = oracle.mask_build(parent, tree_off, 256)
        assert status.tolist() == [0]
        R = _closure(parent)
        dense = np.stack([_bits_to_dense(mask[u], n) for u in range(n)]).astype(bool)
        assert np.array_equal(dense, R)
        assert np.array_equal(depth, R.sum(axis=1) - 1)
        # words beyond n are zero
        for u in range(n):
            for v in range(n, 256):
                assert (int(mask[u][v // 64]) >> (v % 64)) & 1 == 0
    del rng


def test_mask_ragged_batch_and_bad_trees(oracle):
    trees = [np.array([-1, 0, 0], np.int32), np.array([0, 0], np.int32),  # root not -1
             np.array([-1, 1], np.int32),  # parent not before child
             np.zeros(0, np.int32), np.array([-1, 0, 1, 2, 3], np.int32)]
    parent = np.concatenate(trees)
    tree_off = np.cumsum([0] + [len(t) for t in trees]).astype(np.int32)
    mask, depth, status = oracle.mask_build(parent, tree_off, 4)  # last tree exceeds n_max = 4
    assert status.tolist() == [0, oracle.ST_BAD_TREE, oracle.ST_BAD_TREE, 0, oracle.ST_BAD_TREE]
    assert depth[:3].tolist() == [0, 1, 1]
    assert depth[3:7].tolist() == [-1] * 4 and (mask[3:7] == 0).all()
    assert depth[7:].tolist() == [-1] * 5


# ----------------------------------------------------------- attention ----

def _gathered_causal_reference(w, out_rows=None):
    """Independent fp64 routine: for node u, gather the sequence S_u = prefix
    followed by the root path to u (K/V rows in sequence order) and take the
    last position of plain causal attention over it."""
    def f64(t):
        return t.to(torch.float64).numpy()
    q, k, v = f64(w.q), f64(w.k_cache), f64(w.v_cache)
    bt, bs, g = w.block_table.numpy(), w.block_size, w.Hq // w.Hkv
    res = {}
    for b in range(w.B):
        off, n, P = int(w.tree_off[b]), int(w.tree_off[b + 1] - w.tree_off[b]), int(w.prefix_len[b])
        par = w.parent[off:off + n].numpy()
        for u in range(n):
            path = []
            c = u
            while c != -1:
                path.append(c)
                c = par[c]
            seq_slots = list(range(P)) + [P + x for x in reversed(path)]
            blk = bt[b][np.array(seq_slots) // bs]
            row = np.array(seq_slots) % bs
            for h in range(w.Hq):
                t = (off + u) * w.Hq + h
                if out_rows is not None and t not in out_rows:
                    continue
                K = k[blk, h // g, row]
                Vv = v[blk, h // g, row]
                s = K @ q[off + u, h] * w.scale
                p = np.exp(s - s.max())
                res[t] = (p / p.sum()) @ Vv
    return res


def _run_oracle_attn(oracle, w, rows=None):
    def arr(t):
        return t.numpy() if w.dtype == W.F32 else t.view(torch.int16).numpy().view(np.uint16)
    return oracle.tree_attention(arr(w.q), arr(w.k_cache), arr(w.v_cache), w.block_table.numpy(), w.block_size,
                                 w.prefix_len.numpy(), w.tree_off.numpy(), w.parent.numpy(), w.n_max, w.Hq, w.Hkv,
                                 w.D, w.dtype, w.scale, rows=rows, want_f64=True)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_attention_equals_causal_attention_over_gathered_sequence(oracle, dtype):
    w = W.small_random(11, B=3, n_range=(1, 12), prefix_range=(0, 40), Hq=4, Hkv=2, D=16, dtype=dtype, block_size=8)
    out, out64, status = _run_oracle_attn(oracle, w)
    assert status.tolist() == [0, 0, 0]
    ref = _gathered_causal_reference(w)
    got = out64.reshape(-1, w.D)
    for t, r in ref.items():
        np.testing.assert_allclose(got[t], r, rtol=0, atol=1e-12)


def test_attention_chain_with_empty_prefix_is_causal_self_attention(oracle):
    """A chain tree with no prefix is textbook causal self-attention."""
    n, Hq, Hkv, D = 23, 4, 4, 16
    gen = np.random.Generator(np.random.PCG64(3))
    w = W.gen._pack("chain", 1, Hq, Hkv, D, W.F32, 7, n, 8, [W.chain_tree(n)],
                    [torch.zeros(n, dtype=torch.int32)], [0], gen, None, None)
    out, out64, status = _run_oracle_attn(oracle, w)
    # sequence order: slot i holds chain node i
    K = torch.stack([w.k_cache[w.block_table[0, i // 8], :, i % 8] for i in range(n)], 1)  # [Hkv, n, D]
    V = torch.stack([w.v_cache[w.block_table[0, i // 8], :, i % 8] for i in range(n)], 1)
    Q = w.q.permute(1, 0, 2)  # [Hq, n, D]
    ref = torch.nn.functional.scaled_dot_product_attention(Q.double(), K.double(), V.double(), is_causal=True)
    np.testing.assert_allclose(out64.transpose(1, 0, 2), ref.numpy(), rtol=0, atol=1e-12)


def test_attention_zero_query_is_mean_of_visible_values(oracle):
    w = W.small_random(12, B=2, n_range=(3, 9), prefix_range=(0, 20), Hq=2, Hkv=1, D=8, dtype=W.F32, block_size=4)
    w.q.zero_()
    out, out64, status = _run_oracle_attn(oracle, w)
    vv = w.v_cache.double().numpy()
    for b in range(w.B):
        off, n, P = int(w.tree_off[b]), int(w.tree_off[b + 1] - w.tree_off[b]), int(w.prefix_len[b])
        par = w.parent[off:off + n].numpy()
        for u in range(n):
            anc = {u}
            c = par[u]
            while c != -1:
                anc.add(c)
                c = par[c]
            slots = list(range(P)) + [P + a for a in sorted(anc)]
            rows = np.stack([vv[w.block_table[b, s // 4], 0, s % 4] for s in slots])
            for h in range(2):
                np.testing.assert_allclose(out64[off + u, h], rows.mean(0), rtol=0, atol=1e-12)


def test_attention_row_subset_and_bad_requests(oracle):
    w = W.small_random(13, B=3, n_range=(2, 6), prefix_range=(5, 30), Hq=4, Hkv=2, D=8, dtype=W.BF16, block_size=8)
    full, _, st = _run_oracle_attn(oracle, w)
    rows = np.array([0, 5, w.T * 4 - 1], np.int64)
    sub, _, st2 = _run_oracle_attn(oracle, w, rows=rows)
    flat_f, flat_s = full.reshape(-1, 8), sub.reshape(-1, 8)
    for r in rows:
        assert np.array_equal(flat_f[r], flat_s[r])
    # capacity: prefix beyond the block table; bad block id
    w.prefix_len[0] = w.block_table.shape[1] * 8
    w.block_table[1, 0] = w.num_blocks + 3
    _, _, st3 = _run_oracle_attn(oracle, w)
    assert st3[0] & oracle.ST_CAPACITY and st3[1] & oracle.ST_BAD_BLOCK and st3[2] == 0


def test_bf16_rounding_is_exact_round_to_nearest_even(oracle):
    rng = np.random.default_rng(9)
    xs = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000))
    # ties between two bf16 values: odd and even lower neighbours
    xs += [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -133 * 1.5, 2.0 ** -133 * 2.5,
           2.0 ** -133 * 0.5, 2.0 ** -134 * 1.0000001, 3.3895313892515355e38, 3.39e38, 0.0]

    def bf16_value(bits):
        f = np.array([bits << 16], np.uint32).view(np.float32)[0]
        return Fraction(float(f))

    for x in xs:
        bits = oracle.f64_to_bf16_bits(x)
        fx = Fraction(x)
        if abs(x) > 3.3895313892515355e38 * (1 + 2 ** -9):
            assert bits & 0x7fff == 0x7f80
            continue
        got = bf16_value(bits)
        # neighbours one bf16 ulp away (bit patterns are monotone in magnitude)
        mag = bits & 0x7fff
        sign = bits & 0x8000
        cands = [m for m in (mag - 1, mag, mag + 1) if 0 <= m < 0x7f80]
        errs = [abs(bf16_value(sign | m) - fx) for m in cands]
        best = min(errs)
        assert abs(got - fx) == best
        if errs.count(best) > 1:  # exact tie: even mantissa wins
            assert mag % 2 == 0


# -------------------------------------------------------------- greedy ----

def test_greedy_adapted_harness_example(oracle):
    g = dict(read_golden("specinfer_greedy_harness.txt")[:3])
    entries = read_golden("specinfer_greedy_harness.txt")
    V = int(g["vocab"][0])
    parent = np.array([int(x) for x in g["parent"]], np.int32)
    tokens = np.array([int(x) for x in g["tokens"]], np.int32)
    logits = np.random.default_rng(0).standard_normal((3, V)).astype(np.float32)
    for k, v in entries:
        if k == "peak":
            logits[int(v[0]), int(v[1])] = float(v[2])
    exp_path = [int(x) for k, v in entries if k == "expect_path" for x in v]
    exp_emit = [int(x) for k, v in entries if k == "expect_emitted" for x in v]
    r = oracle.verify_greedy(logits, tokens, parent, [0, 3], 3)
    assert r["status"].tolist() == [0]
    assert r["accept_len"][0] == len(exp_path) and r["n_emitted"][0] == len(exp_emit)
    assert r["path"][0, :len(exp_path)].tolist() == exp_path
    assert r["emitted"][0, :len(exp_emit)].tolist() == exp_emit


def test_greedy_bruteforce_longest_matching_root_path(oracle):
    """Enumerate every root path; the accepted one is the longest whose
    tokens follow the target argmax chain (ties: lowest end-node index)."""
    rng = np.random.default_rng(21)
    for trial in range(300):
        n = int(rng.integers(1, 14))
        V = int(rng.integers(2, 5))
        gen = np.random.Generator(np.random.PCG64(trial))
        parent = W.random_parent_tree(n, gen).numpy()
        tokens = rng.integers(0, V, n).astype(np.int32)
        logits = rng.integers(-3, 3, (n, V)).astype(np.float32)  # many ties
        a = [int(np.flatnonzero(row == row.max())[0]) for row in logits]
        best, best_len = 0, 1
        for u in range(n):
            path = []
            c = u
            while c != -1:
                path.append(c)
                c = parent[c]
            path.reverse()
            if all(tokens[path[i + 1]] == a[path[i]] for i in range(len(path) - 1)) and len(path) > best_len:
                best, best_len = u, len(path)
        path = []
        c = best
        while c != -1:
            path.append(c)
            c = parent[c]
        path.reverse()
        r = oracle.verify_greedy(logits, tokens, parent, [0, n], n)
        assert r["accept_len"][0] == best_len
        assert r["path"][0, :best_len].tolist() == path
        assert r["emitted"][0, :best_len].tolist() == [int(tokens[p]) for p in path[1:]] + [a[best]]
        assert (r["path"][0, best_len:] == -1).all()


def test_greedy_chain_is_linear_greedy_speculation(oracle):
    rng = np.random.default_rng(4)
    for _ in range(100):
        K, V = int(rng.integers(1, 9)), 5
        n = K + 1
        logits = rng.standard_normal((n, V)).astype(np.float32)
        a = logits.argmax(1)
        tokens = np.where(rng.random(n) < 0.7, np.r_[0, a[:-1]], rng.integers(0, V, n)).astype(np.int32)
        accepted = 0
        while accepted < K and tokens[accepted + 1] == a[accepted]:
            accepted += 1
        r = oracle.verify_greedy(logits, tokens, W.chain_tree(n).numpy(), [0, n], n)
        assert r["accept_len"][0] == accepted + 1
        assert r["emitted"][0, accepted] == a[accepted]


def test_greedy_rejects_bad_tokens_and_trees(oracle):
    logits = np.zeros((5, 4), np.float32)
    parent = np.array([-1, 0, -1, 0, 1], np.int32)
    tokens = np.array([0, 1, 0, 9, 0], np.int32)
    r = oracle.verify_greedy(logits, tokens, parent, [0, 2, 3, 5], 3)
    assert r["status"].tolist() == [0, 0, oracle.ST_BAD_TOKEN | oracle.ST_BAD_TREE]
    assert r["accept_len"].tolist() == [1, 1, 0] and r["n_emitted"][2] == 0
    assert (r["path"][2] == -1).all() and (r["emitted"][2] == -1).all()


# ---------------------------------------------------------- stochastic ----

def _acc_word(u):
    """Raw acceptance word whose uniform (w >> 8) * 2^-24 equals u (u a multiple of 2^-24)."""
    return np.uint32(int(round(u * 2 ** 24)) << 8)


def _one_child_case(oracle, p, q, x, u_acc, U):
    V = len(p)
    logits = np.log(np.array([p, p], np.float64)).astype(np.float32)
    qp = np.array([q, q], np.float32)
    uni = np.array([[0, 0], [_acc_word(u_acc), 0]], np.uint32)
    uni[0, 1] = U
    r = oracle.verify_stochastic(logits, qp, np.array([0, x], np.int32), np.array([-1, 0], np.int32), [0, 2], uni, 2)
    return r


@pytest.mark.parametrize("example", ["a", "b"])
def test_stochastic_per_token_examples(oracle, example):
    ents = read_golden("inference_opt_accept_examples.txt")
    start = ents.index(("example", [example]))
    d = dict(ents[start + 1:start + 6])
    q = [float(v) for v in d["q"]]
    p = [float(v) for v in d["p"]]
    x = int(d["x"][0])
    acc = float(d["accept_prob"][0])
    resid = np.array([float(v) for v in d["residual"]])
    # acceptance probability: accepted just below it, rejected just above
    below, above = acc - 2 ** -10, acc + 2 ** -10
    assert _one_child_case(oracle, p, q, x, below, 0)["path"][0, 1] == 1
    rej = _one_child_case(oracle, p, q, x, above, 0)
    assert rej["accept_len"][0] == 1
    # residual after the rejection (C5 values within a few fp32 ulp)
    logits = np.log(np.array(p, np.float64)).astype(np.float32)
    r1, d1, S1 = oracle.residual(logits, np.array(q, np.float32), 1)
    np.testing.assert_allclose(r1, resid, rtol=0, atol=4e-7)
    # the resample follows the residual: the emitted token's CDF interval holds U
    cdf = np.cumsum(resid)
    for U in [0, 1, 2 ** 31, 2 ** 32 - 1] + list(np.random.default_rng(1).integers(0, 2 ** 32, 200)):
        tok = _one_child_case(oracle, p, q, x, above, np.uint32(U))["emitted"][0, 0]
        u = int(U) / 2 ** 32
        expect = int(np.searchsorted(cdf, u, side="right"))
        if min(abs(cdf - u)) > 1e-6:
            assert tok == expect
        assert resid[tok] > 0


def _p_row(key, V):
    rng = np.random.default_rng(key)
    return rng.dirichlet(np.full(V, 0.7))


def mc_tree_inputs(n_trials, V, root_kids, kid_kids, seed, per_child=False):
    """Inputs of n_trials depth-2 trees whose draft tokens are i.i.d. draws
    from the parent's draft row; p and q rows are fixed functions of the token
    path.  Returns (dict of verifier inputs, table of p rows by path).
    per_child: each sibling is drawn from a row of its own (the i-th child
    of a node from draft model i, as in a merged tree), and q_probs row c is
    the row child c was drawn from."""
    if per_child:
        return _mc_tree_inputs_per_child(n_trials, V, root_kids, kid_kids, seed)
    rng = np.random.default_rng(seed)
    key0 = seed * 1000

    def p_of(path):
        return _p_row((key0, 1) + tuple(path), V)

    def q_of(path):
        return _p_row((key0, 2) + tuple(path), V)

    n = 1 + root_kids + root_kids * kid_kids
    parent = [-1] + [0] * root_kids + [1 + i for i in range(root_kids) for _ in range(kid_kids)]
    parent = np.array(parent, np.int32)
    P1 = {(): p_of(())}
    Q1 = {(): q_of(())}
    for a in range(V):
        P1[(a,)] = p_of((a,))
        Q1[(a,)] = q_of((a,))
        for b in range(V):
            P1[(a, b)] = p_of((a, b))
    # draft tokens
    t1 = np.stack([rng.choice(V, n_trials, p=Q1[()]) for _ in range(root_kids)], 1)  # [N, root_kids]
    t2 = np.zeros((n_trials, root_kids, kid_kids), np.int64)
    for a in range(V):
        sel = t1 == a
        cnt = int(sel.sum())
        t2[sel] = rng.choice(V, (cnt, kid_kids), p=Q1[(a,)])
    tokens = np.concatenate([np.zeros((n_trials, 1), np.int64), t1, t2.reshape(n_trials, -1)], 1).astype(np.int32)
    # rows: p_logits = log p(.|S_u), q_probs = q(.|S_u)
    logp = np.zeros((n_trials, n, V), np.float32)
    qpr = np.zeros((n_trials, n, V), np.float32)
    logp[:, 0] = np.log(P1[()])
    qpr[:, 0] = Q1[()]
    for a in range(V):
        logp[:, 1:1 + root_kids][t1 == a] = np.log(P1[(a,)])
        qpr[:, 1:1 + root_kids][t1 == a] = Q1[(a,)]
    for a in range(V):
        for b in range(V):
            sel = (t1[:, :, None] == a) & (t2 == b)
            flat = sel.reshape(n_trials, -1)
            logp[:, 1 + root_kids:][flat] = np.log(P1[(a, b)])
    uni = rng.integers(0, 2 ** 32, (n_trials * n, 2), dtype=np.uint64).astype(np.uint32)
    inputs = dict(p_logits=logp.reshape(-1, V), q_probs=qpr.reshape(-1, V), tokens=tokens.reshape(-1),
                  parent=np.tile(parent, n_trials), tree_off=np.arange(0, n * n_trials + 1, n, dtype=np.int32),
                  uniforms=uni, n_max=n)
    return inputs, P1


def _mc_tree_inputs_per_child(n_trials, V, root_kids, kid_kids, seed):
    rng = np.random.default_rng(seed)
    key0 = seed * 1000 + 500

    def p_of(path):
        return _p_row((key0, 1) + tuple(path), V)

    def qk(i, path):  # draft model i's row after the token path
        return _p_row((key0, 3, i) + tuple(path), V)

    n = 1 + root_kids + root_kids * kid_kids
    parent = np.array([-1] + [0] * root_kids + [1 + i for i in range(root_kids) for _ in range(kid_kids)], np.int32)
    P1 = {(): p_of(())}
    for a in range(V):
        P1[(a,)] = p_of((a,))
        for b in range(V):
            P1[(a, b)] = p_of((a, b))
    t1 = np.stack([rng.choice(V, n_trials, p=qk(i, ())) for i in range(root_kids)], 1)
    t2 = np.zeros((n_trials, root_kids, kid_kids), np.int64)
    for a in range(V):
        sel = t1 == a
        cnt = int(sel.sum())
        t2[sel] = np.stack([rng.choice(V, cnt, p=qk(j, (a,))) for j in range(kid_kids)], 1)
    tokens = np.concatenate([np.zeros((n_trials, 1), np.int64), t1, t2.reshape(n_trials, -1)], 1).astype(np.int32)
    logp = np.zeros((n_trials, n, V), np.float32)
    qpr = np.zeros((n_trials, n, V), np.float32)
    logp[:, 0] = np.log(P1[()])
    qpr[:, 0] = 1.0 / V  # the root's own row is never read
    for i in range(root_kids):
        qpr[:, 1 + i] = qk(i, ())
    for a in range(V):
        logp[:, 1:1 + root_kids][t1 == a] = np.log(P1[(a,)])
        for i in range(root_kids):
            for j in range(kid_kids):
                qpr[t1[:, i] == a, 1 + root_kids + i * kid_kids + j] = qk(j, (a,))
        for b in range(V):
            flat = ((t1[:, :, None] == a) & (t2 == b)).reshape(n_trials, -1)
            logp[:, 1 + root_kids:][flat] = np.log(P1[(a, b)])
    uni = rng.integers(0, 2 ** 32, (n_trials * n, 2), dtype=np.uint64).astype(np.uint32)
    inputs = dict(p_logits=logp.reshape(-1, V), q_probs=qpr.reshape(-1, V), tokens=tokens.reshape(-1),
                  parent=np.tile(parent, n_trials), tree_off=np.arange(0, n * n_trials + 1, n, dtype=np.int32),
                  uniforms=uni, n_max=n)
    return inputs, P1


def _run_mc_tree(oracle, n_trials, V, root_kids, kid_kids, seed):
    inputs, P1 = mc_tree_inputs(n_trials, V, root_kids, kid_kids, seed)
    return oracle.verify_stochastic(**inputs), P1


def _chisq_pvalue(counts, probs):
    from scipy.special import gammaincc
    N = counts.sum()
    exp = probs * N
    keep = exp > 0
    stat = float((((counts - exp) ** 2)[keep] / exp[keep]).sum())
    dof = int(keep.sum()) - 1
    return float(gammaincc(dof / 2.0, stat / 2.0))


@pytest.mark.parametrize("seed,root_kids,kid_kids", [(1, 3, 2), (2, 3, 2), (3, 2, 3), (4, 1, 2), (5, 3, 1)])
def test_stochastic_emits_target_distribution(oracle, seed, root_kids, kid_kids):
    """Monte-Carlo check of losslessness ("Inference Optimization Techniques",
    the two-case proof in the "Misconception" section): the first emitted token
    follows p(.|root), and, when the first token was an accepted draft x, the
    second follows p(.|x)."""
    V, N = 8, 200_000
    r, P = _run_mc_tree(oracle, N, V, root_kids, kid_kids, seed)
    assert (r["status"] == 0).all()
    first = r["emitted"][:, 0]
    assert _chisq_pvalue(np.bincount(first, minlength=V), P[()]) > 1e-4
    cont = r["accept_len"] >= 2
    for x in range(V):
        sel = cont & (first == x)
        if sel.sum() < 2000:
            continue
        second = r["emitted"][sel, 1]
        assert _chisq_pvalue(np.bincount(second, minlength=V), P[(x,)]) > 1e-4, x


def _tempered(p, tau):
    w = np.asarray(p, np.float64) ** tau
    return w / w.sum()


def _softmax64(l, tau=1.0):
    z = np.asarray(l, np.float64) * tau
    e = np.exp(z - z.max())
    return e / e.sum()


@pytest.mark.parametrize("tau", [0.25, 0.5, 1.0, 2.0, 3.7])
def test_temperature_target_is_tempered_softmax(oracle, tau):
    """Sampling at temperature T ("Stochastic Verification Algorithm"): the
    row's target is softmax(l / T), here with tau = 1/T; after a rejection the
    residual is norm(max(softmax(l tau) - q, 0)) (fp64 closed forms)."""
    rng = np.random.default_rng(int(tau * 100))
    V = 1000
    l = (3.0 * rng.standard_normal(V)).astype(np.float32)
    q = rng.dirichlet(np.full(V, 0.3)).astype(np.float32)
    r0, _, _ = oracle.residual(l, q, 0, tau)
    ref0 = _softmax64(l, tau)
    np.testing.assert_allclose(r0, ref0, rtol=2e-5, atol=1e-12)
    r1, _, _ = oracle.residual(l, q, 1, tau)
    d = np.maximum(ref0 - q.astype(np.float64), 0)
    np.testing.assert_allclose(r1, d / d.sum(), rtol=0, atol=2e-6)


def test_per_child_residuals_follow_each_siblings_row(oracle):
    """Merged trees ("Merge-Based Tree Construction"): siblings drawn from
    different draft rows; each rejection subtracts the rejected child's own
    row: r_2 = norm(max(norm(max(p - q1, 0)) - q2, 0)) (fp64 closed form)."""
    rng = np.random.default_rng(12)
    V = 500
    l = (2.0 * rng.standard_normal(V)).astype(np.float32)
    q1 = rng.dirichlet(np.full(V, 0.5)).astype(np.float32)
    q2 = rng.dirichlet(np.full(V, 0.5)).astype(np.float32)
    r2, _, _ = oracle.residual(l, np.stack([q1, q2]), 2)
    p = _softmax64(l)
    d1 = np.maximum(p - q1, 0)
    r1 = d1 / d1.sum()
    d2 = np.maximum(r1 - q2, 0)
    np.testing.assert_allclose(r2, d2 / d2.sum(), rtol=0, atol=2e-6)
    # and the other order gives the other closed form
    r2b, _, _ = oracle.residual(l, np.stack([q2, q1]), 2)
    d1b = np.maximum(p - q2, 0)
    d2b = np.maximum(d1b / d1b.sum() - q1, 0)
    np.testing.assert_allclose(r2b, d2b / d2b.sum(), rtol=0, atol=2e-6)


@pytest.mark.parametrize("tau", [0.5, 2.0])
def test_stochastic_with_temperature_emits_tempered_target(oracle, tau):
    """Losslessness at temperature T: the first emitted token follows
    p(.|root)^(1/T) normalised, the second p(.|x)^(1/T) normalised."""
    V, N = 8, 200_000
    inputs, P = mc_tree_inputs(N, V, 3, 2, 11)
    r = oracle.verify_stochastic(**inputs, inv_temp=np.full(N, tau, np.float32))
    assert (r["status"] == 0).all()
    first = r["emitted"][:, 0]
    assert _chisq_pvalue(np.bincount(first, minlength=V), _tempered(P[()], tau)) > 1e-4
    # the untempered target is rejected at this sample size
    assert _chisq_pvalue(np.bincount(first, minlength=V), P[()]) < 1e-6
    cont = r["accept_len"] >= 2
    for x in range(V):
        sel = cont & (first == x)
        if sel.sum() < 2000:
            continue
        assert _chisq_pvalue(np.bincount(r["emitted"][sel, 1], minlength=V), _tempered(P[(x,)], tau)) > 1e-4, x


@pytest.mark.parametrize("seed,root_kids,kid_kids", [(21, 3, 2), (22, 2, 3), (23, 4, 1)])
def test_stochastic_per_child_rows_emit_target_distribution(oracle, seed, root_kids, kid_kids):
    """Losslessness with siblings from different draft models (each child
    tested against, and on rejection subtracted as, its own row)."""
    V, N = 8, 200_000
    inputs, P = mc_tree_inputs(N, V, root_kids, kid_kids, seed, per_child=True)
    r = oracle.verify_stochastic(**inputs, q_per_child=True)
    assert (r["status"] == 0).all()
    first = r["emitted"][:, 0]
    assert _chisq_pvalue(np.bincount(first, minlength=V), P[()]) > 1e-4
    cont = r["accept_len"] >= 2
    for x in range(V):
        sel = cont & (first == x)
        if sel.sum() < 2000:
            continue
        assert _chisq_pvalue(np.bincount(r["emitted"][sel, 1], minlength=V), P[(x,)]) > 1e-4, x


def test_per_child_rows_copied_from_parents_equal_per_parent_mode(oracle):
    """Special case: when every child's row is its parent's row, the per-child
    layout is the per-parent one, outcome for outcome; and tau = 1 given
    explicitly is the default."""
    inputs, _ = mc_tree_inputs(3000, 8, 3, 2, 5)
    r0 = oracle.verify_stochastic(**inputs)
    par = inputs["parent"]
    n = inputs["n_max"]
    qc = inputs["q_probs"].copy()
    for g in range(len(par)):
        if par[g] >= 0:
            qc[g] = inputs["q_probs"][(g // n) * n + par[g]]
    r1 = oracle.verify_stochastic(**dict(inputs, q_probs=qc), q_per_child=True)
    r2 = oracle.verify_stochastic(**inputs, inv_temp=np.ones(3000, np.float32))
    for k in r0:
        assert np.array_equal(r0[k], r1[k]) and np.array_equal(r0[k], r2[k]), k


def test_bad_inverse_temperature_is_flagged(oracle):
    logits = np.zeros((10, 4), np.float32)
    qp = np.full((10, 4), 0.25, np.float32)
    tokens = np.array([0, 1] * 4 + [0, 7], np.int32)
    parent = np.array([-1, 0] * 5, np.int32)
    uni = np.zeros((10, 2), np.uint32)
    tau = np.array([0.0, -1.0, np.inf, np.nan, np.inf], np.float32)
    r = oracle.verify_stochastic(logits, qp, tokens, parent, [0, 2, 4, 6, 8, 10], uni, 2, inv_temp=tau)
    assert r["status"].tolist() == [oracle.ST_BAD_TEMP] * 4 + [oracle.ST_BAD_TEMP | oracle.ST_BAD_TOKEN]
    assert (r["accept_len"] == 0).all() and (r["path"] == -1).all()


def test_stochastic_chain_matches_closed_form_expected_tokens(oracle):
    """E[T] = (1 - a^(g+1)) / (1 - a) for a chain of g i.i.d. drafts with
    per-draft acceptance a (the "Worked Example" section); the page's printed
    values are checked against the formula, then the verifier against both."""
    ents = read_golden("inference_opt_accept_examples.txt")
    cases = [(float(v[0]), int(v[1]), float(v[2])) for k, v in ents if k == "expected_tokens"]
    ex_b = dict(ents[ents.index(("example", ["b"])) + 1:])
    rng = np.random.default_rng(77)
    N = 200_000
    for alpha, gamma, printed in cases:
        closed = (1 - alpha ** (gamma + 1)) / (1 - alpha)
        assert abs(closed - printed) < 1e-3
        if alpha == 0.7:
            p = np.array([float(v) for v in ex_b["p"]])
            q = np.array([float(v) for v in ex_b["q"]])
            assert abs(np.minimum(p, q).sum() - 0.7) < 1e-12
        else:
            p, q = np.array([alpha, 1 - alpha]), np.array([1.0, 0.0])
        V, n = len(p), gamma + 1
        tokens = rng.choice(V, (N, n), p=q).astype(np.int32)
        logits = np.tile(np.log(np.maximum(p, 1e-300)).astype(np.float32), (N * n, 1))
        qp = np.tile(q.astype(np.float32), (N * n, 1))
        uni = rng.integers(0, 2 ** 32, (N * n, 2), dtype=np.uint64).astype(np.uint32)
        r = oracle.verify_stochastic(logits, qp, tokens.reshape(-1), np.tile(W.chain_tree(n).numpy(), N),
                                     np.arange(0, N * n + 1, n, dtype=np.int32), uni, n)
        T = r["n_emitted"].astype(np.float64)
        assert abs(T.mean() - closed) <= 4 * T.std() / math.sqrt(N), (alpha, gamma, T.mean(), closed)


def test_stochastic_width1_stops_at_first_rejection(oracle):
    """On a chain (linear speculation, "Misconception" section): once a draft
    is rejected nothing after it is kept, the emitted count is the accepted
    prefix plus one, and a fully accepted chain ends with a bonus token."""
    rng = np.random.default_rng(8)
    V, n, N = 6, 6, 2000
    logits = rng.standard_normal((N * n, V)).astype(np.float32)
    qp = rng.dirichlet(np.ones(V), N * n).astype(np.float32)
    tokens = rng.integers(0, V, N * n).astype(np.int32)
    uni = rng.integers(0, 2 ** 32, (N * n, 2), dtype=np.uint64).astype(np.uint32)
    r = oracle.verify_stochastic(logits, qp, tokens, np.tile(W.chain_tree(n).numpy(), N),
                                 np.arange(0, N * n + 1, n, dtype=np.int32), uni, n)
    for b in range(N):
        L = r["accept_len"][b]
        assert r["path"][b, :L].tolist() == list(range(L))
        assert r["emitted"][b, :L - 1].tolist() == tokens[b * n + 1:b * n + L].tolist()


def test_stochastic_zero_draft_probability_is_accepted_and_bad_inputs(oracle):
    logits = np.zeros((2, 4), np.float32)
    qp = np.array([[0.5, 0.5, 0.0, 0.0]] * 2, np.float32)
    uni = np.array([[0, 0], [0xffffffff, 0]], np.uint32)
    r = oracle.verify_stochastic(logits, qp, np.array([0, 3], np.int32), np.array([-1, 0], np.int32), [0, 2], uni, 2)
    assert r["accept_len"][0] == 2
    r = oracle.verify_stochastic(logits, qp, np.array([0, 4], np.int32), np.array([-1, 0], np.int32), [0, 2], uni, 2)
    assert r["status"][0] == oracle.ST_BAD_TOKEN and r["accept_len"][0] == 0


# ------------------------------------------------ arithmetic contract ----

def test_canonical_exp_within_2_ulp_of_libm():
    import oracle as o
    rng = np.random.default_rng(0)
    xs = np.concatenate([np.linspace(-87.0, 0.0, 1_000_001, dtype=np.float64).astype(np.float32),
                         -rng.random(500_000, dtype=np.float32) * 87.0,
                         -(rng.random(200_000, dtype=np.float32) * 1e-3),
                         np.array([0.0, -0.0, -1e-30, -87.0, -86.99999], np.float32)])
    got = o.canon_exp(xs)
    ref = np.exp(xs.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    err = np.abs(got.astype(np.float64) - ref) / ulp
    assert err.max() <= 2.0, float(err.max())
    assert o.canon_exp(np.array([0.0], np.float32))[0] == 1.0
    assert (o.canon_exp(np.array([-87.0001, -88.0, -1e30, -np.inf], np.float32)) == 0).all()


def test_fx_is_exact_truncation():
    import oracle as o
    rng = np.random.default_rng(1)
    vals = list(rng.random(2000, dtype=np.float32) * 2) + [0.0, 2 ** -46, 2 ** -47, 1.0, 1.9999999]
    for v in vals:
        v32 = float(np.float32(v))
        assert o.fx(v32) == math.floor(Fraction(v32) * 2 ** 46)
    arr = np.array(vals + [np.float32(2 ** -126), np.float32(1.4e-45)], np.float32)
    got = o.fx_array(arr)
    assert got.dtype == np.uint64
    assert [int(x) for x in got] == [math.floor(Fraction(float(v)) * 2 ** 46) for v in arr]


def _is_rn_f32(x, exact):
    """x (fp32) is the round-to-nearest-even fp32 value of the rational `exact`."""
    x = np.float32(x)
    lo, hi = np.nextafter(x, np.float32(-np.inf)), np.nextafter(x, np.float32(np.inf))
    e = abs(Fraction(float(x)) - exact)
    for y in (lo, hi):
        ey = abs(Fraction(float(y)) - exact)
        if ey < e or (ey == e and int(np.float32(y).view(np.uint32)) % 2 == 0):
            return False
    return True


def test_residual_step_is_rounded_quotient_then_rounded_difference():
    """C5 one entry: r = RN(d / Z), then RN(r - q) clamped at zero, checked
    against exact rationals (Z of the form fp32(S) * 2^-46 as the sums make
    them, d and q probabilities, zeros)."""
    import oracle as o
    rng = np.random.default_rng(7)
    n = 3000
    d = (rng.random(n) ** 6).astype(np.float32)
    d[::17] = 0.0
    q = (rng.random(n) ** 3).astype(np.float32)
    S = rng.integers(1, 2 ** 62, size=(n + 1) // 2, dtype=np.int64) >> rng.integers(0, 60, size=(n + 1) // 2)
    Zp = (np.maximum(S, 1).astype(np.float32) * np.float32(2.0 ** -46)).astype(np.float32)
    got = o.resid_step(d, q, Zp)
    for i in range(n):
        Z = Fraction(float(Zp[i // 2]))
        r = np.float32(d[i]) / np.float32(Zp[i // 2])
        assert _is_rn_f32(r, Fraction(float(d[i])) / Z)
        diff = np.float32(r) - np.float32(q[i])
        assert _is_rn_f32(diff, Fraction(float(r)) - Fraction(float(q[i])))
        want = diff if diff > 0 else np.float32(0.0)
        assert got[i].view(np.uint32) == np.float32(want).view(np.uint32), i


# --------------------------------------------------------------- commit ----

def _elems(t, dtype):
    return t.numpy() if dtype == W.F32 else t.view(torch.int16).numpy().view(np.uint16)


def _as_f64(a, dtype):
    return a.astype(np.float64) if dtype == W.F32 else (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_append_then_attention_is_causal_attention_over_callers_rows(oracle, dtype):
    """[SpecInfer guide] "Depth-First Flattening and KV Cache Reuse": the tree
    tokens' keys and values are appended to the active cache after the
    prefix, in node order.  After the append (over a cache whose tree slots
    held garbage), the oracle's attention must equal causal attention over
    prefix + root path where the prefix K/V come from the cache and the tree
    K/V straight from the caller's [T][Hkv][D] rows (independent fp64)."""
    w = W.small_random(21, B=3, n_range=(1, 11), prefix_range=(0, 30), Hq=4, Hkv=2, D=16, dtype=dtype, block_size=8)
    g = np.random.default_rng(5)
    tdt = w.torch_dtype
    k_new = torch.from_numpy(g.standard_normal((w.T, w.Hkv, w.D))).to(tdt)
    v_new = torch.from_numpy(g.standard_normal((w.T, w.Hkv, w.D))).to(tdt)
    kc, vc = w.k_cache.clone(), w.v_cache.clone()
    bt, bs = w.block_table.numpy(), w.block_size
    for b in range(w.B):  # garbage in the tree slots
        P, n = int(w.prefix_len[b]), int(w.tree_off[b + 1] - w.tree_off[b])
        for s_ in range(P, P + n):
            kc[bt[b, s_ // bs], :, s_ % bs] = 1e3
            vc[bt[b, s_ // bs], :, s_ % bs] = -1e3
    k_out, v_out, st = oracle.kv_append(_elems(k_new, dtype), _elems(v_new, dtype), _elems(kc, dtype),
                                        _elems(vc, dtype), bt, bs, w.prefix_len.numpy(), w.tree_off.numpy(), w.n_max,
                                        w.Hkv, w.D, dtype, np.zeros(w.B, np.int32))
    assert st.tolist() == [0] * w.B
    _, out64, status = oracle.tree_attention(_elems(w.q, dtype), k_out, v_out, bt, bs, w.prefix_len.numpy(),
                                             w.tree_off.numpy(), w.parent.numpy(), w.n_max, w.Hq, w.Hkv, w.D, dtype,
                                             w.scale, want_f64=True)
    assert status.tolist() == [0] * w.B
    kpre, vpre = kc.double().numpy(), vc.double().numpy()
    kt, vt = k_new.double().numpy(), v_new.double().numpy()
    q = w.q.double().numpy()
    grp = w.Hq // w.Hkv
    for b in range(w.B):
        off, n, P = int(w.tree_off[b]), int(w.tree_off[b + 1] - w.tree_off[b]), int(w.prefix_len[b])
        par = w.parent[off:off + n].numpy()
        for u in range(n):
            path, c = [], u
            while c != -1:
                path.append(c)
                c = par[c]
            path.reverse()
            for h in range(w.Hq):
                kvh = h // grp
                Kp = np.array([kpre[bt[b, s_ // bs], kvh, s_ % bs] for s_ in range(P)]).reshape(P, w.D)
                Vp = np.array([vpre[bt[b, s_ // bs], kvh, s_ % bs] for s_ in range(P)]).reshape(P, w.D)
                K = np.concatenate([Kp, kt[off + np.array(path), kvh]])
                V = np.concatenate([Vp, vt[off + np.array(path), kvh]])
                sc = K @ q[off + u, h] * w.scale
                p = np.exp(sc - sc.max())
                np.testing.assert_allclose(out64[off + u, h], (p / p.sum()) @ V, rtol=0, atol=1e-12)


def test_append_into_one_page_per_request_is_a_plain_slice(oracle):
    """With one page per request (page b holds request b's slots), the tree
    rows of kv-head h are exactly cache[b, h, P:P+n] and nothing else moves."""
    B, Hkv, D, bs = 3, 2, 8, 64
    g = np.random.default_rng(8)
    n = np.array([5, 0, 17])
    tree_off = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    P = np.array([10, 3, 47], np.int32)
    T = int(tree_off[-1])
    kc = g.standard_normal((B, Hkv, bs, D)).astype(np.float32)
    vc = g.standard_normal((B, Hkv, bs, D)).astype(np.float32)
    k_new = g.standard_normal((T, Hkv, D)).astype(np.float32)
    v_new = g.standard_normal((T, Hkv, D)).astype(np.float32)
    bt = np.arange(B, dtype=np.int32).reshape(B, 1)
    k_out, v_out, st = oracle.kv_append(k_new, v_new, kc, vc, bt, bs, P, tree_off, 32, Hkv, D, W.F32,
                                        np.zeros(B, np.int32))
    assert st.tolist() == [0, 0, 0]
    k_ref, v_ref = kc.copy(), vc.copy()
    for b in range(B):
        for h in range(Hkv):
            k_ref[b, h, P[b]:P[b] + n[b]] = k_new[tree_off[b]:tree_off[b + 1], h]
            v_ref[b, h, P[b]:P[b] + n[b]] = v_new[tree_off[b]:tree_off[b + 1], h]
    assert np.array_equal(k_out, k_ref) and np.array_equal(v_out, v_ref)


def test_append_keeps_other_slots_and_rejects_bad_requests(oracle):
    w = W.small_random(22, B=5, n_range=(1, 9), prefix_range=(0, 40), Hq=4, Hkv=2, D=8, dtype=W.BF16, block_size=8)
    g = np.random.default_rng(9)
    k_new = g.integers(0, 2 ** 16, size=(w.T, w.Hkv, w.D), dtype=np.uint16)
    v_new = g.integers(0, 2 ** 16, size=(w.T, w.Hkv, w.D), dtype=np.uint16)
    bt = w.block_table.numpy().copy()
    P = w.prefix_len.numpy().copy()
    tree_off = w.tree_off.numpy()
    P[1] = bt.shape[1] * 8 - int(tree_off[2] - tree_off[1]) + 1  # last tree slot past the table
    bt[2, P[2] // 8] = w.num_blocks + 4                           # a bad id among the tree's pages
    st_in = np.zeros(w.B, np.int32)
    k0, v0 = _elems(w.k_cache, W.BF16), _elems(w.v_cache, W.BF16)
    k_out, v_out, st = oracle.kv_append(k_new, v_new, k0, v0, bt, 8, P, tree_off, w.n_max, w.Hkv, w.D, W.BF16,
                                        st_in)
    assert st[1] == oracle.ST_CAPACITY and st[2] == oracle.ST_BAD_BLOCK and st[0] == st[3] == st[4] == 0
    written = np.zeros(k0.shape[:3], bool)  # [block][head][row]
    for b in (0, 3, 4):
        for u in range(int(tree_off[b + 1] - tree_off[b])):
            s_ = int(P[b]) + u
            written[bt[b, s_ // 8], :, s_ % 8] = True
            for h in range(w.Hkv):
                assert np.array_equal(k_out[bt[b, s_ // 8], h, s_ % 8], k_new[tree_off[b] + u, h])
                assert np.array_equal(v_out[bt[b, s_ // 8], h, s_ % 8], v_new[tree_off[b] + u, h])
    assert np.array_equal(k_out[~written], k0[~written]) and np.array_equal(v_out[~written], v0[~written])
    # a tree larger than n_max is flagged and nothing is written
    _, _, st2 = oracle.kv_append(k_new, v_new, k0, v0, w.block_table.numpy(), 8, w.prefix_len.numpy(), tree_off, 1,
                                 w.Hkv, w.D, W.BF16, np.zeros(w.B, np.int32))
    assert all((st2[b] == oracle.ST_BAD_TREE) == (tree_off[b + 1] - tree_off[b] > 1) for b in range(w.B))


def test_commit_moves_path_rows_and_keeps_the_rest(oracle):
    rng = np.random.default_rng(3)
    w = W.small_random(31, B=4, n_range=(3, 20), prefix_range=(0, 50), Hq=4, Hkv=2, D=8, dtype=W.BF16, block_size=4)
    kc = w.k_cache.view(torch.int16).numpy().view(np.uint16)
    vc = w.v_cache.view(torch.int16).numpy().view(np.uint16)
    path = np.full((w.B, w.n_max), -1, np.int32)
    alen = np.zeros(w.B, np.int32)
    for b in range(w.B):
        n = int(w.tree_off[b + 1] - w.tree_off[b])
        par = w.parent[int(w.tree_off[b]):int(w.tree_off[b + 1])].numpy()
        u = int(rng.integers(0, n))
        p = []
        while u != -1:
            p.append(u)
            u = par[u]
        p.reverse()
        path[b, :len(p)] = p
        alen[b] = len(p)
    status = np.zeros(w.B, np.int32)
    status[3] = oracle.ST_BAD_TOKEN  # a failed request stays untouched
    k2, v2, new_len, st = oracle.kv_commit(kc, vc, w.block_table.numpy(), w.block_size, w.prefix_len.numpy(), path,
                                           alen, w.Hkv, w.D, W.BF16, status)
    P = w.prefix_len.numpy()
    assert new_len.tolist() == [int(P[b] + alen[b]) for b in range(3)] + [int(P[3])]
    assert st.tolist() == [0, 0, 0, oracle.ST_BAD_TOKEN]
    bt, bs = w.block_table.numpy(), w.block_size

    def rowv(c, b, s):
        return c[bt[b, s // bs], :, s % bs]
    touched = set()
    for b in range(3):
        for i in range(alen[b]):
            assert np.array_equal(rowv(k2, b, P[b] + i), rowv(kc, b, P[b] + path[b, i]))
            assert np.array_equal(rowv(v2, b, P[b] + i), rowv(vc, b, P[b] + path[b, i]))
            touched.add((bt[b, (P[b] + i) // bs], (P[b] + i) % bs))
    for blk in range(kc.shape[0]):
        for s in range(bs):
            if (blk, s) not in touched:
                assert np.array_equal(k2[blk, :, s], kc[blk, :, s]) and np.array_equal(v2[blk, :, s], vc[blk, :, s])


def test_commit_rejects_bad_paths(oracle):
    w = W.small_random(32, B=2, n_range=(4, 4), prefix_range=(3, 3), Hq=2, Hkv=1, D=8, dtype=W.F32, block_size=4)
    kc, vc = w.k_cache.numpy(), w.v_cache.numpy()
    path = np.array([[0, 2, 1, -1], [1, 2, -1, -1]], np.int32)
    k2, v2, new_len, st = oracle.kv_commit(kc, vc, w.block_table.numpy(), 4, w.prefix_len.numpy(), path,
                                           np.array([3, 2], np.int32), 1, 8, W.F32, np.zeros(2, np.int32))
    assert st.tolist() == [oracle.ST_BAD_PATH] * 2 and new_len.tolist() == [3, 3]
    assert np.array_equal(k2, kc) and np.array_equal(v2, vc)


def _random_paths(w, rng):
    path = np.full((w.B, w.n_max), -1, np.int32)
    alen = np.zeros(w.B, np.int32)
    for b in range(w.B):
        par = w.parent[int(w.tree_off[b]):int(w.tree_off[b + 1])].numpy()
        u = int(rng.integers(0, len(par)))
        p = []
        while u != -1:
            p.append(u)
            u = par[u]
        path[b, :len(p)] = p[::-1]
        alen[b] = len(p)
    return path, alen


def test_release_of_a_printed_page_layout(oracle):
    """Pages of 4 slots; prefix 5 and a 10-node tree fill slots 5..14 (pages
    1..3).  Three accepted nodes give new length 8: pages 0 and 1 stay, pages
    2 and 3 lie wholly past it and go back to the pool; page 4 was never the
    tree's."""
    bt = np.array([[10, 11, 12, 13, 14]], np.int32)
    out, pool, cnt, st = oracle.kv_release(bt, 4, [5], [0, 10], [8], [0], 16)
    assert out.tolist() == [[10, 11, -1, -1, 14]] and pool.tolist() == [12, 13] and cnt == 2 and st.tolist() == [0]
    # everything accepted into the last page: nothing is past the new length
    out, pool, cnt, _ = oracle.kv_release(bt, 4, [5], [0, 10], [15], [0], 16)
    assert cnt == 0 and out.tolist() == bt.tolist()
    # a failed request keeps every page
    out, pool, cnt, st = oracle.kv_release(bt, 4, [5], [0, 10], [8], [oracle.ST_BAD_TOKEN], 16)
    assert cnt == 0 and st.tolist() == [oracle.ST_BAD_TOKEN]
    # a pool that cannot take every page of the call takes none, and the
    # requests that had pages to release are flagged
    bt2 = np.array([[10, 11, 12, 13, 14], [20, 21, 22, 23, 24]], np.int32)
    out, pool, cnt, st = oracle.kv_release(bt2, 4, [5, 5], [0, 10, 20], [8, 8], [0, 0], 3)
    assert cnt == 0 and out.tolist() == bt2.tolist() and st.tolist() == [oracle.ST_CAPACITY] * 2
    # a failed request's pages do not count
    out, pool, cnt, st = oracle.kv_release(bt2, 4, [5, 5], [0, 10, 20], [8, 8], [0, oracle.ST_BAD_TOKEN], 3)
    assert cnt == 2 and pool.tolist() == [12, 13] and st.tolist() == [0, oracle.ST_BAD_TOKEN]
    # appends after the pool's current count, in request then page order
    out, pool, cnt, st = oracle.kv_release(bt2, 4, [5, 5], [0, 10, 20], [8, 8], [0, 0], 5, free_count=1)
    assert cnt == 5 and pool.tolist()[1:] == [12, 13, 22, 23] and (st == 0).all()
    assert out.tolist() == [[10, 11, -1, -1, 14], [20, 21, -1, -1, 24]]


def test_release_invariants_on_random_batches(oracle):
    """Every released id is a page wholly past the new length inside the
    tree's span, listed in request then page order; every other entry of the
    block table is unchanged."""
    rng = np.random.default_rng(9)
    for seed in range(6):
        w = W.small_random(40 + seed, B=7, n_range=(1, 40), prefix_range=(0, 60), Hq=2, Hkv=1, D=8, dtype=W.F32,
                           block_size=int(rng.choice([4, 8, 16])))
        path, alen = _random_paths(w, rng)
        P, bs = w.prefix_len.numpy(), w.block_size
        new_len = (P + alen).astype(np.int32)
        bt = w.block_table.numpy()
        out, pool, cnt, st = oracle.kv_release(bt, bs, P, w.tree_off.numpy(), new_len, np.zeros(w.B, np.int32), 10000)
        expect = []
        for b in range(w.B):
            n = int(w.tree_off[b + 1] - w.tree_off[b])
            keep, span = -(-int(new_len[b]) // bs), min(bt.shape[1], -(-(int(P[b]) + n) // bs))
            for i in range(bt.shape[1]):
                if keep <= i < span:
                    expect.append(int(bt[b, i]))
                    assert out[b, i] == -1
                else:
                    assert out[b, i] == bt[b, i]
        assert pool.tolist() == expect and cnt == len(expect) and (st == 0).all()
        assert len(set(expect)) == len(expect)


def test_layered_commit_moves_each_layers_rows(oracle):
    """Three layers with different contents: each layer's rows move per the
    path (numpy gather of that layer's snapshot), the release follows."""
    rng = np.random.default_rng(4)
    w = W.small_random(33, B=4, n_range=(3, 20), prefix_range=(0, 50), Hq=4, Hkv=2, D=8, dtype=W.BF16, block_size=4)
    path, alen = _random_paths(w, rng)
    layers_k = [(w.k_cache.view(torch.int16).numpy().view(np.uint16) + 3 * l).astype(np.uint16) for l in range(3)]
    layers_v = [(w.v_cache.view(torch.int16).numpy().view(np.uint16) + 5 * l).astype(np.uint16) for l in range(3)]
    ks, vs, new_len, st, bt_out, pool, cnt = oracle.kv_commit_layers(
        layers_k, layers_v, w.block_table.numpy(), w.block_size, w.prefix_len.numpy(), w.tree_off.numpy(), path, alen,
        w.Hkv, w.D, W.BF16, np.zeros(w.B, np.int32), 1000)
    P, bt, bs = w.prefix_len.numpy(), w.block_table.numpy(), w.block_size
    assert new_len.tolist() == (P + alen).tolist() and (st == 0).all()
    for l in range(3):
        for b in range(w.B):
            for i in range(alen[b]):
                d, src = P[b] + i, P[b] + path[b, i]
                assert np.array_equal(ks[l][bt[b, d // bs], :, d % bs], layers_k[l][bt[b, src // bs], :, src % bs])
                assert np.array_equal(vs[l][bt[b, d // bs], :, d % bs], layers_v[l][bt[b, src // bs], :, src % bs])
    assert cnt == len(pool) and all(int(x) >= 0 for x in pool)


# --------------------------------------------------------------- Philox ----

_PHILOX_CPP = r"""
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdio>
#include <cstdint>
int main() {
  const uint64_t seeds[] = {0ull, 1ull, 0x123456789abcdef0ull, 0xffffffffffffffffull};
  const uint64_t offs[] = {0ull, 1ull, 0x00000007fffffffeull, 0xdeadbeefcafebabeull};
  const uint64_t subs[] = {0ull, 3ull, 0xffffffff00000001ull};
  for (uint64_t s : seeds) for (uint64_t o : offs) for (uint64_t q : subs) {
    at::Philox4_32 e(s, q, o);  // key = seed; counter words 0,1 = offset, words 2,3 = subsequence
    uint32_t w0 = e(), w1 = e(), w2 = e(), w3 = e();
    std::printf("%llu %llu %llu %u %u %u %u\n", (unsigned long long)s, (unsigned long long)o,
                (unsigned long long)q, w0, w1, w2, w3);
  }
  return 0;
}
"""


# ----------------------------------------------------- tree construction ----

def _rank_order(row):
    """Tokens of a score row best first: larger value, then lower id; NaN last; -0 == +0."""
    r = np.asarray(row, np.float64) + 0.0  # -0 -> +0
    nan = np.isnan(r)
    return np.lexsort((np.arange(len(r)), -np.where(nan, 0, r), nan))


def _depths(parent, lo, hi):
    d = []
    for u in range(hi - lo):
        c, k = u, 0
        while parent[lo + c] != -1:
            c = parent[lo + c]
            k += 1
        d.append(k)
    return np.array(d)


def test_expansion_of_the_printed_schedule(oracle):
    """"Method A": schedule <3, 2, 1, 1> gives 3 nodes at depth 1, 6 at depth 2
    and 6 at depths 3 and 4; every node's children are the top-k of its row
    in rank order, appended level by level (parents before children)."""
    rng = np.random.default_rng(31)
    B, V, sched = 3, 50, [3, 2, 1, 1]
    rows = {}

    def level_scores(lev, ids):
        out = rng.standard_normal((B * len(ids), V)).astype(np.float32)
        out[:, 7] = out[:, 8]  # ties between tokens 7 and 8
        for b in range(B):
            for i, u in enumerate(ids):
                rows[(b, int(u))] = out[b * len(ids) + i]
        return out

    parent, tokens, tree_off = oracle.tree_expand(np.array([4, 5, 6]), level_scores, sched, V)
    n = 1 + 3 + 6 + 6 + 6
    assert tree_off.tolist() == [0, n, 2 * n, 3 * n]
    for b in range(B):
        lo = b * n
        par = parent[lo:lo + n]
        assert par[0] == -1 and all(0 <= par[u] < u for u in range(1, n))
        assert np.bincount(_depths(parent, lo, lo + n)).tolist() == [1, 3, 6, 6, 6]
        assert tokens[lo] == [4, 5, 6][b]
        for u in range(n):
            kids = [c for c in range(1, n) if par[c] == u]
            if not kids:
                continue
            want = _rank_order(rows[(b, u)])[:len(kids)]
            assert [tokens[lo + c] for c in kids] == want.tolist()
            assert kids == list(range(kids[0], kids[0] + len(kids)))


def test_expansion_rank_order_ties_nan_and_signed_zero(oracle):
    V = 9
    row = np.array([0.5, np.nan, 0.5, -0.0, 0.0, np.inf, -np.inf, 0.5, np.nan], np.float32)
    parent = np.full(1 + V, -1, np.int32)
    tokens = np.zeros(1 + V, np.int32)
    oracle.tree_expand_level(row[None], 1, V, 0, parent, tokens, 1 + V)
    assert tokens[1:].tolist() == [5, 0, 2, 7, 3, 4, 6, 1, 8]
    assert tokens[1:].tolist() == _rank_order(row).tolist()
    # random rows with many ties against the numpy order
    rng = np.random.default_rng(3)
    rows = rng.integers(0, 5, (40, 300)).astype(np.float32)
    rows[rng.random(rows.shape) < 0.05] = np.nan
    parent = np.full(40 * 8, -1, np.int32)
    tokens = np.zeros(40 * 8, np.int32)
    oracle.tree_expand_level(rows, 1, 7, 0, parent, tokens, 8)
    for b in range(40):
        assert tokens[b * 8 + 1:b * 8 + 8].tolist() == _rank_order(rows[b])[:7].tolist()
        assert parent[b * 8 + 1:b * 8 + 8].tolist() == [0] * 7


def _root_path_tokens(parent, tokens, lo, u):
    out = []
    while parent[lo + u] != -1:
        out.append(int(tokens[lo + u]))
        u = parent[lo + u]
    return tuple(out[::-1])


def test_merge_is_the_union_of_prefixes(oracle):
    """"Method B": every prefix of every candidate sequence is exactly one
    node whose token path is that prefix (S_v = S_u), no two nodes share a
    path, and nodes are numbered in first-appearance order."""
    rng = np.random.default_rng(17)
    B, M, m, V = 6, 5, 7, 3  # a small vocabulary: many shared prefixes
    seqs = rng.integers(0, V, (B, M, m)).astype(np.int32)
    seqs[:, 3] = seqs[:, 1]  # an identical sequence
    lens = rng.integers(0, m + 1, (B, M)).astype(np.int32)
    r = oracle.tree_merge(seqs, lens, np.arange(B) % V, V)
    assert (r["status"] == 0).all()
    for b in range(B):
        lo, hi = r["tree_off"][b], r["tree_off"][b + 1]
        par = r["parent"][lo:hi]
        assert par[0] == -1 and all(0 <= par[u] < u for u in range(1, hi - lo))
        paths = [_root_path_tokens(r["parent"], r["tokens"], lo, u) for u in range(hi - lo)]
        assert len(set(paths)) == len(paths)  # no duplicate token paths
        order = []
        for s in range(M):
            for j in range(lens[b, s]):
                pre = tuple(seqs[b, s, :j + 1].tolist())
                assert paths[r["node_of"][b, s, j]] == pre
                if pre not in order:
                    order.append(pre)
            assert (r["node_of"][b, s, lens[b, s]:] == -1).all()
        assert paths[1:] == order  # insertion order, and nothing else
        for u in range(1, hi - lo):
            s, j = divmod(int(r["src"][lo + u]), m)
            assert tuple(seqs[b, s, :j + 1].tolist()) == paths[u]


def test_merge_special_cases_and_bad_inputs(oracle):
    seq = np.array([[[1, 2, 3, 4]]], np.int32)
    r = oracle.tree_merge(seq, [[4]], [0], 10)  # one sequence: a chain
    assert r["parent"].tolist() == [-1, 0, 1, 2, 3] and r["tokens"].tolist() == [0, 1, 2, 3, 4]
    r = oracle.tree_merge(np.repeat(seq, 3, 1), [[4, 4, 4]], [0], 10)  # identical drafts: still one chain
    assert r["parent"].tolist() == [-1, 0, 1, 2, 3]
    r = oracle.tree_merge(np.repeat(seq, 3, 0), [[5], [4], [4]], [0, 0, 12], 10)
    assert r["status"].tolist() == [oracle.ST_BAD_TREE, 0, oracle.ST_BAD_TOKEN]
    assert r["tree_off"].tolist() == [0, 1, 6, 7] and (r["node_of"][0] == -1).all()


# -------------------------------------------------- dynamic draft length ----

def test_graph_keys_of_the_printed_example(oracle):
    d = dict(read_golden("dsd_graph_keys.txt"))
    max_k, tokens = int(d["max_k"][0]), int(d["tokens"][0])
    keys = oracle.dsd_graph_keys(tokens, max_k)
    assert [k for t, k in keys if t == tokens] == [int(v) for v in d["dynamic_k"]]
    assert int(d["fixed_k"][0]) in [k for t, k in keys if t == tokens]
    # brute force over a wider range: exactly the divisible pairs, in order
    keys = oracle.dsd_graph_keys(200, 9)
    assert keys == [(t, k) for t in range(1, 201) for k in range(1, 10) if t % (k + 1) == 0]


def _al_closed(alpha, K):
    return (1 - alpha ** (K + 1)) / (1 - alpha)


def test_optimal_k_maximises_goodput_and_falls_with_batch_size(oracle):
    """goodput = AL / ITL with AL the closed form of "Inference Optimization
    Techniques" (E[T] = (1 - a^(K+1)) / (1 - a)) and a dense-model cost ITL =
    c0 + c1 * BS * (K + 1): the table equals a brute-force argmax, and the
    optimal K does not grow with the batch size (the page's dense-model
    statement)."""
    ks = np.arange(1, 9, dtype=np.int32)
    bss = np.array([1, 2, 4, 8, 16, 32, 64, 128, 256, 512])
    for alpha, c0, c1 in [(0.8, 10.0, 0.05), (0.6, 5.0, 0.2), (0.9, 20.0, 0.01)]:
        al = np.array([[_al_closed(alpha, k) for k in ks] for _ in bss])
        itl = np.array([[c0 + c1 * bs * (k + 1) for k in ks] for bs in bss])
        kopt = oracle.dsd_optimal_k(al, itl, ks)
        brute = [int(ks[int(np.argmax(al[i] / itl[i]))]) for i in range(len(bss))]
        assert kopt.tolist() == brute
        assert all(a >= b for a, b in zip(kopt[:-1], kopt[1:])), kopt
        assert kopt[0] > kopt[-1]


def test_optimal_k_ties_invalid_cells_and_lookup(oracle):
    ks = np.array([1, 2, 3], np.int32)
    al = np.array([[2.0, 4.0, 6.0], [1.0, np.nan, 5.0], [1.0, 2.0, 3.0], [np.inf, 1.0, 1.0]])
    itl = np.array([[1.0, 2.0, 3.0], [1.0, 1.0, 0.0], [-1.0, 0.0, np.nan], [1.0, 1.0, 2.0]])
    assert oracle.dsd_optimal_k(al, itl, ks).tolist() == [1, 1, -1, 2]
    bs_tab, k_tab = [1, 4, 32, 128], [6, 5, 3, 1]
    for bs, want in [(0, 6), (1, 6), (3, 6), (4, 5), (31, 5), (32, 3), (127, 3), (128, 1), (10 ** 6, 1)]:
        assert oracle.dsd_select_k(bs_tab, k_tab, bs) == want
    assert oracle.dsd_select_k([], [], 5) == -1


def test_blend_is_an_exponential_moving_average(oracle):
    x = np.nan
    samples = [3.0, 5.0, 4.0, 10.0]
    w = 0.25
    ref = samples[0]
    x = oracle.dsd_blend(x, samples[0], w)
    assert x == ref
    for smp in samples[1:]:
        ref = (1 - w) * ref + w * smp
        x = oracle.dsd_blend(x, smp, w)
        assert abs(x - ref) < 1e-15
    assert oracle.dsd_blend(7.0, 1.0, 1.0) == 1.0


def test_philox_matches_pytorch_engine(oracle):
    """Philox4x32-10 against the independent engine in PyTorch's public
    headers (ATen/core/PhiloxRNGEngine.h): key = seed, counter = (offset lo,
    offset hi, subsequence lo, subsequence hi)."""
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    if not os.path.exists(os.path.join(inc, "ATen", "core", "PhiloxRNGEngine.h")):
        pytest.skip("PyTorch headers not installed")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "p.cpp"), os.path.join(d, "p")
        open(src, "w").write(_PHILOX_CPP)
        subprocess.check_call(["g++", "-std=c++17", "-O1", "-I", inc, src, "-o", exe])
        lines = subprocess.check_output([exe]).decode().split("\n")
    n = 0
    for line in lines:
        if not line.strip():
            continue
        s, o, q, *w = [int(x) for x in line.split()]
        ctr = [o & 0xffffffff, o >> 32, q & 0xffffffff, q >> 32]
        key = [s & 0xffffffff, s >> 32]
        assert oracle.philox4x32_10(ctr, key).tolist() == w
        n += 1
    assert n == 48


def test_philox_uniform_layout(oracle):
    tree_off = np.array([0, 3, 3, 7], np.int32)
    out = oracle.philox_uniforms(0xabcdef0123, 5, tree_off)
    for b in range(3):
        for t in range(tree_off[b], tree_off[b + 1]):
            w = oracle.philox4x32_10([t - tree_off[b], b, 5, 0], [0xabcdef0123 & 0xffffffff, 0xabcdef0123 >> 32])
            assert out[t].tolist() == w[:2].tolist()


def test_stochastic_children_tried_in_increasing_index(oracle):
    """Reading of the multi-sibling rule: the children of a node are tested in
    increasing node index.  With every acceptance uniform at 0 each test
    passes, so the walk takes the lowest-index child at every level."""
    #        0
    #      / | \
    #     1  4  6        node 1 has children 2, 3; node 4 has child 5
    parent = np.array([-1, 0, 1, 1, 0, 4, 0], np.int32)
    V = 5
    logits = np.zeros((7, V), np.float32)
    qp = np.full((7, V), 1.0 / V, np.float32)
    tokens = np.array([0, 1, 2, 3, 4, 0, 2], np.int32)
    uni = np.zeros((7, 2), np.uint32)
    r = oracle.verify_stochastic(logits, qp, tokens, parent, [0, 7], uni, 7)
    assert r["path"][0, :3].tolist() == [0, 1, 2] and r["accept_len"][0] == 3
    # reject child 1 (largest acceptance word) -> child 4 is tried next
    uni[1, 0] = 0xffffffff
    logits[0] = [0.0, -30.0, 0.0, 0.0, 0.0]
    r = oracle.verify_stochastic(logits, qp, tokens, parent, [0, 7], uni, 7)
    assert r["path"][0, :3].tolist() == [0, 4, 5]


def test_stochastic_zero_sum_residual_keeps_the_target(oracle):
    """Reading of the residual step when max(r - q, 0) sums to zero (q >= r
    everywhere: impossible for two normalised distributions except through
    rounding): the target stays r, so the walk samples from p itself."""
    V = 6
    logits = np.log(np.array([0.3, 0.25, 0.2, 0.1, 0.1, 0.05])).astype(np.float32)
    r0, _, _ = oracle.residual(logits, np.zeros(V, np.float32), 0)
    q = (r0 * np.float32(1.001)).astype(np.float32)
    parent = np.array([-1, 0, 0], np.int32)
    tokens = np.array([0, 1, 2], np.int32)
    rows = np.stack([logits] * 3)
    qp = np.stack([q] * 3)
    # both children rejected (largest acceptance word), then the sample
    cdf = np.cumsum(r0.astype(np.float64))
    for frac in [0.0, 0.1, 0.29, 0.31, 0.5, 0.6, 0.74, 0.8, 0.9, 0.96, 0.999]:
        U = int(frac * 2 ** 32)
        uni = np.array([[0, U], [0xffffffff, 0], [0xffffffff, 0]], np.uint32)
        r = oracle.verify_stochastic(rows, qp, tokens, parent, [0, 3], uni, 3)
        expect = int(np.searchsorted(cdf, U / 2 ** 32, side="right"))
        assert r["accept_len"][0] == 1 and r["emitted"][0, 0] == expect, frac
