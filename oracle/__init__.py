"""CPU oracle for one tree-verification pass (numpy front end over oracle.c).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product (the CUDA library and its binding) never imports it,
and has no CPU fallback.

What each function follows (page title, section):
  * mask_build        -- "SpecInfer Guide: Tree-Based Speculative LLM Serving",
                         "The Topology-Aware 2D Causal Mask"
  * tree_attention    -- same page, "Generalizing Attention to Tree Topologies"
                         and "Depth-First Flattening and KV Cache Reuse"
  * verify_greedy     -- same page, "Greedy Verification Algorithm"
  * verify_stochastic -- same page, "Stochastic Verification Algorithm", with
                         the accept / residual rule of "Inference Optimization
                         Techniques: Speed and Efficiency" (the
                         "Misconception" section and its traced example)
  * kv_append         -- SpecInfer guide, "Depth-First Flattening and KV Cache
                         Reuse" (tree K/V appended after the prefix)
  * kv_commit         -- SpecInfer guide, "Depth-First Flattening and KV Cache
                         Reuse" and "PagedKV Allocation with Zero-Copy Pruning"
  * tree_expand_level / tree_expand -- SpecInfer guide, "Method A:
                         Expansion-Based Tree Construction"
  * tree_merge        -- same page, "Method B: Merge-Based Tree Construction"
  * philox_uniforms   -- Philox4x32-10 (Salmon et al., SC'11)
  * dsd_*             -- "Hardware-aware dynamic speculative decoding":
                         goodput = AL / ITL, the offline K table, its
                         runtime lookup, live statistics, and the graph keys
                         <tokens, K> of "Compatibility with full CUDA Graph"

Pins (in tests/test_oracle_pins.py, all ``-m "not gpu"``):
  * mask: the 6-node matrix printed on the SpecInfer guide (tests/golden),
    chain tree == lower-triangular causal mask, brute-force ancestor sets;
  * attention: every node equals plain causal attention over the gathered
    sequence prefix + root path (independent fp64 routine, 1e-12); chain tree
    with an empty prefix == torch scaled_dot_product_attention(is_causal);
    q = 0 gives the mean of the visible values; bf16 rounding vs exact
    rational rounding;
  * greedy: brute force over all root paths; the adapted harness example of
    the SpecInfer guide (tests/golden);
  * stochastic: the two per-token examples of the "Inference Optimization
    Techniques" page (tests/golden), a Monte-Carlo chi-square test that the
    emitted tokens follow p, and the closed form E[T] = (1-a^(g+1))/(1-a) of
    the same page on chains; with an inverse temperature tau the target is
    softmax(l tau) and its residual (fp64 closed forms), and the emitted
    tokens follow p^tau normalised (Monte Carlo); with per-child draft rows
    the residuals after two rejections match the fp64 closed form in either
    order, the emitted tokens follow p (Monte Carlo), and children whose
    rows copy their parent's reproduce the per-parent mode exactly;
  * canonical exp: <= 2 ulp from libm's fp64 exp;
  * FX sums: equal to exact integer sums; the array form equals the scalar;
  * one residual step: the correctly rounded quotient d / Z, then the
    correctly rounded difference with q, clamped at zero (exact rationals);
  * append: attention over the appended cache equals causal attention over
    prefix + root path with the tree K/V taken straight from the caller's
    rows; with one contiguous page the tree rows are a plain slice; nothing
    else changes; bad requests are untouched;
  * commit: invariants against a snapshot gather;
  * expansion: the page's schedule <3, 2, 1, 1> gives levels of 3, 6, 6, 6
    nodes; children are the top-k of their row in numpy's lexicographic
    order (value, then token id; NaN last), level by level;
  * merge: brute force over the page's condition: every prefix of every
    sequence is one node with that token path, no two nodes share a path,
    first-appearance numbering; chains and identical drafts;
  * Philox: equal to the Philox4x32-10 engine shipped in PyTorch's headers.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
ST_BAD_TREE, ST_BAD_TOKEN, ST_CAPACITY, ST_BAD_BLOCK, ST_BAD_PATH, ST_BAD_TEMP = 1, 2, 4, 16, 32, 64

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, u32, u64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double
        L.oracle_tree_mask_build.argtypes = [P, P, i32, i32, P, P, P]
        L.oracle_tree_attention.argtypes = [P, P, P, P, i32, i32, i32, P, P, P, i32, i32, i32, i32, i32, i32,
                                            f64, P, i64, P, P, P]
        L.oracle_verify_greedy.argtypes = [P, P, P, P, i32, i32, i32, P, P, P, P, P]
        L.oracle_verify_stochastic.argtypes = [P, P, P, P, P, P, i32, i32, i32, P, i32, P, P, P, P, P]
        L.oracle_kv_commit.argtypes = [P, P, i64, P, i32, i32, i32, P, P, i32, P, i32, i32, i32, i32, P, P]
        L.oracle_kv_append.argtypes = [P, P, P, P, P, i32, i32, i32, P, P, i32, i32, i32, i32, i32, P]
        L.oracle_kv_release.argtypes = [P, i32, i32, P, P, P, P, i32, P, i32, P]
        L.oracle_tree_expand_level.argtypes = [P, i32, i32, i32, i32, i32, i32, P, P]
        L.oracle_tree_merge.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P, P, P]
        L.oracle_dsd_optimal_k.argtypes = [P, P, i32, i32, P, P]
        L.oracle_dsd_select_k.argtypes = [P, P, i32, i32]
        L.oracle_dsd_graph_keys.argtypes = [i32, i32, P, P, i32]
        L.oracle_dsd_blend.argtypes = [f64, f64, f64]
        L.oracle_dsd_blend.restype = f64
        L.oracle_philox4x32_10.argtypes = [P, P, P]
        L.oracle_philox_uniforms.argtypes = [u64, u32, P, i32, P]
        L.oracle_canon_exp.argtypes = [ctypes.c_float]
        L.oracle_canon_exp.restype = ctypes.c_float
        L.oracle_canon_exp_array.argtypes = [P, P, i64]
        L.oracle_fx_array.argtypes = [P, P, i64]
        L.oracle_resid_step_array.argtypes = [P, P, P, P, i64]
        L.oracle_fx.argtypes = [ctypes.c_float]
        L.oracle_fx.restype = u64
        L.oracle_f64_to_bf16.argtypes = [f64]
        L.oracle_f64_to_bf16.restype = ctypes.c_uint16
        L.oracle_residual.argtypes = [P, P, i32, i32, ctypes.c_float, P, P, P]
        _lib = L
    return _lib


def _c(a, dtype):
    """Contiguous numpy array of the given dtype (no copy when already so)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def mask_build(parent, tree_off, n_max):
    parent, tree_off = _c(parent, np.int32), _c(tree_off, np.int32)
    B, T, W = len(tree_off) - 1, int(tree_off[-1]), (n_max + 63) // 64
    mask = np.zeros((T, W), np.uint64)
    depth = np.zeros(T, np.int32)
    status = np.zeros(B, np.int32)
    lib().oracle_tree_mask_build(_p(parent), _p(tree_off), B, n_max, _p(mask), _p(depth), _p(status))
    return mask, depth, status


def tree_attention(q, k_cache, v_cache, block_table, block_size, prefix_len, tree_off, parent, n_max,
                   Hq, Hkv, D, dtype, scale, rows=None, want_f64=False):
    """q, k_cache, v_cache: float32 arrays, or uint16 arrays of bfloat16 bits
    when dtype == BF16.  Returns (out, out_f64 or None, status)."""
    edt = np.float32 if dtype == F32 else np.uint16
    q, k_cache, v_cache = _c(q, edt), _c(k_cache, edt), _c(v_cache, edt)
    block_table = _c(block_table, np.int32)
    prefix_len, tree_off, parent = _c(prefix_len, np.int32), _c(tree_off, np.int32), _c(parent, np.int32)
    B, T = len(tree_off) - 1, int(tree_off[-1])
    max_blocks = block_table.shape[1] if block_table.ndim == 2 else block_table.size // max(B, 1)
    num_blocks = k_cache.size // (Hkv * block_size * D)
    out = np.zeros((T, Hq, D), edt)
    out64 = np.zeros((T, Hq, D), np.float64) if want_f64 else None
    status = np.zeros(B, np.int32)
    rows_a = _c(rows, np.int64) if rows is not None else None
    lib().oracle_tree_attention(_p(q), _p(k_cache), _p(v_cache), _p(block_table), max_blocks, block_size, num_blocks,
                                _p(prefix_len), _p(tree_off), _p(parent), B, n_max, Hq, Hkv, D, dtype, float(scale),
                                _p(rows_a), 0 if rows_a is None else len(rows_a), _p(out), _p(out64), _p(status))
    return out, out64, status


def _verify_outputs(B, n_max):
    return (np.full((B, n_max), -1, np.int32), np.zeros(B, np.int32), np.full((B, n_max), -1, np.int32),
            np.zeros(B, np.int32), np.zeros(B, np.int32))


def verify_greedy(p_logits, tokens, parent, tree_off, n_max):
    p_logits = _c(p_logits, np.float32)
    tokens, parent, tree_off = _c(tokens, np.int32), _c(parent, np.int32), _c(tree_off, np.int32)
    B, V = len(tree_off) - 1, p_logits.shape[-1]
    path, alen, emitted, nem, status = _verify_outputs(B, n_max)
    lib().oracle_verify_greedy(_p(p_logits), _p(tokens), _p(parent), _p(tree_off), B, n_max, V,
                               _p(path), _p(alen), _p(emitted), _p(nem), _p(status))
    return dict(path=path, accept_len=alen, emitted=emitted, n_emitted=nem, status=status)


def verify_stochastic(p_logits, q_probs, tokens, parent, tree_off, uniforms, n_max, inv_temp=None,
                      q_per_child=False):
    """inv_temp: per-request inverse temperatures (None: 1); q_per_child:
    q_probs row c is child c's own draft distribution (else row u serves
    every child of u)."""
    p_logits, q_probs = _c(p_logits, np.float32), _c(q_probs, np.float32)
    tokens, parent, tree_off = _c(tokens, np.int32), _c(parent, np.int32), _c(tree_off, np.int32)
    uniforms = _c(uniforms, np.uint32)
    B, V = len(tree_off) - 1, p_logits.shape[-1]
    tau = None if inv_temp is None else _c(inv_temp, np.float32)
    path, alen, emitted, nem, status = _verify_outputs(B, n_max)
    lib().oracle_verify_stochastic(_p(p_logits), _p(q_probs), _p(tokens), _p(parent), _p(tree_off), _p(uniforms),
                                   B, n_max, V, None if tau is None else _p(tau), int(bool(q_per_child)),
                                   _p(path), _p(alen), _p(emitted), _p(nem), _p(status))
    return dict(path=path, accept_len=alen, emitted=emitted, n_emitted=nem, status=status)


def kv_commit(k_cache, v_cache, block_table, block_size, prefix_len, path, accept_len, Hkv, D, dtype, status):
    """Returns (k_new, v_new, new_len, status_out); the inputs are not modified."""
    edt = np.float32 if dtype == F32 else np.uint16
    k_new, v_new = np.array(k_cache, dtype=edt, copy=True, order="C"), np.array(v_cache, dtype=edt, copy=True, order="C")
    block_table = _c(block_table, np.int32)
    prefix_len, path, accept_len = _c(prefix_len, np.int32), _c(path, np.int32), _c(accept_len, np.int32)
    st = np.array(status, dtype=np.int32, copy=True)
    B = len(prefix_len)
    max_blocks = block_table.shape[1]
    num_blocks = k_new.size // (Hkv * block_size * D)
    new_len = np.zeros(B, np.int32)
    lib().oracle_kv_commit(_p(k_new), _p(v_new), k_new.size, _p(block_table), max_blocks, block_size, num_blocks,
                           _p(prefix_len), _p(path), path.shape[1], _p(accept_len), B, Hkv, D, dtype,
                           _p(new_len), _p(st))
    return k_new, v_new, new_len, st


def kv_append(k_new, v_new, k_cache, v_cache, block_table, block_size, prefix_len, tree_off, n_max, Hkv, D, dtype,
              status):
    """Tree K/V rows [T][Hkv][D] appended after each request's prefix.
    Returns (k_cache_new, v_cache_new, status_out); the inputs are not modified."""
    edt = np.float32 if dtype == F32 else np.uint16
    k_out = np.array(k_cache, dtype=edt, copy=True, order="C")
    v_out = np.array(v_cache, dtype=edt, copy=True, order="C")
    k_new, v_new = _c(k_new, edt), _c(v_new, edt)
    block_table, prefix_len, tree_off = _c(block_table, np.int32), _c(prefix_len, np.int32), _c(tree_off, np.int32)
    st = np.array(status, dtype=np.int32, copy=True)
    B = len(prefix_len)
    assert k_new.size == v_new.size == int(tree_off[-1]) * Hkv * D
    num_blocks = k_out.size // (Hkv * block_size * D)
    lib().oracle_kv_append(_p(k_new), _p(v_new), _p(k_out), _p(v_out), _p(block_table), block_table.shape[1],
                           block_size, num_blocks, _p(prefix_len), _p(tree_off), B, n_max, Hkv, D, dtype, _p(st))
    return k_out, v_out, st


def kv_release(block_table, block_size, prefix_len, tree_off, new_len, status, free_cap, free_count=0):
    """Page release after a commit.  Returns (block_table_out, free_pool[:count],
    count, status_out); the inputs are not modified."""
    bt = np.array(block_table, dtype=np.int32, copy=True, order="C")
    st = np.array(status, dtype=np.int32, copy=True)
    prefix_len, tree_off, new_len = _c(prefix_len, np.int32), _c(tree_off, np.int32), _c(new_len, np.int32)
    pool = np.full(max(int(free_cap), 1), -1, np.int32)
    cnt = np.array([free_count], np.int32)
    lib().oracle_kv_release(_p(bt), bt.shape[1], block_size, _p(prefix_len), _p(tree_off), _p(new_len), _p(st),
                            len(prefix_len), _p(pool), int(free_cap), _p(cnt))
    return bt, pool[:int(cnt[0])], int(cnt[0]), st


def kv_commit_layers(k_caches, v_caches, block_table, block_size, prefix_len, tree_off, path, accept_len, Hkv, D,
                     dtype, status, free_cap, free_count=0):
    """Every layer's commit (the single-layer commit per layer, each starting
    from the same status), then the page release.  Returns (k_list, v_list,
    new_len, status_out, block_table_out, free_pool, count)."""
    ks, vs = [], []
    new_len, st = None, None
    for k, v in zip(k_caches, v_caches):
        k2, v2, nl, s2 = kv_commit(k, v, block_table, block_size, prefix_len, path, accept_len, Hkv, D, dtype, status)
        ks.append(k2)
        vs.append(v2)
        new_len, st = nl, s2
    bt, pool, cnt, st = kv_release(block_table, block_size, prefix_len, tree_off, new_len, st, free_cap, free_count)
    return ks, vs, new_len, st, bt, pool, cnt


def tree_expand_level(scores, F, k, level_start, parent, tokens, n_total):
    """Appends level level_start + F .. of every request (see oracle.c);
    parent/tokens are [B * n_total] int32 arrays, updated in place."""
    scores = _c(scores, np.float32)
    V = scores.shape[-1]
    B = scores.size // (F * V) if F > 0 else 0
    assert parent.dtype == np.int32 and tokens.dtype == np.int32
    rc = lib().oracle_tree_expand_level(_p(scores), B, F, V, k, level_start, n_total, _p(parent), _p(tokens))
    assert rc == 0
    return parent, tokens


def tree_expand(root_tokens, level_scores, schedule, V):
    """A whole expansion tree: level_scores(level, frontier_node_ids) gives the
    [B * F, V] score rows of that level's frontier.  Returns (parent, tokens,
    tree_off) packed, each request's tree 1 + k1 + k1 k2 + ... nodes."""
    B = len(root_tokens)
    sizes = [1]
    for k in schedule:
        sizes.append(sizes[-1] * k)
    n_total = sum(sizes)
    parent = np.full(B * n_total, -1, np.int32)
    tokens = np.zeros(B * n_total, np.int32)
    tokens[::n_total] = root_tokens
    start = 0
    for lev, k in enumerate(schedule):
        F = sizes[lev]
        tree_expand_level(level_scores(lev, np.arange(start, start + F)), F, k, start, parent, tokens, n_total)
        start += F
    return parent, tokens, np.arange(0, B * n_total + 1, n_total, dtype=np.int32)


def tree_merge(seqs, lens, root_tok, V):
    """seqs [B, M, m] int32, lens [B, M], root_tok [B].  Returns dict of
    tree_off, parent, tokens, src (packed, trimmed to tree_off[-1]), node_of
    [B, M, m] and status [B]."""
    seqs, lens, root_tok = _c(seqs, np.int32), _c(lens, np.int32), _c(root_tok, np.int32)
    B, M, m = seqs.shape
    cap = B * (1 + M * m)
    tree_off = np.zeros(B + 1, np.int32)
    parent, tokens, src = np.zeros(cap, np.int32), np.zeros(cap, np.int32), np.zeros(cap, np.int32)
    node_of, status = np.zeros((B, M, m), np.int32), np.zeros(B, np.int32)
    lib().oracle_tree_merge(_p(seqs), _p(lens), _p(root_tok), B, M, m, V, _p(tree_off), _p(parent), _p(tokens),
                            _p(src), _p(node_of), _p(status))
    T = int(tree_off[-1])
    return dict(tree_off=tree_off, parent=parent[:T], tokens=tokens[:T], src=src[:T], node_of=node_of,
                status=status)


def dsd_optimal_k(al, itl, k_values):
    """al, itl: [n_bs, n_k]; returns the K of highest AL / ITL per row (-1: none)."""
    al, itl = _c(al, np.float64), _c(itl, np.float64)
    k_values = _c(k_values, np.int32)
    n_bs, n_k = al.shape
    out = np.zeros(n_bs, np.int32)
    lib().oracle_dsd_optimal_k(_p(al), _p(itl), n_bs, n_k, _p(k_values), _p(out))
    return out


def dsd_select_k(bs_table, k_table, bs):
    bs_table, k_table = _c(bs_table, np.int32), _c(k_table, np.int32)
    return int(lib().oracle_dsd_select_k(_p(bs_table), _p(k_table), len(bs_table), int(bs)))


def dsd_graph_keys(max_tokens, max_k):
    n = lib().oracle_dsd_graph_keys(max_tokens, max_k, None, None, 0)
    t, k = np.zeros(max(n, 1), np.int32), np.zeros(max(n, 1), np.int32)
    lib().oracle_dsd_graph_keys(max_tokens, max_k, _p(t), _p(k), n)
    return list(zip(t[:n].tolist(), k[:n].tolist()))


def dsd_blend(cell, sample, w):
    return float(lib().oracle_dsd_blend(float(cell), float(sample), float(w)))


def philox4x32_10(ctr, key):
    ctr, key = _c(ctr, np.uint32), _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_p(ctr), _p(key), _p(out))
    return out


def philox_uniforms(seed, round_, tree_off):
    tree_off = _c(tree_off, np.int32)
    B, T = len(tree_off) - 1, int(tree_off[-1])
    out = np.zeros((T, 2), np.uint32)
    lib().oracle_philox_uniforms(ctypes.c_uint64(seed), ctypes.c_uint32(round_), _p(tree_off), B, _p(out))
    return out


def canon_exp(x):
    x = _c(x, np.float32)
    y = np.empty_like(x)
    lib().oracle_canon_exp_array(_p(x), _p(y), x.size)
    return y


def fx(v):
    return int(lib().oracle_fx(ctypes.c_float(v)))


def fx_array(v):
    """C3 weights trunc(v * 2^46) of a float32 array, as uint64."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint64)
    lib().oracle_fx_array(_p(v), _p(out), v.size)
    return out


def resid_step(d, q, Zp):
    """One C5 residual step per entry: max(d / Z - q, 0), Z = Zp[i // 2]."""
    d, q, Zp = _c(d, np.float32), _c(q, np.float32), _c(Zp, np.float32)
    assert d.shape == q.shape and Zp.size >= (d.size + 1) // 2
    out = np.empty_like(d)
    lib().oracle_resid_step_array(_p(d), _p(q), _p(Zp), _p(out), d.size)
    return out


def f64_to_bf16_bits(x):
    return int(lib().oracle_f64_to_bf16(float(x)))


def residual(l, q, j, inv_temp=1.0):
    """Target distribution r_j and weights d_j of one row after j rejections:
    q is one draft row (used j times) or j rows [j][V], one per rejection."""
    l, q = _c(l, np.float32), _c(q, np.float32)
    V = l.size
    if q.ndim == 1:
        q = np.ascontiguousarray(np.tile(q, (max(j, 1), 1)))
    assert q.shape[0] >= j
    r, d, S = np.zeros(V, np.float32), np.zeros(V, np.float32), np.zeros(1, np.uint64)
    lib().oracle_residual(_p(l), _p(q), V, j, ctypes.c_float(inv_temp), _p(r), _p(d), _p(S))
    return r, d, int(S[0])
