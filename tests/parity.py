"""Helpers shared by the GPU parity tests: run the oracle and the CUDA path on
the same seeded workload and compare."""
import numpy as np
import torch

import oracle as O
import workloads as W


def np_elems(t, dtype):
    """CPU tensor -> numpy array the oracle takes (fp32, or raw bf16 bits)."""
    t = t.detach().cpu().contiguous()
    return t.numpy() if dtype == W.F32 else t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(a):
    return (a.astype(np.uint32) << 16).view(np.float32)


def out_as_f32(t, dtype):
    t = t.detach().cpu().contiguous()
    return t.numpy() if dtype == W.F32 else t.float().numpy()


def oracle_mask(w):
    return O.mask_build(w.parent.numpy(), w.tree_off.numpy(), w.n_max)


def oracle_attention(w, rows=None):
    return O.tree_attention(np_elems(w.q, w.dtype), np_elems(w.k_cache, w.dtype), np_elems(w.v_cache, w.dtype),
                            w.block_table.numpy(), w.block_size, w.prefix_len.numpy(), w.tree_off.numpy(),
                            w.parent.numpy(), w.n_max, w.Hq, w.Hkv, w.D, w.dtype, w.scale, rows=rows)


def oracle_greedy(w):
    return O.verify_greedy(w.p_logits.numpy(), w.tokens.numpy(), w.parent.numpy(), w.tree_off.numpy(), w.n_max)


def oracle_stochastic(w):
    return O.verify_stochastic(w.p_logits.numpy(), w.q_probs.numpy(), w.tokens.numpy(), w.parent.numpy(),
                               w.tree_off.numpy(), w.uniforms.numpy().view(np.uint32), w.n_max)


def attn_tolerance_ok(got, ref, dtype):
    """fp32: max-abs 1e-5.  bf16 inputs: |got - ref| <= 2e-2 + 1e-2 |ref|."""
    if dtype == W.F32:
        return np.abs(got - ref) <= 1e-5
    return np.abs(got - ref) <= 2e-2 + 1e-2 * np.abs(ref)


# ----------------------------------------------------- parallel oracle ----
# Full-size attention checks run the oracle on every row (or many rows): the
# rows are split over spawned host processes (never forked: the parent holds a
# CUDA context), which read the inputs from memory-mapped .npy files.

_ATTN_KEYS = ("q", "k_cache", "v_cache", "block_table", "prefix_len", "tree_off", "parent")


def _attn_rows_worker(job):
    import numpy as _np
    import oracle as _O
    folder, meta, rows = job
    a = {k: _np.load(f"{folder}/{k}.npy", mmap_mode="r") for k in _ATTN_KEYS}
    out, _, st = _O.tree_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], meta["block_size"],
                                   a["prefix_len"], a["tree_off"], a["parent"], meta["n_max"], meta["Hq"],
                                   meta["Hkv"], meta["D"], meta["dtype"], meta["scale"], rows=rows)
    return out.reshape(-1, meta["D"])[rows], st


def host_workers():
    import os
    return max(1, min(16, os.cpu_count() or 1))


def oracle_attention_rows(w, rows, workers=None, caches=None):
    """Oracle attention of the flat rows t * Hq + h listed in `rows` (sorted
    int64), computed in parallel: returns (out [len(rows)][D] in the oracle's
    element type, status[B]).  caches: (k, v) oracle element arrays to use
    instead of the workload's own."""
    import multiprocessing as mp
    import tempfile
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    workers = workers or host_workers()
    kc, vc = caches if caches is not None else (np_elems(w.k_cache, w.dtype), np_elems(w.v_cache, w.dtype))
    arrays = dict(q=np_elems(w.q, w.dtype), k_cache=kc, v_cache=vc,
                  block_table=w.block_table.numpy(), prefix_len=w.prefix_len.numpy(), tree_off=w.tree_off.numpy(),
                  parent=w.parent.numpy())
    meta = dict(block_size=w.block_size, n_max=w.n_max, Hq=w.Hq, Hkv=w.Hkv, D=w.D, dtype=w.dtype, scale=w.scale)
    with tempfile.TemporaryDirectory() as folder:
        for k, v in arrays.items():
            np.save(f"{folder}/{k}.npy", np.ascontiguousarray(v))
        parts = [p for p in np.array_split(rows, workers * 4) if p.size]
        with mp.get_context("spawn").Pool(min(workers, len(parts))) as pool:
            res = pool.map(_attn_rows_worker, [(folder, meta, p) for p in parts])
    out = np.concatenate([r[0] for r in res]) if res else np.zeros((0, w.D))
    st = res[0][1] if res else np.zeros(w.B, np.int32)
    return out, st


def rows_covering(w, k, seed):
    """At least k flat (node, head) rows, sorted, that include rows of every
    request and of every kv-head of each request: each request's first and
    last node on every kv-head, then uniform picks."""
    g = np.random.default_rng(seed)
    tree_off = w.tree_off.numpy()
    grp = w.Hq // w.Hkv
    pick = set()
    for b in range(w.B):
        lo, hi = int(tree_off[b]), int(tree_off[b + 1])
        if hi <= lo:
            continue
        for kvh in range(w.Hkv):
            for t in {lo, hi - 1, int(g.integers(lo, hi))}:
                pick.add(t * w.Hq + kvh * grp + int(g.integers(0, grp)))
    total = w.T * w.Hq
    extra = max(0, k - len(pick))
    if extra:
        pick.update(g.choice(total, size=min(extra * 2, total), replace=False).tolist())
    return np.array(sorted(pick), dtype=np.int64)
