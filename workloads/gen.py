"""Seeded synthetic inputs for one tree-verification pass.

This module only draws inputs: trees, tokens, query and key/value tensors,
target logits and draft probabilities.  It holds none of the verification
arithmetic, and both the CUDA path and the CPU oracle consume what it makes.
Everything is created on the CPU from a seeded numpy Generator (PCG64).

N(mu, v) below is mean mu and VARIANCE v (the mathematical convention).

The five workload families:
  0  tiny: B=1, 4/4 heads, D=64, fp32, prefix 128, 16-node tree with
     parent[i] ~ U[0, i-1], tokens ~ U[0, 512), logits ~ N(0, 2),
     draft = softmax(logits + N(0, 1)).
  1  Llama-style decode layer: B=8, 32/8 heads, D=128, bf16, prefix 2048,
     64-node expansion tree with per-depth widths (4,2,2,1,1,1,1,1) cut at 64
     in BFS order and renumbered depth-first; children of u are the top-k
     tokens of the draft row of u; V=32000, logits ~ N(0, 3) plus +8 on one
     random token per row, draft = softmax(logits + N(0, 1.5)).
  2  wide ensemble: B=1, 64/8 heads, D=128, bf16, prefix 8192, 256-node trie
     merge of 4 random trees of depth 8 (branching U{1,2,3}, child tokens the
     first b entries of a per-path candidate list shared by all trees),
     V=128256, logits ~ N(0, 3), draft = softmax(logits + N(0, 1.5)).
  3  batched serving: B=64, 32/8 heads, D=128, bf16, 16-token pages with a
     random block table, prefix ~ U[256, 16384], trees of U[8, 64] nodes with
     random parents, children = the top tokens of the parent's draft row by
     sibling rank, V=32000, logits as in 1.
  4  linear-vs-tree sweep point: chains of K+1 nodes or random trees of K+1
     nodes, B in {1, 4, 16, 64, 256}, 32/8 heads, D=128, bf16, prefix 4096,
     V=32000, logits as in 1, draft = (1-a) p + a softmax(N(0, 3)), child
     tokens sampled from the parent's draft row.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

F32, BF16 = 0, 1


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    dtype: int            # F32 or BF16
    V: int
    n_max: int
    block_size: int
    parent: torch.Tensor  # int32 [T]  local parent index, -1 at each root
    tree_off: torch.Tensor  # int32 [B+1]
    tokens: torch.Tensor  # int32 [T]
    prefix_len: torch.Tensor  # int32 [B]
    block_table: torch.Tensor  # int32 [B, max_blocks]
    num_blocks: int
    q: torch.Tensor        # [T, Hq, D] float32 / bfloat16
    k_cache: torch.Tensor  # [num_blocks, Hkv, block_size, D]
    v_cache: torch.Tensor
    p_logits: Optional[torch.Tensor]  # float32 [T, V]
    q_probs: Optional[torch.Tensor]   # float32 [T, V]
    uniforms: torch.Tensor  # int32 [T, 2]: raw 32-bit words (bit patterns)
    philox_seed: int = 0
    philox_round: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def T(self):
        return int(self.tree_off[-1])

    @property
    def max_blocks(self):
        return self.block_table.shape[1]

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == F32 else torch.bfloat16

    @property
    def scale(self):
        return 1.0 / float(np.sqrt(self.D))


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _randint(gen, lo, hi):
    """Uniform integer in [lo, hi)."""
    return int(gen.integers(lo, hi))


_CHUNK = 1 << 24  # elements per independently seeded stream of a large normal fill
_PARALLEL_MIN = 1 << 26  # fills at least this large use the chunked streams


def _normal(gen, shape, var, dtype=torch.float32):
    """N(0, var) samples.  Tensors of 2^26 elements or more (the GB-sized
    caches of the serving and sweep workloads) are filled in fixed chunks of
    2^24 elements, chunk i from its own PCG64 stream seeded by a draw of `gen`,
    on a thread pool: the values depend only on `gen`'s state, not on the
    threads.  Smaller tensors are drawn from `gen` directly."""
    n = int(np.prod(shape)) if len(shape) else 1
    if n < _PARALLEL_MIN:
        x = torch.from_numpy(gen.standard_normal(shape, dtype=np.float32))
        if var != 1.0:
            x.mul_(float(np.sqrt(var)))
        return x.to(dtype)
    from concurrent.futures import ThreadPoolExecutor
    import os
    nchunks = (n + _CHUNK - 1) // _CHUNK
    seeds = gen.integers(0, 2**63, nchunks)
    out = torch.empty(n, dtype=dtype)
    sd = float(np.sqrt(var))

    def fill(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        x = torch.from_numpy(np.random.Generator(np.random.PCG64(int(seeds[i]))).standard_normal(hi - lo,
                                                                                                dtype=np.float32))
        if var != 1.0:
            x.mul_(sd)
        out[lo:hi] = x.to(dtype)

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        list(ex.map(fill, range(nchunks)))
    return out.view(shape)


def random_parent_tree(n, gen):
    """parent[0] = -1, parent[i] uniform in [0, i-1]."""
    par = torch.full((n,), -1, dtype=torch.int32)
    for i in range(1, n):
        par[i] = _randint(gen, 0, i)
    return par


def chain_tree(n):
    return torch.arange(-1, n - 1, dtype=torch.int32)


def bfs_to_dfs(parent_bfs):
    """Renumber a tree given in BFS order (parent before child) to depth-first
    preorder, children visited in their original order.  Returns (parent_dfs,
    perm) with perm[new] = old."""
    n = len(parent_bfs)
    children = [[] for _ in range(n)]
    for i in range(1, n):
        children[int(parent_bfs[i])].append(i)
    order, stack = [], [0]
    while stack:
        u = stack.pop()
        order.append(u)
        stack.extend(reversed(children[u]))
    new_of = {old: new for new, old in enumerate(order)}
    par = torch.full((n,), -1, dtype=torch.int32)
    for new, old in enumerate(order):
        if old != 0:
            par[new] = new_of[int(parent_bfs[old])]
    return par, torch.tensor(order, dtype=torch.long)


def expansion_tree_bfs(widths, n_cap):
    """Parent array (BFS order) of an expansion tree: the root, then widths[d]
    children for every node of depth d, cut at n_cap nodes."""
    parent, level = [-1], [0]
    for w in widths:
        nxt = []
        for u in level:
            for _ in range(w):
                if len(parent) >= n_cap:
                    break
                parent.append(u)
                nxt.append(len(parent) - 1)
        level = nxt
        if len(parent) >= n_cap or not level:
            break
    return torch.tensor(parent, dtype=torch.int32)


def _splitmix64(x):
    x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return x ^ (x >> 31)


def _path_key(path):
    key = 0x1234567
    for t in path:
        key = _splitmix64(key ^ t)
    return key


def _candidates(path_key, V, k, shared_seed):
    out, i = [], 0
    while len(out) < k:
        t = _splitmix64(path_key ^ _splitmix64(shared_seed + i)) % V
        if t not in out:
            out.append(int(t))
        i += 1
    return out


def merged_ensemble_tree(n_trees, depth, V, n_cap, gen, shared_seed=12345):
    """Trie merge of n_trees random trees (branching U{1,2,3} per node, child
    tokens the first b entries of a candidate list that depends only on the
    token path), identical paths deduplicated; BFS order, cut at n_cap.
    Returns (parent_bfs, tokens_bfs, root_token)."""
    root_tok = _randint(gen, 0, V)
    # merged trie: key = token path tuple
    index = {(): 0}
    parent, tokens = [-1], [root_tok]
    frontier = [()]  # paths at the current depth, BFS order
    tree_levels = [[()] for _ in range(n_trees)]
    for d in range(depth):
        new_levels = []
        for t in range(n_trees):
            nxt = []
            for path in tree_levels[t]:
                b = _randint(gen, 1, 4)
                key = _path_key(path)
                for tok in _candidates(key, V, b, shared_seed):
                    nxt.append(path + (tok,))
            new_levels.append(nxt[:4 * n_cap])
        tree_levels = new_levels
        # add this depth's nodes to the trie in BFS order (tree order, then rank)
        for t in range(n_trees):
            for path in tree_levels[t]:
                if path not in index and len(parent) < n_cap and path[:-1] in index:
                    index[path] = len(parent)
                    parent.append(index[path[:-1]])
                    tokens.append(path[-1])
        if len(parent) >= n_cap:
            break
    return torch.tensor(parent, dtype=torch.int32), torch.tensor(tokens, dtype=torch.int32)


def _paged_cache(gen, B, Hkv, D, block_size, seq_lens, dtype, spare_blocks=0):
    """K/V ~ N(0, 1) in pages of block_size slots; the block table is a random
    permutation of a pool of sum(ceil(len/bs)) (+ spare) blocks."""
    need = [(int(s) + block_size - 1) // block_size for s in seq_lens]
    num_blocks = sum(need) + spare_blocks
    max_blocks = max(need) if need else 1
    perm = torch.from_numpy(gen.permutation(num_blocks).astype(np.int32))
    bt = torch.zeros((B, max(max_blocks, 1)), dtype=torch.int32)
    pos = 0
    for b in range(B):
        bt[b, :need[b]] = perm[pos:pos + need[b]]
        pos += need[b]
    shape = (num_blocks, Hkv, block_size, D)
    k = _normal(gen, shape, 1.0, dtype)
    v = _normal(gen, shape, 1.0, dtype)
    return bt, num_blocks, k, v


def _target_and_draft(gen, T, V, var, spike, noise_var):
    logits = _normal(gen, (T, V), var)
    if spike:
        idx = torch.from_numpy(gen.integers(0, V, T))
        logits[torch.arange(T), idx] += spike
    draft = torch.softmax((logits.double() + _normal(gen, (T, V), noise_var).double()), dim=-1).float()
    return logits, draft


def _random_words(gen, T):
    return torch.from_numpy(gen.integers(0, 2**32, (T, 2), dtype=np.uint64).astype(np.uint32).view(np.int32))


def _pack(name, B, Hq, Hkv, D, dtype, V, n_max, block_size, parents, toks, prefix, gen, logits, draft,
          spare_blocks=0, meta=None):
    tree_off = torch.zeros(B + 1, dtype=torch.int32)
    for b in range(B):
        tree_off[b + 1] = tree_off[b] + len(parents[b])
    T = int(tree_off[-1])
    parent = torch.cat(parents) if T else torch.zeros(0, dtype=torch.int32)
    tokens = torch.cat(toks) if T else torch.zeros(0, dtype=torch.int32)
    prefix_len = torch.tensor(prefix, dtype=torch.int32)
    seq = [prefix[b] + len(parents[b]) for b in range(B)]
    tdt = torch.float32 if dtype == F32 else torch.bfloat16
    bt, nblk, k, v = _paged_cache(gen, B, Hkv, D, block_size, seq, tdt, spare_blocks)
    q = _normal(gen, (T, Hq, D), 1.0, tdt)
    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype, V=V, n_max=n_max, block_size=block_size,
                    parent=parent, tree_off=tree_off, tokens=tokens, prefix_len=prefix_len, block_table=bt,
                    num_blocks=nblk, q=q, k_cache=k, v_cache=v, p_logits=logits, q_probs=draft,
                    uniforms=_random_words(gen, T), meta=meta or {})


def config0(seed=1000):
    g = _rng(seed)
    n, V = 16, 512
    par = random_parent_tree(n, g)
    toks = torch.from_numpy(g.integers(0, V, n).astype(np.int32))
    logits, draft = _target_and_draft(g, n, V, 2.0, 0.0, 1.0)
    return _pack("tiny: B=1, 4/4 heads, D=64, fp32, prefix 128, 16-node random tree, V=512",
                 1, 4, 4, 64, F32, V, n, 16, [par], [toks], [128], g, logits, draft)


def _expansion_request(g, widths, n_cap, V):
    par_bfs = expansion_tree_bfs(widths, n_cap)
    n = len(par_bfs)
    logits, draft = _target_and_draft(g, n, V, 3.0, 8.0, 1.5)
    toks = torch.zeros(n, dtype=torch.int32)
    toks[0] = _randint(g, 0, V)
    # children of u = the top-k tokens of draft[u], k = number of children
    kids = [[] for _ in range(n)]
    for i in range(1, n):
        kids[int(par_bfs[i])].append(i)
    for u in range(n):
        if kids[u]:
            top = torch.topk(draft[u], len(kids[u])).indices
            for r, c in enumerate(kids[u]):
                toks[c] = int(top[r])
    par, perm = bfs_to_dfs(par_bfs)
    return par, toks[perm], logits[perm], draft[perm]


def config1(seed=1001, B=8, prefix=2048, widths=(4, 2, 2, 1, 1, 1, 1, 1), n_cap=64, V=32000, block_size=256):
    g = _rng(seed)
    pars, toks, ls, ds = [], [], [], []
    for _ in range(B):
        p, t, l, d = _expansion_request(g, widths, n_cap, V)
        pars.append(p), toks.append(t), ls.append(l), ds.append(d)
    return _pack("Llama-style decode layer: B=8, 32/8 heads, D=128, bf16, prefix 2048, 64-node expansion tree "
                 "(4,2,2,1,1,1,1,1), V=32000", B, 32, 8, 128, BF16, V, n_cap, block_size, pars, toks,
                 [prefix] * B, g, torch.cat(ls), torch.cat(ds))


def config2(seed=1002, n_cap=256, V=128256, prefix=8192, block_size=256):
    g = _rng(seed)
    par_bfs, tok_bfs = merged_ensemble_tree(4, 8, V, n_cap, g)
    par, perm = bfs_to_dfs(par_bfs)
    toks = tok_bfs[perm]
    n = len(par)
    logits, draft = _target_and_draft(g, n, V, 3.0, 0.0, 1.5)
    return _pack("wide ensemble: B=1, 64/8 heads, D=128, bf16, prefix 8192, 256-node merged tree, V=128256",
                 1, 64, 8, 128, BF16, V, n_cap, block_size, [par], [toks], [prefix], g, logits, draft)


def _ranked_children_tokens(par, draft_rows, V, g):
    n = len(par)
    toks = torch.zeros(n, dtype=torch.int32)
    toks[0] = _randint(g, 0, V)
    kids = [[] for _ in range(n)]
    for i in range(1, n):
        kids[int(par[i])].append(i)
    for u in range(n):
        if kids[u]:
            top = torch.topk(draft_rows[u], len(kids[u])).indices
            for r, c in enumerate(kids[u]):
                toks[c] = int(top[r])
    return toks


def config3(seed=1003, B=64, p_lo=256, p_hi=16384, n_lo=8, n_hi=64, V=32000, block_size=16, with_logits=True):
    g = _rng(seed)
    pars, toks, ls, ds, prefix = [], [], [], [], []
    for _ in range(B):
        prefix.append(_randint(g, p_lo, p_hi + 1))
        n = _randint(g, n_lo, n_hi + 1)
        par = random_parent_tree(n, g)
        if with_logits:
            l, d = _target_and_draft(g, n, V, 3.0, 8.0, 1.5)
            ls.append(l), ds.append(d)
            toks.append(_ranked_children_tokens(par, d, V, g))
        else:
            toks.append(torch.from_numpy(g.integers(0, V, n).astype(np.int32)))
        pars.append(par)
    logits = torch.cat(ls) if with_logits else None
    draft = torch.cat(ds) if with_logits else None
    return _pack("batched serving: B=64, 32/8 heads, D=128, bf16, 16-token pages, prefix U[256,16384], "
                 "trees U[8,64] nodes, V=32000", B, 32, 8, 128, BF16, V, n_hi, block_size, pars, toks, prefix, g,
                 logits, draft)


def config4(K=4, B=16, tree="chain", alpha=0.3, seed=1004, prefix=4096, V=32000, block_size=16):
    """One point of the linear-vs-tree sweep (chain or random tree of K+1 nodes)."""
    g = _rng(seed + 7919 * K + 104729 * B + int(alpha * 1000) + (0 if tree == "chain" else 1))
    n = K + 1
    pars = [chain_tree(n) if tree == "chain" else random_parent_tree(n, g) for _ in range(B)]
    T = B * n
    logits = _normal(g, (T, V), 3.0)
    idx = torch.from_numpy(g.integers(0, V, T))
    logits[torch.arange(T), idx] += 8.0
    p = torch.softmax(logits.double(), -1)
    r = torch.softmax(_normal(g, (T, V), 3.0).double(), -1)
    draft = ((1 - alpha) * p + alpha * r).float()
    del p, r
    # child tokens: inverse-CDF draws from the parent's draft row
    toks = []
    for b in range(B):
        t = torch.zeros(n, dtype=torch.int32)
        t[0] = _randint(g, 0, V)
        rows = draft[[b * n + int(pars[b][c]) for c in range(1, n)]].double().numpy()
        cdf = np.cumsum(rows, axis=1)
        u = g.random(n - 1)[:, None] * cdf[:, -1:]
        t[1:] = torch.from_numpy(np.minimum((cdf <= u).sum(axis=1), V - 1).astype(np.int32))
        toks.append(t)
    return _pack(f"sweep point: {tree} K={K}, B={B}, alpha={alpha}, 32/8 heads, D=128, bf16, prefix 4096, V=32000",
                 B, 32, 8, 128, BF16, V, n, block_size, pars, toks, [prefix] * B, g, logits, draft,
                 meta=dict(K=K, tree=tree, alpha=alpha))


def chain_prefix(w, n):
    """The first n nodes of every request of a chain workload (a chain's
    prefix is a chain): the same requests, prefixes and cache with K = n - 1
    drafts."""
    assert 1 <= n <= w.n_max and all(int(w.tree_off[b + 1] - w.tree_off[b]) == w.n_max for b in range(w.B))
    rows = torch.cat([torch.arange(b * w.n_max, b * w.n_max + n) for b in range(w.B)])
    meta = dict(w.meta, K=n - 1)
    return Workload(name=w.name.replace(f"K={w.n_max - 1}", f"K={n - 1}"), B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D,
                    dtype=w.dtype, V=w.V, n_max=n, block_size=w.block_size, parent=torch.cat([chain_tree(n)] * w.B),
                    tree_off=torch.arange(0, w.B * n + 1, n, dtype=torch.int32), tokens=w.tokens[rows].contiguous(),
                    prefix_len=w.prefix_len, block_table=w.block_table, num_blocks=w.num_blocks,
                    q=w.q[rows].contiguous(), k_cache=w.k_cache, v_cache=w.v_cache,
                    p_logits=w.p_logits[rows].contiguous(), q_probs=w.q_probs[rows].contiguous(),
                    uniforms=w.uniforms[rows].contiguous(), meta=meta)


def make_config(i, **kw):
    return [config0, config1, config2, config3, config4][i](**kw)


def tree_kv_rows(w, seed):
    """Keys and values of the tree tokens as the target model would hand them
    over: [T][Hkv][D] ~ N(0, 1) in the workload's dtype, one pair per seed."""
    g = _rng(seed)
    k = _normal(g, (w.T, w.Hkv, w.D), 1.0, w.torch_dtype)
    v = _normal(g, (w.T, w.Hkv, w.D), 1.0, w.torch_dtype)
    return k, v


def small_random(seed, B=3, n_range=(1, 40), prefix_range=(0, 300), Hq=8, Hkv=2, D=64, dtype=BF16, V=97,
                 block_size=16, n_max=None):
    """Small ragged case for parity tests: several tiles, ragged tails."""
    g = _rng(seed)
    pars, toks, prefix = [], [], []
    for _ in range(B):
        n = _randint(g, n_range[0], n_range[1] + 1)
        pars.append(random_parent_tree(n, g) if n > 0 else torch.zeros(0, dtype=torch.int32))
        toks.append(torch.from_numpy(g.integers(0, V, n).astype(np.int32)))
        prefix.append(_randint(g, prefix_range[0], prefix_range[1] + 1))
    T = sum(len(p) for p in pars)
    logits, draft = _target_and_draft(g, T, V, 3.0, 0.0, 1.0)
    nm = n_max if n_max is not None else max([len(p) for p in pars] + [1])
    return _pack(f"small ragged: B={B}, {Hq}/{Hkv} heads, D={D}", B, Hq, Hkv, D, dtype, V, nm, block_size, pars, toks,
                 prefix, g, logits, draft)
