"""GPU parity: every step of the pass through the C ABI against the CPU oracle
on the same seeded inputs.  Bit-exact for masks, depths, uniforms, paths,
emitted tokens, commit results and status words; attention within max-abs
1e-5 (fp32) or 2e-2 + 1e-2 |ref| (bf16 inputs)."""
import functools

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
import tree_speculative_verification_spec_gb300 as S
from tree_speculative_verification_spec_gb300.pipeline import DeviceBatch, VerifyPass
from parity import (attn_tolerance_ok, bf16_bits_to_f32, np_elems, oracle_attention, oracle_attention_rows,
                    oracle_greedy, oracle_mask, oracle_stochastic, out_as_f32, rows_covering)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_speculative_verification_spec_gb300 import build
    build.build()
    S.lib()


def _pass(w, **kw):
    vp = VerifyPass(DeviceBatch.from_workload(w, **kw))
    return vp


@functools.lru_cache(maxsize=None)
def _workload(which, **kw):
    """Full-size workloads, generated once per test session (read-only here)."""
    return W.make_config(which, **kw)


# sweep points of the linear-vs-tree workload: (K, B, tree, alpha)
SWEEP_POINTS = [(1, 4, "chain", 0.1), (4, 16, "chain", 0.3), (8, 64, "chain", 0.5), (8, 64, "random", 0.3),
                (3, 256, "random", 0.1)]


# ------------------------------------------------------------------ mask ----

def _ragged_trees(seed, sizes, n_max):
    g = np.random.Generator(np.random.PCG64(seed))
    pars = [W.random_parent_tree(n, g) if n > 0 else torch.zeros(0, dtype=torch.int32) for n in sizes]
    return pars


@pytest.mark.parametrize("sizes,n_max", [([16], 16), ([1, 64, 65, 0, 130], 130), ([1024], 1024),
                                         ([300, 7, 0, 0, 257], 300)])
def test_mask_build_parity(sizes, n_max):
    pars = _ragged_trees(sum(sizes), sizes, n_max)
    parent = torch.cat(pars)
    tree_off = torch.tensor(np.cumsum([0] + sizes), dtype=torch.int32)
    if len(sizes) > 2:  # plant a bad tree in request 1
        parent[tree_off[1] + 3] = 70
    m_ref, d_ref, s_ref = O.mask_build(parent.numpy(), tree_off.numpy(), n_max)
    B, T, Wd = len(sizes), int(tree_off[-1]), (n_max + 63) // 64
    mask = torch.zeros((T, Wd), dtype=torch.int64, device="cuda")
    depth = torch.zeros(T, dtype=torch.int32, device="cuda")
    status = torch.full((B,), 99, dtype=torch.int32, device="cuda")
    S.spec_tree_mask_build(parent.cuda(), tree_off.cuda(), B, n_max, mask, depth, status)
    torch.cuda.synchronize()
    assert np.array_equal(mask.cpu().numpy().view(np.uint64), m_ref)
    assert np.array_equal(depth.cpu().numpy(), d_ref)
    assert np.array_equal(status.cpu().numpy(), s_ref)


def test_mask_build_chain_and_printed_example():
    parent = torch.tensor([-1, 0, 0, 1, 1, 2] + list(range(-1, 99)), dtype=torch.int32)
    tree_off = torch.tensor([0, 6, 106], dtype=torch.int32)
    m_ref, d_ref, s_ref = O.mask_build(parent.numpy(), tree_off.numpy(), 100)
    mask = torch.zeros((106, 2), dtype=torch.int64, device="cuda")
    depth = torch.zeros(106, dtype=torch.int32, device="cuda")
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    S.spec_tree_mask_build(parent.cuda(), tree_off.cuda(), 2, 100, mask, depth, status)
    assert np.array_equal(mask.cpu().numpy().view(np.uint64), m_ref)
    assert np.array_equal(depth.cpu().numpy(), d_ref)


# ---------------------------------------------------------------- Philox ----

@pytest.mark.parametrize("seed,rnd", [(0, 0), (0xdeadbeefcafef00d, 7), (12345, 0xffffffff)])
def test_philox_parity(seed, rnd):
    tree_off = torch.tensor([0, 16, 16, 80, 1104], dtype=torch.int32)
    ref = O.philox_uniforms(seed, rnd, tree_off.numpy())
    out = torch.zeros((1104, 2), dtype=torch.int32, device="cuda")
    S.spec_philox_uniforms(seed, rnd, tree_off.cuda(), 4, 1024, out)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref)


# ---------------------------------------------------------------- verify ----

def _gpu_verify(w, mode):
    vp = _pass(w)
    vp.mask_build()
    vp.verify(mode)
    torch.cuda.synchronize()
    return dict(path=vp.path.cpu().numpy(), accept_len=vp.accept_len.cpu().numpy(),
                emitted=vp.emitted.cpu().numpy(), n_emitted=vp.n_emitted.cpu().numpy(),
                status=vp.status.cpu().numpy())


def _assert_verify_equal(got, ref, B):
    for k in ("path", "accept_len", "emitted", "n_emitted", "status"):
        assert np.array_equal(got[k][:B], ref[k][:B]), (k, got[k][:B], ref[k][:B])


SMALL_VERIFY = [dict(seed=s, B=B, n_range=nr, V=V) for s, B, nr, V in [
    (1, 4, (1, 12), 2), (2, 6, (1, 40), 7), (3, 5, (0, 64), 64), (4, 3, (1, 300), 513), (5, 2, (60, 90), 1000),
    (6, 8, (1, 30), 4099), (7, 2, (10, 30), 32000), (8, 1, (5, 9), 40000), (9, 2, (3, 20), 128256),
    (10, 1, (3, 12), 131072),  # the largest vocabulary the library takes
    (11, 12, (1, 40), 32000), (12, 7, (2, 20), 131072)]]  # 12-CTA clusters (5 to 12 requests)


@pytest.mark.parametrize("cfg", SMALL_VERIFY, ids=lambda c: f"V{c['V']}_s{c['seed']}")
@pytest.mark.parametrize("mode", ["greedy", "stochastic"])
def test_verify_parity_random_trees(cfg, mode):
    w = W.small_random(cfg["seed"], B=cfg["B"], n_range=cfg["n_range"], prefix_range=(0, 4), Hq=2, Hkv=1, D=64,
                       V=cfg["V"], block_size=16)
    if mode == "greedy":
        # make matches likely: child tokens copy the parent's argmax half of the time
        am = w.p_logits.argmax(1)
        g = np.random.default_rng(cfg["seed"])
        for b in range(w.B):
            off = int(w.tree_off[b])
            for u in range(1, int(w.tree_off[b + 1]) - off):
                if g.random() < 0.6:
                    w.tokens[off + u] = am[off + int(w.parent[off + u])]
        ref = oracle_greedy(w)
    else:
        ref = oracle_stochastic(w)
    got = _gpu_verify(w, mode)
    _assert_verify_equal(got, ref, w.B)


@pytest.mark.parametrize("mode", ["greedy", "stochastic"])
def test_verify_parity_many_siblings_and_duplicates(mode):
    """A star root with 200 children whose tokens repeat: long sibling loops,
    many residual updates, equal sibling tokens."""
    n, V, B = 201, 33, 3
    g = np.random.default_rng(3)
    parent = torch.tensor([-1] + [0] * (n - 1), dtype=torch.int32)
    w = W.small_random(40, B=B, n_range=(n, n), prefix_range=(0, 1), Hq=2, Hkv=1, D=64, V=V, block_size=16)
    w.parent = torch.cat([parent] * B)
    w.tokens = torch.from_numpy(g.integers(0, 4, B * n).astype(np.int32))
    # draft rows far from the target: rejections are frequent
    w.q_probs = torch.softmax(torch.from_numpy(g.standard_normal((B * n, V)).astype(np.float32)) * 4, -1)
    ref = oracle_greedy(w) if mode == "greedy" else oracle_stochastic(w)
    got = _gpu_verify(w, mode)
    _assert_verify_equal(got, ref, B)


def test_verify_zero_sum_residual_fallback():
    """q >= r everywhere at some nodes: the first rejection leaves a zero-sum
    residual and the state must stay r (then a sample from p)."""
    w = W.small_random(44, B=6, n_range=(2, 40), prefix_range=(0, 1), Hq=2, Hkv=1, D=64, V=33000, block_size=16)
    g = np.random.default_rng(5)
    for t in range(w.T):
        if g.random() < 0.5:
            r0, _, _ = O.residual(w.p_logits[t].numpy(), np.zeros(w.V, np.float32), 0)
            w.q_probs[t] = torch.from_numpy((r0 * np.float32(1.001)).astype(np.float32))
    w.uniforms[:, 0] = -1  # every acceptance word at its maximum: many rejections
    ref = oracle_stochastic(w)
    got = _gpu_verify(w, "stochastic")
    _assert_verify_equal(got, ref, w.B)


@pytest.mark.parametrize("mode", ["greedy", "stochastic"])
def test_verify_bad_inputs(mode):
    w = W.small_random(41, B=4, n_range=(3, 8), prefix_range=(0, 1), Hq=2, Hkv=1, D=64, V=50, block_size=16)
    off = w.tree_off.numpy()
    w.tokens[off[1] + 1] = 50          # out of range token
    w.tokens[off[2]] = -3              # bad root token
    w.parent[off[3] + 2] = 2           # parent not before child
    ref = oracle_greedy(w) if mode == "greedy" else oracle_stochastic(w)
    got = _gpu_verify(w, mode)
    _assert_verify_equal(got, ref, w.B)
    assert got["status"][0] == 0 and got["status"][1] == S.SPEC_DEV_BAD_TOKEN
    assert got["status"][3] & S.SPEC_DEV_BAD_TREE


def test_verify_empty_requests():
    """Requests with no tree nodes are idle: accept_len 0, rows of -1, status 0."""
    g = np.random.Generator(np.random.PCG64(42))
    sizes = [0, 5, 0, 0, 3]
    pars = [W.random_parent_tree(n, g) if n else torch.zeros(0, dtype=torch.int32) for n in sizes]
    toks = [torch.from_numpy(g.integers(0, 50, n).astype(np.int32)) for n in sizes]
    T = sum(sizes)
    logits = torch.from_numpy(g.standard_normal((T, 50)).astype(np.float32))
    draft = torch.softmax(logits + 1, -1)
    w = W.gen._pack("empty requests", len(sizes), 2, 1, 64, W.BF16, 50, 8, 16, pars, toks, [3] * len(sizes), g,
                    logits, draft)
    for mode in ("greedy", "stochastic"):
        ref = oracle_greedy(w) if mode == "greedy" else oracle_stochastic(w)
        got = _gpu_verify(w, mode)
        _assert_verify_equal(got, ref, w.B)
        assert got["accept_len"].tolist() == [0, ref["accept_len"][1], 0, 0, ref["accept_len"][4]]


@pytest.mark.parametrize("which", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("mode", ["greedy", "stochastic"])
def test_verify_parity_workloads(which, mode):
    """The pages' workloads at full size (configs 0-3; 4 = its default sweep point)."""
    w = _workload(which)
    ref = oracle_greedy(w) if mode == "greedy" else oracle_stochastic(w)
    got = _gpu_verify(w, mode)
    _assert_verify_equal(got, ref, w.B)
    assert (got["status"][:w.B] == 0).all()


def test_verify_philox_uniforms_from_both_sides():
    """Workload 0 as specified: stochastic verification with Philox words from
    seed 0 (each side generates its own; the words match bit for bit)."""
    w = W.make_config(0)
    w.uniforms = torch.from_numpy(O.philox_uniforms(0, 0, w.tree_off.numpy()).view(np.int32))
    ref = oracle_stochastic(w)
    vp = _pass(w)
    S.spec_philox_uniforms(0, 0, vp.batch.tree_off, w.B, w.n_max, vp.batch.uniforms)
    vp.mask_build()
    vp.verify("stochastic")
    torch.cuda.synchronize()
    assert vp.path.cpu().numpy()[0].tolist() == ref["path"][0].tolist()
    assert vp.emitted.cpu().numpy()[0].tolist() == ref["emitted"][0].tolist()


def test_stochastic_gpu_matches_oracle_on_monte_carlo_trees():
    """The oracle's Monte-Carlo losslessness workload through the GPU verifier:
    identical emitted tokens trial by trial (hence the same distribution)."""
    from test_oracle_pins import mc_tree_inputs
    V, N = 8, 20000
    c, _ = mc_tree_inputs(N, V, 3, 2, 11)
    r = O.verify_stochastic(**c)
    B, n_max, dev = len(c["tree_off"]) - 1, c["n_max"], "cuda"
    path = torch.zeros((B, n_max), dtype=torch.int32, device=dev)
    alen = torch.zeros(B, dtype=torch.int32, device=dev)
    emit = torch.zeros((B, n_max), dtype=torch.int32, device=dev)
    nem = torch.zeros(B, dtype=torch.int32, device=dev)
    st = torch.zeros(B, dtype=torch.int32, device=dev)
    ws = torch.empty(S.spec_verify_workspace_size(B, n_max, V), dtype=torch.uint8, device=dev)

    def d(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    S.spec_tree_verify_stochastic(d(c["p_logits"]), d(c["q_probs"]), d(c["tokens"]), d(c["parent"]),
                                  d(c["tree_off"]), d(c["uniforms"].view(np.int32)), B, n_max, V, path, alen, emit,
                                  nem, ws, st)
    torch.cuda.synchronize()
    assert np.array_equal(emit.cpu().numpy(), r["emitted"])
    assert np.array_equal(alen.cpu().numpy(), r["accept_len"])


# ------------------------------------ temperature and per-child draft rows ----

def _gpu_verify_opts(w, inv_temp=None, q_layout=S.SPEC_Q_PER_PARENT, ws_bytes=None):
    vp = _pass(w)
    if ws_bytes is not None:  # 256 bytes: no room for row statistics, the walk makes them
        vp.verify_ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    vp.mask_build()
    tau = None if inv_temp is None else torch.from_numpy(np.asarray(inv_temp, np.float32)).cuda()
    vp.verify("stochastic", inv_temp=tau, q_layout=q_layout)
    torch.cuda.synchronize()
    return dict(path=vp.path.cpu().numpy(), accept_len=vp.accept_len.cpu().numpy(),
                emitted=vp.emitted.cpu().numpy(), n_emitted=vp.n_emitted.cpu().numpy(),
                status=vp.status.cpu().numpy())


def _oracle_opts(w, inv_temp=None, q_per_child=False):
    return O.verify_stochastic(w.p_logits.numpy(), w.q_probs.numpy(), w.tokens.numpy(), w.parent.numpy(),
                               w.tree_off.numpy(), w.uniforms.numpy().view(np.uint32), w.n_max,
                               inv_temp=inv_temp, q_per_child=q_per_child)


OPTS_VERIFY = [c for c in SMALL_VERIFY if c["V"] in (7, 64, 1000, 4099, 32000, 128256)]


@pytest.mark.parametrize("cfg", OPTS_VERIFY, ids=lambda c: f"V{c['V']}_s{c['seed']}")
@pytest.mark.parametrize("ws", ["full", "256"])
@pytest.mark.parametrize("layout", [S.SPEC_Q_PER_PARENT, S.SPEC_Q_PER_CHILD])
def test_stochastic_temperature_and_layout_parity(cfg, ws, layout):
    """Per-request inverse temperatures (0.3 ... 4) and both draft-row
    layouts, with and without row statistics: every output bit-exact."""
    w = W.small_random(cfg["seed"] + 100, B=cfg["B"], n_range=cfg["n_range"], prefix_range=(0, 4), Hq=2, Hkv=1,
                       D=64, V=cfg["V"], block_size=16)
    g = np.random.default_rng(cfg["seed"])
    # draft rows away from the target: rejections, and several residual steps per node, are common
    w.q_probs = torch.softmax(torch.from_numpy(g.standard_normal((w.T, w.V)).astype(np.float32)) * 3, -1)
    tau = g.choice(np.array([0.3, 0.7, 1.0, 1.6, 4.0], np.float32), w.B)
    ref = _oracle_opts(w, tau, layout == S.SPEC_Q_PER_CHILD)
    got = _gpu_verify_opts(w, tau, layout, None if ws == "full" else 256)
    _assert_verify_equal(got, ref, w.B)
    assert (got["status"][:w.B] == 0).all()


@pytest.mark.parametrize("ws", ["full", "256"])
def test_per_child_star_with_frozen_residuals(ws):
    """A 120-child star per request with per-child rows; a third of the
    children have an all-ones row, so rejecting them leaves a zero-sum
    residual (the state freezes after a varying number of steps), and every
    acceptance word is at its maximum."""
    n, V, B = 121, 4099, 3
    g = np.random.default_rng(9)
    w = W.small_random(45, B=B, n_range=(n, n), prefix_range=(0, 1), Hq=2, Hkv=1, D=64, V=V, block_size=16)
    w.parent = torch.cat([torch.tensor([-1] + [0] * (n - 1), dtype=torch.int32)] * B)
    q = torch.softmax(torch.from_numpy(g.standard_normal((w.T, V)).astype(np.float32)) * 3, -1)
    ones = torch.from_numpy(g.random(w.T) < 0.33)
    q[ones] = 1.0
    w.q_probs = q
    w.uniforms[:, 0] = -1
    ref = _oracle_opts(w, None, True)
    got = _gpu_verify_opts(w, None, S.SPEC_Q_PER_CHILD, None if ws == "full" else 256)
    _assert_verify_equal(got, ref, B)


@pytest.mark.parametrize("which", [1, 2])
def test_temperature_and_per_child_at_full_size(which):
    """The decode-layer and ensemble workloads at full size, verified at
    per-request temperatures and with per-child draft rows: bit-exact."""
    w = _workload(which)
    g = np.random.default_rng(which)
    tau = g.choice(np.array([0.5, 0.8, 1.25, 2.0], np.float32), w.B)
    for layout in (S.SPEC_Q_PER_PARENT, S.SPEC_Q_PER_CHILD):
        ref = _oracle_opts(w, tau, layout == S.SPEC_Q_PER_CHILD)
        got = _gpu_verify_opts(w, tau, layout)
        _assert_verify_equal(got, ref, w.B)
        assert (got["status"][:w.B] == 0).all()


def test_bad_inverse_temperature_status():
    w = W.small_random(46, B=6, n_range=(2, 9), prefix_range=(0, 1), Hq=2, Hkv=1, D=64, V=1000, block_size=16)
    tau = np.array([0.0, -1.0, np.inf, np.nan, 1.0, 0.5], np.float32)
    ref = _oracle_opts(w, tau)
    got = _gpu_verify_opts(w, tau)
    _assert_verify_equal(got, ref, w.B)
    assert got["status"].tolist()[:4] == [S.SPEC_DEV_BAD_TEMP] * 4 and got["status"][4] == got["status"][5] == 0


def test_per_child_gpu_matches_oracle_on_monte_carlo_trees():
    """The oracle's per-child Monte-Carlo workload (siblings from different
    draft rows) through the GPU verifier, trial by trial, at tau = 1 and 2."""
    from test_oracle_pins import mc_tree_inputs
    V, N = 8, 20000
    c, _ = mc_tree_inputs(N, V, 3, 2, 21, per_child=True)
    B, n_max, dev = len(c["tree_off"]) - 1, c["n_max"], "cuda"

    def d(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    for tau_v in (1.0, 2.0):
        tau = np.full(B, tau_v, np.float32)
        r = O.verify_stochastic(**c, inv_temp=tau, q_per_child=True)
        outs = [torch.zeros((B, n_max), dtype=torch.int32, device=dev), torch.zeros(B, dtype=torch.int32, device=dev),
                torch.zeros((B, n_max), dtype=torch.int32, device=dev), torch.zeros(B, dtype=torch.int32, device=dev)]
        st = torch.zeros(B, dtype=torch.int32, device=dev)
        ws = torch.empty(S.spec_verify_workspace_size(B, n_max, V), dtype=torch.uint8, device=dev)
        S.spec_tree_verify_stochastic(d(c["p_logits"]), d(c["q_probs"]), d(c["tokens"]), d(c["parent"]),
                                      d(c["tree_off"]), d(c["uniforms"].view(np.int32)), B, n_max, V, *outs, ws, st,
                                      inv_temp=d(tau), q_layout=S.SPEC_Q_PER_CHILD)
        torch.cuda.synchronize()
        assert np.array_equal(outs[2].cpu().numpy(), r["emitted"])
        assert np.array_equal(outs[1].cpu().numpy(), r["accept_len"])


# ----------------------------------------------------- tree construction ----

def _t(x, dtype=None):
    return torch.from_numpy(np.ascontiguousarray(x if dtype is None else x.astype(dtype))).cuda()


@pytest.mark.parametrize("B,F,V,k,kind", [(3, 1, 64, 4, "ints"), (5, 3, 1001, 3, "nan"), (2, 7, 32000, 8, "normal"),
                                          (4, 2, 517, 17, "ints"), (1, 5, 4096, 32, "zeros"), (2, 4, 7, 7, "normal"),
                                          (6, 2, 128256, 16, "normal"), (3, 3, 33, 1, "ints")])
def test_expand_level_parity(B, F, V, k, kind):
    """One expansion level: every child's parent and token equal the
    oracle's (ties by token id, NaN last, -0 == +0), aligned and unaligned rows."""
    g = np.random.default_rng(B * 100 + k)
    if kind == "ints":
        sc = g.integers(-3, 3, (B * F, V)).astype(np.float32)
    elif kind == "zeros":
        sc = np.where(g.random((B * F, V)) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
        sc[:, 100] = 1.0
    else:
        sc = g.standard_normal((B * F, V)).astype(np.float32)
    if kind == "nan":
        sc[g.random(sc.shape) < 0.3] = np.nan
        sc[0, :] = np.nan
    level_start = 1
    n_total = level_start + F + F * k + 2
    par = np.full(B * n_total, -5, np.int32)
    tok = np.full(B * n_total, -5, np.int32)
    O.tree_expand_level(sc, F, k, level_start, par, tok, n_total)
    gp, gt = _t(np.full(B * n_total, -5, np.int32)), _t(np.full(B * n_total, -5, np.int32))
    S.spec_tree_expand_level(_t(sc), B, F, V, k, level_start, n_total, gp, gt)
    torch.cuda.synchronize()
    assert gp.cpu().numpy().tolist() == par.tolist()
    assert gt.cpu().numpy().tolist() == tok.tolist()


def test_expansion_schedule_then_verify():
    """The decode layer's schedule <4,2,2,1,1,1,1,1> (V = 32000, 8 requests)
    built level by level on the device from per-level draft rows, equal to
    the oracle's tree; the built trees then go through mask build and greedy
    verification."""
    B, V, sched = 8, 32000, [4, 2, 2, 1, 1, 1, 1, 1]
    g = np.random.default_rng(77)
    sizes = [1]
    for k in sched:
        sizes.append(sizes[-1] * k)
    n_total = sum(sizes)
    rows = [g.standard_normal((B * sizes[lev], V)).astype(np.float32) for lev in range(len(sched))]
    roots = g.integers(0, V, B).astype(np.int32)
    par_ref, tok_ref, off_ref = O.tree_expand(roots, lambda lev, ids: rows[lev], sched, V)
    tree_off = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    par = torch.full((B * n_total,), -9, dtype=torch.int32, device="cuda")
    tok = torch.full((B * n_total,), -9, dtype=torch.int32, device="cuda")
    S.spec_tree_init(_t(roots), B, n_total, tree_off, par, tok)
    start = 0
    for lev, k in enumerate(sched):
        S.spec_tree_expand_level(_t(rows[lev]), B, sizes[lev], V, k, start, n_total, par, tok)
        start += sizes[lev]
    torch.cuda.synchronize()
    assert tree_off.cpu().tolist() == off_ref.tolist()
    assert par.cpu().numpy().tolist() == par_ref.tolist()
    assert tok.cpu().numpy().tolist() == tok_ref.tolist()
    # the built trees are valid input for the rest of the pass
    w = W.small_random(78, B=B, n_range=(n_total, n_total), prefix_range=(0, 1), Hq=2, Hkv=1, D=64, V=V,
                       block_size=16)
    w.parent, w.tokens = torch.from_numpy(par_ref), torch.from_numpy(tok_ref)
    got = _gpu_verify(w, "greedy")
    ref = oracle_greedy(w)
    _assert_verify_equal(got, ref, B)
    assert (got["status"][:B] == 0).all()


def _merge_gpu(seqs, lens, roots, V):
    B, M, m = seqs.shape
    cap = max(1, B * (1 + M * m))
    out = dict(tree_off=torch.full((B + 1,), -3, dtype=torch.int32, device="cuda"),
               parent=torch.full((cap,), -3, dtype=torch.int32, device="cuda"),
               tokens=torch.full((cap,), -3, dtype=torch.int32, device="cuda"),
               src=torch.full((cap,), -3, dtype=torch.int32, device="cuda"),
               node_of=torch.full((max(1, B * M * m),), -3, dtype=torch.int32, device="cuda"),
               status=torch.full((max(B, 1),), -3, dtype=torch.int32, device="cuda"))
    S.spec_tree_merge(_t(seqs, np.int32) if seqs.size else None, _t(lens, np.int32) if lens.size else None,
                      _t(roots, np.int32) if B else None, B, M, m, V, out["tree_off"], out["parent"],
                      out["tokens"], out["src"], out["node_of"], out["status"])
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in out.items()}
    T = int(got["tree_off"][-1])
    for k in ("parent", "tokens", "src"):
        got[k] = got[k][:T]
    got["node_of"] = got["node_of"][:B * M * m].reshape(B, M, m)
    got["status"] = got["status"][:B]
    return got


@pytest.mark.parametrize("B,M,m,V", [(5, 4, 8, 3), (1500, 3, 5, 4), (7, 31, 33, 2), (2, 31, 33, 100000),
                                     (3, 1, 9, 50), (4, 16, 1, 5), (2, 0, 4, 5), (0, 4, 4, 5)])
def test_merge_parity(B, M, m, V):
    """Merged trees equal the oracle's: offsets, parents, tokens, sources,
    the prefix-to-node map and statuses (bad lengths and tokens included;
    1500 requests take the offset scan over two rounds; 31 full sequences of
    33 distinct tokens come close to the 1024-node limit)."""
    g = np.random.default_rng(B + M + m)
    seqs = g.integers(0, V, (B, M, m)).astype(np.int32)
    lens = g.integers(0, m + 1, (B, M)).astype(np.int32)
    if V >= 100000:
        lens[:] = m
    if B > 3 and M > 0:
        lens[1, 0] = m + 1          # bad length
        seqs[2, 0, 0] = V           # bad token (inside the length)
        lens[2, 0] = max(lens[2, 0], 1)
        seqs[3, M - 1, m - 1] = -1  # outside the length: ignored
        lens[3, M - 1] = m - 1
    if B > 0 and M > 1:
        seqs[0, 1] = seqs[0, 0]     # an identical draft
    roots = g.integers(0, V, B).astype(np.int32)
    ref = O.tree_merge(seqs, lens, roots, V)
    got = _merge_gpu(seqs, lens, roots, V)
    for k in ("tree_off", "parent", "tokens", "src", "node_of", "status"):
        assert np.array_equal(got[k], ref[k]), k
    if B > 3 and M > 0:
        assert ref["status"][1] == S.SPEC_DEV_BAD_TREE and ref["status"][2] == S.SPEC_DEV_BAD_TOKEN


# --------------------------------------------- graphs per <tokens, K> ----

def test_graph_cache_per_tokens_and_k():
    """Full graphs of the pass for the <tokens, K> keys with tokens divisible
    by K + 1: each key's first use captures, a replay verifies its batch as
    the oracle does, and new inputs copied into the same buffers replay
    correctly as well."""
    from tree_speculative_verification_spec_gb300.dynamic_k import GraphCache
    keys = [key for key in S.spec_dsd_graph_keys(12, 3) if key[0] in (8, 12)]
    assert keys == [(8, 1), (8, 3), (12, 1), (12, 2), (12, 3)]
    works = {}

    def make(tokens, K):
        w = W.config4(K=K, B=tokens // (K + 1), tree="chain", alpha=0.3, seed=60, prefix=80, V=1000)
        works[(tokens, K)] = w
        return VerifyPass(DeviceBatch.from_workload(w))

    cache = GraphCache(make)
    for key in keys:
        vp = cache.replay(*key)
        torch.cuda.synchronize()
        w = works[key]
        ref = oracle_stochastic(w)
        got = dict(path=vp.path.cpu().numpy(), accept_len=vp.accept_len.cpu().numpy(),
                   emitted=vp.emitted.cpu().numpy(), n_emitted=vp.n_emitted.cpu().numpy(),
                   status=vp.status.cpu().numpy())
        _assert_verify_equal(got, ref, w.B)
    assert cache.keys() == keys
    # new inputs into the captured buffers of one key
    key = (12, 2)
    w2 = W.config4(K=2, B=4, tree="chain", alpha=0.3, seed=61, prefix=80, V=1000)
    vp = cache.pass_for(*key)
    for name in ("tokens", "p_logits", "q_probs", "uniforms", "q"):
        getattr(vp.batch, name).copy_(getattr(w2, name))
    vp = cache.replay(*key)
    torch.cuda.synchronize()
    ref = oracle_stochastic(w2)
    assert np.array_equal(vp.emitted.cpu().numpy()[:4], ref["emitted"][:4])
    assert np.array_equal(vp.accept_len.cpu().numpy()[:4], ref["accept_len"][:4])


# ------------------------------------------------------------- attention ----

def _gpu_attention(w, flags=S.SPEC_ATTN_AUTO, max_prefix=None):
    vp = _pass(w, max_prefix=max_prefix)
    vp.mask_build()
    vp.attention(flags)
    torch.cuda.synchronize()
    return out_as_f32(vp.out, w.dtype), vp.status.cpu().numpy()


ATTN_CASES = [
    dict(seed=1, B=3, n_range=(1, 40), prefix_range=(0, 300), Hq=8, Hkv=2, D=64, dtype=W.F32, block_size=16),
    dict(seed=2, B=2, n_range=(1, 20), prefix_range=(100, 700), Hq=4, Hkv=4, D=128, dtype=W.F32, block_size=8),
    dict(seed=3, B=3, n_range=(1, 70), prefix_range=(0, 900), Hq=8, Hkv=2, D=128, dtype=W.BF16, block_size=16),
    dict(seed=4, B=2, n_range=(30, 130), prefix_range=(0, 1500), Hq=32, Hkv=8, D=128, dtype=W.BF16,
         block_size=128),
    dict(seed=5, B=4, n_range=(1, 9), prefix_range=(1, 520), Hq=16, Hkv=2, D=64, dtype=W.BF16, block_size=64),
    dict(seed=6, B=1, n_range=(200, 200), prefix_range=(0, 0), Hq=8, Hkv=1, D=128, dtype=W.BF16, block_size=256),
]


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: f"s{c['seed']}_D{c['D']}_{'f32' if c['dtype'] == 0 else 'bf16'}")
@pytest.mark.parametrize("flags", [S.SPEC_ATTN_AUTO, S.SPEC_ATTN_CUDA_CORE, S.SPEC_ATTN_TCGEN05])
def test_attention_parity_small(case, flags):
    if flags == S.SPEC_ATTN_TCGEN05 and case["dtype"] != W.BF16:
        pytest.skip("the tensor-core path takes bf16")
    c = dict(case)
    w = W.small_random(c.pop("seed"), V=16, **c)
    ref, _, s_ref = oracle_attention(w)
    got, st = _gpu_attention(w, flags)
    assert np.array_equal(st[:w.B], s_ref)
    ref32 = ref.astype(np.float32) if w.dtype == W.F32 else (ref.astype(np.uint32) << 16).view(np.float32)
    ok = attn_tolerance_ok(got.reshape(ref32.shape), ref32, w.dtype)
    assert ok.all(), float(np.abs(got.reshape(ref32.shape) - ref32).max())


TC_CASES = [  # (B, n_range, prefix_range, Hq, Hkv, D, block_size)
    (2, (1, 40), (0, 0), 8, 2, 128, 8),
    (3, (20, 64), (100, 600), 32, 8, 128, 16),
    (2, (1, 33), (120, 129), 16, 4, 128, 32),
    (2, (60, 200), (0, 400), 8, 1, 128, 64),
    (1, (30, 40), (3000, 5000), 32, 8, 128, 256),  # long prefix: several key splits
    (2, (5, 90), (200, 700), 16, 4, 64, 16),
    (1, (128, 128), (127, 127), 4, 1, 64, 512),
    (4, (1, 3), (1, 2000), 32, 8, 128, 128),        # few rows: padded 128-row tile
    # more CTAs than SMs (the multi-wave instantiation): D 64 with Q by TMA,
    # and g = 3 (Q staged by the threads)
    (64, (20, 60), (50, 300), 16, 4, 64, 16),
    (48, (10, 40), (30, 200), 12, 4, 128, 16),
    (2, (5, 40), (50, 300), 6, 2, 128, 16),          # one wave, g = 3 (Q staged by the threads)
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: f"B{c[0]}_D{c[5]}_bs{c[6]}_P{c[2][1]}")
def test_attention_tcgen05_layouts(case):
    B, nr, pr, Hq, Hkv, D, bs = case
    w = W.small_random(sum(nr) + pr[1] + bs, B=B, n_range=nr, prefix_range=pr, Hq=Hq, Hkv=Hkv, D=D, dtype=W.BF16,
                       V=16, block_size=bs)
    ref, _, s_ref = oracle_attention(w)
    got, st = _gpu_attention(w, S.SPEC_ATTN_TCGEN05)
    assert (st[:w.B] == 0).all() and (s_ref == 0).all()
    ref32 = (ref.astype(np.uint32) << 16).view(np.float32)
    g = got.reshape(ref32.shape)
    bad = ~attn_tolerance_ok(g, ref32, w.dtype)
    assert not bad.any(), (int(bad.sum()), float(np.abs(g - ref32).max()), np.argwhere(bad)[:5].tolist())


def test_attention_parity_workload0():
    w = W.make_config(0)
    ref, _, s_ref = oracle_attention(w)
    got, st = _gpu_attention(w)
    assert (st[:1] == 0).all()
    assert np.abs(got.reshape(ref.shape) - ref).max() <= 1e-5


def test_attention_capacity_and_bad_blocks():
    w = W.small_random(9, B=3, n_range=(3, 9), prefix_range=(10, 60), Hq=4, Hkv=2, D=64, dtype=W.BF16, V=16,
                       block_size=16)
    w.prefix_len[0] = w.block_table.shape[1] * 16  # beyond the block table
    w.block_table[1, 0] = w.num_blocks + 5         # bad block id
    _, _, s_ref = oracle_attention(w)
    got, st = _gpu_attention(w, max_prefix=int(w.prefix_len.max()))
    assert st[0] & S.SPEC_DEV_CAPACITY and st[1] & S.SPEC_DEV_BAD_BLOCK and st[2] == 0
    assert s_ref[0] & O.ST_CAPACITY and s_ref[1] & O.ST_BAD_BLOCK


@pytest.mark.parametrize("extra", [0, 1])
def test_attention_one_wave_boundary(extra):
    # exactly one CTA per SM (the one-wave instantiation), then one more (the
    # multi-wave one): one kv-head and at most 128 rows per request, so the
    # grid has B CTAs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    w = W.small_random(40 + extra, B=sms + extra, n_range=(1, 32), prefix_range=(1, 200), Hq=4, Hkv=1, D=128,
                       dtype=W.BF16, V=16, block_size=16)
    ref, _, s_ref = oracle_attention(w)
    got, st = _gpu_attention(w, S.SPEC_ATTN_TCGEN05)
    assert (st[:w.B] == 0).all() and (s_ref == 0).all()
    ref32 = (ref.astype(np.uint32) << 16).view(np.float32)
    g = got.reshape(ref32.shape)
    bad = ~attn_tolerance_ok(g, ref32, w.dtype)
    assert not bad.any(), (int(bad.sum()), float(np.abs(g - ref32).max()))


def test_attention_capacity_and_bad_blocks_multi_wave():
    # 200 requests x 2 kv-heads: more CTAs than SMs
    w = W.small_random(10, B=200, n_range=(2, 6), prefix_range=(10, 60), Hq=4, Hkv=2, D=128, dtype=W.BF16, V=16,
                       block_size=16)
    w.prefix_len[7] = w.block_table.shape[1] * 16  # beyond the block table
    w.block_table[150, 0] = w.num_blocks + 5       # bad block id
    ref, _, s_ref = oracle_attention(w)
    got, st = _gpu_attention(w, S.SPEC_ATTN_TCGEN05, max_prefix=int(w.prefix_len.max()))
    flagged = {7: S.SPEC_DEV_CAPACITY, 150: S.SPEC_DEV_BAD_BLOCK}
    for b in range(w.B):
        assert st[b] == flagged.get(b, 0), (b, int(st[b]))
    assert s_ref[7] & O.ST_CAPACITY and s_ref[150] & O.ST_BAD_BLOCK
    # rows of the other requests match the oracle
    ref32 = (ref.astype(np.uint32) << 16).view(np.float32)
    g = got.reshape(ref32.shape)
    to = w.tree_off.numpy()
    keep = np.ones(w.T, bool)
    for b in flagged:
        keep[to[b]:to[b + 1]] = False
    bad = ~attn_tolerance_ok(g[keep], ref32[keep], w.dtype)
    assert not bad.any(), int(bad.sum())


def _sampled_rows(w, k, seed):
    g = np.random.default_rng(seed)
    return np.sort(g.choice(w.T * w.Hq, size=min(k, w.T * w.Hq), replace=False)).astype(np.int64)


@pytest.mark.parametrize("which", [1, 2, 3, 4])
def test_attention_parity_workloads_full_size(which):
    """Full-size workloads in the launch configuration of the benchmark.  The
    decode layer (16 384 rows) and the wide ensemble (16 384 rows over 8448
    keys) are checked on EVERY (node, head) row; batched serving (73k rows,
    prefixes up to 16k) and the sweep point on at least 1024 rows that include
    the first and last node of every request on every kv-head.  The oracle
    rows are computed in parallel host processes."""
    w = _workload(which)
    rows = np.arange(w.T * w.Hq, dtype=np.int64) if which in (1, 2) else rows_covering(w, 1024, which)
    assert rows.size >= 1024
    ref, s_ref = oracle_attention_rows(w, rows)
    got, st = _gpu_attention(w)
    assert (st[:w.B] == 0).all() and (s_ref == 0).all()
    ref32 = bf16_bits_to_f32(ref)
    g = got.reshape(-1, w.D)[rows]
    bad = ~attn_tolerance_ok(g, ref32, w.dtype)
    assert not bad.any(), (int(bad.sum()), float(np.abs(g - ref32).max()),
                           [divmod(int(rows[i]), w.Hq) for i in np.flatnonzero(bad.any(axis=1))[:5]])


@pytest.mark.parametrize("point", SWEEP_POINTS, ids=lambda p: f"{p[2]}_K{p[0]}_B{p[1]}_a{p[3]}")
def test_sweep_points_parity(point):
    """Linear-vs-tree sweep points (chains and random trees of K+1 nodes, small
    query-row groups on the padded tensor-core tile): sampled attention rows,
    greedy and stochastic verification exact."""
    K, B, tree, alpha = point
    w = W.config4(K=K, B=B, tree=tree, alpha=alpha)
    rows = _sampled_rows(w, 48, K * 1000 + B)
    ref, _, s_ref = oracle_attention(w, rows=rows)
    got, st = _gpu_attention(w)
    assert (st[:w.B] == 0).all() and (s_ref == 0).all()
    ref32 = (ref.astype(np.uint32) << 16).view(np.float32).reshape(-1, w.D)[rows]
    assert attn_tolerance_ok(got.reshape(-1, w.D)[rows], ref32, w.dtype).all()
    for mode in ("greedy", "stochastic"):
        ref_v = oracle_greedy(w) if mode == "greedy" else oracle_stochastic(w)
        _assert_verify_equal(_gpu_verify(w, mode), ref_v, w.B)


@pytest.mark.parametrize("tree", ["chain", "random"])
def test_stochastic_with_and_without_row_statistics(tree):
    """Large batches verify with precomputed row statistics (a workspace of
    spec_verify_workspace_size bytes); a 256-byte workspace makes the walk
    compute them itself.  Both equal the oracle bit for bit."""
    w = W.config4(K=6, B=80, tree=tree, alpha=0.4, prefix=16)
    ref = oracle_stochastic(w)
    d = DeviceBatch.from_workload(w)
    full = S.spec_verify_workspace_size(d.B, d.n_max, d.V)
    assert full > 256
    for ws_bytes in (full, 256):
        i32 = dict(dtype=torch.int32, device="cuda")
        path, emit = torch.full((d.B, d.n_max), 7, **i32), torch.full((d.B, d.n_max), 7, **i32)
        alen, nem, st = torch.zeros(d.B, **i32), torch.zeros(d.B, **i32), torch.zeros(d.B, **i32)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        S.spec_tree_verify_stochastic(d.p_logits, d.q_probs, d.tokens, d.parent, d.tree_off, d.uniforms, d.B,
                                      d.n_max, d.V, path, alen, emit, nem, ws, st)
        torch.cuda.synchronize()
        got = dict(path=path.cpu().numpy(), accept_len=alen.cpu().numpy(), emitted=emit.cpu().numpy(),
                   n_emitted=nem.cpu().numpy(), status=st.cpu().numpy())
        _assert_verify_equal(got, ref, w.B)


def test_workspace_canary_changes_nothing(monkeypatch):
    """With SPECTREE_WORKSPACE_CANARY=1 every workspace is filled with 0xFF
    (NaN) before use: split-KV attention (long prefix, several key splits)
    and stochastic verification with row statistics still equal the oracle,
    so neither reads scratch it did not write."""
    monkeypatch.setenv("SPECTREE_WORKSPACE_CANARY", "1")
    B, nr, pr, Hq, Hkv, D, bs = TC_CASES[4]
    w = W.small_random(sum(nr) + pr[1] + bs, B=B, n_range=nr, prefix_range=pr, Hq=Hq, Hkv=Hkv, D=D, dtype=W.BF16,
                       V=16, block_size=bs)
    d = DeviceBatch.from_workload(w)
    assert S.spec_attention_workspace_size(d.B, d.T, d.n_max, d.max_prefix, d.Hq, d.Hkv, d.D) > 256  # splits
    ref, _, _ = oracle_attention(w)
    got, st = _gpu_attention(w, S.SPEC_ATTN_TCGEN05)
    ref32 = (ref.astype(np.uint32) << 16).view(np.float32)
    assert attn_tolerance_ok(got.reshape(ref32.shape), ref32, w.dtype).all() and (st[:w.B] == 0).all()
    w2 = W.config4(K=6, B=80, tree="random", alpha=0.4, prefix=16)
    ref2 = oracle_stochastic(w2)
    got2 = _gpu_verify(w2, "stochastic")  # full workspace: row statistics
    _assert_verify_equal(got2, ref2, w2.B)


# ---------------------------------------------------------------- append ----

def _oracle_append(w, k_new, v_new, status=None):
    st = np.zeros(w.B, np.int32) if status is None else status
    return O.kv_append(np_elems(k_new, w.dtype), np_elems(v_new, w.dtype), np_elems(w.k_cache, w.dtype),
                       np_elems(w.v_cache, w.dtype), w.block_table.numpy(), w.block_size, w.prefix_len.numpy(),
                       w.tree_off.numpy(), w.n_max, w.Hkv, w.D, w.dtype, st)


@pytest.mark.parametrize("dtype,D,bs", [(W.BF16, 128, 16), (W.F32, 64, 8), (W.BF16, 64, 256), (W.F32, 128, 512)])
def test_kv_append_parity(dtype, D, bs):
    """Tree K/V rows into slots prefix + u, byte-exact against the oracle:
    ragged and empty trees, a request past its block table, a bad block id
    among a tree's pages."""
    w = W.small_random(40 + bs, B=7, n_range=(0, 70), prefix_range=(0, 600), Hq=8, Hkv=2, D=D, dtype=dtype,
                       block_size=bs, n_max=80)
    k_new, v_new = W.tree_kv_rows(w, bs)
    n = (w.tree_off[1:] - w.tree_off[:-1]).numpy()
    big = [b for b in range(w.B) if n[b] > 0]
    w.prefix_len[big[0]] = w.block_table.shape[1] * bs - int(n[big[0]]) + 1  # last tree slot past the table
    b2 = big[1]
    w.block_table[b2, (int(w.prefix_len[b2]) + int(n[b2]) - 1) // bs] = w.num_blocks + 3
    k_ref, v_ref, st_ref = _oracle_append(w, k_new, v_new)
    assert st_ref[big[0]] == O.ST_CAPACITY and st_ref[b2] == O.ST_BAD_BLOCK
    d = DeviceBatch.from_workload(w)
    vp = VerifyPass(d)
    vp.status.zero_()
    vp.append(k_new.cuda(), v_new.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(vp.status.cpu().numpy()[:w.B], st_ref)
    assert np.array_equal(np_elems(d.k_cache, w.dtype), k_ref)
    assert np.array_equal(np_elems(d.v_cache, w.dtype), v_ref)


def test_kv_append_rejects_oversized_trees_and_bad_arguments():
    w = W.small_random(47, B=3, n_range=(3, 9), prefix_range=(0, 40), Hq=4, Hkv=2, D=64, dtype=W.BF16, block_size=16)
    k_new, v_new = W.tree_kv_rows(w, 1)
    d = DeviceBatch.from_workload(w)
    vp = VerifyPass(d)
    vp.status.zero_()
    k0 = d.k_cache.clone()
    S.spec_kv_append(k_new.cuda(), v_new.cuda(), d.k_cache, d.v_cache, d.block_table, d.max_blocks, d.block_size,
                     d.num_blocks, d.prefix_len, d.tree_off, d.B, 2, d.Hkv, d.D, vp.status)  # n_max 2 < n_b
    torch.cuda.synchronize()
    assert (vp.status.cpu().numpy()[:w.B] == S.SPEC_DEV_BAD_TREE).all()
    assert torch.equal(d.k_cache, k0)
    with pytest.raises(S.SpecError) as e:  # unaligned rows
        S.spec_kv_append(k_new.cuda().view(-1)[1:1 + k_new.numel() - 8].view(-1), v_new.cuda(), d.k_cache, d.v_cache,
                         d.block_table, d.max_blocks, d.block_size, d.num_blocks, d.prefix_len, d.tree_off, d.B,
                         d.n_max, d.Hkv, d.D, vp.status)
    assert e.value.code == S.SPEC_ERR_INVALID_ARG


@pytest.mark.parametrize("case", [TC_CASES[1], TC_CASES[4], TC_CASES[7]], ids=["paged16", "splits", "padded"])
def test_mask_append_attention_chain(case):
    """mask build -> append -> attention, each launched right after the other
    (the append and the tensor-core attention start before their predecessor
    ends): over a cache whose tree slots hold garbage, attention must see the
    appended rows, as the oracle's append followed by its attention does."""
    B, nr, pr, Hq, Hkv, D, bs = case
    w = W.small_random(sum(nr) + pr[1] + bs + 7, B=B, n_range=nr, prefix_range=pr, Hq=Hq, Hkv=Hkv, D=D,
                       dtype=W.BF16, V=16, block_size=bs)
    k_new, v_new = W.tree_kv_rows(w, 77)
    k_ref, v_ref, _ = _oracle_append(w, k_new, v_new)
    ref, _, s_ref = O.tree_attention(np_elems(w.q, w.dtype), k_ref, v_ref, w.block_table.numpy(), w.block_size,
                                     w.prefix_len.numpy(), w.tree_off.numpy(), w.parent.numpy(), w.n_max, w.Hq,
                                     w.Hkv, w.D, w.dtype, w.scale)
    d = DeviceBatch.from_workload(w)  # caches as generated: the tree slots hold other values
    vp = VerifyPass(d)
    kn, vn = k_new.cuda(), v_new.cuda()
    torch.cuda.synchronize()
    vp.mask_build()
    vp.append(kn, vn)
    vp.attention()
    torch.cuda.synchronize()
    assert (vp.status.cpu().numpy()[:w.B] == 0).all() and (s_ref == 0).all()
    ref32 = bf16_bits_to_f32(ref).reshape(-1, w.D)
    got = out_as_f32(vp.out, w.dtype).reshape(-1, w.D)
    bad = ~attn_tolerance_ok(got, ref32, w.dtype)
    assert not bad.any(), (int(bad.sum()), float(np.abs(got - ref32).max()))
    assert np.array_equal(np_elems(d.k_cache, w.dtype), k_ref) and np.array_equal(np_elems(d.v_cache, w.dtype), v_ref)


# ---------------------------------------------------------------- commit ----

def _oracle_commit(w, ref_v):
    st = np.zeros(w.B, np.int32)
    return O.kv_commit(np_elems(w.k_cache, w.dtype), np_elems(w.v_cache, w.dtype), w.block_table.numpy(),
                       w.block_size, w.prefix_len.numpy(), ref_v["path"], ref_v["accept_len"], w.Hkv, w.D, w.dtype,
                       st)


@pytest.mark.parametrize("dtype,D,bs", [(W.BF16, 128, 16), (W.F32, 64, 8), (W.BF16, 64, 256)])
def test_commit_parity(dtype, D, bs):
    w = W.small_random(51, B=5, n_range=(1, 70), prefix_range=(0, 200), Hq=4, Hkv=2, D=D, dtype=dtype, V=3,
                       block_size=bs)
    # tokens copy the argmax chain so paths are long
    am = w.p_logits.argmax(1)
    for b in range(w.B):
        off = int(w.tree_off[b])
        for u in range(1, int(w.tree_off[b + 1]) - off):
            w.tokens[off + u] = am[off + int(w.parent[off + u])]
    ref_v = oracle_greedy(w)
    k_ref, v_ref, nl_ref, st_ref = _oracle_commit(w, ref_v)
    vp = _pass(w)
    vp.mask_build()
    vp.verify("greedy")
    vp.commit()
    torch.cuda.synchronize()
    assert np.array_equal(vp.accept_len.cpu().numpy(), ref_v["accept_len"])
    assert (ref_v["accept_len"] > 2).any()
    assert np.array_equal(np_elems(vp.batch.k_cache, dtype), k_ref)
    assert np.array_equal(np_elems(vp.batch.v_cache, dtype), v_ref)
    assert np.array_equal(vp.new_len.cpu().numpy(), nl_ref)
    assert np.array_equal(vp.status.cpu().numpy(), st_ref)


def test_commit_bad_paths_and_failed_requests():
    w = W.small_random(52, B=3, n_range=(6, 6), prefix_range=(5, 5), Hq=2, Hkv=1, D=64, dtype=W.BF16, V=3,
                       block_size=8)
    d = DeviceBatch.from_workload(w)
    path = torch.tensor([[0, 2, 1, -1, -1, -1], [0, 1, 3, -1, -1, -1], [0, 1, -1, -1, -1, -1]], dtype=torch.int32)
    alen = torch.tensor([3, 3, 2], dtype=torch.int32)
    status = torch.tensor([0, 0, S.SPEC_DEV_BAD_TOKEN], dtype=torch.int32)
    k0, v0 = d.k_cache.clone(), d.v_cache.clone()
    new_len = torch.zeros(3, dtype=torch.int32, device="cuda")
    st = status.cuda()
    S.spec_kv_commit(d.k_cache, d.v_cache, d.block_table, d.max_blocks, d.block_size, d.num_blocks, d.prefix_len,
                     path.cuda(), 6, alen.cuda(), 3, 1, 64, new_len, st)
    torch.cuda.synchronize()
    k_ref, v_ref, nl_ref, st_ref = O.kv_commit(np_elems(w.k_cache, w.dtype), np_elems(w.v_cache, w.dtype),
                                               w.block_table.numpy(), 8, w.prefix_len.numpy(), path.numpy(),
                                               alen.numpy(), 1, 64, W.BF16, status.numpy())
    assert st.cpu().tolist() == st_ref.tolist() == [S.SPEC_DEV_BAD_PATH, 0, S.SPEC_DEV_BAD_TOKEN]
    assert new_len.cpu().tolist() == nl_ref.tolist()
    assert np.array_equal(np_elems(d.k_cache, W.BF16), k_ref)
    assert np.array_equal(np_elems(d.v_cache, W.BF16), v_ref)


def _root_paths(w, rng):
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


@pytest.mark.parametrize("dtype,D,bs,cap,B", [(W.BF16, 128, 16, 4096, 6), (W.F32, 64, 8, 4096, 6),
                                              (W.BF16, 64, 8, 3, 6), (W.BF16, 128, 16, 8192, 70)])
def test_commit_layers_and_page_release(dtype, D, bs, cap, B):
    """Three layers committed in one launch, then the page release: every
    layer's cache, new lengths, statuses, the block table and the free list
    (order included) exactly as the oracle; a short pool releases nothing.
    With 70 requests x 2 kv-heads one CTA moves several of the six caches."""
    rng = np.random.default_rng(61)
    w = W.small_random(62, B=B, n_range=(2, 60), prefix_range=(0, 90), Hq=4, Hkv=2, D=D, dtype=dtype, V=3,
                       block_size=bs)
    path, alen = _root_paths(w, rng)
    path[4, :3] = [0, 2, 1]  # not increasing: BAD_PATH, untouched
    alen[4] = 3
    status = np.zeros(w.B, np.int32)
    status[5] = S.SPEC_DEV_BAD_TOKEN  # failed upstream: untouched, keeps its pages
    L = 3
    k_layers = [np_elems(w.k_cache, dtype) for _ in range(L)]
    v_layers = [np_elems(w.v_cache, dtype) for _ in range(L)]
    for l in range(L):  # different contents per layer
        if dtype == W.F32:
            k_layers[l] = k_layers[l] + l
            v_layers[l] = v_layers[l] - l
        else:
            k_layers[l] = (k_layers[l] ^ np.uint16(l)).astype(np.uint16)
            v_layers[l] = (v_layers[l] ^ np.uint16(3 * l)).astype(np.uint16)
    ks, vs, nl_ref, st_ref, bt_ref, pool_ref, cnt_ref = O.kv_commit_layers(
        k_layers, v_layers, w.block_table.numpy(), bs, w.prefix_len.numpy(), w.tree_off.numpy(), path, alen, w.Hkv,
        D, dtype, status, cap, free_count=1)
    dev = "cuda"
    tdt = torch.float32 if dtype == W.F32 else torch.int16
    kd = [torch.from_numpy(k.view(np.int16) if dtype == W.BF16 else k).to(dev) for k in k_layers]
    vd = [torch.from_numpy(v.view(np.int16) if dtype == W.BF16 else v).to(dev) for v in v_layers]
    kp = torch.tensor([t.data_ptr() for t in kd], dtype=torch.int64, device=dev)
    vp = torch.tensor([t.data_ptr() for t in vd], dtype=torch.int64, device=dev)
    bt = w.block_table.to(dev).contiguous()
    pool = torch.full((cap,), -7, dtype=torch.int32, device=dev)
    cnt = torch.tensor([1], dtype=torch.int32, device=dev)
    new_len = torch.zeros(w.B, dtype=torch.int32, device=dev)
    st = torch.from_numpy(status).to(dev)
    S.spec_kv_commit_layers(kp, vp, L, bt, bt.shape[1], bs, w.num_blocks, w.prefix_len.to(dev), w.tree_off.to(dev),
                            torch.from_numpy(path).to(dev), path.shape[1], torch.from_numpy(alen).to(dev), w.B,
                            w.Hkv, D, dtype, new_len, pool, cnt, st)
    torch.cuda.synchronize()
    for l in range(L):
        got_k = kd[l].cpu().numpy().view(np.uint16) if dtype == W.BF16 else kd[l].cpu().numpy()
        got_v = vd[l].cpu().numpy().view(np.uint16) if dtype == W.BF16 else vd[l].cpu().numpy()
        assert np.array_equal(got_k, ks[l]) and np.array_equal(got_v, vs[l]), l
    assert new_len.cpu().tolist() == nl_ref.tolist()
    assert st.cpu().tolist() == st_ref.tolist()
    assert bt.cpu().numpy().tolist() == bt_ref.tolist()
    assert int(cnt.item()) == cnt_ref
    assert pool.cpu().numpy()[1:cnt_ref].tolist() == pool_ref[1:].tolist()
    if cap == 3:
        assert cnt_ref == 1 and any(x & S.SPEC_DEV_CAPACITY for x in st_ref)
    else:
        assert cnt_ref > 1


# ------------------------------------------------------------- full pass ----

@pytest.mark.parametrize("mode", ["stochastic", "greedy"])
def test_full_pass_workload1(mode):
    """The benchmark's pass (workload 1) end to end: mask, attention, verify,
    commit; verify and commit exact, attention on the first and last node of
    every request on every kv-head plus uniform picks."""
    w = W.make_config(1)
    ref_m = oracle_mask(w)
    ref_v = oracle_greedy(w) if mode == "greedy" else oracle_stochastic(w)
    rows = rows_covering(w, 256, 17)
    ref_a, _ = oracle_attention_rows(w, rows)
    k_ref, v_ref, nl_ref, st_ref = _oracle_commit(w, ref_v)
    vp = _pass(w)
    vp.run(mode)
    torch.cuda.synchronize()
    assert np.array_equal(vp.mask.cpu().numpy().view(np.uint64), ref_m[0])
    for k in ("path", "accept_len", "emitted", "n_emitted"):
        assert np.array_equal(getattr(vp, k).cpu().numpy(), ref_v[k]), k
    got = out_as_f32(vp.out, w.dtype).reshape(-1, w.D)[rows]
    assert attn_tolerance_ok(got, bf16_bits_to_f32(ref_a), w.dtype).all()
    assert np.array_equal(np_elems(vp.batch.k_cache, w.dtype), k_ref)
    assert np.array_equal(np_elems(vp.batch.v_cache, w.dtype), v_ref)
    assert np.array_equal(vp.new_len.cpu().numpy(), nl_ref)


def test_full_pass_workload3_greedy_then_commit():
    """The batched-serving workload as specified: 64 requests on 16-token pages
    with a random block table, greedy verification, then the KV commit: mask,
    verify, commit and new lengths exact, attention on the first and last node
    of every request on every kv-head."""
    w = _workload(3)
    ref_m = oracle_mask(w)
    ref_v = oracle_greedy(w)
    rows = rows_covering(w, 256, 33)
    ref_a, _ = oracle_attention_rows(w, rows)
    k_ref, v_ref, nl_ref, st_ref = _oracle_commit(w, ref_v)
    vp = _pass(w)
    vp.run("greedy")
    torch.cuda.synchronize()
    assert np.array_equal(vp.mask.cpu().numpy().view(np.uint64), ref_m[0])
    for k in ("path", "accept_len", "emitted", "n_emitted"):
        assert np.array_equal(getattr(vp, k).cpu().numpy(), ref_v[k]), k
    assert (ref_v["accept_len"] > 1).sum() > 0
    got = out_as_f32(vp.out, w.dtype).reshape(-1, w.D)[rows]
    assert attn_tolerance_ok(got, bf16_bits_to_f32(ref_a), w.dtype).all()
    assert np.array_equal(np_elems(vp.batch.k_cache, w.dtype), k_ref)
    assert np.array_equal(np_elems(vp.batch.v_cache, w.dtype), v_ref)
    assert np.array_equal(vp.new_len.cpu().numpy(), nl_ref)
    assert np.array_equal(vp.status.cpu().numpy()[:w.B], st_ref)


def test_full_pass_workload3_with_tree_kv_append():
    """The batched-serving pass starting from tree K/V handed over by the
    caller: mask, append, attention, greedy verification, commit.  The caches
    after the append and after the commit are byte-exact, verification exact,
    attention on the first and last node of every request on every kv-head."""
    w = _workload(3)
    k_new, v_new = W.tree_kv_rows(w, 303)
    k_app, v_app, st_app = _oracle_append(w, k_new, v_new)
    assert (st_app == 0).all()
    rows = rows_covering(w, 1024, 34)
    ref_a, _ = oracle_attention_rows(w, rows, caches=(k_app, v_app))
    ref_v = oracle_greedy(w)
    k_ref, v_ref, nl_ref, st_ref = O.kv_commit(k_app, v_app, w.block_table.numpy(), w.block_size,
                                               w.prefix_len.numpy(), ref_v["path"], ref_v["accept_len"], w.Hkv, w.D,
                                               w.dtype, np.zeros(w.B, np.int32))
    del k_app, v_app
    vp = _pass(w)
    vp.mask_build()
    vp.append(k_new.cuda(), v_new.cuda())
    vp.attention()
    got = out_as_f32(vp.out, w.dtype).reshape(-1, w.D)[rows]  # synchronises
    vp.verify("greedy")
    vp.commit()
    torch.cuda.synchronize()
    assert attn_tolerance_ok(got, bf16_bits_to_f32(ref_a), w.dtype).all()
    for k in ("path", "accept_len", "emitted", "n_emitted"):
        assert np.array_equal(getattr(vp, k).cpu().numpy(), ref_v[k]), k
    assert np.array_equal(np_elems(vp.batch.k_cache, w.dtype), k_ref)
    assert np.array_equal(np_elems(vp.batch.v_cache, w.dtype), v_ref)
    assert np.array_equal(vp.new_len.cpu().numpy(), nl_ref)
    assert np.array_equal(vp.status.cpu().numpy()[:w.B], st_ref)


# ---------------------------------------------------------- failure detection ----

def test_bounded_wait_expires_with_a_timeout_status_and_the_context_survives():
    """A wait on a barrier nothing completes ends after its limit with
    SPEC_DEV_TIMEOUT; the next call on the same context works normally."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    S.spec_selftest_bounded_wait(st, 4096)
    torch.cuda.synchronize()
    assert st.item() == S.SPEC_DEV_TIMEOUT
    test_philox_parity(0, 0)
