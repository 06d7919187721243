"""The library's dynamic-K host functions against the oracle (no GPU: these
calls launch nothing).  Integer outputs exactly; the moving average within
1e-12 relative (the two sides round the blend differently)."""
import numpy as np
import pytest

import oracle as O
import tree_speculative_verification_spec_gb300 as S


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tree_speculative_verification_spec_gb300 import build
    build.build()
    S.lib()


def test_optimal_k_matches_oracle_on_random_tables():
    rng = np.random.default_rng(4)
    for _ in range(200):
        n_bs, n_k = int(rng.integers(1, 12)), int(rng.integers(1, 10))
        al = rng.uniform(0.5, 6, (n_bs, n_k))
        itl = rng.uniform(-0.5, 3, (n_bs, n_k))
        al[rng.random(al.shape) < 0.1] = np.nan
        itl[rng.random(itl.shape) < 0.05] = np.inf
        tie = rng.random(n_bs) < 0.2  # first and last columns equal: a goodput tie
        itl[tie, 0] = itl[tie, -1]
        al[tie, 0] = al[tie, -1]
        ks = np.sort(rng.choice(np.arange(1, 20), n_k, replace=False)).astype(np.int32)
        got = np.zeros(n_bs, np.int32)
        S.spec_dsd_optimal_k(np.ascontiguousarray(al), np.ascontiguousarray(itl), ks, got)
        assert got.tolist() == O.dsd_optimal_k(al, itl, ks).tolist()


def test_select_k_matches_oracle_and_rejects_unsorted_tables():
    rng = np.random.default_rng(5)
    for _ in range(100):
        n = int(rng.integers(1, 10))
        bs = np.sort(rng.choice(np.arange(1, 600), n, replace=False)).astype(np.int32)
        ks = rng.integers(1, 9, n).astype(np.int32)
        for q in list(rng.integers(0, 700, 20)) + list(bs) + [0, int(bs[0]) - 1]:
            assert S.spec_dsd_select_k(bs, ks, int(q)) == O.dsd_select_k(bs, ks, int(q))
    with pytest.raises(S.SpecError):
        S.spec_dsd_select_k(np.array([4, 4], np.int32), np.array([1, 2], np.int32), 4)
    with pytest.raises(S.SpecError):
        S.spec_dsd_select_k(np.zeros(0, np.int32), np.zeros(0, np.int32), 4)


def test_graph_keys_match_oracle():
    for mt, mk in [(8, 3), (1, 5), (0, 3), (300, 7), (64, 1), (1000, 16)]:
        assert S.spec_dsd_graph_keys(mt, mk) == O.dsd_graph_keys(mt, mk)


def test_update_matches_the_oracle_blend():
    rng = np.random.default_rng(6)
    al = np.full((3, 4), np.nan)
    itl = np.full((3, 4), np.nan)
    ref_al, ref_itl = al.copy(), itl.copy()
    for _ in range(300):
        b, j = int(rng.integers(0, 3)), int(rng.integers(0, 4))
        a_s, t_s, w = float(rng.uniform(1, 5)), float(rng.uniform(0.1, 2)), float(rng.uniform(0.01, 1))
        S.spec_dsd_update(al, itl, b, j, a_s, t_s, w)
        ref_al[b, j] = O.dsd_blend(ref_al[b, j], a_s, w)
        ref_itl[b, j] = O.dsd_blend(ref_itl[b, j], t_s, w)
        np.testing.assert_allclose(al, ref_al, rtol=1e-12, equal_nan=True)
        np.testing.assert_allclose(itl, ref_itl, rtol=1e-12, equal_nan=True)
    with pytest.raises(S.SpecError):
        S.spec_dsd_update(al, itl, 0, 0, 1.0, 1.0, 0.0)
    with pytest.raises(S.SpecError):
        S.spec_dsd_update(al, itl, 3, 0, 1.0, 1.0, 0.5)


def test_dynamic_k_table_selects_the_goodput_optimum():
    """The policy object: measured cells (closed-form AL, a dense cost model),
    a moving-average refresh, and the runtime lookup by batch size."""
    from tree_speculative_verification_spec_gb300.dynamic_k import DynamicK
    bss, ks = [1, 8, 64, 256], [1, 2, 3, 4, 5, 6, 7]
    pol = DynamicK(bss, ks)
    with pytest.raises(ValueError):
        pol.select(4)
    alpha = 0.8
    for i, bs in enumerate(bss):
        for j, k in enumerate(ks):
            pol.record(i, j, (1 - alpha ** (k + 1)) / (1 - alpha), 10.0 + 0.05 * bs * (k + 1))
    k_opt = pol.optimal_k()
    al, itl = pol.al.copy(), pol.itl.copy()
    assert k_opt.tolist() == O.dsd_optimal_k(al, itl, np.array(ks, np.int32)).tolist()
    assert k_opt[0] >= k_opt[-1]
    assert pol.select(1) == k_opt[0] and pol.select(100) == k_opt[2] and pol.select(10 ** 4) == k_opt[3]
    # live statistics: K = 1 at batch size 1 suddenly becomes very fast
    for _ in range(40):
        pol.record(0, 0, 1.8, 0.5, weight=0.25)
    assert pol.select(1) == 1


def test_chain_prefix_keeps_each_requests_first_nodes():
    """The dynamic-K profile cuts one set of chains to every K: a chain's
    first K + 1 nodes, with the rows, tokens and uniforms of those nodes."""
    import workloads as W
    full = W.config4(K=4, B=3, tree="chain", alpha=0.3, prefix=32, V=500)
    for n in (1, 2, 5):
        w = W.chain_prefix(full, n)
        assert w.n_max == n and w.tree_off.tolist() == list(range(0, 3 * n + 1, n))
        assert w.parent.tolist() == ([-1] + list(range(n - 1))) * 3
        for b in range(3):
            src = slice(b * 5, b * 5 + n)
            dst = slice(b * n, b * n + n)
            assert np.array_equal(w.tokens[dst].numpy(), full.tokens[src].numpy())
            assert np.array_equal(w.p_logits[dst].numpy(), full.p_logits[src].numpy())
            assert np.array_equal(w.q_probs[dst].numpy(), full.q_probs[src].numpy())
            assert np.array_equal(w.uniforms[dst].numpy(), full.uniforms[src].numpy())
        assert w.k_cache is full.k_cache and w.meta["K"] == n - 1
