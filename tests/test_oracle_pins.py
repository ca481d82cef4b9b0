"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks one oracle function against something it does not compute
itself: a closed form, a hand-worked case, a library routine, an invariant of
the definitions, or brute force on tiny inputs.  Definitions followed: page
"MiniCPM4: Ultra-Efficient LLMs on End Devices" (paper-graph-ui digest),
section "InfLLM v2".
"""

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import synthetic_inputs as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- kernels ----

@pytest.mark.parametrize("L,expect", [(0, 0), (31, 0), (32, 1), (47, 1), (48, 2), (4096, 255),
                                      (32768, 2047), (131072, 8191), (131080, 8191)])
def test_kernel_count_closed_form(L, expect):
    # S_j = K[j s : j s + p] must fit in L keys: j s + p <= L.
    assert O.n_complete_kernels(L, 32, 16) == expect
    assert expect == sum(1 for j in range(L) if j * 16 + 32 <= L)


def test_compress_keys_prefix_sum_closed_form():
    rng = np.random.default_rng(5)
    for (L, p, s) in [(200, 32, 16), (97, 8, 3), (64, 64, 64), (31, 32, 16)]:
        K = rng.standard_normal((L, 6))
        Kc = O.compress_keys(K, p, s)
        P = np.concatenate([np.zeros((1, 6)), np.cumsum(K, axis=0)])
        n = O.n_complete_kernels(L, p, s)
        ref = np.array([(P[j * s + p] - P[j * s]) / p for j in range(n)]).reshape(n, 6)
        assert Kc.shape == (n, 6)
        np.testing.assert_allclose(Kc, ref, rtol=1e-12, atol=1e-12)


def test_compress_keys_arithmetic_ramp():
    # K[t] = t: the mean of t = js .. js+p-1 is js + (p-1)/2.
    L, p, s = 300, 32, 16
    K = np.arange(L, dtype=np.float64)[:, None]
    Kc = O.compress_keys(K, p, s)
    assert np.array_equal(Kc[:, 0], np.array([j * s + (p - 1) / 2 for j in range(Kc.shape[0])]))


# ------------------------------------------------------ kernel softmax ----

def test_kernel_softmax_matches_torch_softmax():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((16, 300)) * 7.0
    ref = torch.softmax(torch.from_numpy(z), dim=1).numpy()
    np.testing.assert_allclose(O.kernel_softmax(z), ref, rtol=1e-13, atol=0)


def test_group_relevance_is_head_mean_and_sums_to_one():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((16, 77))
    g = O.group_relevance(z)
    ref = torch.softmax(torch.from_numpy(z), dim=1).mean(dim=0).numpy()
    np.testing.assert_allclose(g, ref, rtol=1e-13)
    assert abs(g.sum() - 1.0) < 1e-12


# ------------------------------------------------------- block relevance ----

def _block_relevance_brute(g, i, m, p, s):
    """Max over kernels whose key set meets the block's key set (set intersection)."""
    c = i // m
    r = []
    for j in range(c + 1):
        bkeys = set(range(j * m, (j + 1) * m))
        vals = [g[k] for k in range(len(g)) if bkeys & set(range(k * s, k * s + p))]
        r.append(max(vals) if vals else -math.inf)
    return np.array(r)


@pytest.mark.parametrize("m,p,s", [(64, 32, 16), (16, 8, 4), (32, 32, 16), (8, 12, 5)])
def test_block_relevance_brute_force(m, p, s):
    rng = np.random.default_rng(m * 100 + p + s)
    for i in [0, 5, p - 1, p, m - 1, m, 3 * m + 7, 6 * m - 1, 400]:
        nv = O.visible_kernel_count(i, p, s)
        g = rng.random(nv)
        np.testing.assert_array_equal(O.block_relevance(g, i, m, p, s),
                                      _block_relevance_brute(g, i, m, p, s))


def test_block_relevance_recommended_shape_uses_kernels_4j_minus_1_to_4j_plus_3():
    i = 64 * 20 + 40
    nv = O.visible_kernel_count(i, 32, 16)
    g = np.random.default_rng(3).random(nv)
    r = O.block_relevance(g, i, 64, 32, 16)
    for j in range(r.shape[0]):
        ks = [k for k in range(4 * j - 1, 4 * j + 4) if 0 <= k < nv]
        expect = max(g[k] for k in ks) if ks else -math.inf
        assert r[j] == expect


# --------------------------------------------------------- forced blocks ----

@pytest.mark.parametrize("i,expect", [(0, [0]), (63, [0]), (64, [0, 1]), (127, [0, 1]),
                                      (128, [0, 1, 2]), (1000, [0, 14, 15]),
                                      (131071, [0, 2046, 2047])])
def test_forced_blocks_hand_cases(i, expect):
    assert O.forced_blocks(i, 64, 1, 2) == expect


# ----------------------------------------------------------------- top-k ----

def _topk_brute(r, forced, topk, includes_forced):
    """Enumerate every subset of candidates; keep those that dominate the rest."""
    fset = set(forced)
    cand = [j for j in range(len(r)) if j not in fset and np.isfinite(r[j])]
    n = max(0, (topk - len(forced)) if includes_forced else topk)
    n = min(n, len(cand))
    key = {j: (r[j], -j) for j in cand}
    good = []
    for sub in itertools.combinations(cand, n):
        rest = [j for j in cand if j not in sub]
        if all(key[a] > key[b] for a in sub for b in rest):
            good.append(sorted(fset | set(sub)))
    assert len(good) == 1
    return good[0]


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(11)
    for trial in range(60):
        nb = int(rng.integers(1, 11))
        r = rng.integers(0, 4, nb).astype(np.float64) / 4.0   # many exact ties
        r[rng.random(nb) < 0.15] = -np.inf
        i = nb * 64 - 1
        forced = O.forced_blocks(i, 64, 1, 2)
        for topk in (3, 4, 6):
            for inc in (True, False):
                got = O.top_k_blocks(r, forced, topk, inc).tolist()
                assert got == _topk_brute(r, forced, topk, inc)


def test_hand_worked_selections():
    spec = json.load(open(os.path.join(GOLDEN, "hand_selection.json")))
    st_ = spec["settings"]
    for case in spec["cases"]:
        K = np.zeros((st_["L"], st_["d"]))
        for a, b in case["spans"]:
            K[a:b, 0] = math.log(4.0)
        q = np.array(case["q_heads"], dtype=np.float64)
        Kc = O.compress_keys(K, st_["kernel"], st_["stride"])
        for topk_s, expect in case["select"].items():
            st = O.Settings(block=st_["block"], kernel=st_["kernel"], stride=st_["stride"],
                            topk=int(topk_s), n_init=st_["n_init"], n_local=st_["n_local"],
                            includes_forced=True, score_scale=st_["score_scale"])
            sel = O.select_for_query(q, Kc, st_["i"], st)
            want = [float(Fraction(a, b)) for a, b in zip(case["r_block_num"], case["r_block_den"])]
            np.testing.assert_allclose(sel.r, want, rtol=1e-14)
            assert sel.blocks.tolist() == expect, (case["name"], topk_s)
            bnd = case["boundary"][topk_s]
            if bnd is None:
                assert math.isnan(sel.boundary), (case["name"], topk_s, sel.boundary)
            else:
                assert abs(sel.boundary - float(Fraction(*bnd))) <= 1e-14, (case["name"], topk_s, sel.boundary)


# --------------------------------------------------- selection invariants ----

def _rand_case(seed, L=1500, G=16, d=8):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((G, d)), rng.standard_normal((L, d))


def test_selection_key_shift_invariance():
    q, K = _rand_case(4)
    st = O.Settings(topk=8, score_scale=1.0)
    i = K.shape[0] - 1
    base = O.select_for_query(q, O.compress_keys(K, 32, 16), i, st)
    shifted = O.select_for_query(q, O.compress_keys(K + np.array([0.5, -1.25, 2.0, 0, 0, 1, 0, -3.0]), 32, 16), i, st)
    np.testing.assert_allclose(shifted.r, base.r, rtol=1e-9)
    assert shifted.blocks.tolist() == base.blocks.tolist()


def test_selection_head_permutation_invariance():
    q, K = _rand_case(5)
    st = O.Settings(topk=8)
    Kc = O.compress_keys(K, 32, 16)
    i = K.shape[0] - 1
    base = O.select_for_query(q, Kc, i, st)
    perm = O.select_for_query(q[np.random.default_rng(0).permutation(16)], Kc, i, st)
    np.testing.assert_allclose(perm.r, base.r, rtol=1e-12)
    assert perm.blocks.tolist() == base.blocks.tolist()


def test_selection_structural_invariants():
    q, K = _rand_case(6, L=2000)
    Kc = O.compress_keys(K, 32, 16)
    for inc in (True, False):
        st = O.Settings(topk=10, includes_forced=inc)
        for i in [0, 20, 31, 63, 64, 100, 640, 1999]:
            sel = O.select_for_query(q, Kc, i, st)
            c = i // 64
            forced = O.forced_blocks(i, 64, 1, 2)
            assert set(forced) <= set(sel.blocks.tolist())
            assert sel.blocks.max() <= c and sel.blocks.tolist() == sorted(set(sel.blocks.tolist()))
            n_vis_blocks = c + 1
            want = min(10, n_vis_blocks) if inc else min(10 + len(forced), n_vis_blocks)
            assert len(sel.blocks) == want, (i, inc)


# ------------------------------------------- coarse-LSE approximation ----

def test_window_means_prefix_sum_and_ramp():
    # Coarse kernels: means of non-overlapping windows of s_c keys.
    rng = np.random.default_rng(11)
    K = rng.standard_normal((300, 5))
    P = np.concatenate([np.zeros((1, 5)), np.cumsum(K, axis=0)])
    for size in (64, 128):
        W = O.window_means(K, size, size)
        n = 300 // size
        ref = np.array([(P[(j + 1) * size] - P[j * size]) / size for j in range(n)]).reshape(n, 5)
        np.testing.assert_allclose(W, ref, rtol=1e-12, atol=1e-12)
    ramp = O.window_means(np.arange(256, dtype=np.float64)[:, None], 64, 64)[:, 0]
    assert ramp.tolist() == [31.5, 95.5, 159.5, 223.5]
    # (p, s) windows are exactly the semantic kernels.
    np.testing.assert_array_equal(O.window_means(K, 32, 16), O.compress_keys(K, 32, 16))


def test_log_sum_exp_against_torch():
    z = np.random.default_rng(12).standard_normal((16, 77)) * 9.0
    ref = torch.logsumexp(torch.from_numpy(z), dim=1).numpy()
    np.testing.assert_allclose(O.log_sum_exp(z), ref, rtol=1e-13)


def test_coarse_lse_with_fine_kernels_is_the_exact_selection():
    # Feeding the fine kernels as the "coarse" set (their LSE is the exact
    # one) must reproduce the exact path bit for bit.
    q, K = _rand_case(13, L=1200)
    Kc = O.compress_keys(K, 32, 16)
    i = 1199
    exact = O.select_for_query(q, Kc, i, O.Settings(topk=8))
    st = O.Settings(topk=8, coarse=16)   # visible-window rule of 16-key windows
    n16 = O.visible_kernel_count(i, 16, 16)
    assert n16 >= Kc.shape[0]
    fine_as_coarse = O.select_for_query(q, Kc, i, st, Kcc=Kc)
    np.testing.assert_allclose(fine_as_coarse.r, exact.r, rtol=1e-12)
    assert fine_as_coarse.blocks.tolist() == exact.blocks.tolist()


def test_coarse_lse_is_a_common_per_head_normaliser():
    # g = mean_h exp(z_h - lse_h): the coarse path equals the definition with
    # lse from the coarse windows, and a constant added to every head's lse
    # scales g uniformly, leaving the block order unchanged.
    q, K = _rand_case(14, L=2000)
    Kc = O.compress_keys(K, 32, 16)
    Kcc = O.window_means(K, 64, 64)
    i, d = 1999, q.shape[1]
    st = O.Settings(topk=10, coarse=64)
    sel = O.select_for_query(q, Kc, i, st, Kcc=Kcc)
    n_vis = O.visible_kernel_count(i, 32, 16)
    z = O.kernel_logits(q, Kc[:n_vis], st.sscale(d))
    zc = O.kernel_logits(q, Kcc[:O.visible_kernel_count(i, 64, 64)], st.sscale(d))
    lse = torch.logsumexp(torch.from_numpy(zc), dim=1).numpy()
    g = (np.exp(z - lse[:, None])).mean(axis=0)
    np.testing.assert_allclose(sel.g, g, rtol=1e-12)
    g_shift = O.group_relevance_given_lse(z, lse + 3.7)
    np.testing.assert_allclose(g_shift, g * math.exp(-3.7), rtol=1e-12)
    r_shift = O.block_relevance(g_shift, i, 64, 32, 16)
    blocks_shift = O.top_k_blocks(r_shift, O.forced_blocks(i, 64, 1, 2), 10, True)
    assert blocks_shift.tolist() == sel.blocks.tolist()


def test_coarse_lse_keeps_exact_lse_before_first_coarse_window():
    q, K = _rand_case(15, L=200)
    Kc = O.compress_keys(K, 32, 16)
    Kcc = O.window_means(K, 64, 64)
    for i in (31, 40, 62):
        a = O.select_for_query(q, Kc, i, O.Settings(topk=4))
        b = O.select_for_query(q, Kc, i, O.Settings(topk=4, coarse=64), Kcc=Kcc)
        np.testing.assert_array_equal(a.r, b.r)


def test_planted_blocks_are_selected_on_4k_decode_workload():
    inp = S.make_inputs(S.WORKLOADS["decode_4k"])
    st = O.Settings(topk=16)
    sel = O.run_selection(inp, st)[(0, 0, 0)]
    assert set(inp.planted[0, 0].tolist()) <= set(sel.blocks.tolist())
    assert len(sel.blocks) == 16


# ------------------------------------------------------------- attention ----

def test_attention_dense_degeneracy_matches_torch_sdpa():
    # With every visible block selected the method is exact dense causal
    # attention ("Initial and local tokens always selected": l <= k m).
    rng = np.random.default_rng(8)
    G, d, L = 16, 128, 300
    q_all = rng.standard_normal((L, G, d))
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    qt = torch.from_numpy(q_all).permute(1, 0, 2)[None]            # [1, G, L, d]
    kt = torch.from_numpy(K)[None, None].expand(1, G, L, d)
    vt = torch.from_numpy(V)[None, None].expand(1, G, L, d)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)[0]  # [G, L, d]
    for i in [0, 1, 63, 64, 150, 299]:
        blocks = np.arange(i // 64 + 1)
        out, lse = O.sparse_attention(q_all[i], K, V, blocks, i, 64, 1 / math.sqrt(d))
        np.testing.assert_allclose(out, ref[:, i].numpy(), rtol=1e-10, atol=1e-12)
        sc = (q_all[i] @ K[: i + 1].T) / math.sqrt(d)
        np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(sc), dim=1).numpy(), rtol=1e-13)


def test_attention_block_mask_matches_torch_sdpa_with_mask():
    rng = np.random.default_rng(9)
    G, d, L = 16, 32, 640
    q = rng.standard_normal((G, d))
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    i = 600
    blocks = np.array([0, 3, 5, 8, 9])
    mask = np.zeros(L, dtype=bool)
    for j in blocks:
        mask[j * 64:(j + 1) * 64] = True
    mask[i + 1:] = False
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None], torch.from_numpy(K)[None, None].expand(1, G, L, d),
        torch.from_numpy(V)[None, None].expand(1, G, L, d),
        attn_mask=torch.from_numpy(mask)[None, None, None], scale=0.3)[0, :, 0]
    out, _ = O.sparse_attention(q, K, V, blocks, i, 64, 0.3)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-11, atol=1e-13)


def test_attention_split_merge_identity():
    # Softmax over a union equals the lse-weighted merge of its parts: the
    # identity the split-KV combine relies on.
    rng = np.random.default_rng(10)
    G, d, L = 16, 16, 1024
    q, K, V = rng.standard_normal((G, d)), rng.standard_normal((L, d)), rng.standard_normal((L, d))
    i = L - 1
    all_b = np.array([0, 2, 3, 7, 11, 12, 15])
    o_all, l_all = O.sparse_attention(q, K, V, all_b, i, 64, 0.25)
    parts = [all_b[:3], all_b[3:5], all_b[5:]]
    res = [O.sparse_attention(q, K, V, p_, i, 64, 0.25) for p_ in parts]
    M = np.max([r[1] for r in res], axis=0)
    w = [np.exp(r[1] - M) for r in res]
    merged = sum(wi[:, None] * r[0] for wi, r in zip(w, res)) / sum(w)[:, None]
    np.testing.assert_allclose(merged, o_all, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(M + np.log(sum(w)), l_all, rtol=1e-13)


# ------------------------------------------------- attention backward ----

def _grad_case(seed=20, G=4, d=6, L=300):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((G, d)), rng.standard_normal((L, d)), rng.standard_normal((L, d)),
            rng.standard_normal((G, d)))


def test_attention_grad_matches_torch_autograd(grad_fn=None):
    q, K, V, dO = _grad_case()
    blocks, i, m, scale = np.array([0, 2, 4]), 290, 64, 0.37
    dq, dK, dV = (grad_fn or O.sparse_attention_grad)(q, K, V, blocks, i, m, scale, dO)
    qt = torch.from_numpy(q).requires_grad_()
    Kt = torch.from_numpy(K).requires_grad_()
    Vt = torch.from_numpy(V).requires_grad_()
    mask = torch.zeros(K.shape[0], dtype=torch.bool)
    for j in blocks:
        mask[j * m:(j + 1) * m] = True
    mask[i + 1:] = False
    s = scale * (qt @ Kt.T)
    s = s.masked_fill(~mask[None, :], float("-inf"))
    out = torch.softmax(s, dim=1) @ Vt
    out.backward(torch.from_numpy(dO))
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dK, Kt.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dV, Vt.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_attention_grad_finite_differences():
    q, K, V, dO = _grad_case(seed=21, G=2, d=3, L=140)
    blocks, i, m, scale = np.array([0, 2]), 135, 64, 0.5
    dq, dK, dV = O.sparse_attention_grad(q, K, V, blocks, i, m, scale, dO)

    def f(q_, K_, V_):
        return float((O.sparse_attention(q_, K_, V_, blocks, i, m, scale)[0] * dO).sum())

    eps = 1e-6
    for (arr, grad, idxs) in ((q, dq, [(0, 0), (1, 2)]), (K, dK, [(3, 1), (130, 0), (70, 2)]),
                              (V, dV, [(5, 0), (135, 2), (100, 1)])):
        for ix in idxs:
            plus, minus = arr.copy(), arr.copy()
            plus[ix] += eps
            minus[ix] -= eps
            args_p = [plus if arr is x else x for x in (q, K, V)]
            args_m = [minus if arr is x else x for x in (q, K, V)]
            num = (f(*args_p) - f(*args_m)) / (2 * eps)
            assert abs(num - grad[ix]) <= 1e-6 * (1 + abs(num)), (ix, num, grad[ix])
    # keys outside the attended set get no gradient
    assert np.all(dK[64:128] == 0) and np.all(dV[136:] == 0)


def _block_grad_case(seed=22, G=4, d=6, L=300, m=64, T=9):
    """Queries at scattered positions, each with its own block set (its own
    block always in it): the key-centric gradients of every block against
    the per-query gradients summed."""
    rng = np.random.default_rng(seed)
    K, V = rng.standard_normal((L, d)), rng.standard_normal((L, d))
    Q, dO, X = (rng.standard_normal((T, G, d)) for _ in range(3))
    pos = np.sort(rng.choice(np.arange(40, L), size=T, replace=False))
    nb = (L + m - 1) // m
    sets = []
    for t in range(T):
        own = pos[t] // m
        others = [j for j in range(own) if rng.random() < 0.5]
        sets.append(np.array(sorted(set(others + [own]))))
    return K, V, Q, dO, X, pos, sets, nb


def test_block_grad_kv_matches_per_query_sums(fn=None):
    fn = fn or O.block_grad_kv
    K, V, Q, dO, X, pos, sets, nb = _block_grad_case()
    m, scale = 64, 0.41
    T = Q.shape[0]
    lse, D = np.zeros(Q.shape[:2]), np.zeros(Q.shape[:2])
    ref_k, ref_v, ref_x = np.zeros(K.shape), np.zeros(K.shape), np.zeros(K.shape)
    for t in range(T):
        o, lse[t] = O.sparse_attention(Q[t], K, V, sets[t], pos[t], m, scale)
        D[t] = (dO[t] * o).sum(axis=1)
        _, keys, gk, gv = O.sparse_attention_grad_selected(Q[t], K, V, sets[t], pos[t], m, scale, dO[t])
        ref_k[keys] += gk
        ref_v[keys] += gv
        ref_x[keys] += O.sparse_attention_grad_selected(Q[t], K, V, sets[t], pos[t], m, scale, X[t])[3]
    for j in range(nb):
        sel = np.array([t for t in range(T) if j in set(sets[t].tolist())], dtype=int)
        rows = slice(j * m, min((j + 1) * m, K.shape[0]))
        if sel.size == 0:
            continue
        dk, dv, dx = fn(Q[sel], dO[sel], lse[sel], D[sel], pos[sel], K[rows], V[rows], j * m, scale, X[sel])
        np.testing.assert_allclose(dk, ref_k[rows], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dv, ref_v[rows], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dx, ref_x[rows], rtol=1e-10, atol=1e-12)


def _planted_block_grad_mistakes():
    good = O.block_grad_kv

    def no_causal_mask(Q, dO, lse, D, pos, Kj, Vj, key0, scale, extra=None):   # keys after the query counted
        return good(Q, dO, lse, D, pos + 10 ** 6, Kj, Vj, key0, scale, extra)

    def no_d_term(Q, dO, lse, D, pos, Kj, Vj, key0, scale, extra=None):        # dS = P dP
        return good(Q, dO, lse, np.zeros_like(D), pos, Kj, Vj, key0, scale, extra)

    def no_scale(Q, dO, lse, D, pos, Kj, Vj, key0, scale, extra=None):         # dK without the softmax scale
        dk, dv, dx = good(Q, dO, lse, D, pos, Kj, Vj, key0, scale, extra)
        return dk / scale, dv, dx

    def shifted_keys(Q, dO, lse, D, pos, Kj, Vj, key0, scale, extra=None):     # block credited one key off
        return good(Q, dO, lse, D, pos, Kj, Vj, key0 + 1, scale, extra)

    return [no_causal_mask, no_d_term, no_scale, shifted_keys]


@pytest.mark.parametrize("bad", _planted_block_grad_mistakes())
def test_planted_block_grad_mistakes_are_caught(bad):
    with pytest.raises(AssertionError):
        test_block_grad_kv_matches_per_query_sums(bad)


# ------------------------------------------------ the pins catch mistakes ----

def _planted_mistakes():
    orig_br = O.block_relevance

    def br_off_by_one(g, i, m, p, s):                  # kernel range shifted by one
        r = orig_br(np.roll(g, 1), i, m, p, s)
        return r

    def gr_max_not_mean(z):                            # max over heads instead of mean
        return O.kernel_softmax(z).max(axis=0)

    def ks_no_norm(z):                                 # dropped normaliser
        return np.exp(z - z.max(axis=1, keepdims=True))

    def forced_no_prev(i, m, n_init, n_local):         # local window of one block
        c = i // m
        return sorted({0, c})

    orig_wm = O.window_means

    def wm_half_stride(K, size, stride):               # overlapping coarse windows
        return orig_wm(K, size, max(1, stride // 2) if size == stride else stride)

    def lse_plain_max(z):                              # max instead of log-sum-exp
        return z.max(axis=1)

    def bnd_max_not_min(r, blocks, forced):            # best taken score instead of the last
        scored = [int(j) for j in blocks if int(j) not in set(forced)]
        return float(max(r[j] for j in scored)) if scored else float("nan")

    def bnd_with_forced(r, blocks, forced):            # forced blocks counted in
        return float(min(r[int(j)] for j in blocks)) if len(blocks) else float("nan")

    def bnd_first_not_taken(r, blocks, forced):        # best score left out instead
        rest = [j for j in range(r.shape[0]) if j not in set(int(b) for b in blocks) and np.isfinite(r[j])]
        return float(max(r[j] for j in rest)) if rest else float("nan")

    return [("block_relevance", br_off_by_one), ("group_relevance", gr_max_not_mean),
            ("kernel_softmax", ks_no_norm), ("forced_blocks", forced_no_prev),
            ("window_means", wm_half_stride), ("log_sum_exp", lse_plain_max),
            ("boundary_score", bnd_max_not_min), ("boundary_score", bnd_with_forced),
            ("boundary_score", bnd_first_not_taken)]


@pytest.mark.parametrize("name,bad", _planted_mistakes(), ids=lambda x: x if isinstance(x, str) else x.__name__)
def test_planted_oracle_mistakes_are_caught(monkeypatch, name, bad):
    monkeypatch.setattr(O.infllmv2_oracle, name, bad)
    monkeypatch.setattr(O, name, bad)
    checks = [test_hand_worked_selections, test_group_relevance_is_head_mean_and_sums_to_one,
              test_selection_structural_invariants,
              lambda: test_block_relevance_brute_force(64, 32, 16),
              lambda: test_forced_blocks_hand_cases(1000, [0, 14, 15]),
              test_window_means_prefix_sum_and_ramp, test_log_sum_exp_against_torch]
    failed = 0
    for chk in checks:
        try:
            chk()
        except AssertionError:
            failed += 1
    assert failed > 0, f"planted mistake in {name} went unnoticed"


def _planted_grad_mistakes():
    good = O.sparse_attention_grad

    def no_scale_dq(q, K, V, b, i, m, s, dO):          # dropped softmax scale on dq
        dq, dK, dV = good(q, K, V, b, i, m, s, dO)
        return dq / s, dK, dV

    def no_d_term(q, K, V, b, i, m, s, dO):            # dS = P * dP, the row term dropped
        dq, dK, dV = good(q, K, V, b, i, m, s, dO)
        _, lse = O.sparse_attention(q, K, V, b, i, m, s)
        mask = np.zeros(K.shape[0], dtype=bool)
        for j in b:
            mask[j * m:(j + 1) * m] = True
        mask[i + 1:] = False
        P = np.exp(s * (q @ K[mask].T) - lse[:, None])
        dS = P * (dO @ V[mask].T)
        dq = s * (dS @ K[mask])
        return dq, dK, dV

    def shifted_dk(q, K, V, b, i, m, s, dO):           # gradient credited to the wrong key
        dq, dK, dV = good(q, K, V, b, i, m, s, dO)
        return dq, np.roll(dK, 1, axis=0), dV

    def dv_uses_ds(q, K, V, b, i, m, s, dO):           # dV built from the wrong factor
        dq, dK, dV = good(q, K, V, b, i, m, s, dO)
        return dq, dK, dK / s

    return [no_scale_dq, no_d_term, shifted_dk, dv_uses_ds]


@pytest.mark.parametrize("bad", _planted_grad_mistakes())
def test_planted_grad_mistakes_are_caught(bad):
    with pytest.raises(AssertionError):
        test_attention_grad_matches_torch_autograd(bad)
