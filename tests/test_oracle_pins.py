"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each test ties one oracle routine to an independent library routine, a brute-force enumeration,
a closed form, a hand-derived sequence (``tests/golden/``) or an identity of the mathematics, so
that a dropped term, a wrong sign or index, or a transposed operand in the oracle fails here.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import oracle.dsa_oracle as OD

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng


def _sdpa(q, keys, values, scale, mask=None):
    """torch's float64 scaled-dot-product attention: an independent softmax implementation."""
    qt = torch.from_numpy(q)[None, :, None, :]            # [1, G, 1, D]
    kt = torch.from_numpy(keys)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(values)[None, None].expand(1, q.shape[0], -1, -1)
    am = None if mask is None else torch.from_numpy(mask)[None, None, None, :]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=am, scale=scale)
    return out[0, :, 0].numpy()


# ------------------------------------------------------------------------------------ attention

@pytest.mark.parametrize("G,L", [(1, 37), (4, 300), (16, 129)])
def test_attend_matches_library_softmax(G, L):
    r = rng(G * 1000 + L)
    D = 128
    q, K, V = r.normal(size=(G, D)), r.normal(size=(L, D)), r.normal(size=(L, D))
    scale = 1 / math.sqrt(D)
    Out, m, l = O.attend(q, K, V, np.arange(L), scale)
    np.testing.assert_allclose(Out, _sdpa(q, K, V, scale), rtol=1e-12, atol=1e-12)
    lse = torch.logsumexp(torch.from_numpy(scale * q @ K.T), dim=1).numpy()
    np.testing.assert_allclose(m + np.log(l), lse, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(m, (scale * q @ K.T).max(1), rtol=1e-14, atol=1e-14)


def test_attend_subset_matches_masked_library_softmax():
    r = rng(7)
    G, L, D = 4, 200, 128
    q, K, V = r.normal(size=(G, D)), r.normal(size=(L, D)), r.normal(size=(L, D))
    ids = np.sort(r.choice(L, 57, replace=False))
    mask = np.full(L, -np.inf)
    mask[ids] = 0.0
    Out, _, _ = O.attend(q, K, V, ids, 0.1)
    np.testing.assert_allclose(Out, _sdpa(q, K, V, 0.1, mask), rtol=1e-12, atol=1e-12)


def test_attend_empty_set_is_merge_identity():
    q = np.ones((2, 8))
    Out, m, l = O.attend(q, np.zeros((4, 8)), np.zeros((4, 8)), [], 1.0)
    assert np.all(Out == 0) and np.all(m == -np.inf) and np.all(l == 0)


def test_full_budget_topk_equals_dense_attention_with_ragged_tail():
    """Top-K with K >= number of pages attends to every token: equals dense softmax attention."""
    r = rng(11)
    G, D, page, L = 4, 128, 16, 16 * 9 + 5
    q, K, V = r.normal(size=(G, D)), r.normal(size=(L, D)), r.normal(size=(L, D))
    kmax, kmin = O.page_meta_minmax(K, page)
    S = O.score_pages_minmax(O.representative_query(q), kmax, kmin)
    sel = O.select_topk(O.pad_scores(S, 32), 1000)
    assert sel == list(range(10))
    Out, _, _ = O.attend(q, K, V, O.page_token_ids(sel, page, L), 1 / math.sqrt(D))
    np.testing.assert_allclose(Out, _sdpa(q, K, V, 1 / math.sqrt(D)), rtol=1e-12, atol=1e-12)


def test_page_token_ids_clip_to_length():
    assert list(O.page_token_ids([2, 0], 4, 10)) == [8, 9, 0, 1, 2, 3]


@pytest.mark.parametrize("seed", range(4))
def test_merge_of_disjoint_parts_equals_attention_over_union(seed):
    """PRR §3.3 recurrence: merging partials of disjoint sets, in any order, is attention over the
    union; an empty part is the identity."""
    r = rng(100 + seed)
    G, L, D = 3, 150, 16
    q, K, V = r.normal(size=(G, D)) * 3, r.normal(size=(L, D)), r.normal(size=(L, D))
    ids = r.permutation(L)
    cuts = sorted(r.choice(np.arange(1, L), 3, replace=False))
    sets = np.split(ids, cuts)
    parts = [O.attend(q, K, V, s, 0.5) for s in sets] + [O.attend(q, K, V, [], 0.5)]
    whole = O.attend(q, K, V, np.arange(L), 0.5)
    for order in (parts, parts[::-1], [parts[2], parts[4], parts[0], parts[3], parts[1]]):
        got = O.merge_partials(order)
        for a, b in zip(got, whole):
            np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------ metadata

def test_minmax_meta_bounds_and_is_attained():
    r = rng(3)
    K = r.normal(size=(16 * 5 + 3, 32))
    kmax, kmin = O.page_meta_minmax(K, 16)
    assert kmax.shape == (6, 32)
    for j in range(6):
        seg = K[j * 16:(j + 1) * 16]
        assert np.all(seg <= kmax[j]) and np.all(seg >= kmin[j])
        assert np.all(np.any(seg == kmax[j], axis=0)) and np.all(np.any(seg == kmin[j], axis=0))
    assert np.all(kmax[5] >= kmin[5])


def test_mean_meta_closed_forms():
    K = np.zeros((16 * 3 + 2, 8))
    K[0:16] = 2.0
    K[16:32] = np.arange(16)[:, None]          # 0..15 -> mean 7.5
    K[32:48] = -1.0
    K[48:50] = [[4.0] * 8, [6.0] * 8]          # ragged block of 2 -> mean 5
    mean = O.page_meta_mean(K, 16)
    np.testing.assert_array_equal(mean[:, 0], [2.0, 7.5, -1.0, 5.0])


# ------------------------------------------------------------------------------------ scoring

@pytest.mark.parametrize("seed", range(3))
def test_quest_score_is_maximum_over_box_corners(seed):
    """S^j = max over the corners x of the box [kmin, kmax] of q . x (the box's support value),
    enumerated exhaustively for D = 6."""
    r = rng(50 + seed)
    D = 6
    K = r.normal(size=(8 * 4, D))
    q = r.normal(size=(1, D))
    kmax, kmin = O.page_meta_minmax(K, 8)
    S = O.score_pages_minmax(O.representative_query(q), kmax, kmin)
    for j in range(4):
        corners = [np.where(bits, kmax[j], kmin[j]) for bits in itertools.product([0, 1], repeat=D)]
        best = max(float(q[0] @ c) for c in corners)
        assert abs(S[j] - best) <= 1e-12 * max(1.0, abs(best))


@pytest.mark.parametrize("G", [1, 4, 16])
def test_quest_score_bounds_every_token(G):
    """LServe §4.2: the page score bounds q_bar . k_t from above for every token of the page, and
    is tight for single-token pages."""
    r = rng(G)
    D, page, L = 128, 16, 16 * 20 + 7
    q, K = r.normal(size=(G, D)), r.normal(size=(L, D))
    qbar = O.representative_query(q)
    kmax, kmin = O.page_meta_minmax(K, page)
    S = O.score_pages_minmax(qbar, kmax, kmin)
    dots = K @ qbar
    for j in range(len(S)):
        assert S[j] >= dots[j * page:(j + 1) * page].max() - 1e-12
    k1max, k1min = O.page_meta_minmax(K, 1)
    np.testing.assert_allclose(O.score_pages_minmax(qbar, k1max, k1min), dots, rtol=1e-12, atol=1e-12)
    phys = O.physical_scores(S, 4)
    for P in range(len(phys)):
        assert phys[P] >= dots[P * 64:(P + 1) * 64].max() - 1e-12


def test_representative_query_is_group_mean():
    r = rng(9)
    q1 = r.normal(size=(1, 128))
    np.testing.assert_allclose(O.representative_query(np.repeat(q1, 8, 0)), q1[0], rtol=1e-15, atol=0)
    q = r.normal(size=(4, 128))
    np.testing.assert_allclose(O.representative_query(q), (q[0] + q[1] + q[2] + q[3]) / 4, rtol=1e-14)


def test_mean_score_is_mean_of_token_dots():
    r = rng(12)
    K = r.normal(size=(16 * 6 + 9, 128))
    q = r.normal(size=128)
    S = O.score_pages_mean(q, O.page_meta_mean(K, 16))
    dots = K @ q
    ref = [dots[j * 16:(j + 1) * 16].mean() for j in range(7)]
    np.testing.assert_allclose(S, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------ selection

def _brute_topk(s, k):
    """Max-sum subset of size min(k, #valid); ties -> lexicographically smallest index set."""
    valid = [j for j in range(len(s)) if s[j] > -np.inf]
    kk = min(k, len(valid))
    best = None
    for comb in itertools.combinations(valid, kk):
        key = (-sum(s[j] for j in comb), comb)
        if best is None or key < best:
            best = key
    return list(best[1]) if best else []


@pytest.mark.parametrize("seed", range(40))
def test_topk_matches_brute_force_with_planted_ties(seed):
    r = rng(seed)
    n = int(r.integers(1, 13))
    k = int(r.integers(0, 5))
    s = r.integers(-3, 4, size=n).astype(float)          # small integers: many exact ties
    s[r.random(n) < 0.2] = -np.inf
    assert O.select_topk(s, k) == _brute_topk(s, k)


@pytest.mark.parametrize("seed", range(20))
def test_hier_matches_brute_force_over_physical_pages(seed):
    r = rng(200 + seed)
    g = int(r.integers(1, 5))
    n_log = int(r.integers(1, 13))
    k = int(r.integers(0, 4))
    s = r.integers(-3, 4, size=n_log).astype(float)
    s[r.random(n_log) < 0.15] = -np.inf
    n_phys = -(-n_log // g)
    phys = [max(s[p * g:(p + 1) * g]) for p in range(n_phys)]
    assert O.select_hier(s, g, k) == _brute_topk(phys, k)


def test_hier_with_one_logical_per_physical_is_flat_topk():
    r = rng(5)
    s = r.normal(size=300)
    assert O.select_hier(s, 1, 40) == O.select_topk(s, 40)


def test_rank_order_descending_ties_to_lower_index():
    assert O.rank_pages([1.0, 3.0, 3.0, -np.inf, 2.0]) == [1, 2, 4, 0]


# ------------------------------------------------------------------------------------ streaming

def test_streaming_window_covering_everything_is_dense():
    r = rng(21)
    L, D = 300, 32
    q, K, V = r.normal(size=(2, D)), r.normal(size=(L, D)), r.normal(size=(L, D))
    ids = O.streaming_token_ids(L, 64, 256)
    assert list(ids) == list(range(L))
    np.testing.assert_allclose(O.attend(q, K, V, ids, 0.2)[0], _sdpa(q, K, V, 0.2), rtol=1e-12)


def test_streaming_window_matches_lambda_mask():
    r = rng(22)
    L, D = 1000, 32
    q, K, V = r.normal(size=(2, D)), r.normal(size=(L, D)), r.normal(size=(L, D))
    t = np.arange(L)
    mask = np.where((t < 64) | (t >= L - 256), 0.0, -np.inf)
    ids = O.streaming_token_ids(L, 64, 256)
    assert len(ids) == 320
    np.testing.assert_allclose(O.attend(q, K, V, ids, 0.2)[0], _sdpa(q, K, V, 0.2, mask), rtol=1e-12)
    assert list(O.streaming_token_ids(10, 4, 0)) == [0, 1, 2, 3]
    assert list(O.streaming_token_ids(10, 0, 3)) == [7, 8, 9]


# ------------------------------------------------------------------------------------ PSA

def _zipf_row(n_blocks, block, s, D=128, seed=0):
    """Blocks whose tokens all share the logit -s ln r (r = rank); block order shuffled."""
    r = rng(seed)
    rank = r.permutation(n_blocks) + 1
    q = np.zeros((1, D))
    q[0, 0] = 1.0
    K = np.zeros((n_blocks * block, D))
    for j in range(n_blocks):
        K[j * block:(j + 1) * block, 0] = -s * math.log(rank[j])
        K[j * block:(j + 1) * block, 1] = rank[j]         # orthogonal to q: no effect on logits
    V = r.normal(size=(n_blocks * block, D))
    scores = -np.log(rank.astype(float))                # any order-preserving criticality
    return q, K, V, scores, rank


def test_psa_stop_count_matches_zipf_closed_form():
    gold = json.load(open(os.path.join(GOLDEN, "psa_zipf_stop.json")))
    q, K, V, scores, rank = _zipf_row(200, 16, gold["zipf_s"])
    res = O.psa_progressive(q, K, V, scores, 16, 200 * 16, gold["tau"], 1024, 1.0)
    assert len(res["ranked"]) == gold["stop_blocks"]
    assert [int(rank[j]) for j in res["ranked"]] == list(range(1, 8))
    assert abs(res["ratios"][-2][0] - gold["ratio_before_stop"]) < 1e-4
    assert abs(res["ratios"][-1][0] - gold["ratio_at_stop"]) < 1e-4


def test_psa_needs_two_blocks_above_half_and_one_at_or_below():
    gold = json.load(open(os.path.join(GOLDEN, "psa_zipf_stop.json")))
    q, K, V, scores, _ = _zipf_row(50, 16, 0.0, seed=3)      # equal masses
    assert len(O.psa_progressive(q, K, V, scores, 16, 800, 0.51, 99, 1.0)["ranked"]) == \
        gold["min_blocks_for_tau_above_half"]
    assert len(O.psa_progressive(q, K, V, scores, 16, 800, 0.5, 99, 1.0)["ranked"]) == 1
    # equal masses: ratio after n blocks is n / (n + 1) -> tau 0.9 needs 9 blocks
    assert len(O.psa_progressive(q, K, V, scores, 16, 800, 0.9, 99, 1.0)["ranked"]) == 9


def test_psa_tau_one_visits_everything_and_equals_dense():
    r = rng(31)
    G, D, block, L = 2, 64, 16, 16 * 12 + 3
    q, K, V = r.normal(size=(G, D)), r.normal(size=(L, D)), r.normal(size=(L, D))
    scores = O.score_pages_mean(O.representative_query(q), O.page_meta_mean(K, block))
    res = O.psa_progressive(q, K, V, scores, block, L, 1.0, 10_000, 0.125)
    assert sorted(res["ranked"]) == list(range(13))
    np.testing.assert_allclose(res["O_fused"], _sdpa(q, K, V, 0.125), rtol=1e-12, atol=1e-12)


def _gqa_psa_row():
    gold = json.load(open(os.path.join(GOLDEN, "psa_gqa_stop.json")))
    a = np.asarray(gold["masses_head0"], dtype=np.float64)
    n = len(a)
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    K = np.stack([np.log(a), np.zeros(n)], axis=1)
    V = rng(5).normal(size=(n, 2))
    scores = np.arange(n, 0, -1, dtype=np.float64)      # visit in index order
    return gold, q, K, V, scores


def test_psa_group_stops_when_every_head_satisfies_the_rule():
    """A group of two query heads on one KV head: one head satisfies the stop rule after 4 blocks,
    the other after 9; the walk stops after 9 (tests/golden/psa_gqa_stop.json)."""
    gold, q, K, V, scores = _gqa_psa_row()
    n = len(scores)
    res = O.psa_progressive(q, K, V, scores, 1, n, gold["tau"], 100, 1.0)
    assert res["ranked"] == list(range(gold["stop_blocks_every_head"]))
    np.testing.assert_allclose(res["ratios"][-1], [gold["ratio_head0_at_stop"],
                                                   gold["ratio_head1_at_stop"]], rtol=1e-12)
    np.testing.assert_allclose(res["ratios"][3][0], 15 / 16, rtol=1e-12)
    np.testing.assert_allclose(res["ratios"][7][1], 8 / 9, rtol=1e-12)


@pytest.mark.parametrize("tau,cap", [(0.95, 100), (0.99, 5), (0.8, 100)])
def test_psa_fused_output_is_attention_over_visited_blocks(tau, cap):
    """PSA §3.2 weighted fusion is exact: it equals softmax attention over the union of visited
    blocks, and the visit order is the criticality ranking."""
    r = rng(int(tau * 100) + cap)
    G, D, block, L = 1, 128, 16, 16 * 40
    q, K, V = r.normal(size=(G, D)), r.normal(size=(L, D)), r.normal(size=(L, D))
    K[16 * 7:16 * 8] += 1.5 * q[0] / np.linalg.norm(q[0])
    scores = O.score_pages_mean(q[0], O.page_meta_mean(K, block))
    res = O.psa_progressive(q, K, V, scores, block, L, tau, cap, 1 / math.sqrt(D))
    n = len(res["ranked"])
    assert 1 <= n <= cap
    assert res["ranked"] == O.rank_pages(scores)[:n]
    ids = O.page_token_ids(res["ranked"], block, L)
    Oref, mref, lref = O.attend(q, K, V, ids, 1 / math.sqrt(D))
    np.testing.assert_allclose(res["O_fused"], Oref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["m"], mref, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(res["l"], lref, rtol=1e-12)
    if n < cap:
        assert res["ratios"][-1][0] >= tau and all(x[0] < tau for x in res["ratios"][:-1])


def test_psa_nleft_variant_is_stricter():
    q, K, V, scores, _ = _zipf_row(64, 16, 1.1, seed=4)
    lit = O.psa_progressive(q, K, V, scores, 16, 64 * 16, 0.95, 999, 1.0)
    nl = O.psa_progressive(q, K, V, scores, 16, 64 * 16, 0.95, 999, 1.0, use_nleft=True)
    assert len(nl["ranked"]) > len(lit["ranked"])
    # with N_left the rule bounds the unvisited mass: it holds at the end when every block is in
    full = O.psa_progressive(q, K, V, scores, 16, 64 * 16, 0.999999, 999, 1.0, use_nleft=True)
    assert full["ratios"][-1][0] == 1.0 or len(full["ranked"]) <= 64


# ------------------------------------------------------------------------------------ EMA

def test_ema_hand_sequence():
    gold = json.load(open(os.path.join(GOLDEN, "ema_hand_sequence.json")))
    ell = np.array([gold["initial_level"]])
    v = np.array([gold["initial_trend"]])
    for t, s in enumerate(gold["scores"]):
        ell, v = O.ema_update(np.array([s]), ell, v, gold["alpha"], gold["beta"])
        assert abs(ell[0] - gold["level"][t]) < 1e-12
        assert abs(v[0] - gold["trend"][t]) < 1e-12
        assert abs(O.ema_predict(ell, v, gold["gamma"])[0] - gold["prediction_next"][t]) < 1e-12


def test_ema_constant_scores_are_a_fixed_point_and_init_predicts_last_scores():
    IS = np.array([3.0, -1.0, -np.inf, 0.5])
    ell, v = O.ema_init(IS)
    np.testing.assert_array_equal(O.ema_predict(ell, v, 0.5), IS)
    for _ in range(5):
        ell, v = O.ema_update(IS, ell, v, 0.6, 0.3)
    np.testing.assert_array_equal(ell, IS)
    np.testing.assert_array_equal(v, [0, 0, 0, 0])


def test_ema_page_without_history_starts_like_init():
    ell = np.array([1.0, -np.inf, -np.inf])
    v = np.array([0.5, 0.0, 0.0])
    l2, v2 = O.ema_update(np.array([2.0, 4.0, -np.inf]), ell, v, 0.6, 0.3)
    np.testing.assert_allclose(l2, [0.6 * 2 + 0.4 * 1, 4.0, -np.inf])
    np.testing.assert_allclose(v2, [0.3 * (2 - 1) + 0.7 * 0.5, 0.0, 0.0])


def test_ema_prediction_ranking_invariant_under_positive_affine_scores():
    r = rng(41)
    traj = [r.normal(size=50) for _ in range(6)]
    ell, v = O.ema_init(traj[0])
    ell2, v2 = O.ema_init(3.0 * traj[0] + 7.0)
    for IS in traj[1:]:
        ell, v = O.ema_update(IS, ell, v, 0.6, 0.3)
        ell2, v2 = O.ema_update(3.0 * IS + 7.0, ell2, v2, 0.6, 0.3)
    assert O.select_topk(O.ema_predict(ell, v, 0.5), 10) == O.select_topk(O.ema_predict(ell2, v2, 0.5), 10)


def test_calibration_grid_has_eighty_candidates():
    grid = O.calibration_grid()
    assert len(grid) == 80
    assert sorted({round(a, 6) for a, _, _ in grid}) == [0.2, 0.4, 0.6, 0.8]
    assert sorted({round(b, 6) for _, b, _ in grid}) == [0.1, 0.2, 0.3, 0.4, 0.5]
    assert sorted({round(c, 6) for _, _, c in grid}) == [0.0, 0.25, 0.5, 0.75]


def test_calibration_prefers_trend_when_rankings_cross():
    """Pages whose scores move linearly and cross over time: a trend-following predictor
    (gamma > 0) covers the next top set strictly better than any level-only one (gamma = 0)."""
    n = 40
    slope = np.linspace(-1, 1, n)
    traj = [20 - 6 * slope + slope * t + 0.001 * np.arange(n) for t in range(12)]
    best, Hs = O.calibrate_ema(traj, 5, 6)
    level_only = max(h for (_, _, c), h in zip(O.calibration_grid(), Hs) if c == 0)
    assert best[2] > 0
    assert max(Hs) > level_only + 0.05


def test_calibration_hand_derived_hit_rates():
    """H of two grid points on a 3-step, 5-page trajectory, worked by hand
    (tests/golden/ema_calibration_hand.json): the mean over steps 1..T-1 of the covered share of
    the true set's score mass."""
    gold = json.load(open(os.path.join(GOLDEN, "ema_calibration_hand.json")))
    traj = [np.asarray(x, dtype=np.float64) for x in gold["trajectory"]]
    _, Hs = O.calibrate_ema(traj, gold["k"], gold["k_pred"])
    grid = O.calibration_grid()
    for c, h in gold["H"].items():
        np.testing.assert_allclose(grid[int(c)], gold["points"][c], rtol=1e-12)
        assert abs(Hs[int(c)] - h) < 1e-12, (c, Hs[int(c)], h)


# ------------------------------------------------------------------------------------ PRR

@pytest.mark.parametrize("case", ["random", "disjoint", "superset_of_A", "equal", "empty_P"])
def test_spec_plus_repair_equals_attention_over_true_set(case):
    r = rng(hash(case) % 1000)
    G, D, page, L = 4, 64, 8, 8 * 30 + 5
    q, K, V = r.normal(size=(G, D)), r.normal(size=(L, D)), r.normal(size=(L, D))
    A = sorted(r.choice(31, 10, replace=False))
    if case == "random":
        P = sorted(r.choice(31, 12, replace=False))
    elif case == "disjoint":
        P = [j for j in range(31) if j not in A][:12]
    elif case == "superset_of_A":
        P = sorted(set(A) | {j for j in range(31) if j not in A and j % 3 == 0})
    elif case == "equal":
        P = list(A)
    else:
        P = []
    ref = O.attend(q, K, V, O.page_token_ids(A, page, L), 0.3)
    got = O.spec_repair(q, K, V, page, L, P, A, 0.3)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    union = sorted(set(A) | set(P))
    ref_u = O.attend(q, K, V, O.page_token_ids(union, page, L), 0.3)
    got_u = O.spec_repair(q, K, V, page, L, P, A, 0.3, superset=True)
    for a, b in zip(got_u, ref_u):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_hit_rates():
    assert O.hit_rate([1, 2, 3], [2, 3, 4, 5]) == 0.5
    assert O.score_weighted_hit([1, 2], [2, 3], np.array([0, 3.0, 1.0, 3.0])) == 0.25


# ------------------------------------------------------------------------------------ paging

def test_request_tokens_follow_page_table():
    pool = torch.arange(6 * 2 * 4 * 3, dtype=torch.float32).reshape(6, 2, 4, 3).to(torch.bfloat16)
    table = torch.tensor([[4, 1, 3]], dtype=torch.int32)
    got = O.request_tokens(pool, table, 10, 0, 1)
    assert got.shape == (10, 3)
    np.testing.assert_array_equal(got[0], pool[4, 1, 0].double().numpy())
    np.testing.assert_array_equal(got[5], pool[1, 1, 1].double().numpy())
    np.testing.assert_array_equal(got[9], pool[3, 1, 1].double().numpy())


# ------------------------------------------------------------------------------------ planted mistakes

def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle (on the CPU) and check a pin above fails for each."""
    gold = json.load(open(os.path.join(GOLDEN, "ema_hand_sequence.json")))

    def holt_update(IS, ell, v, alpha, beta):               # trend reads the new level
        l_new = alpha * IS + (1 - alpha) * ell
        return l_new, beta * (l_new - ell) + (1 - beta) * v
    ell, v = holt_update(np.array([1.0]), np.array([0.0]), np.array([0.0]), 0.6, 0.3)
    assert abs(v[0] - gold["trend"][0]) > 0.1

    r = rng(77)
    q, K = r.normal(size=(1, 6)), r.normal(size=(8, 6))
    kmax, kmin = O.page_meta_minmax(K, 8)
    swapped = np.minimum(q * kmax, q * kmin).sum()           # min instead of max
    assert swapped < (K @ q[0]).max()                         # violates the bound pin

    s = np.array([1.0, 2.0, 2.0, 0.5])
    assert sorted(sorted(range(4), key=lambda j: (-s[j], -j))[:1]) != _brute_topk(s, 1)

    # PSA with a query group: stopping when ANY head satisfies the rule (instead of every head)
    gold, q, K, V, scores = _gqa_psa_row()
    with monkeypatch.context() as mp:
        mp.setattr(OD.np, "all", np.any)
        res = O.psa_progressive(q, K, V, scores, 1, len(scores), gold["tau"], 100, 1.0)
    assert len(res["ranked"]) == gold["stop_blocks_any_head"] != gold["stop_blocks_every_head"]

    # calibration: averaging over all T steps, or counting hits instead of score mass
    cal = json.load(open(os.path.join(GOLDEN, "ema_calibration_hand.json")))
    traj = [np.asarray(x, dtype=np.float64) for x in cal["trajectory"]]
    _, Hs = O.calibrate_ema(traj, cal["k"], cal["k_pred"])
    assert abs(Hs[79] * 2 / 3 - cal["H"]["79"]) > 0.05
    with monkeypatch.context() as mp:
        mp.setattr(OD, "score_weighted_hit", lambda P, A, IS: OD.hit_rate(P, A))
        _, Hs_count = O.calibrate_ema(traj, cal["k"], cal["k_pred"])
    assert abs(Hs_count[79] - cal["H"]["79"]) > 0.01

    # KV4: rounding half away from zero, or the odd dim in the low nibble
    kv4 = json.load(open(os.path.join(GOLDEN, "kv4_hand_row.json")))
    row = np.array([kv4["row"]], dtype=np.float32)
    with monkeypatch.context() as mp:
        mp.setattr(OD.np, "rint", lambda y: np.sign(y) * np.floor(np.abs(y) + 0.5))
        assert O.kv4_encode_rows(row)[0][0].tolist() != kv4["bytes"]
    packed, _ = O.kv4_encode_rows(row)
    swapped = ((packed >> 4) | ((packed & 15) << 4)).astype(np.uint8)
    assert swapped[0].tolist() != kv4["bytes"]



def _plant(mp, name, fn):
    """Replaces one oracle routine (package and module names alike) for the context's duration."""
    mp.setattr(O, name, fn)
    mp.setattr(OD, name, fn)


def _pin_fails(pin, *cases):
    """True when the pin raises on at least one of its cases."""
    for args in cases:
        try:
            pin(*args)
        except AssertionError:
            return True
    return False


def test_pins_catch_planted_mistakes_in_metadata_selection_and_merge(monkeypatch):
    """More plausible mistakes, each planted in the oracle (on the CPU): the pin named beside each
    must fail with it in place (and passes without it, as the pins above show)."""
    orig_repair = OD.spec_repair

    def merge_wrong_sign(parts):  # the rescale exponents taken the wrong way round
        parts = list(parts)
        G, D = parts[0][0].shape
        Om, m, l = np.zeros((G, D)), np.full(G, -np.inf), np.zeros(G)
        for (Op, mp_, lp) in parts:
            for g in range(G):
                if lp[g] == 0.0:
                    continue
                if l[g] == 0.0:
                    Om[g], m[g], l[g] = Op[g], mp_[g], lp[g]
                    continue
                m_new = max(m[g], mp_[g])
                a = math.exp(m_new - m[g]) * l[g]
                b = math.exp(m_new - mp_[g]) * lp[g]
                Om[g] = (a * Om[g] + b * Op[g]) / (a + b)
                m[g], l[g] = m_new, a + b
        return Om, m, l

    plants = [
        # LServe §4.2: a physical page's importance is the max of its logical pages, not the mean
        ("physical_scores",
         lambda s, g: np.array([np.asarray(s, dtype=np.float64)[p * g:(p + 1) * g].mean()
                                for p in range(-(-len(s) // g))]),
         test_hier_matches_brute_force_over_physical_pages, [(i,) for i in range(20)]),
        # PSA §5: a ragged last block averages over its valid tokens, not the full block size
        ("page_meta_mean",
         lambda K, b: np.stack([K[j * b:(j + 1) * b].sum(axis=0) / b for j in range(-(-len(K) // b))]),
         test_mean_meta_closed_forms, [()]),
        # LServe §4.2: the max is taken per channel, not once over two whole dot products
        ("score_pages_minmax",
         lambda qb, kmax, kmin: np.maximum(kmax @ qb, kmin @ qb),
         test_quest_score_is_maximum_over_box_corners, [(i,) for i in range(3)]),
        # PRR §3.3: the running maximum rescales both parts by exp(m_old - m_new)
        ("merge_partials", merge_wrong_sign,
         test_merge_of_disjoint_parts_equals_attention_over_union, [(i,) for i in range(4)]),
        # LServe §4.1: the local window ends at the current token
        ("streaming_token_ids",
         lambda L, sink, local: np.asarray(sorted(set(range(min(sink, L))) |
                                                  set(range(max(0, L - local - 1), L - 1))),
                                           dtype=np.int64),
         test_streaming_window_matches_lambda_mask, [()]),
        # PRR §3.1: the prediction scales the trend by gamma, not the level
        ("ema_predict",
         lambda ell, v, gamma: gamma * np.asarray(ell, dtype=np.float64) + np.asarray(v),
         test_ema_hand_sequence, [()]),
        # PRR §5: the group's representative query is the mean of its heads, not the sum
        ("representative_query",
         lambda qg: OD.to_f64(qg).sum(axis=0),
         test_representative_query_is_group_mean, [()]),
        # PRR §3.3 exact mode: speculative parts of pages outside A are dropped, not merged
        ("spec_repair",
         lambda *a, superset=False, **kw: orig_repair(*a, superset=True, **kw),
         test_spec_plus_repair_equals_attention_over_true_set, [("random",), ("disjoint",)]),
    ]
    for name, wrong, pin, cases in plants:
        with monkeypatch.context() as mp:
            _plant(mp, name, wrong)
            assert _pin_fails(pin, *cases), f"{pin.__name__} does not catch a wrong {name}"
    for name, _, pin, cases in plants:  # and every pin passes on the oracle as it stands
        assert not _pin_fails(pin, *cases), f"{pin.__name__} fails on the unchanged oracle"
    # PSA §3.2: the stop rule compares against the smallest block mass seen, not the largest
    with monkeypatch.context() as mp:
        mp.setattr(OD.np, "minimum", np.maximum)
        assert _pin_fails(test_psa_stop_count_matches_zipf_closed_form, ())
    assert not _pin_fails(test_psa_stop_count_matches_zipf_closed_form, ())


# ------------------------------------------------------------------------------------ KV8

def test_kv8_codes_match_the_e4m3_format():
    """The e4m3 rounding step against the format's own values: exponent bias 7, 3 mantissa bits,
    448 = 0x7E the largest finite, 2^-9 the smallest subnormal, ties to even."""
    rows = np.array([[448.0, 1.0, -2.0, 0.0, 2.0 ** -9, 1.0625, 1.1875, -0.0]], dtype=np.float32)
    codes, scale = O.kv8_encode_rows(rows)
    assert scale[0] == np.float32(1.0)           # max |x| = 448 maps to scale 1
    assert codes[0].tolist() == [0x7E, 0x38, 0xC0, 0x00, 0x01, 0x38, 0x3A, 0x80]
    dec = O.kv8_decode_rows(codes, scale)
    assert dec[0].tolist() == [448.0, 1.0, -2.0, 0.0, 2.0 ** -9, 1.0, 1.25, -0.0]


def test_kv8_round_trip_error_is_bounded():
    """Decoded rows stay within half an e4m3 step of the input: relative 2^-4 for values in the
    normal range of the row's scale, absolute 2^-10 * scale below it; a zero row decodes to zero."""
    r = rng(3)
    x = r.normal(size=(50, 128)).astype(np.float32) * r.uniform(0.01, 30, size=(50, 1)).astype(np.float32)
    x[7] = 0.0
    codes, scale = O.kv8_encode_rows(x)
    dec = O.kv8_decode_rows(codes, scale)
    assert scale[7] == 0 and np.all(dec[7] == 0)
    err = np.abs(dec - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, scale[:, None] * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(err <= bound)
    # the largest magnitude of every row is represented exactly (it maps to 448)
    for i in range(50):
        if scale[i] > 0:
            j = int(np.argmax(np.abs(x[i])))
            assert abs(dec[i, j] - x[i, j]) <= abs(x[i, j]) * 1e-6


# ------------------------------------------------------------------------------------ KV4

def test_kv4_codes_match_the_hand_row():
    """Scale, rounding (ties to even), offset-8 nibbles and their order in a byte against a row
    worked by hand (tests/golden/kv4_hand_row.json)."""
    g = json.load(open(os.path.join(GOLDEN, "kv4_hand_row.json")))
    row = np.array([g["row"]], dtype=np.float32)
    packed, scale = O.kv4_encode_rows(row)
    assert scale[0] == np.float32(g["scale"])
    assert packed[0].tolist() == g["bytes"]
    assert O.kv4_decode_rows(packed, scale)[0].tolist() == g["decoded"]
    # a power-of-two factor moves the scale only
    p2, s2 = O.kv4_encode_rows(row * np.float32(0.125))
    assert p2[0].tolist() == g["bytes"] and s2[0] == np.float32(0.125)
    pz, sz = O.kv4_encode_rows(np.zeros((1, 8), dtype=np.float32))
    assert sz[0] == 0 and pz[0].tolist() == [g["zero_row_byte"]] * 4


def test_kv4_round_trip_error_is_half_a_step():
    """Decoded values stay within half a code step (scale / 2) of the input; the largest magnitude
    of a row decodes to 7 * scale (within fp32 rounding of max|x| / 7); codes stay in [-7, 7]."""
    r = rng(5)
    x = r.normal(size=(60, 128)).astype(np.float32) * r.uniform(0.01, 30, size=(60, 1)).astype(np.float32)
    x[11] = 0.0
    packed, scale = O.kv4_encode_rows(x)
    dec = O.kv4_decode_rows(packed, scale)
    assert scale[11] == 0 and np.all(dec[11] == 0)
    err = np.abs(dec - x)
    assert np.all(err <= scale[:, None] * (0.5 + 1e-6))
    nib = np.stack([packed & 15, packed >> 4], axis=-1)
    assert nib.min() >= 1 and nib.max() <= 15
    for i in range(60):
        if scale[i] > 0:
            j = int(np.argmax(np.abs(x[i])))
            assert abs(abs(dec[i, j]) - abs(x[i, j])) <= abs(x[i, j]) * 1e-6

