"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``check_*`` helper raises AssertionError when the oracle breaks one fact:
a closed form, an invariant, a special case that reduces to a textbook
definition, brute force over every K-subset of a tiny row, or central finite
differences.  The same helpers run against deliberately broken copies of the
oracle (``test_pins_catch_planted_mistakes``) to show that each plausible
mistake fails at least one pin.
"""
import itertools
import math

import numpy as np
import pytest

import oracle.router_oracle as O


# --------------------------------------------------------------------------
# score functions: closed forms
# --------------------------------------------------------------------------
def check_softmax_closed_form():
    # logits ln(1..4): softmax is exactly (1, 2, 3, 4) / 10
    x = np.log(np.array([1.0, 2.0, 3.0, 4.0]))
    s = O.score_row(x, "softmax")
    assert np.allclose(s, [0.1, 0.2, 0.3, 0.4], rtol=0, atol=1e-15), s
    # invariant under a shift of the whole row
    s2 = O.score_row(x + 37.25, "softmax")
    assert np.allclose(s, s2, rtol=0, atol=1e-15)
    # two experts: softmax of (a, b) equals sigmoid(a - b)
    a, b = 0.7, -1.9
    s3 = O.score_row(np.array([a, b]), "softmax")
    assert abs(s3[0] - 1.0 / (1.0 + math.exp(-(a - b)))) < 1e-15
    # random rows sum to one
    rng = np.random.default_rng(1)
    for E in (1, 3, 64, 2304):
        s = O.score_row(rng.normal(0, 2, E), "softmax")
        assert abs(s.sum() - 1.0) < 1e-12
        assert np.all(s > 0)


def check_sigmoid_closed_form():
    s = O.score_row(np.array([0.0, math.log(3.0), -math.log(3.0)]), "sigmoid")
    assert np.allclose(s, [0.5, 0.75, 0.25], rtol=0, atol=1e-15), s
    x = np.random.default_rng(2).normal(0, 3, 1000)
    assert np.allclose(O.score_row(x, "sigmoid") + O.score_row(-x, "sigmoid"), 1.0,
                       rtol=0, atol=1e-15)
    assert np.all(np.diff(O.score_row(np.sort(x), "sigmoid")) >= 0)


def test_softmax_closed_form():
    check_softmax_closed_form()


def test_sigmoid_closed_form():
    check_sigmoid_closed_form()


# --------------------------------------------------------------------------
# top-K selection: brute force over all subsets
# --------------------------------------------------------------------------
def brute_force_topk(keys, K, allowed=None):
    """The K-subset of allowed experts whose smallest key is >= every key left
    out, choosing among valid subsets the lexicographically smallest sorted
    index tuple (= ties to the lower index)."""
    E = len(keys)
    idx = [i for i in range(E) if allowed is None or allowed[i]]
    for sub in itertools.combinations(idx, K):  # lexicographic order
        inside = min(keys[i] for i in sub)
        outside = [keys[i] for i in idx if i not in sub]
        if not outside or inside >= max(outside):
            return set(sub)
    raise AssertionError("no valid subset")


def brute_force_groups(keys, K, G, gk):
    """Group-limited pre-selection by enumeration: a group's score is the
    largest sum over its (K/gk)-subsets; kept groups are the valid gk-subset
    of groups with the lexicographically smallest tuple."""
    E = len(keys)
    eg = E // G
    M = K // gk
    gs = [max(sum(c) for c in itertools.combinations(keys[g * eg:(g + 1) * eg], M))
          for g in range(G)]
    kept = brute_force_topk(gs, gk)
    allowed = [(i // eg) in kept for i in range(E)]
    return allowed


def _rows_for_brute_force(rng, E):
    yield rng.integers(-2, 3, E).astype(float)         # heavy ties
    yield rng.normal(0, 1, E)                          # distinct
    yield np.zeros(E)                                  # all equal
    yield np.where(rng.random(E) < 0.5, 0.0, -0.0)     # signed zeros only
    yield np.round(rng.normal(0, 1, E), 1)             # some ties


def check_topk_brute_force():
    rng = np.random.default_rng(3)
    for E in range(1, 9):
        for x in _rows_for_brute_force(rng, E):
            for sf in ("softmax", "sigmoid"):
                for bias in (None, rng.integers(-1, 2, E) * 0.25):
                    s = O.score_row(x, sf)
                    key = s + (0 if bias is None else bias)
                    for K in range(1, E + 1):
                        _, m, _, _ = O.topk_fwd_row(x, K, sf, expert_bias=bias)
                        want = brute_force_topk(list(key), K)
                        got = set(np.nonzero(m)[0].tolist())
                        assert got == want, (E, K, sf, x, bias, got, want)


def check_grouped_brute_force():
    rng = np.random.default_rng(4)
    for E, G in ((4, 2), (6, 3), (8, 4), (8, 2), (9, 3)):
        for x in _rows_for_brute_force(rng, E):
            for bias in (None, rng.uniform(-0.1, 0.1, E)):
                s = O.score_row(x, "sigmoid")
                key = s + (0 if bias is None else bias)
                for gk in range(1, G + 1):
                    for K in range(gk, gk * (E // G) + 1, gk):
                        _, m, _, _ = O.topk_fwd_row(x, K, "sigmoid", G, gk,
                                                    expert_bias=bias)
                        allowed = brute_force_groups(list(key), K, G, gk)
                        want = brute_force_topk(list(key), K, allowed)
                        got = set(np.nonzero(m)[0].tolist())
                        assert got == want, (E, G, gk, K, x, got, want)


def test_topk_brute_force():
    check_topk_brute_force()


def test_grouped_brute_force():
    check_grouped_brute_force()


# --------------------------------------------------------------------------
# probabilities: closed forms and special cases
# --------------------------------------------------------------------------
def check_probs_closed_forms():
    rng = np.random.default_rng(5)
    for E, K in ((16, 1), (64, 4), (512, 22), (300, 36)):
        x = rng.normal(0, 1.5, E)
        c = 2.5
        p, m, s, _ = O.topk_fwd_row(x, K, "sigmoid", scaling_factor=c)
        assert abs(p.sum() - c) < 1e-12                    # renormalised to c
        assert m.sum() == K and np.all(p[m] > 0) and np.all(p[~m] == 0)
        p, m, s, _ = O.topk_fwd_row(x, K, "softmax", scaling_factor=c)
        assert abs(p.sum() - c * s[m].sum()) < 1e-12
        assert np.allclose(p[m], c * s[m], rtol=0, atol=0)
        assert m.sum() == K and np.all(p[~m] == 0)
        # softmax keyed on the raw logits picks the K largest logits
        assert set(np.nonzero(m)[0]) == set(np.argsort(-x, kind="stable")[:K])
    # K = E: softmax probs are c * softmax; sigmoid probs equal c * aux scores
    x = rng.normal(0, 1, 40)
    p, m, s, _ = O.topk_fwd_row(x, 40, "softmax", scaling_factor=1.5)
    assert np.allclose(p, 1.5 * O.score_row(x, "softmax"), rtol=0, atol=1e-15)
    p, _, _, _ = O.topk_fwd_row(x, 40, "sigmoid", scaling_factor=1.5)
    q, _, _ = O.aux_scores_fwd_row(x, 3, "sigmoid")
    assert np.allclose(p, 1.5 * q, rtol=1e-14, atol=0)
    # an all-equal row selects experts 0..K-1 and softmax probs are c / E
    p, m, _, _ = O.topk_fwd_row(np.full(24, 0.3), 5, "softmax", scaling_factor=2.0)
    assert np.array_equal(np.nonzero(m)[0], np.arange(5))
    assert np.allclose(p[:5], 2.0 / 24, rtol=0, atol=1e-16)
    # K = 1 sigmoid: the single probability is c
    p, m, _, _ = O.topk_fwd_row(x, 1, "sigmoid", scaling_factor=2.5)
    assert p[m][0] == 2.5


def check_grouping_identities():
    rng = np.random.default_rng(6)
    for _ in range(20):
        E, G = 64, 8
        x = rng.normal(0, 1, E)
        b = rng.uniform(-0.1, 0.1, E)
        for sf in ("softmax", "sigmoid"):
            ref = O.topk_fwd_row(x, 8, sf, 0, 0, 2.0, b)
            for ng, gk in ((1, 1), (G, G), (4, 4)):
                got = O.topk_fwd_row(x, 8, sf, ng, gk, 2.0, b)
                assert np.array_equal(got[1], ref[1])
                assert np.array_equal(got[0], ref[0])
            # a constant bias does not change the selection
            m0 = O.topk_fwd_row(x, 8, sf, G, 4, 2.0, None)[1]
            m1 = O.topk_fwd_row(x, 8, sf, G, 4, 2.0, np.full(E, 0.07))[1]
            assert np.array_equal(m0, m1)
    # a hand-built grouped row: group 0 holds the single largest key, but
    # groups 1 and 2 have larger top-2 sums, so group 0 is dropped
    x = np.array([5.0, -5.0, 3.0, 3.0, 2.9, 2.9, 0.0, 0.0])
    _, m, _, _ = O.topk_fwd_row(x, 2, "sigmoid", 4, 1)
    assert np.array_equal(np.nonzero(m)[0], [2, 3])
    _, m, _, _ = O.topk_fwd_row(x, 4, "sigmoid", 4, 2)
    assert np.array_equal(np.nonzero(m)[0], [2, 3, 4, 5])


def check_softmax_post():
    """Post-softmax probs equal c times the softmax of the selected logits
    alone (computed here directly from its definition), select like softmax,
    sum to c, and equal the pre-softmax probs when K = E."""
    rng = np.random.default_rng(11)
    for E, K in ((8, 3), (64, 8), (512, 22), (300, 36)):
        x = rng.normal(0, 1.5, E)
        p, m, s, _ = O.topk_fwd_row(x, K, "softmax_post", scaling_factor=2.5)
        _, m_pre, s_pre, _ = O.topk_fwd_row(x, K, "softmax", scaling_factor=2.5)
        assert np.array_equal(m, m_pre) and np.allclose(s, s_pre, rtol=0, atol=0)
        sel = np.nonzero(m)[0]
        xs = x[sel]
        want = 2.5 * np.exp(xs - xs.max()) / np.exp(xs - xs.max()).sum()
        assert np.allclose(p[sel], want, rtol=1e-13, atol=0)
        assert abs(p.sum() - 2.5) < 1e-12 and np.all(p[~m] == 0)
    x = rng.normal(0, 1, 20)
    assert np.allclose(O.topk_fwd_row(x, 20, "softmax_post")[0],
                       O.topk_fwd_row(x, 20, "softmax")[0], rtol=1e-14, atol=0)


def check_aux_loss():
    """Perfectly balanced routing with uniform scores gives exactly coeff (the
    loss's minimum for balanced assignments); a hand-worked 2 x 2 case; the
    gradient matches central differences; routing every token to one expert
    with all its score there gives coeff * E."""
    T, E, K = 8, 4, 2
    q = np.full((T, E), 1.0 / E)
    m = np.zeros((T, E), bool)
    for t in range(T):                       # each expert gets T K / E tokens
        m[t, [t % E, (t + 1) % E]] = True
    loss, tok = O.aux_loss_fwd(q, m, K, 0.01)
    assert np.array_equal(tok, [4, 4, 4, 4]) and abs(loss - 0.01) < 1e-15
    # 2 tokens x 2 experts, K = 1: tokens = (2, 0), sum_t q = (1.3, 0.7):
    # loss = c * 2 / (1 * 4) * (1.3 * 2 + 0.7 * 0) = c * 1.3
    q = np.array([[0.6, 0.4], [0.7, 0.3]])
    m = np.array([[1, 0], [1, 0]], bool)
    loss, tok = O.aux_loss_fwd(q, m, 1, 2.0)
    assert np.array_equal(tok, [2, 0]) and abs(loss - 2.6) < 1e-15
    # all tokens on expert 0 with q concentrated there: coeff * E
    q = np.zeros((5, 6)); q[:, 0] = 1.0
    m = np.zeros((5, 6), bool); m[:, 0] = True
    assert abs(O.aux_loss_fwd(q, m, 1, 0.5)[0] - 0.5 * 6) < 1e-14
    # gradient
    rng = np.random.default_rng(12)
    T, E, K = 6, 5, 2
    q = rng.random((T, E))
    m = np.zeros((T, E), bool)
    for t in range(T):
        m[t, rng.choice(E, K, replace=False)] = True
    _, tok = O.aux_loss_fwd(q, m, K, 0.3)
    g = O.aux_loss_bwd(1.7, tok, T, K, 0.3)
    h = 1e-6
    for t in range(T):
        for e in range(E):
            qp = q.copy(); qp[t, e] += h
            qm = q.copy(); qm[t, e] -= h
            fd = 1.7 * (O.aux_loss_fwd(qp, m, K, 0.3)[0] - O.aux_loss_fwd(qm, m, K, 0.3)[0]) / (2 * h)
            assert abs(fd - g[t, e]) < 1e-8


def check_compact():
    """Compact outputs: a hand-worked row (ties to the lower index), an
    all-equal row, a biased row whose rank order differs from the weight
    order, the expanded-row index k T + t, and agreement with the dense map
    on random grouped/biased rows (keys non-increasing along k, equal keys in
    increasing index order)."""
    x = np.array([[1.0, 3.0, 3.0, 0.0, 2.0], [0.0, 0.0, 0.0, 0.0, 0.0]])
    o = O.topk_fwd_compact(x, 3, "softmax")
    assert o["topk_indices"].tolist() == [[1, 2, 4], [0, 1, 2]]
    z = np.exp(x[0] - 3.0).sum()
    assert np.allclose(o["topk_weights"][0], np.exp(np.array([3.0, 3.0, 2.0]) - 3.0) / z,
                       rtol=1e-15, atol=0)
    assert np.allclose(o["topk_weights"][1], 0.2, rtol=1e-15, atol=0)
    assert o["token_expert_indices"].tolist() == [[0, 2, 4], [1, 3, 5]]
    # softmax scores (0.665, 0.245, 0.090), bias (0, 1, 0): keys put expert 1
    # first although its weight is the smaller
    o = O.topk_fwd_compact(np.array([[2.0, 1.0, 0.0]]), 2, "softmax",
                           expert_bias=np.array([0.0, 1.0, 0.0]))
    assert o["topk_indices"].tolist() == [[1, 0]]
    assert o["topk_weights"][0, 0] < o["topk_weights"][0, 1]
    rng = np.random.default_rng(13)
    T, E, K = 7, 24, 6
    for sf in ("softmax", "sigmoid", "softmax_post"):
        x = rng.integers(-3, 4, (T, E)).astype(float)      # many ties
        b = rng.uniform(-0.1, 0.1, E)
        d = O.topk_fwd(x, K, sf, 4, 2, 1.5, b)
        o = O.topk_fwd_compact(x, K, sf, 4, 2, 1.5, b)
        assert sorted(o["token_expert_indices"].ravel().tolist()) == list(range(T * K))
        for t in range(T):
            idx = o["topk_indices"][t]
            assert sorted(idx.tolist()) == np.nonzero(d["routing_map"][t])[0].tolist()
            assert np.array_equal(o["topk_weights"][t], d["probs"][t][idx])
            key = d["scores"][t][idx] + b[idx]
            for k in range(K - 1):
                assert key[k] > key[k + 1] or (key[k] == key[k + 1] and idx[k] < idx[k + 1])


def test_compact():
    check_compact()


def check_expert_maps():
    """A hand-worked 3 x 2 case (expert 0 taken by token 0 at k = 1 before
    token 1 at k = 0: token order, not k order), then invariants on random
    routings: the maps are inverse permutations, each permuted row's expert
    and column recover the (t, k) choice through the reverse-permute
    formula, offsets are the histogram's prefix sums, and tokens rise inside
    each expert's range."""
    m = O.expert_maps(np.array([[2, 0], [0, 1], [2, 1]]), 4)
    assert m["permuted_to_unpermuted"].tolist() == [3, 1, 4, 5, 0, 2]
    assert m["unpermuted_to_permuted"].tolist() == [4, 1, 5, 0, 2, 3]
    assert m["permuted_experts"].tolist() == [0, 0, 1, 1, 2, 2]
    assert m["expert_first_token_offset"].tolist() == [0, 2, 4, 6, 6]
    rng = np.random.default_rng(14)
    for T, E, K in ((1, 8, 3), (5, 6, 6), (40, 64, 8), (33, 300, 36)):
        idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)])
        m = O.expert_maps(idx, E)
        p2u, u2p = m["permuted_to_unpermuted"], m["unpermuted_to_permuted"]
        off, ex = m["expert_first_token_offset"], m["permuted_experts"]
        n = T * K
        assert sorted(p2u.tolist()) == list(range(n))
        assert np.array_equal(u2p[p2u], np.arange(n))
        assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(idx.ravel(), minlength=E))]))
        for t in range(T):
            for k in range(K):
                p = u2p[t + k * T]
                e = ex[p]
                assert e == idx[t, k] and off[e] <= p < off[e + 1]
        tok = p2u % T
        for e in range(E):
            assert np.all(np.diff(tok[off[e]:off[e + 1]]) > 0)


def test_expert_maps():
    check_expert_maps()


def test_aux_loss():
    check_aux_loss()


def test_probs_closed_forms():
    check_probs_closed_forms()


def test_softmax_post():
    check_softmax_post()


def test_grouping_identities():
    check_grouping_identities()


# --------------------------------------------------------------------------
# backward: central finite differences of L = sum g * p(x)
# --------------------------------------------------------------------------
def _fd_grad(f, x, h):
    gx = np.zeros_like(x)
    for j in range(x.size):
        e = np.zeros_like(x)
        e[j] = h
        gx[j] = (f(x + e) - f(x - e)) / (2 * h)
    return gx


def check_topk_bwd_finite_differences():
    rng = np.random.default_rng(7)
    h = 1e-4
    checked = 0
    for sf in ("softmax", "sigmoid", "softmax_post"):
        for E, K, c, ng, gk, use_b in ((12, 1, 1.0, 0, 0, False), (12, 3, 2.5, 0, 0, True),
                                       (32, 5, 1.0, 0, 0, False), (32, 8, 2.5, 4, 2, True),
                                       (40, 40, 1.0, 0, 0, False)):
            for _ in range(3):
                x = rng.normal(0, 1.5, E)
                b = rng.uniform(-0.1, 0.1, E) if use_b else None
                g = rng.normal(0, 1, E)
                p, m, s, _ = O.topk_fwd_row(x, K, sf, ng, gk, c, b)

                def loss(xx):
                    pp, mm, _, _ = O.topk_fwd_row(xx, K, sf, ng, gk, c, b)
                    assert np.array_equal(mm, m)
                    return float(np.dot(g, pp))
                try:
                    fd = _fd_grad(loss, x, h)
                except AssertionError:
                    continue  # the selection moved under +-h: not a smooth point
                an = O.topk_bwd_row(g, m, s, sf, c)
                assert np.all(np.abs(fd - an) <= 1e-3 * np.maximum(1, np.abs(an))), \
                    (sf, E, K, np.max(np.abs(fd - an)))
                # tighter than the stated bound: the formula is exact
                assert np.max(np.abs(fd - an)) < 1e-6
                if sf == "softmax":
                    assert abs(an.sum()) < 1e-12   # constants are in the kernel
                if sf in ("sigmoid", "softmax_post") and K == 1:
                    assert np.all(an == 0)
                if sf == "softmax_post":
                    assert abs(an.sum()) < 1e-12   # invariant under a shift of x
                checked += 1
    assert checked >= 20


def check_aux_closed_forms_and_fd():
    rng = np.random.default_rng(8)
    h = 1e-4
    for sf in ("softmax", "sigmoid"):
        for E, K in ((7, 2), (64, 8), (300, 36)):
            x = rng.normal(0, 1.5, E)
            q, m, saved = O.aux_scores_fwd_row(x, K, sf)
            assert abs(q.sum() - 1) < 1e-12
            assert m.sum() == K
            assert set(np.nonzero(m)[0]) == set(np.argsort(-x, kind="stable")[:K])
            if sf == "sigmoid":
                assert np.allclose(saved, 1 / (1 + np.exp(-x)), rtol=0, atol=1e-15)
            if E <= 64:
                g = rng.normal(0, 1, E)
                fd = _fd_grad(lambda xx: float(np.dot(g, O.aux_scores_fwd_row(xx, K, sf)[0])),
                              x, h)
                an = O.aux_scores_bwd_row(g, saved, sf)
                assert np.max(np.abs(fd - an)) < 1e-6, (sf, E, np.max(np.abs(fd - an)))
    # uniform logits: q is uniform, the map is experts 0..K-1
    for sf in ("softmax", "sigmoid"):
        q, m, _ = O.aux_scores_fwd_row(np.full(10, -0.4), 3, sf)
        assert np.allclose(q, 0.1, rtol=0, atol=1e-16)
        assert np.array_equal(np.nonzero(m)[0], [0, 1, 2])


def test_topk_bwd_finite_differences():
    check_topk_bwd_finite_differences()


def test_aux_closed_forms_and_fd():
    check_aux_closed_forms_and_fd()


# --------------------------------------------------------------------------
# output rounding to bf16 (nearest, ties to even)
# --------------------------------------------------------------------------
def check_bf16_rounding():
    u = 2.0 ** -7  # bf16 spacing in [1, 2)
    cases = {1.0: 1.0, 1 + u / 2: 1.0, 1 + 1.5 * u: 1 + 2 * u, 1 + 0.49 * u: 1.0,
             1 + 0.51 * u: 1 + u, -3.0: -3.0, 0.0: 0.0, 255.5: 256.0, 254.5: 254.0,
             2 - u / 4: 2.0}
    for v, want in cases.items():
        assert O.round_to_bf16(np.array([v]))[0] == want, (v, want)
    # agrees with torch's fp32 -> bf16 conversion on fp32 inputs
    import torch
    x = np.random.default_rng(9).normal(0, 10, 10000).astype(np.float32)
    t = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_to_bf16(x.astype(np.float64)), t)


def test_bf16_rounding():
    check_bf16_rounding()


# --------------------------------------------------------------------------
# near ties: which rows may legitimately select differently.  The rule: a
# row is a near tie when the keys on either side of its top-K boundary (or the
# group scores on either side of its group boundary) are distinct and within
# 1e-6 relative; exact ties are not near ties.  Every row below is built by
# hand so that its status follows from that rule and the arithmetic of exp:
# for softmax keys, logits d apart give keys whose relative gap is
# 1 - exp(-d), i.e. d to within d^2 / 2; for sigmoid keys at x = 0 the relative
# gap of logits d apart is d / 2 to first order.
# --------------------------------------------------------------------------
_TAIL = [-1.0, 0.0, -2.0]   # three experts far below every boundary here


def _near_rows():
    """(name, logits row, K, score function, bias, groups, want near_tie)."""
    rows = [
        # K-th and (K+1)-th logits equal: an exact tie, decided by index
        ("exact tie at the boundary", [3.0, 1.0, 1.0] + _TAIL, 2, "softmax", None, None, False),
        # 5e-7 apart: relative key gap 4.9999988e-7 <= 1e-6
        ("5e-7 at the boundary", [3.0, 1.0, 1.0 - 5e-7] + _TAIL, 2, "softmax", None, None, True),
        # 2e-6 apart: relative key gap 1.999998e-6 > 1e-6
        ("2e-6 at the boundary", [3.0, 1.0, 1.0 - 2e-6] + _TAIL, 2, "softmax", None, None, False),
        # the near pair is ranks 1 and 2, both selected; the boundary (rank 2
        # against rank 3) is 2 logits wide
        ("near pair inside the top-K", [3.0, 3.0 - 5e-7, 1.0] + _TAIL, 2, "softmax", None,
         None, False),
        # the near pair is ranks 3 and 4, both left out
        ("near pair below the boundary", [3.0, 2.0, 1.0, 1.0 - 5e-7, -2.0, -3.0], 2,
         "softmax", None, None, False),
        # keys near 0.1 that differ by about 5e-7 in absolute terms but by
        # 5e-6 relative: not near (the rule is relative)
        ("small keys, 5e-6 relative", [3.0, 1.0, 1.0 - 5e-6] + _TAIL, 2, "softmax", None,
         None, False),
        # sigmoid keys 0.5 and sigmoid(-1e-6): relative gap 5e-7
        ("sigmoid, 5e-7 at the boundary", [0.0, -1e-6, -3.0, -4.0], 1, "sigmoid", None,
         None, True),
        # equal scores (all logits 0: s = 1/4), keys s + b differ by 3e-7
        # absolute at 0.75, i.e. 4e-7 relative: the key decides, not the score
        ("biased keys 4e-7 apart", [0.0, 0.0, 0.0, 0.0], 1, "softmax",
         [0.0, 0.5, 0.5 - 3e-7, 0.0], None, True),
    ]
    # four groups of two, keep two, K = 2: a group scores its largest key.
    # Kept: groups 0 and 1; the expert boundary (s(3) against s(0)) is wide.
    rows += [
        ("group scores 5e-7 apart at the group boundary",
         [5.0, 0.0, 3.0, -1.0, 3.0 - 5e-7, -1.0, -2.0, -2.0], 2, "softmax", None, (4, 2), True),
        ("group scores tied exactly at the group boundary",
         [5.0, 0.0, 3.0, -1.0, 3.0, -1.0, -2.0, -2.0], 2, "softmax", None, (4, 2), False),
        ("group scores 2e-6 apart at the group boundary",
         [5.0, 0.0, 3.0, -1.0, 3.0 - 2e-6, -1.0, -2.0, -2.0], 2, "softmax", None, (4, 2), False),
        # the near groups (0 and 1) are both kept; groups 2 and 3 are far below
        ("near groups both kept",
         [3.0, -1.0, 3.0 - 5e-7, -1.0, 1.0, -2.0, -2.0, -3.0], 2, "softmax", None, (4, 2), False),
        # keeping every group leaves no group boundary; K = 4 puts the
        # expert boundary between s(0) and s(-1)
        ("every group kept",
         [5.0, 0.0, 3.0, -1.0, 3.0 - 5e-7, -1.0, -2.0, -2.0], 4, "softmax", None, (4, 4), False),
    ]
    return rows


def check_near_tie_classifier():
    for name, x, K, sf, b, grp, want in _near_rows():
        logits = np.array([x], dtype=np.float64)
        bias = None if b is None else np.array(b, dtype=np.float64)
        ng, gk = grp if grp is not None else (0, 0)
        got = O.topk_fwd(logits, K, sf, ng, gk, 1.0, bias)["near_tie"][0]
        assert got == want, (name, got, want)
        got_c = O.topk_fwd_compact(logits, K, sf, ng, gk, 1.0, bias)["near_tie"][0]
        assert got_c == want, (name, "compact", got_c, want)
    # aux scores: the same boundary rule on q (softmax; sigmoid / sum sigmoid,
    # whose relative gaps are those of the sigmoid)
    aux = [
        ([3.0, 1.0, 1.0] + _TAIL, 2, "softmax", False),
        ([3.0, 1.0, 1.0 - 5e-7] + _TAIL, 2, "softmax", True),
        ([3.0, 1.0, 1.0 - 2e-6] + _TAIL, 2, "softmax", False),
        ([3.0, 2.0, 1.0, 1.0 - 5e-7, -2.0, -3.0], 2, "softmax", False),
        ([0.0, -1e-6, -3.0, -4.0], 1, "sigmoid", True),
        ([0.0, 0.0, -3.0, -4.0], 1, "sigmoid", False),
    ]
    for x, K, sf, want in aux:
        got = O.aux_scores_fwd(np.array([x]), K, sf)["near_tie"][0]
        assert got == want, ("aux", x, K, sf, got, want)
    # K = E: no boundary at all
    assert not O.topk_fwd(np.array([[1.0, 1.0 - 5e-7]]), 2)["near_tie"][0]
    # several rows at once: the flags line up with their rows
    rows = _near_rows()[:3]
    batch = np.array([r[1] for r in rows])
    assert list(O.topk_fwd(batch, 2)["near_tie"]) == [r[6] for r in rows]


def test_near_tie_classifier():
    check_near_tie_classifier()


def test_near_tie_rows_select_by_the_rule():
    # the exact-tie row selects the lower index (not exempt); the 5e-7 row
    # selects the larger key, index 1, like any other row
    r = O.topk_fwd(np.array([[3.0, 1.0, 1.0] + _TAIL]), 2)
    assert list(np.nonzero(r["routing_map"][0])[0]) == [0, 1]
    r = O.topk_fwd(np.array([[3.0, 1.0 - 5e-7, 1.0] + _TAIL]), 2)
    assert list(np.nonzero(r["routing_map"][0])[0]) == [0, 2]


# --------------------------------------------------------------------------
# the pins catch plausible mistakes planted in the oracle (CPU only)
# --------------------------------------------------------------------------
def _wrong_order(keys):  # ties to the HIGHER index
    keys = np.asarray(keys, dtype=np.float64)
    return np.lexsort((-np.arange(keys.size), -keys))


def _wrong_softmax_score(x, sf):
    x = np.asarray(x, dtype=np.float64)
    if sf == "softmax":
        e = np.exp(x - x.max())
        return e / e.max()          # normalised by the max, not the sum
    return 1 / (1 + np.exp(-x))


def _wrong_sigmoid_sign(x, sf):
    x = np.asarray(x, dtype=np.float64)
    if sf == "sigmoid":
        return 1 / (1 + np.exp(x))
    e = np.exp(x - x.max())
    return e / e.sum()


def _wrong_group_scores(keys, G, per_group):  # strided instead of contiguous
    return np.array([np.sort(keys[g::G])[::-1][:per_group].sum() for g in range(G)])


def _wrong_group_scores_max(keys, G, per_group):  # max instead of top-M sum
    eg = keys.size // G
    return np.array([keys[g * eg:(g + 1) * eg].max() for g in range(G)])


_orig_topk_bwd_row = O.topk_bwd_row


def _wrong_bwd_no_d(g, m, s, sf, c=1.0):
    g = np.asarray(g, float)
    s = np.asarray(s, float)
    mm = np.asarray(m, bool).astype(float)
    if sf == "softmax":
        return s * (c * mm * g)     # drops the -D term
    return _orig_topk_bwd_row(g, m, s, sf, c)


def _wrong_bwd_sigmoid_scale(g, m, s, sf, c=1.0):
    if sf == "sigmoid":
        return _orig_topk_bwd_row(g, m, s, sf, 1.0)   # drops c
    return _orig_topk_bwd_row(g, m, s, sf, c)


_orig_fwd_row = O.topk_fwd_row


def _wrong_no_renorm(x, K, score_func, num_groups=0, group_topk=0,
                     scaling_factor=1.0, expert_bias=None):
    p, m, s, n = _orig_fwd_row(x, K, score_func, num_groups, group_topk,
                               scaling_factor, expert_bias)
    if score_func == "sigmoid":
        p = np.where(m, scaling_factor * s, 0.0)
    return p, m, s, n


_orig_aux_bwd = O.aux_scores_bwd_row


def _wrong_aux_bwd(g, saved, sf):
    if sf == "sigmoid":
        v = np.asarray(saved, float)
        Z = v.sum()
        return (np.asarray(g, float) - np.sum(g * v) / Z) / Z * v   # drops (1 - v)
    return _orig_aux_bwd(g, saved, sf)


def _wrong_bf16(x):
    return np.asarray(x, np.float64).astype(np.float32).view(np.uint32) \
        .__and__(np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)  # truncation


def _wrong_post_bwd(g, m, s, sf, c=1.0):
    if sf == "softmax_post":
        return _orig_topk_bwd_row(g, m, s, "sigmoid", c)   # sigmoid's extra (1 - s)
    return _orig_topk_bwd_row(g, m, s, sf, c)


_orig_aux_loss = O.aux_loss_fwd


def _wrong_aux_loss(q, m, K, coeff):   # divides by T instead of T^2
    loss, tok = _orig_aux_loss(q, m, K, coeff)
    return loss * np.asarray(q).shape[0], tok


_orig_compact = O.topk_fwd_compact


def _wrong_compact_by_weight(logits, K, sf="softmax", ng=0, gk=0, c=1.0, expert_bias=None):
    o = _orig_compact(logits, K, sf, ng, gk, c, expert_bias)   # ranks by weight, not key
    order = np.argsort(-o["topk_weights"], axis=1, kind="stable")
    o["topk_indices"] = np.take_along_axis(o["topk_indices"], order, 1)
    o["topk_weights"] = np.take_along_axis(o["topk_weights"], order, 1)
    return o


def _wrong_compact_tei(logits, K, sf="softmax", ng=0, gk=0, c=1.0, expert_bias=None):
    o = _orig_compact(logits, K, sf, ng, gk, c, expert_bias)   # t K + k instead of k T + t
    T = np.asarray(logits).shape[0]
    o["token_expert_indices"] = np.arange(T * K).reshape(T, K)
    return o


_orig_expert_maps = O.expert_maps


def _wrong_maps_k_order(idx, E):   # sorts by (expert, k, token)
    idx = np.asarray(idx)
    T, K = idx.shape
    out = _orig_expert_maps(idx, E)
    choices = sorted((int(idx[t, k]), k, t) for t in range(T) for k in range(K))
    out["permuted_to_unpermuted"] = np.array([t + k * T for _, k, t in choices])
    out["unpermuted_to_permuted"][out["permuted_to_unpermuted"]] = np.arange(T * K)
    return out


def _wrong_maps_row_major(idx, E):   # expanded row t K + k instead of t + k T
    idx = np.asarray(idx)
    T, K = idx.shape
    out = _orig_expert_maps(idx, E)
    p2u = out["permuted_to_unpermuted"]
    t, k = p2u % T, p2u // T
    out["permuted_to_unpermuted"] = t * K + k
    out["unpermuted_to_permuted"][out["permuted_to_unpermuted"]] = np.arange(T * K)
    return out


def _wrong_near_exact_ties(a, b):   # exempts exact ties too
    d = abs(a - b)
    return 0.0 <= d <= O.NEAR_TIE_REL * max(abs(a), abs(b))


def _wrong_near_absolute(a, b):   # absolute instead of relative
    d = abs(a - b)
    return 0.0 < d <= O.NEAR_TIE_REL


def _wrong_boundary_one_below(ranked_keys, K):   # (K+1)-th against (K+2)-th
    if K + 1 >= ranked_keys.size:
        return False
    return O._near(ranked_keys[K], ranked_keys[K + 1])


def _wrong_boundary_inside(ranked_keys, K):   # (K-1)-th against K-th
    if K >= ranked_keys.size or K < 2:
        return False
    return O._near(ranked_keys[K - 2], ranked_keys[K - 1])


def _wrong_group_near_dropped(gs, group_topk):   # the group boundary ignored
    return False


PLANTED = [
    ("_near", _wrong_near_exact_ties, [check_near_tie_classifier]),
    ("_near", _wrong_near_absolute, [check_near_tie_classifier]),
    ("boundary_near_tie", _wrong_boundary_one_below, [check_near_tie_classifier]),
    ("boundary_near_tie", _wrong_boundary_inside, [check_near_tie_classifier]),
    ("group_near_tie", _wrong_group_near_dropped, [check_near_tie_classifier]),
    ("expert_maps", _wrong_maps_k_order, [check_expert_maps]),
    ("expert_maps", _wrong_maps_row_major, [check_expert_maps]),
    ("topk_fwd_compact", _wrong_compact_by_weight, [check_compact]),
    ("topk_fwd_compact", _wrong_compact_tei, [check_compact]),
    ("order_desc", _wrong_order, [check_topk_brute_force]),
    ("score_row", _wrong_softmax_score, [check_softmax_closed_form]),
    ("score_row", _wrong_sigmoid_sign, [check_sigmoid_closed_form]),
    ("group_scores", _wrong_group_scores, [check_grouped_brute_force]),
    ("group_scores", _wrong_group_scores_max, [check_grouped_brute_force]),
    ("topk_bwd_row", _wrong_bwd_no_d, [check_topk_bwd_finite_differences]),
    ("topk_bwd_row", _wrong_bwd_sigmoid_scale, [check_topk_bwd_finite_differences]),
    ("topk_bwd_row", _wrong_post_bwd, [check_topk_bwd_finite_differences]),
    ("topk_fwd_row", _wrong_no_renorm, [check_probs_closed_forms]),
    ("aux_scores_bwd_row", _wrong_aux_bwd, [check_aux_closed_forms_and_fd]),
    ("round_to_bf16", _wrong_bf16, [check_bf16_rounding]),
    ("aux_loss_fwd", _wrong_aux_loss, [check_aux_loss]),
]


@pytest.mark.parametrize("name,wrong,checks", PLANTED,
                         ids=[f"{p[0]}-{p[1].__name__}" for p in PLANTED])
def test_pins_catch_planted_mistakes(monkeypatch, name, wrong, checks):
    monkeypatch.setattr(O, name, wrong)
    for check in checks:
        with pytest.raises(AssertionError):
            check()
