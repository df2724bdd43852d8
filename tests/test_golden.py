"""The oracle against the hand-worked fixtures in tests/golden/."""
import numpy as np
import pytest

import oracle.router_oracle as O
from golden_cases import all_cases

CASES = all_cases()


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_oracle_matches_hand_worked_case(case):
    op = case["op"]
    if op == "maps":
        r = O.expert_maps(case["topk_indices"].astype(np.int64), case["E"])
        for name in ("expert_first_token_offset", "permuted_to_unpermuted",
                     "unpermuted_to_permuted", "permuted_experts"):
            assert np.array_equal(r[name], case[name].astype(np.int64)), name
        return
    K = case["K"]
    if op == "aux_loss":
        q, m = case["scores"], case["routing_map"].astype(bool)
        loss, tokens = O.aux_loss_fwd(q, m, K, case["coeff"])
        assert abs(loss - case["loss"][0]) <= 1e-15
        assert np.array_equal(tokens, case["tokens"].astype(np.int64))
        g = O.aux_loss_bwd(case["grad_loss"][0], tokens, q.shape[0], K, case["coeff"])
        assert np.allclose(g, case["grad_scores"], rtol=0, atol=1e-15)
        return
    sf = case["score_func"]
    if op == "compact":
        r = O.topk_fwd_compact(case["logits"], K, sf, case["num_groups"], case["group_topk"],
                               case["scaling_factor"])
        assert np.array_equal(r["topk_indices"], case["topk_indices"].astype(np.int64))
        assert np.allclose(r["topk_weights"], case["topk_weights"], rtol=0, atol=1e-15)
        assert np.array_equal(r["token_expert_indices"],
                              case["token_expert_indices"].astype(np.int64))
        assert not r["near_tie"].any()
        return
    x = case["logits"][None, :]
    if op == "topk_fwd":
        r = O.topk_fwd(x, K, sf, case["num_groups"], case["group_topk"],
                       case["scaling_factor"])
        assert np.array_equal(r["routing_map"][0], case["routing_map"].astype(bool))
        if "scores" in case:
            assert np.allclose(r["scores"][0], case["scores"], rtol=0, atol=1e-15)
        if "probs" in case:
            assert np.allclose(r["probs"][0], case["probs"], rtol=0, atol=1e-15)
    elif op == "topk_bwd":
        r = O.topk_fwd(x, K, sf, scaling_factor=case["scaling_factor"])
        assert np.array_equal(r["routing_map"][0], case["routing_map"].astype(bool))
        gx = O.topk_bwd(case["grad_probs"][None, :], r["routing_map"], r["scores"], sf,
                        case["scaling_factor"])
        assert np.allclose(gx[0], case["grad_logits"], rtol=0, atol=1e-15)
    elif op == "aux":
        r = O.aux_scores_fwd(x, K, sf)
        assert np.allclose(r["scores"][0], case["scores"], rtol=0, atol=1e-15)
        assert np.array_equal(r["routing_map"][0], case["routing_map"].astype(bool))
        if "intermediate" in case:
            assert np.allclose(r["saved"][0], case["intermediate"], rtol=0, atol=1e-15)
        gx = O.aux_scores_bwd(case["grad_scores"][None, :], r["saved"], sf)
        assert np.allclose(gx[0], case["grad_logits"], rtol=0, atol=1e-15)
    else:
        raise AssertionError(op)


# Mistakes planted in the oracle, each of which the named hand-worked fixture
# must catch.
_orig_aux_loss_fwd = O.aux_loss_fwd
_orig_aux_loss_bwd = O.aux_loss_bwd
_orig_compact = O.topk_fwd_compact
_orig_maps = O.expert_maps
_orig_bwd_row = O.topk_bwd_row


def _aux_loss_over_t(q, m, K, coeff):          # divides by T, not T^2
    loss, tokens = _orig_aux_loss_fwd(q, m, K, coeff)
    return loss * np.asarray(q).shape[0], tokens


def _aux_loss_without_k(q, m, K, coeff):       # f_e = tokens / T, K dropped
    loss, tokens = _orig_aux_loss_fwd(q, m, K, coeff)
    return loss * K, tokens


def _aux_loss_bwd_without_k(grad_loss, tokens, T, K, coeff):
    return _orig_aux_loss_bwd(grad_loss, tokens, T, 1, coeff)


def _compact_row_major_tei(logits, K, sf="softmax", ng=0, gk=0, c=1.0, expert_bias=None):
    out = _orig_compact(logits, K, sf, ng, gk, c, expert_bias)   # t K + k
    T = np.asarray(logits).shape[0]
    out["token_expert_indices"] = np.arange(T * K).reshape(T, K)
    return out


def _order_ties_to_higher(keys):
    keys = np.asarray(keys, dtype=np.float64)
    return np.lexsort((-np.arange(keys.size), -keys))


def _maps_by_choice_index(idx, E):             # (expert, k, token) order
    idx = np.asarray(idx)
    T, K = idx.shape
    out = _orig_maps(idx, E)
    choices = sorted((int(idx[t, k]), k, t) for t in range(T) for k in range(K))
    out["permuted_to_unpermuted"] = np.array([t + k * T for _, k, t in choices])
    out["unpermuted_to_permuted"][out["permuted_to_unpermuted"]] = np.arange(T * K)
    return out


def _post_bwd_with_sigmoid_factor(g, m, s, sf, c=1.0):
    if sf == "softmax_post":
        return _orig_bwd_row(g, m, s, "sigmoid", c)   # an extra (1 - s)
    return _orig_bwd_row(g, m, s, sf, c)


PLANTED = [
    ("aux_loss_fwd", _aux_loss_over_t, "aux_loss_k1.txt"),
    ("aux_loss_fwd", _aux_loss_without_k, "aux_loss_k2.txt"),
    ("aux_loss_bwd", _aux_loss_bwd_without_k, "aux_loss_k2.txt"),
    ("topk_fwd_compact", _compact_row_major_tei, "compact.txt"),
    ("order_desc", _order_ties_to_higher, "compact.txt"),
    ("expert_maps", _maps_by_choice_index, "expert_maps.txt"),
    ("topk_bwd_row", _post_bwd_with_sigmoid_factor, "softmax_post_bwd.txt"),
]
BY_NAME = {c["name"]: c for c in CASES}


@pytest.mark.parametrize("name,wrong,fixture", PLANTED,
                         ids=[f"{p[2]}-{p[1].__name__}" for p in PLANTED])
def test_fixture_catches_planted_mistake(monkeypatch, name, wrong, fixture):
    test_oracle_matches_hand_worked_case(BY_NAME[fixture])   # passes as written
    monkeypatch.setattr(O, name, wrong)
    with pytest.raises(AssertionError):
        test_oracle_matches_hand_worked_case(BY_NAME[fixture])
