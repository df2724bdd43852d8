"""The oracle against the hand-worked fixtures in tests/golden/."""
import numpy as np
import pytest

import oracle.router_oracle as O
from golden_cases import all_cases

CASES = all_cases()


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_oracle_matches_hand_worked_case(case):
    x = case["logits"][None, :]
    sf, K = case["score_func"], case["K"]
    if case["op"] == "topk_fwd":
        r = O.topk_fwd(x, K, sf, case["num_groups"], case["group_topk"],
                       case["scaling_factor"])
        assert np.array_equal(r["routing_map"][0], case["routing_map"].astype(bool))
        if "scores" in case:
            assert np.allclose(r["scores"][0], case["scores"], rtol=0, atol=1e-15)
        if "probs" in case:
            assert np.allclose(r["probs"][0], case["probs"], rtol=0, atol=1e-15)
    elif case["op"] == "topk_bwd":
        r = O.topk_fwd(x, K, sf, scaling_factor=case["scaling_factor"])
        assert np.array_equal(r["routing_map"][0], case["routing_map"].astype(bool))
        gx = O.topk_bwd(case["grad_probs"][None, :], r["routing_map"], r["scores"], sf,
                        case["scaling_factor"])
        assert np.allclose(gx[0], case["grad_logits"], rtol=0, atol=1e-15)
    elif case["op"] == "aux":
        r = O.aux_scores_fwd(x, K, sf)
        assert np.allclose(r["scores"][0], case["scores"], rtol=0, atol=1e-15)
        assert np.array_equal(r["routing_map"][0], case["routing_map"].astype(bool))
        if "intermediate" in case:
            assert np.allclose(r["saved"][0], case["intermediate"], rtol=0, atol=1e-15)
        gx = O.aux_scores_bwd(case["grad_scores"][None, :], r["saved"], sf)
        assert np.allclose(gx[0], case["grad_logits"], rtol=0, atol=1e-15)
    else:
        raise AssertionError(case["op"])
