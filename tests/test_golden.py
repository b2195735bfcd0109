"""The oracle against verification steps worked out by hand from the pages'
rules (tests/golden/hand_cases.json; each case carries its derivation and the
passage it follows)."""
import pytest

import golden_cases as gc

CASES = gc.load()


@pytest.mark.parametrize("case", CASES["sample_cases"], ids=lambda c: c["name"])
def test_sample_hand_cases(orc, case):
    target, draft, tokens, uni = gc.sample_case(case)
    r = orc.verify_sample(target, "f32", draft, "f32", True, tokens, uni, 1.0)
    assert r["out_tokens"][0].tolist() == case["out_tokens"]
    assert int(r["num_accepted"][0]) == case["num_accepted"]
    assert r["near_accept"][0] == -1 and r["near_cdf"][0] == 0


@pytest.mark.parametrize("case", CASES["greedy_cases"], ids=lambda c: c["name"])
def test_greedy_hand_cases(orc, case):
    target, tokens = gc.greedy_case(case)
    out, n = orc.verify_greedy(target, "f32", tokens)
    assert out[0].tolist() == case["out_tokens"]
    assert int(n[0]) == case["num_accepted"]


@pytest.mark.parametrize("case", CASES["tree_cases"], ids=lambda c: c["name"])
def test_tree_hand_cases(orc, case):
    rows, parents, tokens, max_depth = gc.tree_case(case)
    out, n, path = orc.verify_tree_greedy(rows, "f32", parents, tokens, max_depth)
    assert out[0].tolist() == case["out_tokens"]
    assert int(n[0]) == case["num_accepted"]
    assert path[0].tolist() == case["out_path"]
