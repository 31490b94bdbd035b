"""The oracle against hand-derived examples stored under tests/golden/ (each file names the
passage of the pages it follows and shows its derivation). The pages print no worked
example, so these are the definitions applied by hand to small inputs."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_every_fixture_cites_its_source():
    for name in os.listdir(GOLDEN):
        d = load(name)
        assert d["source"] and d["derivation"], name


@pytest.mark.parametrize("case", load("schedule_hand.json")["cases"])
def test_schedule(case):
    slow = oracle.schedule(np.array(case["mask"], np.uint8), case["t_max"])
    assert np.flatnonzero(slow).tolist() == case["slow_steps"]


@pytest.mark.parametrize("case", load("token_schedule_hand.json")["cases"])
def test_token_schedule(case):
    trig = np.array(load("token_schedule_hand.json")["trigger_ids"], np.int32)
    slow = oracle.schedule_tokens(np.array(case["tokens"], np.int32), trig, case["t_max"])
    assert np.flatnonzero(slow).tolist() == case["slow_steps"]


@pytest.mark.parametrize("case", load("sparse_rows_hand.json")["cases"])
def test_sparse_rows(case):
    rows = oracle.sparse_rows(case["L_slow"], case["L_now"], case["S"], case["W"],
                              np.array(case["selected"], np.int32))
    assert rows.tolist() == case["rows"]


@pytest.mark.parametrize("case", load("fused_scores_hand.json")["cases"])
def test_fused_scores(case):
    f = np.array(case["f"], np.float32)
    s = oracle.fused_scores(case["L"], case["S"], case["W"], case["tau"], case["lambda"], f)
    np.testing.assert_array_equal(s, np.array(case["s"], np.float32))
    sel = oracle.select(case["L"], case["S"], case["W"], 2, case["tau"], case["lambda"], f)
    assert sel.tolist() == case["top2"]


@pytest.mark.parametrize("case", load("topk_ties_hand.json")["cases"])
def test_topk_ties(case):
    s = np.array(load("topk_ties_hand.json")["scores"], np.float32)
    assert sorted(oracle.topk(s, case["K"]).tolist()) == case["kept"]
    assert oracle.topk(s, case["K"]).tolist() == case["kept"]
