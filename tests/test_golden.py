"""The oracle against the stored golden cases (hand-derived, and its own regression fixture)."""

import json
import math
import os

import torch

from paged_kv_decode_mapping_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _scatter(k, v, BS=2, seed=0):
    """Dense [L, D] keys/values spread over a shuffled pool of 2L blocks (one kv head)."""
    L, D = k.shape
    nblk = (L + BS - 1) // BS
    NB = 2 * nblk + 1
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(seed))
    table = perm[:nblk].to(torch.int32)[None]
    kc = torch.full((NB, 1, BS, D), float("nan")).to(torch.bfloat16)
    vc = kc.clone()
    for t in range(L):
        kc[int(table[0, t // BS]), 0, t % BS] = k[t]
        vc[int(table[0, t // BS]), 0, t % BS] = v[t]
    return kc, vc, table


def test_closed_form_cases(oracle):
    doc = json.load(open(os.path.join(GOLD, "closed_form_cases.json")))
    scales = {"ln3": math.log(3.0), "ln2": math.log(2.0), "1": 1.0}
    for case in doc["cases"]:
        k = torch.tensor(case["k"]).to(torch.bfloat16)
        v = torch.tensor(case["v"]).to(torch.bfloat16)
        assert torch.equal(k.float(), torch.tensor(case["k"]))  # exactly representable
        assert torch.equal(v.float(), torch.tensor(case["v"]))
        q = torch.tensor(case["q"]).to(torch.bfloat16)[None, None]
        for seed in range(3):
            kc, vc, table = _scatter(k, v, seed=seed)
            out = oracle.decode(q, kc, vc, table, torch.tensor([len(k)], dtype=torch.int32),
                                scales[case["scale"]])
            assert torch.allclose(out[0, 0], torch.tensor(case["out"], dtype=torch.float64),
                                  atol=1e-12), case["name"]


def test_regression_fixture(oracle):
    doc = json.load(open(os.path.join(GOLD, "oracle_small_case.json")))
    spec = dict(doc["spec"])
    spec["lens"] = tuple(spec["lens"])
    inp = W.make_inputs(W.small_workload(**spec))
    out, _, _ = oracle.step(inp)
    assert torch.allclose(out, torch.tensor(doc["out"], dtype=torch.float64), atol=1e-12)
