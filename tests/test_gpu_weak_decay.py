"""Weak decay over a long sequence: g = logsigmoid(N(mu, 1)) with mu = 8 to
10, so the state keeps tokens for thousands of steps instead of the
workloads' 20 (mu = 3) to 150 (mu = 5).

The relative error of o grows with mu at any length (4.34e-3 at mu = 5,
4.86e-3 at 8, 4.93e-3 at 9, 5.03e-3 at 10, the same at 16 k and 64 k
tokens): when the state dominates o, every bf16 rounding of the method's
precision contract (the intermediates qg, kg, w, u, Aqk; the state and v'
as MMA operands; o itself) weighs a little more.  mu = 8 and 9 are held to
the forward's tolerances; mu = 10 is held to 1.1 times them, the measured
edge of the contract, so that a change that makes the weak-decay error
worse still fails.  One 65 536-token sequence of two heads, every element
against the fp64 recurrence; the figures are printed."""
from __future__ import annotations

import pytest
import torch

from chunked_gated_delta_gb300 import synth
from parity_util import MAXREL_O, REL_HT, REL_O, UNIT_REL, assert_within, compare, oracle_ref, report, run_gpu

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _run(mu):
    x = synth.make_inputs(synth.Workload("weak_decay", B=1, T=65536, H=2, K=128, V=128, mu=mu,
                                         seed=20261214 + int(mu)))
    o, ht = run_gpu(x)
    o_ref, ht_ref = oracle_ref(x)
    res = compare(x, o, ht, o_ref, ht_ref)
    report(f"weak decay mu={mu:g}", res)
    return res


@pytest.mark.parametrize("mu", [8.0, 9.0])
def test_weak_decay_within_tolerance(mu):
    assert_within(_run(mu), f"mu={mu}")


def test_weak_decay_edge_of_the_contract():
    res = _run(10.0)
    f = 1.1
    assert res["rel_o"] <= f * REL_O and res["maxrel_o"] <= f * MAXREL_O, res
    assert res["rel_ht"] <= f * REL_HT and res["unit_rel_o"] <= UNIT_REL, res
