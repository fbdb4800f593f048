"""The parity harness's own logic (CPU): the oracle split across worker processes gives the
trace the serial oracle gives, including the cut at the step where every sentence is done."""

import numpy as np
import torch

from oracle import beam as ob
from tests import harness as hz


def _same_trace(a, b):
    assert len(a.steps) == len(b.steps)
    for x, y in zip(a.steps, b.steps):
        assert (x.beam_idx == y.beam_idx).all() and (x.tokens == y.tokens).all()
        assert (x.scores == y.scores).all() and (x.done == y.done).all() and x.all_done == y.all_done
        assert sorted(x.sentences) == sorted(y.sentences)
    assert a.salts == b.salts and a.seqs == b.seqs
    for hx, hy in zip(a.hyps, b.hyps):
        for p, q in zip(hx, hy):
            assert [(h.ns, h.tokens, h.length, h.serial) for h in p.beams] == \
                   [(h.ns, h.tokens, h.length, h.serial) for h in q.beams]
    for n in (1, a.bs.W):
        ra, rb = a.bs.finalize(n), b.bs.finalize(n)
        assert all(np.array_equal(u, v) for u, v in zip(ra[:3], rb[:3]))


def test_parallel_oracle_equals_serial():
    case = hz.BeamCase("tiny", 9, 3, 6, 16, torch.float32, eos=5, alpha=0.6, seed=5)
    _same_trace(hz.run_oracle(case), hz.run_oracle_parallel(case, workers=3))


def test_parallel_oracle_cuts_at_all_done():
    case = hz.BeamCase("tiny", 6, 3, 8, 30, torch.float32, eos=2, alpha=1.0, early_stopping=ob.ES_TRUE, seed=11)
    a = hz.run_oracle(case)
    assert a.steps[-1].all_done and len(a.steps) < case.T
    _same_trace(a, hz.run_oracle_parallel(case, workers=4))


def test_check_scores_is_relative():
    hz.check_scores([-1.0 - 0.9e-5], [-1.0], "within")
    hz.check_scores([0.0, float("-inf")], [0.0, float("-inf")], "exact")
    for got, ref in (([-1.0 - 1.1e-5], [-1.0]), ([-1e-3 - 2e-8], [-1e-3]), ([1e-12], [0.0]),
                     ([-3.0], [float("-inf")])):
        try:
            hz.check_scores(got, ref, "outside")
        except AssertionError:
            continue
        raise AssertionError(f"{got} vs {ref} passed")
    hz.REL_ERR.pop(hz.CURRENT_TEST[0], None)      # the deliberate misses are not a measurement
