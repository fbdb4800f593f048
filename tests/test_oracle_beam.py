"""Pins of the beam-search oracle against what the pages and the mathematics fix.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, > for >=) fails at least one of them.
"""

import itertools
import math

import numpy as np
import pytest
import torch

import synth
from oracle import beam as ob


# ------------------------------------------------------------------------------
# row log-softmax: a library routine and a closed form
# ------------------------------------------------------------------------------

def test_log_softmax_matches_torch_fp64():
    x = synth.normal_rows(7, 1000, 3.0, seed=1).double()
    x[2, 5] = float("-inf")
    mine = ob.log_softmax_rows(x.numpy())
    ref = torch.log_softmax(x, dim=-1).numpy()
    assert np.allclose(mine, ref, rtol=0, atol=1e-12, equal_nan=False)
    assert np.allclose(np.exp(mine).sum(axis=1), 1.0, atol=1e-12)


def test_log_softmax_shift_invariance_and_uniform_row():
    # closed forms: a uniform row gives -ln V; adding a constant to a row changes nothing
    V = 37
    assert np.allclose(ob.log_softmax_rows(np.zeros((1, V))), -math.log(V), atol=1e-15)
    x = np.random.default_rng(0).normal(size=(3, V))
    assert np.allclose(ob.log_softmax_rows(x), ob.log_softmax_rows(x + 123.25), atol=1e-12)


# ------------------------------------------------------------------------------
# top-k with the tie rule: brute force against a full sort
# ------------------------------------------------------------------------------

@pytest.mark.parametrize("n,M", [(1, 1), (10, 3), (50, 50), (200, 9), (64, 70)])
def test_best_first_equals_full_sort(n, M):
    rng = np.random.default_rng(n * 31 + M)
    v = rng.integers(-4, 4, size=n).astype(np.float64)          # many ties
    v[rng.integers(0, n, size=max(1, n // 10))] = -np.inf
    got = ob.best_first(v, M)
    full = sorted(range(n), key=lambda j: (-v[j], j))[:M]
    assert list(got) == full


# ------------------------------------------------------------------------------
# length penalty: Table 9-6 (all ten numbers and the winners)
# ------------------------------------------------------------------------------

def test_length_penalty_table_9_6(golden):
    g = golden("lp_table_9_6.json")
    s_short = g["short"]["tokens"] * math.log(g["short"]["p"])
    s_long = g["long"]["tokens"] * math.log(g["long"]["p"])
    tol = g["tolerance"]
    assert abs(s_short - g["short"]["sum"]) < tol and abs(s_long - g["long"]["sum"]) < tol
    assert abs(ob.length_penalty(5, 0.6, ob.LP_GNMT) - g["gnmt_lp"]["5"]) < tol
    assert abs(ob.length_penalty(10, 0.6, ob.LP_GNMT) - g["gnmt_lp"]["10"]) < tol
    for row in g["rows"]:
        kind = ob.LP_GNMT if row["kind"] == "gnmt" else ob.LP_POWER
        a = ob.normalized_score(s_short, 5, row["alpha"], kind)
        b = ob.normalized_score(s_long, 10, row["alpha"], kind)
        assert abs(a - row["short"]) < tol, row
        assert abs(b - row["long"]) < tol, row
        # the finished set with room for one hypothesis keeps the table's winner
        h = ob.Hypotheses(1, row["alpha"], kind, ob.ES_FALSE, 10)
        h.add((0,) * 6, s_short, 5)
        h.add((0,) * 11, s_long, 10)
        assert len(h) == 1
        assert len(h.beams[0].tokens) == (6 if row["winner"] == "short" else 11), row


def test_alpha_zero_is_no_normalisation():
    for kind in (ob.LP_GNMT, ob.LP_POWER):
        for n in (1, 7, 200):
            assert ob.normalized_score(-3.25, n, 0.0, kind) == -3.25


# ------------------------------------------------------------------------------
# the worked tree: Figure 9-3 text + Table 9-5
# ------------------------------------------------------------------------------

def _tree_logits(g, step, rows_prefix):
    vocab = g["vocab"]
    V = len(vocab)
    out = np.full((len(rows_prefix), V), -np.inf)
    for r, prefix in enumerate(rows_prefix):
        probs = g["step1_probs"] if step == 1 else g["step2_probs"][vocab[prefix[-1]]]
        for tok, p in probs.items():
            out[r, vocab.index(tok)] = math.log(p)
    return out


def test_tree_table_9_5(golden):
    g = golden("tree_table_9_5.json")
    vocab = g["vocab"]
    V, W, tol = len(vocab), g["W"], g["tolerance"]
    bs = ob.BeamSearch(1, W, V, eos=-1, alpha=0.0, max_len=2, bos=-7)
    r1 = bs.step(_tree_logits(g, 1, [s[1:] or [0] for s in bs.seqs]))
    kept1 = [(vocab[int(t)], s) for t, s in zip(r1.tokens, r1.scores)]
    for (tok, sc), (etok, esc) in zip(kept1, g["step1_kept"]):
        assert tok == etok and abs(sc - esc) < tol
    logits2 = _tree_logits(g, 2, [s[1:] for s in bs.seqs])
    # every candidate of the step-2 table, through the oracle's own score add
    ss = bs.sentence_step(0, logits2, 2)
    cand = {}
    for (rank, j, score) in ss.walked:
        w, v = divmod(j, V)
        cand[vocab[bs.seqs[w][-1]] + " " + vocab[v]] = score
    lsm = ob.log_softmax_rows(logits2)
    for row in g["table_9_5"]:
        parent, tok = row["cand"].split()
        w = [vocab[s[-1]] for s in bs.seqs].index(parent)
        full = bs.scores[0, w] + lsm[w, vocab.index(tok)]
        assert abs(full - row["score"]) < tol, row
        assert abs(lsm[w, vocab.index(tok)] - row["logp"]) < tol, row
        assert abs(math.exp(full) - row["joint"]) < tol, row
        if row["kept"]:
            assert abs(cand[row["cand"]] - row["score"]) < tol
    r2 = bs.step(logits2)
    parents = [vocab[bs.seqs[0][1]], vocab[bs.seqs[1][1]]]
    assert parents == g["step2_beam_idx_parents"]
    assert list(r2.beam_idx) == [1, 0]                    # beam_idx = [B, A]
    assert [vocab[int(t)] for t in r2.tokens] == ["x", "x"]
    assert abs(math.exp(r2.scores[0]) - g["beam_joint"]) < tol
    # greedy = W = 1 reaches A x at 0.200, beam search B x at 0.360 (1.8x)
    gr = ob.BeamSearch(1, 1, V, eos=-1, alpha=0.0, max_len=2, bos=-7)
    gr.step(_tree_logits(g, 1, [[0]]))
    rg = gr.step(_tree_logits(g, 2, [gr.seqs[0][1:]]))
    assert [vocab[t] for t in gr.seqs[0][1:]] == ["A", "x"]
    assert abs(math.exp(rg.scores[0]) - g["greedy_joint"]) < tol
    assert abs(math.exp(r2.scores[0]) / math.exp(rg.scores[0]) - g["ratio"]) < 1e-9 + 0.01


# ------------------------------------------------------------------------------
# the batch layout: batch=3, W=2, V=6
# ------------------------------------------------------------------------------

def test_batch_layout(golden):
    g = golden("batch_layout.json")
    B, W, V = g["batch"], g["W"], g["V"]
    for case in g["cases"]:
        bs = ob.BeamSearch(B, W, V, eos=-1, alpha=0.0, max_len=4)
        bs.scores[:] = 0.0                           # both beams live and equal
        logits = np.zeros((B * W, V))
        w, v = divmod(case["j"], V)
        assert (w, v) == (case["beam"], case["token"])
        logits[case["b"] * W + w, v] = 5.0           # the sentence's single best candidate
        res = bs.step(logits)
        assert res.beam_idx[case["b"] * W] == case["row"]
        assert res.tokens[case["b"] * W] == case["token"]
    # exact ties across rows go to the lower flat index j (R2)
    bs = ob.BeamSearch(B, W, V, eos=-1, alpha=0.0, max_len=4)
    bs.scores[:] = 0.0
    logits = np.zeros((B * W, V))
    logits[:, 3] = 2.0                               # same candidate in both rows of each sentence
    res = bs.step(logits)
    for b in range(B):
        assert list(res.beam_idx[b * W:(b + 1) * W]) == [b * W, b * W + 1]
        assert list(res.tokens[b * W:(b + 1) * W]) == [3, 3]


# ------------------------------------------------------------------------------
# exhaustive enumeration: W = |V|^(n-1) returns the top W of all |V|^n paths
# ------------------------------------------------------------------------------

def _prefix_model(V, seed):
    def f(prefix):
        g = torch.Generator().manual_seed(synth.mix_seed(seed, len(prefix), *prefix))
        return (torch.randn(V, generator=g, dtype=torch.float64) * 2.0).numpy()
    return f


@pytest.mark.parametrize("V,n", [(3, 3), (2, 4), (4, 2), (3, 2)])
def test_exhaustive_enumeration(V, n):
    W = V ** (n - 1)
    model = _prefix_model(V, seed=100 + V * 10 + n)
    bos = 0
    bs = ob.BeamSearch(1, W, V, eos=-1, alpha=0.0, max_len=n, bos=bos)
    for _ in range(n):
        logits = np.stack([model(tuple(s)) for s in bs.seqs])
        res = bs.step(logits)
    paths = ob.exhaustive_paths(model, V, n, bos=bos)
    paths.sort(key=lambda sp: -sp[0])
    top = paths[:W]
    got = sorted(zip(res.scores, [tuple(s) for s in bs.seqs]), key=lambda sp: -sp[0])
    for (gs, gp), (es, ep) in zip(got, top):
        assert gp == ep
        assert abs(gs - es) < 1e-12
    assert abs(sum(math.exp(s) for s, _ in paths) - 1.0) < 1e-12    # the paths form a distribution


def test_beam_one_is_greedy_argmax():
    V, T = 50, 6
    x = [synth.normal_rows(2, V, 2.0, seed=s).numpy() for s in range(T)]
    bs = ob.BeamSearch(2, 1, V, eos=-1, alpha=0.0, max_len=T)
    total = np.zeros(2)
    for t in range(T):
        res = bs.step(x[t])
        am = x[t].argmax(axis=1)
        assert list(res.tokens) == list(am)
        total += ob.log_softmax_rows(x[t])[np.arange(2), am]
        assert list(res.beam_idx) == [0, 1]
    assert np.allclose(res.scores, total, atol=1e-12)


# ------------------------------------------------------------------------------
# the finished set and the stopping rules
# ------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(12))
def test_hypotheses_invariants(seed):
    rng = np.random.default_rng(seed)
    W = int(rng.integers(1, 5))
    n_add = int(rng.integers(1, 14))
    distinct = seed % 2 == 0
    vals = rng.permutation(50)[:n_add] * -0.1 if distinct else rng.integers(-3, 0, n_add) * 1.0
    h = ob.Hypotheses(W, 0.0, ob.LP_GNMT, ob.ES_FALSE, 10)
    for i, v in enumerate(vals):
        h.add((i,), float(v), 1)
    kept = {hy.tokens[0] for hy in h.beams}
    dropped = set(range(n_add)) - kept
    assert len(h) == min(W, n_add)
    assert h.worst == min(hy.ns for hy in h.beams)
    assert all(vals[k] >= vals[d] for k in kept for d in dropped)   # nothing kept is worse
    if distinct:
        assert kept == set(np.argsort(-vals)[:W].tolist())
    # list order is insertion order
    assert [hy.serial for hy in h.beams] == sorted(hy.serial for hy in h.beams)


def test_add_rejects_equal_to_worst_and_evicts_earliest_of_equal():
    h = ob.Hypotheses(2, 0.0, ob.LP_GNMT, ob.ES_FALSE, 10)
    h.add(("a",), -1.0, 1)
    h.add(("b",), -1.0, 1)
    h.add(("c",), -1.0, 1)           # not strictly better than the worst: rejected
    assert [x.tokens for x in h.beams] == [("a",), ("b",)]
    h.add(("d",), -0.5, 1)           # better: evicts the earliest of the two equal worst
    assert [x.tokens for x in h.beams] == [("b",), ("d",)]
    assert h.worst == -1.0


def test_is_done_hand_values():
    # power lp, alpha = 1: bound = best / t
    h = ob.Hypotheses(1, 1.0, ob.LP_POWER, ob.ES_FALSE, 10)
    assert not h.is_done(-2.0, 3)                   # fewer than W finished
    h.add(("a",), -1.0, 2)                          # ns = -0.5
    assert h.is_done(-2.0, 3)                       # -0.5 >= -0.667
    assert not h.is_done(-1.0, 3)                   # -0.5 <  -0.333
    assert h.is_done(-1.5, 3)                       # -0.5 >= -0.5 (inclusive)
    t = ob.Hypotheses(1, 1.0, ob.LP_POWER, ob.ES_TRUE, 10)
    t.add(("a",), -1.0, 2)
    assert t.is_done(-0.001, 3)                     # True mode: as soon as W are finished
    nv = ob.Hypotheses(1, 1.0, ob.LP_POWER, ob.ES_NEVER, 10)
    nv.add(("a",), -1.0, 2)
    assert not nv.is_done(-2.0, 3)                  # bound over max_len: -2/10 = -0.2 > -0.5
    assert nv.is_done(-6.0, 3)                      # -6/10 = -0.6 <= -0.5
    neg = ob.Hypotheses(1, -1.0, ob.LP_POWER, ob.ES_NEVER, 10)
    neg.add(("a",), -1.0, 2)                        # ns = -1 * 2 = -2
    assert neg.is_done(-0.6, 4)                     # alpha <= 0: bound at t: -0.6 * 4 = -2.4


def _tiny_run(mode, seed=7, B=3, W=2, V=6, T=8, eos=5):
    bs = ob.BeamSearch(B, W, V, eos=eos, alpha=0.6, early_stopping=mode, max_len=T, bos=0)
    done_at = [None] * B
    for t in range(1, T + 1):
        x = synth.batch_logits("tiny", B, W, V, seed=seed, step=t).numpy()
        res = bs.step(x)
        for b in range(B):
            if res.done[b] and done_at[b] is None:
                done_at[b] = t
        if res.all_done:
            break
    return [d if d is not None else T + 1 for d in done_at], bs


@pytest.mark.parametrize("seed", range(6))
def test_early_stopping_modes_are_ordered(seed):
    d_true, _ = _tiny_run(ob.ES_TRUE, seed)
    d_false, _ = _tiny_run(ob.ES_FALSE, seed)
    d_never, _ = _tiny_run(ob.ES_NEVER, seed)
    for a, b, c in zip(d_true, d_false, d_never):
        assert a <= b <= c


def test_true_mode_stops_exactly_when_W_finished():
    _, bs = _tiny_run(ob.ES_TRUE, seed=3)
    for b in range(bs.B):
        assert bs.done[b] == (len(bs.hyps[b]) >= bs.W)


def test_finished_hyps_are_eos_hits_of_the_walk():
    # every finished entry was an EOS candidate within the top W of some step:
    # its normalised score is its raw sum over lp(|y|), and |y| = len(tokens)
    _, bs = _tiny_run(ob.ES_NEVER, seed=11)
    for h in bs.hyps:
        for hy in h.beams:
            assert hy.length == len(hy.tokens)        # BOS + (t-1) tokens, EOS scored: |y| = t
            assert abs(hy.ns - hy.sum_logprobs / ob.length_penalty(hy.length, 0.6, ob.LP_GNMT)) < 1e-15


def test_padding_of_done_sentences():
    bs2 = ob.BeamSearch(3, 2, 6, eos=5, alpha=0.6, early_stopping=ob.ES_TRUE, max_len=8, bos=0)
    for t in range(1, 9):
        before = bs2.done.copy()
        res = bs2.step(synth.batch_logits("tiny", 3, 2, 6, seed=3, step=t).numpy())
        for b in range(3):
            sl = slice(b * 2, b * 2 + 2)
            if before[b]:
                assert (res.beam_idx[sl] == -1).all() and (res.tokens[sl] == -1).all()
                assert (res.scores[sl] == 0).all()
            else:
                assert (res.beam_idx[sl] // 2 == b).all()   # parents stay within the sentence


def test_finalize_rules():
    bs = ob.BeamSearch(1, 2, 6, eos=5, alpha=1.0, lp_kind=ob.LP_POWER, max_len=4, bos=9, pad=-1)
    # hand-set state after 4 steps: one finished hyp and two live beams
    bs.t = 4
    bs.hyps[0].add((9, 1, 2), -1.5, 3)          # ns = -0.5, EOS hit at step 3
    bs.seqs = [[9, 1, 2, 3, 4], [9, 2, 2, 2, 2]]
    bs.scores[0] = [-2.0, -8.0]                  # live: ns = -0.5 (tie) and -2
    out, out_len, out_score, hyps = bs.finalize()
    # tie at -0.5 goes to the latest list entry: the live beam added at finalisation
    assert list(out[0]) == [9, 1, 2, 3, 4] and out_len[0] == 5 and out_score[0] == -0.5
    # a shorter winner gets EOS appended, then PAD
    bs.scores[0] = [-4.0, -8.0]
    out, out_len, out_score, _ = bs.finalize()
    assert list(out[0]) == [9, 1, 2, 5, -1] and out_len[0] == 4 and out_score[0] == -0.5


def test_finalize_returns_the_best_n_in_order():
    bs = ob.BeamSearch(1, 2, 6, eos=5, alpha=1.0, lp_kind=ob.LP_POWER, max_len=4, bos=9, pad=-1)
    bs.t = 4
    bs.hyps[0].add((9, 1, 2), -1.5, 3)          # ns = -0.5, EOS hit at step 3
    bs.seqs = [[9, 1, 2, 3, 4], [9, 2, 2, 2, 2]]
    bs.scores[0] = [-2.0, -8.0]                  # live: ns = -0.5 joins (tie), -2 does not (set full)
    out, out_len, out_score, _ = bs.finalize(2)
    # both hypotheses tie at -0.5: the latest list entry first, then the earlier one
    assert [list(r) for r in out] == [[9, 1, 2, 3, 4], [9, 1, 2, 5, -1]]
    assert list(out_len) == [5, 4] and list(out_score) == [-0.5, -0.5]
    one = bs.finalize(1)
    assert list(one[0][0]) == list(out[0]) and one[1][0] == out_len[0]


@pytest.mark.parametrize("es", [ob.ES_FALSE, ob.ES_TRUE, ob.ES_NEVER])
def test_finalize_n_ranks_the_whole_finished_set(es):
    _, bs = _tiny_run(es, seed=21)
    W = bs.W
    out, out_len, out_score, hyps = bs.finalize(W)
    best1 = bs.finalize(1)
    for b in range(bs.B):
        rows = slice(b * W, (b + 1) * W)
        assert (np.diff(out_score[rows]) <= 0).all()                 # best first
        assert sorted(out_score[rows]) == sorted(h.ns for h in hyps[b].beams)
        np.testing.assert_array_equal(out[b * W], best1[0][b])       # the first is the single best
