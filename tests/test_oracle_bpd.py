"""Pins of the blockwise-parallel-decoding oracle."""

import numpy as np
import pytest
import torch

import synth
from oracle import bpd as ob


def test_argmax_ties_to_lowest():
    assert ob.argmax_first([1.0, 3.0, 3.0, 2.0]) == 1
    assert ob.argmax_first([-np.inf, -np.inf, -5.0]) == 2


def test_figure_1(golden):
    g = golden("bpd_figure1.json")
    vocab, k = g["vocab"], g["k"]
    V = len(vocab)
    props = np.array([[vocab.index(t) for t in g["proposals"]]])
    heads = np.full((1, k, k), vocab.index("<other>"))
    # head 0 at position p is the base model's choice after the prefix proposals[0..p]
    heads[0, 0, 0] = vocab.index(g["base_argmax_given_prefix"]["in"])
    heads[0, 1, 0] = vocab.index(g["base_argmax_given_prefix"]["in the"])
    logits = synth.planted_rows(torch.from_numpy(heads), V, seed=5, salt=0,
                                dtype=torch.float32).numpy()
    khat, nxt = ob.verify(logits, props)
    assert khat[0] == g["khat"]
    assert [vocab[t] for t in props[0, :khat[0]]] == g["accepted"]
    assert vocab[nxt[0, 0]] == "car"        # next iteration starts from the base model's choice


def _model(V, seed, agree):
    def first_logits(b):
        truth = synth.prefix_token(b, (), V, seed)
        heads = [truth]
        y = (truth,)
        for h in range(1, K):
            t_next = synth.prefix_token(b, y, V, seed)
            heads.append(synth.proposal_token(b, (), h, t_next, V, seed, agree))
            y = y + (t_next,)
        return synth.planted_rows(torch.tensor(heads), V, seed=seed, salt=b).float().numpy()

    def combined(b, prefix, props):
        # logits[p, h]: head h+1 given prefix + props[0..p]
        out = np.zeros((K, K), dtype=np.int64)
        for p in range(K):
            ctx = prefix + tuple(props[:p + 1])
            truth = []
            y = ctx
            for h in range(K):
                t_next = synth.prefix_token(b, y, V, seed)
                truth.append(t_next)
                y = y + (t_next,)
            out[p, 0] = truth[0]
            for h in range(1, K):
                out[p, h] = synth.proposal_token(b, ctx, h, truth[h], V, seed, agree)
        salt = synth.mix_seed(b, len(prefix), *prefix, *props)
        return synth.planted_rows(torch.from_numpy(out), V, seed=seed, salt=salt).float().numpy()
    return first_logits, combined


K = 4


@pytest.mark.parametrize("agree,eos", [(0.7, -1), (0.0, -1), (1.0, -1), (0.7, 3)])
def test_blockwise_reproduces_greedy(agree, eos):
    V, length = 11, 23
    seed = 77
    first, combined = _model(V, seed, agree)
    for b in range(3):
        greedy = ob.greedy_decode(lambda y: synth.prefix_token(b, y, V, seed), length, eos)
        got, iters, khats = ob.blockwise_decode(lambda: first(b), lambda p, q: combined(b, p, q),
                                                length, K, eos)
        assert got == greedy
        assert all(kh >= 1 for kh in khats)
        if agree == 1.0 and eos < 0:
            assert iters == -(-length // K)        # perfect proposals: ceil(m / k) iterations
        if agree == 0.0 and eos < 0:
            assert iters == length                 # nothing but the free first token


def test_verify_eos_truncates_and_khat_bounds():
    V, k = 9, 5
    heads = np.zeros((2, k, k), dtype=np.int64)
    props = np.array([[1, 2, 3, 4, 6], [1, 2, 3, 4, 6]])
    for p in range(k):
        heads[:, p, 0] = props[0, min(p + 1, k - 1)]          # every proposal verified
    logits = synth.planted_rows(torch.from_numpy(heads), V, seed=1, salt=1).float().numpy()
    kh, _ = ob.verify(logits, props)
    assert list(kh) == [k, k]
    kh, _ = ob.verify(logits, props, eos=3)
    assert list(kh) == [3, 3]                                   # accepted up to and incl. EOS
    kh, _ = ob.verify(logits, props, eos=1)
    assert list(kh) == [1, 1]


# --- §5 approximate criteria (readings A1-A3) ---------------------------------------

def _hand_rows():
    """One element, k = 3, V = 6.  Head 0 at position 0 ranks the tokens 1, 2, 3, 5, 0, 4
    (tokens 2 and 3 tie at 2.0: the lower id ranks first); head 0 at position 1 has argmax 4.
    Heads 1 and 2 have argmax 0 and 1 everywhere."""
    x = np.full((1, 3, 3, 6), -2.0)
    x[0, :, 1, 0] = 5.0
    x[0, :, 2, 1] = 5.0
    x[0, 0, 0] = [0.1, 3.0, 2.0, 2.0, -1.0, 0.5]
    x[0, 1, 0] = [0.0, 0.0, 0.0, 0.0, 1.0, 0.0]
    x[0, 2, 0] = [0.0, 0.0, 0.0, 0.0, 0.0, 1.0]
    return x


def test_rank_counts_larger_and_lower_equal_tokens():
    row = [0.1, 3.0, 2.0, 2.0, -1.0, 0.5]
    assert [ob.rank_of(row, t) for t in range(6)] == [4, 0, 1, 2, 5, 3]


def test_topk_accepts_a_proposal_by_its_rank():
    x = _hand_rows()
    props = np.array([[0, 3, 4]])            # token 3 has rank 2 at position 0; 4 is the argmax at 1
    assert ob.verify(x, props)[0][0] == 1
    assert ob.verify(x, props, criterion=ob.TOPK, param=1)[0][0] == 1
    assert ob.verify(x, props, criterion=ob.TOPK, param=2)[0][0] == 1
    kh, nxt = ob.verify(x, props, criterion=ob.TOPK, param=3)
    assert kh[0] == 3 and list(nxt[0]) == [5, 0, 1]   # next proposals from position 2
    props2 = np.array([[0, 2, 4]])           # token 2 ties token 3 but has the lower id: rank 1
    assert ob.verify(x, props2, criterion=ob.TOPK, param=2)[0][0] == 3


def test_distance_accepts_a_near_token():
    x = _hand_rows()
    props = np.array([[0, 2, 5]])            # |2 - 1| = 1 at position 0, |5 - 4| = 1 at position 1
    assert ob.verify(x, props, criterion=ob.DISTANCE, param=0)[0][0] == 1
    assert ob.verify(x, props, criterion=ob.DISTANCE, param=1)[0][0] == 3
    props = np.array([[0, 3, 4]])            # |3 - 1| = 2
    assert ob.verify(x, props, criterion=ob.DISTANCE, param=1)[0][0] == 1
    assert ob.verify(x, props, criterion=ob.DISTANCE, param=2)[0][0] == 3


def test_minimum_block_and_its_eos_cut():
    x = _hand_rows()
    props = np.array([[0, 5, 5]])            # fails at position 0
    kh, nxt = ob.verify(x, props, min_accept=2)
    assert kh[0] == 2 and list(nxt[0]) == [4, 0, 1]  # next proposals from position 1
    assert ob.verify(x, props, min_accept=3)[0][0] == 3
    assert ob.verify(x, props, min_accept=3, eos=5)[0][0] == 2   # proposal 1 is EOS: stop after it
    assert ob.verify(x, props, min_accept=9)[0][0] == 3          # at most k


def _random_case(seed, B=24, k=5, V=11):
    rng = np.random.default_rng(seed)
    x = np.round(rng.normal(size=(B, k, k, V)) * 2) / 2   # half-integers: ties happen
    g = x[:, :, 0].argmax(-1)
    props = rng.integers(0, V, size=(B, k))
    agree = rng.random((B, k)) < 0.6
    props[:, 1:] = np.where(agree[:, 1:], g[:, :-1], props[:, 1:])
    return x, props


@pytest.mark.parametrize("seed", range(4))
def test_relaxed_criteria_reduce_to_exact(seed):
    x, props = _random_case(seed)
    kh, nx = ob.verify(x, props, eos=3)
    for crit, param in ((ob.TOPK, 1), (ob.DISTANCE, 0)):
        kh2, nx2 = ob.verify(x, props, eos=3, criterion=crit, param=param, min_accept=1)
        np.testing.assert_array_equal(kh2, kh)
        np.testing.assert_array_equal(nx2, nx)


@pytest.mark.parametrize("seed", range(4))
def test_khat_grows_with_the_relaxation(seed):
    x, props = _random_case(seed)
    B, k, _, V = x.shape
    prev = ob.verify(x, props, criterion=ob.TOPK, param=1)[0]
    for param in range(2, V + 1):
        kh = ob.verify(x, props, criterion=ob.TOPK, param=param)[0]
        assert (kh >= prev).all()
        prev = kh
    assert (prev == k).all()                 # every token is in the top V
    prev = ob.verify(x, props, criterion=ob.DISTANCE, param=0)[0]
    for param in range(1, V):
        kh = ob.verify(x, props, criterion=ob.DISTANCE, param=param)[0]
        assert (kh >= prev).all()
        prev = kh
    assert (prev == k).all()
    for m in range(1, k + 1):
        assert (ob.verify(x, props, min_accept=m)[0] >= m).all()
