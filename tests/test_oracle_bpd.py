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
