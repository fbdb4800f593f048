"""Blockwise parallel decoding in fp64 terms: the oracle for propose / verify.

TEST INFRASTRUCTURE.  Imported only by tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference arm; shares no code with the CUDA library.

What it follows: "Blockwise Parallel Decoding for Deep Autoregressive Models"
(papercache notes on Stern, Shazeer, Uszkoreit):

* §2 greedy decoding: y_{j+1} = argmax_y p(y_{j+1} | y<=j), stop at EOS.
* §3 predict / verify / accept: predictions yhat_{j+i} = argmax p_i(. | yhat<=j)
  for i = 1..k; khat is the largest number with yhat_{j+i} equal to the base
  model's argmax given yhat<=j+i-1 for every i <= khat (khat >= 1 always);
  accept yhat_{j+1..j+khat}.
* §4 the combined scoring and proposal model: one call returns
  p_i(y_{j+i0+i} | yhat<=j+i0) for i, i0 = 1..k, so verify n and predict n+1
  share one call.

Readings
--------
B1 (layout) ``logits[b, p, h, :]`` holds head h+1 (p_{h+1}) at proposal position
   p+1, i.e. given the prefix extended by proposals[0..p].  Verify compares
   proposals[b, p+1] with argmax logits[b, p, 0, :] for p = 0..k-2; the next
   proposals are argmax logits[b, khat-1, h, :] for h = 0..k-1.
B2 (ties) argmax breaks ties toward the lower token id.
B3 (EOS) greedy stops at EOS (§2); if an accepted proposal e < khat is EOS,
   khat becomes e + 1.

§5 approximate inference relaxes the verify test; the criteria's formulas are
missing from the pages' text, so these are the readings (exact when the
parameters are 1, 0, 1):
A1 (top-k, §5.1) proposal p+1 passes when it is among the ``param`` best tokens
   of head 0 at position p: its rank, the number of tokens with a larger logit
   or an equal logit and a lower id (B2), is below ``param`` (>= 1).
A2 (distance, §5.2) with d(u, v) = |u - v| on token ids read as intensities,
   proposal p+1 passes when |proposal - argmax| <= ``param`` (>= 0).
A3 (minimum block, §5.3) at least ``min_accept`` (1..k) tokens are accepted:
   khat = max(khat, min_accept), and the EOS cut (B3) applies after it.
   min_accept = k decodes in fixed blocks of k.  The next proposals come from
   position khat - 1 as always.
"""

from __future__ import annotations

import numpy as np


def argmax_first(row) -> int:
    """argmax with ties to the lowest index (numpy returns the first occurrence)."""
    return int(np.argmax(np.asarray(row, dtype=np.float64)))


EXACT, TOPK, DISTANCE = 0, 1, 2


def rank_of(row, tok: int) -> int:
    """How many tokens beat ``tok``: a larger logit, or an equal one at a lower id (B2)."""
    x = np.asarray(row, dtype=np.float64)
    xt = x[tok]
    return int(np.count_nonzero(x > xt) + np.count_nonzero(x[:tok] == xt))


def passes(row, proposal: int, criterion: int = EXACT, param: int = 0) -> bool:
    """The verify test of one proposal against head 0's row (§3, or A1 / A2)."""
    if criterion == EXACT:
        return proposal == argmax_first(row)
    if criterion == TOPK:
        return 0 <= proposal < len(row) and rank_of(row, proposal) < param
    if criterion == DISTANCE:
        return abs(proposal - argmax_first(row)) <= param
    raise ValueError(f"unknown criterion {criterion}")


def propose(logits) -> np.ndarray:
    """Predict sub-step from per-head logits [B, k, V]: proposals[b, h] = argmax_v."""
    x = np.asarray(logits, dtype=np.float64)
    B, k, _ = x.shape
    out = np.zeros((B, k), dtype=np.int64)
    for b in range(B):
        for h in range(k):
            out[b, h] = argmax_first(x[b, h])
    return out


def verify(logits, proposals, eos: int = -1, criterion: int = EXACT, param: int = 0, min_accept: int = 1):
    """Verify + accept on combined-model logits [B, k, k, V] (B1-B3; A1-A3 for the
    approximate criteria).

    Returns (khat [B], next_proposals [B, k]).
    """
    x = np.asarray(logits)
    props = np.asarray(proposals)
    B, k = props.shape
    khat = np.ones(B, dtype=np.int64)
    nxt = np.zeros((B, k), dtype=np.int64)
    for b in range(B):
        n = 1
        for p in range(k - 1):
            if passes(x[b, p, 0], int(props[b, p + 1]), criterion, param):
                n += 1
            else:
                break
        n = max(n, min(min_accept, k))
        if eos >= 0:
            for e in range(n):
                if int(props[b, e]) == eos:
                    n = e + 1
                    break
        khat[b] = n
        for h in range(k):
            nxt[b, h] = argmax_first(x[b, n - 1, h])
    return khat, nxt


def greedy_decode(next_token, length: int, eos: int = -1) -> list:
    """§2 greedy: extend by ``next_token(prefix)`` until ``length`` tokens or EOS."""
    y = []
    while len(y) < length:
        t = int(next_token(tuple(y)))
        y.append(t)
        if t == eos:
            break
    return y


def blockwise_decode(first_logits, combined_logits, length: int, k: int, eos: int = -1):
    """§3-§4 with one combined call per iteration, for one batch element.

    ``first_logits() -> [k, V]``: the predict sub-step of the first iteration.
    ``combined_logits(prefix, proposals) -> [k, k, V]``: the combined model on
    the prefix extended by the k proposals (layout B1).
    Returns (tokens, iterations, khats).
    """
    y: list = []
    props = propose(np.asarray(first_logits())[None])[0]
    khats = []
    while len(y) < length:
        logits = np.asarray(combined_logits(tuple(y), tuple(int(p) for p in props)))
        kh, nxt = verify(logits[None], props[None], eos)
        n = int(kh[0])
        khats.append(n)
        for i in range(n):
            y.append(int(props[i]))
            if len(y) >= length or int(props[i]) == eos:
                return y, len(khats), khats
        props = nxt[0]
    return y, len(khats), khats
