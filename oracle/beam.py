"""Batched beam search in fp64: the oracle for the fused beam step.

TEST INFRASTRUCTURE.  Imported only by tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference arm; shares no code with the CUDA library.

What it follows
---------------
[BS] "Transformers中的Beam Search高效实现" (zhuanzhi.ai), section
     "多个样本同时进行beam search": the batched step (row log-softmax, add the
     beam's cumulative score, view as [batch, W*V], top-k, beam id = j // V,
     token = j mod V, effective row = b*W + beam id), the ``BeamHypotheses``
     class (``add`` / ``is_done``), padding of finished sentences, the all-done
     exit and the final choice of the best hypothesis.
[LM] "9.2 贪心搜索与束搜索：确定性与近似搜索" (llm_internals), §9.2.2 (expand,
     score, prune, retire; Table 9-5; "何时结束": early_stopping True / False /
     "never") and §9.2.3 (length penalty, GNMT form and |y|^alpha; Table 9-6).

Readings taken where the pages are silent, garbled or disagree
--------------------------------------------------------------
R1  The step ranks 2W candidates per sentence.  [BS]'s code asks top-k for W but
    then skips EOS hits at rank >= W and fills "until W" new beams, which only
    makes sense with more than W candidates; each parent row has one EOS token,
    so at most W of the best 2W are EOS and 2W always yield W live beams.
R2  Candidates are ordered by (score desc, flat index j asc).
R3  |y| is the number of scored tokens (EOS included): t for an EOS hit at step
    t, and the number of steps run for a beam still live at finalisation.
R4  ``is_done`` runs once per sentence after the walk, with the best score of the
    step (the rank-0 candidate) and cur_len = t.
R5  A sentence already done emits (score 0, PAD, beam_idx -1) for its W rows;
    its sequences get PAD appended.
R6  Initial scores are 0 for beam 0 and -inf for the others (the text's -inf,
    not the code's -1e9).
R7  Integer division is floor division.
N1  early_stopping "never": stop only when no live beam can still overtake the
    worst finished one.  Log-probabilities are <= 0, so a live sum can only
    fall; its best attainable normalised score is best / lp(L) maximised over
    the lengths L it can still reach: L = max_len when alpha > 0 (lp grows with
    L) and L = t when alpha <= 0.
N2  Finalisation breaks ties of the best normalised score toward the entry
    latest in the finished list ([BS] sorts ascending, stably, then pops).
N3  The output row is the best hypothesis (BOS first), then EOS when shorter
    than max_len + 1 columns, then PAD.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

LP_GNMT = 0
LP_POWER = 1
ES_FALSE = 0
ES_TRUE = 1
ES_NEVER = 2


def length_penalty(n: float, alpha: float, kind: int) -> float:
    """lp(|y|): GNMT ((5 + |y|) / 6)^alpha, or |y|^alpha ([LM] §9.2.3).  alpha = 0 gives 1."""
    if alpha == 0.0:
        return 1.0
    if kind == LP_GNMT:
        return ((5.0 + n) / 6.0) ** alpha
    if kind == LP_POWER:
        return float(n) ** alpha
    raise ValueError(f"unknown length-penalty kind {kind}")


def normalized_score(sum_logprobs: float, n: float, alpha: float, kind: int) -> float:
    """score(y) = log P(y) / lp(y) ([LM] §9.2.3; [BS] BeamHypotheses.add)."""
    return sum_logprobs / length_penalty(n, alpha, kind)


def log_softmax_rows(x) -> np.ndarray:
    """Row log-softmax in fp64: x - (m + ln sum exp(x - m)), m = row max ([BS] F.log_softmax)."""
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=-1, keepdims=True)
    return x - (m + np.log(np.exp(x - m).sum(axis=-1, keepdims=True)))


def best_first(values: np.ndarray, M: int) -> np.ndarray:
    """Indices of the M best entries of a 1-D array, ordered by (value desc, index asc).

    A top-k with a fixed tie rule (R2): the M-th largest value is found with a
    partition, every index reaching it is kept (so ties are never cut
    arbitrarily), and those are sorted by (value desc, index asc).
    """
    values = np.asarray(values)
    n = values.shape[0]
    M = min(M, n)
    if M <= 0:
        return np.zeros(0, dtype=np.int64)
    if M == n:
        sel = np.arange(n)
    else:
        kth = np.partition(values, n - M)[n - M]
        sel = np.nonzero(values >= kth)[0]
    order = np.lexsort((sel, -values[sel]))
    return sel[order][:M]


@dataclass
class Hyp:
    ns: float            # normalised score
    tokens: tuple        # BOS + generated tokens, without EOS
    sum_logprobs: float
    length: int          # |y| (R3)
    serial: int          # insertion counter (list order is by insertion)


class Hypotheses:
    """One sentence's finished set ([BS] class BeamHypotheses).

    ``beams`` keeps list order: appends go to the end, a deletion keeps the
    order of the rest.  ``margins`` (when given a list) collects the gap of
    every floating-point decision taken, for the input generator's checks.
    """

    def __init__(self, W: int, alpha: float, lp_kind: int, early_stopping: int, max_len: int):
        self.W, self.alpha, self.lp_kind = W, alpha, lp_kind
        self.early_stopping, self.max_len = early_stopping, max_len
        self.beams: list[Hyp] = []
        self.worst = 1e9
        self.serial = 0

    def __len__(self):
        return len(self.beams)

    def copy(self) -> "Hypotheses":
        h = Hypotheses(self.W, self.alpha, self.lp_kind, self.early_stopping, self.max_len)
        h.beams = list(self.beams)
        h.worst, h.serial = self.worst, self.serial
        return h

    def add(self, tokens, sum_logprobs: float, length: int, margins=None):
        ns = normalized_score(sum_logprobs, length, self.alpha, self.lp_kind)
        full = len(self.beams) >= self.W
        if full and margins is not None:
            margins.append(_gap(ns, self.worst))
        if not full or ns > self.worst:
            self.beams.append(Hyp(ns, tuple(tokens), sum_logprobs, length, self.serial))
            self.serial += 1
            if len(self.beams) > self.W:
                ranked = sorted((h.ns, i) for i, h in enumerate(self.beams))
                if margins is not None:
                    margins.append(_gap(ranked[0][0], ranked[1][0]))
                del self.beams[ranked[0][1]]
                self.worst = ranked[1][0]
            else:
                self.worst = min(ns, self.worst)

    def is_done(self, best_sum: float, cur_len: int, margins=None) -> bool:
        if len(self.beams) < self.W:
            return False
        if self.early_stopping == ES_TRUE:
            return True
        if self.early_stopping == ES_NEVER and self.alpha > 0.0:
            bound = normalized_score(best_sum, self.max_len, self.alpha, self.lp_kind)
        else:
            bound = normalized_score(best_sum, cur_len, self.alpha, self.lp_kind)
        if margins is not None:
            margins.append(_gap(self.worst, bound))
        return self.worst >= bound


def _gap(a: float, b: float) -> float:
    """|a - b| / (1 + 0.02 max(|a|, |b|)): the gap of one decision, scaled so that a
    threshold of 1e-3 asks for 1e-3 + 2e-5 max(|a|, |b|).  A decision that involves an
    infinity is exact in every precision, so its gap is infinite."""
    if math.isinf(a) or math.isinf(b):
        return math.inf
    return abs(a - b) / (1.0 + 0.02 * max(abs(a), abs(b)))


@dataclass
class SentenceStep:
    new_beams: list            # [(score, token, global parent row)] x W
    hyps: Hypotheses           # the sentence's finished set after this step
    done: bool
    best: float                # rank-0 candidate score
    walked: list = field(default_factory=list)   # [(rank, j, score)] examined by the walk
    margins: list = field(default_factory=list)


@dataclass
class StepResult:
    beam_idx: np.ndarray       # [R] int64, global parent row or -1 (R5)
    tokens: np.ndarray         # [R] int64
    scores: np.ndarray         # [R] fp64, new cumulative scores
    done: np.ndarray           # [B] bool after the step
    all_done: bool
    sentences: dict            # b -> SentenceStep for sentences live at the step


class BeamSearch:
    """Batched beam search over B sentences x W beams ([BS] beam_search, [LM] §9.2.2)."""

    def __init__(self, batch: int, W: int, V: int, eos: int, alpha: float,
                 early_stopping: int = ES_FALSE, lp_kind: int = LP_GNMT, max_len: int = 8,
                 bos: int = 0, pad: int = -1):
        self.B, self.W, self.V = batch, W, V
        self.eos, self.alpha, self.early_stopping = eos, alpha, early_stopping
        self.lp_kind, self.max_len, self.bos, self.pad = lp_kind, max_len, bos, pad
        self.reset()

    def reset(self):
        B, W = self.B, self.W
        self.scores = np.zeros((B, W), dtype=np.float64)
        self.scores[:, 1:] = -np.inf                                          # R6
        self.seqs = [[self.bos] for _ in range(B * W)]
        self.done = np.zeros(B, dtype=bool)
        self.hyps = [Hypotheses(W, self.alpha, self.lp_kind, self.early_stopping, self.max_len)
                     for _ in range(B)]
        self.t = 0

    # -- one sentence, pure: reads the state, changes nothing ----------------------
    def sentence_step(self, b: int, logits_rows, t: int, margins: bool = False) -> SentenceStep:
        W, V = self.W, self.V
        logp = log_softmax_rows(logits_rows)                                   # [W, V]
        cand = (self.scores[b][:, None] + logp).reshape(-1)                    # j = w*V + v
        top = best_first(cand, 2 * W + 1)                                      # R1 (+1 for margins)
        hyps = self.hyps[b].copy()
        mlist = [] if margins else None
        new_beams, walked = [], []
        last_rank = 0
        for rank, j in enumerate(top[: 2 * W]):
            w, v = divmod(int(j), V)                                           # R7
            row = b * W + w
            walked.append((rank, int(j), float(cand[j])))
            last_rank = rank
            if self.eos >= 0 and v == self.eos:
                if rank >= W:
                    continue
                hyps.add(self.seqs[row], float(cand[j]), t, mlist)
            else:
                new_beams.append((float(cand[j]), v, row))
            if len(new_beams) == W:
                break
        assert len(new_beams) == W, "2W candidates always hold W non-EOS ones"
        best = float(cand[top[0]])
        if margins:
            # every adjacent pair the walk relied on, incl. the first one it did not take
            for i in range(min(last_rank + 1, len(top) - 1)):
                ja, jb = int(top[i]), int(top[i + 1])
                if ja // V != jb // V:                                         # same row: exact
                    mlist.append(_gap(float(cand[ja]), float(cand[jb])))
        done = bool(self.done[b]) or hyps.is_done(best, t, mlist)             # R4
        return SentenceStep(new_beams, hyps, done, best, walked, mlist or [])

    # -- whole batch ------------------------------------------------------------------
    def step(self, logits, margins: bool = False, overrides: dict | None = None) -> StepResult:
        """Advance every row by one token.  ``logits`` is [B*W, V] (widened exactly to fp64).

        ``overrides`` maps a sentence to an already computed SentenceStep (used by
        the input generator after re-salting one sentence).
        """
        if self.t >= self.max_len:
            raise RuntimeError("max_len steps already run")
        B, W = self.B, self.W
        R = B * W
        self.t += 1
        t = self.t
        logits = np.asarray(logits)
        beam_idx = np.full(R, -1, dtype=np.int64)
        tokens = np.full(R, self.pad, dtype=np.int64)
        scores = np.zeros(R, dtype=np.float64)
        steps = {}
        for b in range(B):
            if self.done[b]:
                continue                                                       # R5
            if overrides and b in overrides:
                ss = overrides[b]
            else:
                ss = self.sentence_step(b, logits[b * W:(b + 1) * W], t, margins)
            steps[b] = ss
            for i, (sc, v, row) in enumerate(ss.new_beams):
                scores[b * W + i] = sc
                tokens[b * W + i] = v
                beam_idx[b * W + i] = row
        for b, ss in steps.items():
            self.hyps[b] = ss.hyps
            self.done[b] = ss.done
        self.seqs = [self.seqs[p] + [int(tokens[r])] if p >= 0 else self.seqs[r] + [self.pad]
                     for r, p in enumerate(beam_idx)]
        self.scores = scores.reshape(B, W).copy()
        return StepResult(beam_idx, tokens, scores, self.done.copy(), bool(self.done.all()), steps)

    def finalize(self, n_return: int = 1):
        """The best n_return hypotheses per sentence: (out_seqs [B * n, max_len+1],
        out_len [B * n], out_score [B * n], hyps), sentence b's j-th best in row b * n + j.

        Live beams of sentences not done are added first, with |y| = steps run
        (R3); hypotheses rank by normalised score, ties to the latest list entry
        (N2: [BS] sorts ascending, stably, and pops from the end, once per returned
        sequence; [LM] returns the first num_return_sequences by normalised score);
        each row is BOS + tokens, then EOS if shorter than max_len + 1, then PAD (N3).
        """
        B, W = self.B, self.W
        width = self.max_len + 1
        hyps = [h.copy() for h in self.hyps]
        for b in range(B):
            if self.done[b]:
                continue
            for w in range(W):
                row = b * W + w
                hyps[b].add(self.seqs[row], float(self.scores[b, w]), self.t)
        nr = n_return
        out = np.full((B * nr, width), self.pad, dtype=np.int64)
        out_len = np.zeros(B * nr, dtype=np.int64)
        out_score = np.zeros(B * nr, dtype=np.float64)
        for b in range(B):
            ranked = sorted(hyps[b].beams, key=lambda h: h.ns)   # stable: equal scores keep list order
            for j in range(nr):
                best = ranked.pop()
                n = len(best.tokens)
                row = b * nr + j
                out[row, :n] = best.tokens
                if n < width and self.eos >= 0:
                    out[row, n] = self.eos
                    n += 1
                out_len[row] = n
                out_score[row] = best.ns
        return out, out_len, out_score, hyps


def exhaustive_paths(logits_of_prefix, V: int, n: int, bos: int = 0):
    """Every |V|^n path with its summed log-probability ([LM] §9.2.1, brute force).

    ``logits_of_prefix(prefix_tuple) -> [V]`` is the synthetic model.
    Returns a list of (sum_logprobs, tokens) over all paths.
    """
    out = []
    frontier = [((bos,), 0.0)]
    for _ in range(n):
        nxt = []
        for prefix, s in frontier:
            lp = log_softmax_rows(np.asarray(logits_of_prefix(prefix), dtype=np.float64)[None, :])[0]
            for v in range(V):
                nxt.append((prefix + (v,), s + lp[v]))
        frontier = nxt
    return [(s, p) for p, s in frontier]
