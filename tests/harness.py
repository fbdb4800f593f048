"""Parity harness: drive the oracle and the CUDA path on the same seeded inputs.

Inputs come from ``synth`` only.  For every sentence the oracle checks (a
sample, or all), each step's rows are re-salted until every floating-point
decision the oracle takes has a scaled gap >= MIN_GAP (see oracle.beam._gap:
1e-3 + 2e-5 |score|), so that an fp32 kernel and the fp64 oracle decide alike.
Sentences the oracle does not check keep salt 0 and are generated on the
device.  No value computed by the CUDA path ever feeds the oracle.

Score tolerance: every finite score (cumulative scores, normalised scores of
finished hypotheses and of the final choice) must satisfy
|gpu - ref| <= 1e-5 |ref|, the relative bound stated for this path; a score
whose reference is 0 or infinite must be equal.  Each comparison records its
relative error in ``REL_ERR`` (worst value per test), which the test session
prints at its end, so the margin left under the bound is visible.
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from oracle import beam as ob

MIN_GAP = 1e-3
REL_TOL = 1e-5

# worst relative score error seen per test: {test id: (error, where)}; the session prints it
REL_ERR: dict = {}
CURRENT_TEST = ["(outside a test)"]


def score_tol(ref, t=None):
    """The allowed |gpu - ref| for finite references (t is unused: the bound is purely relative)."""
    return REL_TOL * np.abs(ref)


def check_scores(got, ref, what: str):
    """Assert the relative bound on every finite score, equality on the rest; record the worst error."""
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    exact = ~np.isfinite(ref) | (ref == 0)
    assert (got[exact] == ref[exact]).all(), f"{what}: non-finite or zero scores differ: {got[exact]} vs {ref[exact]}"
    fin = ~exact
    if not fin.any():
        return
    rel = np.abs(got[fin] - ref[fin]) / np.abs(ref[fin])
    worst = float(rel.max())
    key = CURRENT_TEST[0]
    if worst > REL_ERR.get(key, (-1.0, ""))[0]:
        REL_ERR[key] = (worst, what)
    assert worst <= REL_TOL, f"{what}: relative score error {worst:.3g} > {REL_TOL:g} (ref {ref[fin]}, got {got[fin]})"


@dataclass
class BeamCase:
    kind: str               # synth recipe: tiny / tbase / llama / sweep
    B: int
    W: int
    V: int
    T: int                  # steps to run
    dtype: torch.dtype
    eos: int = -1
    alpha: float = 0.6
    early_stopping: int = ob.ES_FALSE
    lp_kind: int = ob.LP_GNMT
    max_len: int | None = None
    seed: int = 1234
    bos: int = 0
    pad: int = -1
    checked: list | None = None   # sentences the oracle runs (None = all)
    ld_pad: int = 0               # extra row stride (exercises ld > V)

    @property
    def R(self):
        return self.B * self.W

    @property
    def ML(self):
        return self.max_len or self.T


@dataclass
class OracleTrace:
    bs: ob.BeamSearch                      # the oracle over the checked sentences only
    checked: list
    steps: list = field(default_factory=list)   # per step: StepResult (checked sentences, local rows)
    salts: list = field(default_factory=list)   # per step: {global sentence: salt}
    seqs: list = field(default_factory=list)    # per step: oracle seqs after the step
    hyps: list = field(default_factory=list)    # per step: the finished sets after the step
    done: list = field(default_factory=list)    # per step: done flags after the step


def _rows(case: BeamCase, b: int, step: int, salt: int, bias, device="cpu"):
    return synth.beam_logits(case.kind, case.W, case.V, seed=case.seed, step=step, sentence=b, salt=salt,
                             dtype=case.dtype, eos=case.eos, bias=bias, device=device)


def run_oracle(case: BeamCase, min_gap: float = MIN_GAP, max_salts: int = 200,
               stop_when_done: bool = True) -> OracleTrace:
    checked = list(range(case.B)) if case.checked is None else list(case.checked)
    bias = synth.zipf_bias(case.V, case.seed) if case.kind == "llama" else None
    bs = ob.BeamSearch(len(checked), case.W, case.V, eos=case.eos, alpha=case.alpha,
                       early_stopping=case.early_stopping, lp_kind=case.lp_kind, max_len=case.ML,
                       bos=case.bos, pad=case.pad)
    tr = OracleTrace(bs, checked)
    for t in range(1, case.T + 1):
        overrides, salts = {}, {}
        for i, b in enumerate(checked):
            if bs.done[i]:
                salts[b] = 0
                continue
            for salt in range(max_salts):
                rows = _rows(case, b, t, salt, bias)
                ss = bs.sentence_step(i, rows.float().numpy(), t, margins=True)
                if min(ss.margins, default=math.inf) >= min_gap:
                    break
            else:
                raise RuntimeError(f"no salt gives a {min_gap} gap (step {t}, sentence {b})")
            overrides[i] = ss
            salts[b] = salt
        dummy = np.zeros((len(checked) * case.W, 1))
        res = bs.step(dummy, overrides=overrides)
        tr.steps.append(res)
        tr.salts.append(salts)
        tr.seqs.append([list(s) for s in bs.seqs])
        tr.hyps.append([h.copy() for h in bs.hyps])
        tr.done.append(bs.done.copy())
        if res.all_done and stop_when_done:
            break
    return tr


_POOL: list = []


def _pool_init():
    torch.set_num_threads(1)


def _oracle_pool():
    """One pool of spawned worker processes (one per host core) for the whole session: spawned,
    not forked, because the test process holds a CUDA context; the workers use the CPU only."""
    import atexit
    import multiprocessing as mp
    import os

    if not _POOL:
        size = max(1, os.cpu_count() or 1)
        pool = mp.get_context("spawn").Pool(size, initializer=_pool_init)
        atexit.register(pool.terminate)
        _POOL.append((pool, size))
    return _POOL[0]


def _oracle_chunk(job):
    case, chunk, min_gap, max_salts = job
    return run_oracle(dataclasses.replace(case, checked=list(chunk)), min_gap, max_salts, stop_when_done=False)


def run_oracle_parallel(case: BeamCase, workers: int | None = None, min_gap: float = MIN_GAP,
                        max_salts: int = 200) -> OracleTrace:
    """run_oracle over the checked sentences split across spawned worker processes.

    Sentences are independent, so each worker runs the oracle on a contiguous chunk for
    every step; the chunks' traces are joined sentence-wise and cut at the first step
    where every sentence is done, which is the trace run_oracle gives for the whole set.
    """
    checked = list(range(case.B)) if case.checked is None else list(case.checked)
    pool, size = _oracle_pool()
    n = max(1, min(workers or size, len(checked)))
    bounds = [round(i * len(checked) / n) for i in range(n + 1)]
    chunks = [checked[bounds[i]:bounds[i + 1]] for i in range(n) if bounds[i + 1] > bounds[i]]
    parts = pool.map(_oracle_chunk, [(case, c, min_gap, max_salts) for c in chunks], chunksize=1)
    T = len(parts[0].steps)
    L = next((t + 1 for t in range(T) if all(p.steps[t].all_done for p in parts)), T)
    W = case.W
    bs = ob.BeamSearch(len(checked), W, case.V, eos=case.eos, alpha=case.alpha,
                       early_stopping=case.early_stopping, lp_kind=case.lp_kind, max_len=case.ML,
                       bos=case.bos, pad=case.pad)
    tr = OracleTrace(bs, checked)
    for t in range(L):
        off, bi, tok, sc, dn, sents, salts = 0, [], [], [], [], {}, {}
        seqs, hyps = [], []
        for p in parts:
            r = p.steps[t]
            bi.append(np.where(r.beam_idx >= 0, r.beam_idx + off * W, -1))
            tok.append(r.tokens)
            sc.append(r.scores)
            dn.append(r.done)
            sents.update({off + b: ss for b, ss in r.sentences.items()})
            salts.update(p.salts[t])
            seqs.extend(p.seqs[t])
            hyps.extend(p.hyps[t])
            off += len(p.checked)
        done = np.concatenate(dn)
        tr.steps.append(ob.StepResult(np.concatenate(bi), np.concatenate(tok), np.concatenate(sc), done,
                                      bool(done.all()), sents))
        tr.salts.append(salts)
        tr.seqs.append(seqs)
        tr.hyps.append(hyps)
        tr.done.append(done.copy())
    last = tr.steps[L - 1]
    bs.scores = last.scores.reshape(len(checked), W).copy()
    bs.seqs = [list(s) for s in tr.seqs[L - 1]]
    bs.done = tr.done[L - 1].copy()
    bs.hyps = [h.copy() for h in tr.hyps[L - 1]]
    bs.t = L
    return tr


def step_logits(case: BeamCase, t: int, salts: dict, device, bias_dev=None, bias_cpu=None):
    """The whole batch's logits for step t on the device ([R, V + ld_pad], rows [:, :V] used)."""
    ld = case.V + case.ld_pad
    out = torch.empty(case.R, ld, dtype=case.dtype, device=device)
    for b in range(case.B):
        if b in salts:
            rows = _rows(case, b, t, salts[b], bias_cpu).to(device)
        else:
            rows = _rows(case, b, t, 0, bias_dev, device=device)
        out[b * case.W:(b + 1) * case.W, :case.V] = rows
    if case.ld_pad:
        out[:, case.V:] = float("nan")        # never read
    return out


def compare_step(case, tr: OracleTrace, t: int, gpu_bi, gpu_tok, gpu_sc, gpu_seqs):
    """Compare one step's outputs of the checked sentences (raises AssertionError)."""
    res = tr.steps[t - 1]
    W = case.W
    for i, b in enumerate(tr.checked):
        g = slice(b * W, (b + 1) * W)
        o = slice(i * W, (i + 1) * W)
        ref_bi = res.beam_idx[o]
        exp_bi = np.where(ref_bi >= 0, ref_bi - i * W + b * W, -1)    # local -> global rows
        np.testing.assert_array_equal(gpu_bi[g], exp_bi, err_msg=f"beam_idx step {t} sentence {b}")
        np.testing.assert_array_equal(gpu_tok[g], res.tokens[o], err_msg=f"tokens step {t} sentence {b}")
        check_scores(gpu_sc[g], res.scores[o], f"scores step {t} sentence {b}")
        if gpu_seqs is not None:
            for w in range(W):
                exp = tr.seqs[t - 1][i * W + w]
                got = gpu_seqs[b * W + w, :len(exp)]
                np.testing.assert_array_equal(got, exp, err_msg=f"seqs step {t} row {b * W + w}")


def compare_finished(case, tr: OracleTrace, fin: dict, t: int):
    W = case.W
    count = fin["count"].cpu().numpy()
    ns = fin["ns"].cpu().numpy()
    ln = fin["len"].cpu().numpy()
    ser = fin["serial"].cpu().numpy()
    tok = fin["tokens"].cpu().numpy()
    done = fin["done"].cpu().numpy()
    for i, b in enumerate(tr.checked):
        h = tr.hyps[t - 1][i]
        assert count[b] == len(h), f"finished count sentence {b} step {t}: {count[b]} vs {len(h)}"
        assert bool(done[b]) == bool(tr.done[t - 1][i]), f"done flag sentence {b} step {t}"
        slots = sorted(range(count[b]), key=lambda q: ser[b * W + q])
        for q, hy in zip(slots, h.beams):
            r = b * W + q
            assert ser[r] == hy.serial, f"serial sentence {b}"
            assert ln[r] == hy.length, f"|y| sentence {b}"
            np.testing.assert_array_equal(tok[r, :len(hy.tokens)], hy.tokens, err_msg=f"hyp tokens sentence {b}")
            check_scores([ns[r]], [hy.ns], f"finished ns sentence {b} step {t}")


def run_gpu_case(case: BeamCase, tr: OracleTrace, device="cuda", check_every_step=True, two_pass=False,
                 shards=None):
    """Run the CUDA path over the oracle's steps and compare everything; returns the BeamSearch.
    With two_pass, every step goes through the two-pass coarse-selection ablation; with
    shards (a list of column boundaries 0 < c1 < ... < V), through per-shard partials and
    their merge."""
    import verify_bs_step_gb300 as vbs

    bias_dev = synth.zipf_bias(case.V, case.seed, device) if case.kind == "llama" else None
    bias_cpu = synth.zipf_bias(case.V, case.seed) if case.kind == "llama" else None
    bs = vbs.BeamSearch(case.B, case.W, case.V, eos=case.eos, alpha=case.alpha,
                        early_stopping=case.early_stopping, lp_kind=case.lp_kind, max_len=case.ML,
                        bos=case.bos, pad=case.pad, dtype=case.dtype, device=device)
    for t in range(1, len(tr.steps) + 1):
        logits = step_logits(case, t, tr.salts[t - 1], device, bias_dev, bias_cpu)
        lg = logits[:, :case.V] if case.ld_pad else logits
        if shards:
            cuts = [0] + list(shards) + [case.V]
            parts = [bs.shard_partial(lg[:, c0:c1], c0) for c0, c1 in zip(cuts[:-1], cuts[1:])]
            bi, tok, sc = bs.merge_shards(torch.stack(parts))
        else:
            bi, tok, sc = bs.step_two_pass(lg) if two_pass else bs.step(lg)
        if check_every_step or t == len(tr.steps):
            torch.cuda.synchronize()
            compare_step(case, tr, t, bi.cpu().numpy(), tok.cpu().numpy(), sc.cpu().numpy(),
                         bs.seqs.cpu().numpy())
            if check_every_step or t == len(tr.steps):
                compare_finished(case, tr, bs.finished(), t)
    assert bs.status() == 0, "device status word set"
    return bs


def compare_finalize(case, tr: OracleTrace, bs, n_return: int = 1):
    out, out_len, out_score = bs.finalize(n_return)
    ref_out, ref_len, ref_score, _ = tr.bs.finalize(n_return)
    out, out_len, out_score = out.cpu().numpy(), out_len.cpu().numpy(), out_score.cpu().numpy()
    T = len(tr.steps)
    n = n_return
    for i, b in enumerate(tr.checked):
        for j in range(n):
            g, o = b * n + j, i * n + j
            np.testing.assert_array_equal(out[g], ref_out[o], err_msg=f"final row sentence {b} rank {j}")
            assert out_len[g] == ref_len[o]
            check_scores([out_score[g]], [ref_score[o]], f"final score sentence {b} rank {j}")
