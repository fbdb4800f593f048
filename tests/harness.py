"""Parity harness: drive the oracle and the CUDA path on the same seeded inputs.

Inputs come from ``synth`` only.  For every sentence the oracle checks (a
sample, or all), each step's rows are re-salted until every floating-point
decision the oracle takes has a scaled gap >= MIN_GAP (see oracle.beam._gap:
1e-3 + 2e-5 |score|), so that an fp32 kernel and the fp64 oracle decide alike.
Sentences the oracle does not check keep salt 0 and are generated on the
device.  No value computed by the CUDA path ever feeds the oracle.

Score tolerance, derived from the arithmetic: the kernel forms each candidate
in fp32 as s + ((x - hi) - lo), from the fp32 cumulative score s, the exact
logit x and the row LSE carried as an fp32 pair hi + lo; the LSE's fp32
partial sums carry a relative error of about 1e-6 (about 1e-6 absolute at
|LSE| ~ 10), the subtraction x - hi rounds by at most half an ulp of ~30
(1e-6), and the new score rounds by half an ulp (6e-8 |s|).  Over t steps the
score therefore drifts by at most sum_i (6e-8 |s_i| + 2e-6) <= 3e-8 t |s_t| +
2e-6 t.  The test allows  |gpu - ref| <= 1e-5 |ref| + 4e-6 t  (the relative
part holds the drift for t <= 300, the absolute part covers the per-step error
with a factor 2).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from oracle import beam as ob

MIN_GAP = 1e-3
REL_TOL = 1e-5
ABS_TOL_PER_STEP = 4e-6


def score_tol(ref, t):
    return REL_TOL * np.abs(ref) + ABS_TOL_PER_STEP * t


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


def run_oracle(case: BeamCase, min_gap: float = MIN_GAP, max_salts: int = 200) -> OracleTrace:
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
        if res.all_done:
            break
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
        ref = res.scores[o]
        err = np.abs(gpu_sc[g].astype(np.float64) - ref)
        fin = np.isfinite(ref)
        assert (gpu_sc[g][~fin] == ref[~fin]).all(), f"non-finite scores step {t} sentence {b}"
        assert (err[fin] <= score_tol(ref[fin], t)).all(), \
            f"scores step {t} sentence {b}: max err {err[fin].max()} ref {ref}"
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
            if math.isfinite(hy.ns):
                assert abs(ns[r] - hy.ns) <= score_tol(hy.ns, t), f"ns sentence {b}: {ns[r]} vs {hy.ns}"
            else:
                assert ns[r] == hy.ns


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
            if math.isfinite(ref_score[o]):
                assert abs(out_score[g] - ref_score[o]) <= score_tol(ref_score[o], T) + 1e-7 * abs(ref_score[o])
            else:
                assert out_score[g] == ref_score[o]
