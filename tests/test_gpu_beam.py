"""Parity of the fused beam step (CUDA, through the C ABI) with the fp64 oracle.

Token ids, beam_idx, sequences, finished sets and done flags must be equal;
scores within harness.score_tol.  Inputs are seeded; the oracle guarantees the
decision gap on every sentence it checks (see tests/harness.py).
"""

import math

import numpy as np
import pytest
import torch

import synth
from oracle import beam as ob
from tests import harness as hz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from verify_bs_step_gb300 import _build
    _build.build()
    import verify_bs_step_gb300 as vbs
    return vbs.lib()


def _run(case, finalize=True, every=True, parallel=False):
    tr = hz.run_oracle_parallel(case) if parallel else hz.run_oracle(case)
    bs = hz.run_gpu_case(case, tr, check_every_step=every)
    if finalize:
        hz.compare_finalize(case, tr, bs)
        if case.W > 1:
            hz.compare_finalize(case, tr, bs, n_return=case.W)     # every hypothesis, best first
    bs.close()
    return tr


# ------------------------------------------------------------------------------------
# the tiny batched case: batch 3, W 2, V 6, EOS 5, 8 steps, fp32 N(0, 2)
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("es", [ob.ES_FALSE, ob.ES_TRUE, ob.ES_NEVER])
@pytest.mark.parametrize("lpk,alpha", [(ob.LP_GNMT, 0.6), (ob.LP_GNMT, 0.0), (ob.LP_POWER, 1.0)])
@pytest.mark.parametrize("seed", [1234, 7, 99])
def test_tiny(es, lpk, alpha, seed):
    case = hz.BeamCase("tiny", 3, 2, 6, 8, torch.float32, eos=5, alpha=alpha, early_stopping=es,
                       lp_kind=lpk, seed=seed)
    _run(case)


def test_tiny_more_sentences_and_longer():
    case = hz.BeamCase("tiny", 17, 3, 6, 24, torch.float32, eos=5, alpha=0.6, seed=5)
    _run(case)


# ------------------------------------------------------------------------------------
# the worked tree (Table 9-5) through the kernel, -inf logits included
# ------------------------------------------------------------------------------------

def test_tree_table_9_5(golden):
    import verify_bs_step_gb300 as vbs
    g = golden("tree_table_9_5.json")
    vocab = g["vocab"]
    V = len(vocab)
    bs = vbs.BeamSearch(1, 2, V, eos=-1, alpha=0.0, max_len=2, bos=0, dtype=torch.float32)
    x1 = torch.full((2, V), float("-inf"))
    for tok, p in g["step1_probs"].items():
        x1[:, vocab.index(tok)] = math.log(p)
    bi, tok, sc = bs.step(x1.cuda())
    assert [vocab[t] for t in tok.tolist()] == ["A", "B"]
    assert np.allclose(sc.cpu().numpy(), [-0.693, -0.916], atol=g["tolerance"])
    x2 = torch.full((2, V), float("-inf"))
    for r, parent in enumerate(["A", "B"]):
        for t, p in g["step2_probs"][parent].items():
            x2[r, vocab.index(t)] = math.log(p)
    bi, tok, sc = bs.step(x2.cuda())
    assert bi.tolist() == [1, 0]
    assert [vocab[t] for t in tok.tolist()] == ["x", "x"]
    assert np.allclose(sc.cpu().numpy(), [-1.022, -1.609], atol=g["tolerance"])
    assert abs(math.exp(sc[0].item()) - 0.360) < g["tolerance"]
    assert bs.status() == 0


# ------------------------------------------------------------------------------------
# the batch layout: batch 3, W 2, V 6, both beams live (scores written by the caller)
# ------------------------------------------------------------------------------------

def test_batch_layout(golden):
    import verify_bs_step_gb300 as vbs
    g = golden("batch_layout.json")
    B, W, V = g["batch"], g["W"], g["V"]
    for case in g["cases"]:
        bs = vbs.BeamSearch(B, W, V, eos=-1, alpha=0.0, max_len=4, dtype=torch.float32)
        bs.scores.zero_()
        x = torch.zeros(B * W, V)
        w, v = divmod(case["j"], V)
        x[case["b"] * W + w, v] = 5.0
        bi, tok, _ = bs.step(x.cuda())
        assert bi[case["b"] * W].item() == case["row"]
        assert tok[case["b"] * W].item() == case["token"]
    bs = vbs.BeamSearch(B, W, V, eos=-1, alpha=0.0, max_len=4, dtype=torch.float32)
    bs.scores.zero_()
    x = torch.zeros(B * W, V)
    x[:, 3] = 2.0
    bi, tok, _ = bs.step(x.cuda())
    for b in range(B):
        assert bi[b * W:(b + 1) * W].tolist() == [b * W, b * W + 1]
        assert tok[b * W:(b + 1) * W].tolist() == [3, 3]


# ------------------------------------------------------------------------------------
# exhaustive enumeration and greedy
# ------------------------------------------------------------------------------------

def _prefix_model(V, seed):
    def f(prefix):
        g = torch.Generator().manual_seed(synth.mix_seed(seed, len(prefix), *prefix))
        return torch.randn(V, generator=g) * 2.0
    return f


@pytest.mark.parametrize("V,n", [(3, 3), (2, 4), (4, 2), (2, 5)])
def test_exhaustive_enumeration(V, n):
    import verify_bs_step_gb300 as vbs
    W = V ** (n - 1)
    model = _prefix_model(V, 500 + V * 10 + n)
    bs = vbs.BeamSearch(1, W, V, eos=-1, alpha=0.0, max_len=n, bos=0, dtype=torch.float32)
    ora = ob.BeamSearch(1, W, V, eos=-1, alpha=0.0, max_len=n, bos=0)
    for t in range(1, n + 1):
        x = torch.stack([model(tuple(s)) for s in ora.seqs])
        res = ora.step(x.numpy())
        bi, tok, sc = bs.step(x.cuda())
        assert bi.tolist() == res.beam_idx.tolist()
        assert tok.tolist() == res.tokens.tolist()
        got = sc.cpu().numpy().astype(np.float64)
        fin = np.isfinite(res.scores)
        assert (got[~fin] == res.scores[~fin]).all()
        assert (np.abs(got[fin] - res.scores[fin]) <= hz.score_tol(res.scores[fin], t)).all()
    paths = sorted(ob.exhaustive_paths(lambda p: model(p).numpy(), V, n), key=lambda sp: -sp[0])[:W]
    seqs = bs.seqs.cpu().numpy()
    assert sorted(tuple(r) for r in seqs) == sorted(p for _, p in paths)


def test_beam_one_is_greedy():
    case = hz.BeamCase("sweep", 5, 1, 1000, 12, torch.float32, eos=-1, seed=3)
    tr = _run(case)
    for res in tr.steps:
        assert (res.beam_idx == np.arange(5)).all()


# ------------------------------------------------------------------------------------
# shapes and paths of the kernel: bf16/fp32 vector paths, the element path (V or ld
# not a multiple of the vector), W = 16 (32 candidates per row), padded rows
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("B,W,V,dtype,ld_pad", [
    (4, 4, 32000, torch.bfloat16, 0),
    (4, 4, 32000, torch.float32, 0),
    (3, 16, 5000, torch.bfloat16, 0),
    (2, 4, 1003, torch.bfloat16, 0),      # V % 8 != 0: element path
    (2, 4, 4096, torch.bfloat16, 8),      # ld = V + 8: vector path with a row stride
    (2, 4, 4096, torch.float32, 3),       # ld = V + 3: element path
    (1, 1, 256000, torch.float32, 0),     # one row split across many CTAs
    (7, 3, 777, torch.float32, 0),
])
def test_shapes(B, W, V, dtype, ld_pad):
    case = hz.BeamCase("sweep", B, W, V, 10, dtype, eos=3, seed=B * 1000 + W * 10 + V % 97, ld_pad=ld_pad)
    _run(case)


@pytest.mark.parametrize("B,W,V,dtype", [
    (3, 4, 32000, torch.float32),         # vector path: the queue overflows, rows are rescanned
    (2, 3, 20011, torch.float32),         # element path, ragged tail
    (1, 2, 128256, torch.bfloat16),
])
def test_ascending_rows(B, W, V, dtype):
    case = hz.BeamCase("ramp", B, W, V, 4, dtype, eos=5, seed=B * 31 + V % 1009)
    _run(case)


def test_eos_heavy_until_all_done_and_reset():
    import verify_bs_step_gb300 as vbs
    # V = 8 with EOS: sentences finish within a few steps; then the whole batch is padded
    case = hz.BeamCase("tiny", 6, 3, 8, 30, torch.float32, eos=2, alpha=1.0, early_stopping=ob.ES_TRUE, seed=11)
    tr = hz.run_oracle(case)
    assert tr.steps[-1].all_done and len(tr.steps) < 30
    bs = hz.run_gpu_case(case, tr)
    assert bs.all_done.item() == 1
    hz.compare_finalize(case, tr, bs)
    # a step after all-done pads every row
    logits = torch.zeros(case.R, case.V, device="cuda")
    bi, tok, sc = bs.step(logits)
    assert (bi == -1).all() and (tok == -1).all() and (sc == 0).all()
    # the same context runs a second decode after reset
    bs.reset()
    tr2 = hz.run_oracle(case)
    for t in range(1, len(tr2.steps) + 1):
        x = hz.step_logits(case, t, tr2.salts[t - 1], "cuda")
        bi, tok, sc = bs.step(x)
        torch.cuda.synchronize()
        hz.compare_step(case, tr2, t, bi.cpu().numpy(), tok.cpu().numpy(), sc.cpu().numpy(), bs.seqs.cpu().numpy())
    bs.close()


def test_max_len_is_enforced():
    import verify_bs_step_gb300 as vbs
    bs = vbs.BeamSearch(1, 2, 10, eos=-1, max_len=2, dtype=torch.float32)
    x = torch.randn(2, 10, device="cuda")
    bs.step(x)
    bs.step(x)
    with pytest.raises(vbs.VbsError) as e:
        bs.step(x)
    assert e.value.status == vbs.ESTATE
    bs.close()


# ------------------------------------------------------------------------------------
# the length-penalty / early-stopping grid on a mid-size case with planted EOS hits
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("es", [ob.ES_FALSE, ob.ES_TRUE, ob.ES_NEVER])
@pytest.mark.parametrize("alpha", [0.0, 0.6, 1.0])
def test_sweep_alpha_early_stopping(es, alpha):
    case = hz.BeamCase("sweep", 32, 4, 32000, 50, torch.bfloat16, eos=7, alpha=alpha, early_stopping=es,
                       seed=4000 + es * 10 + int(alpha * 10), checked=list(range(0, 32, 3)))
    _run(case, every=False)


# ------------------------------------------------------------------------------------
# the workloads at full size
# ------------------------------------------------------------------------------------

def test_tbase_full_size():
    """batch 128, W 4, V 32000 bf16 N(0,3) + one +8 spike per row, EOS 2, 64 steps; every
    sentence checked at every step (the oracle runs in a process pool)."""
    case = hz.BeamCase("tbase", 128, 4, 32000, 64, torch.bfloat16, eos=2, alpha=0.6, seed=1235)
    tr = hz.run_oracle_parallel(case)
    bs = hz.run_gpu_case(case, tr, check_every_step=True)
    hz.compare_finalize(case, tr, bs)
    hz.compare_finalize(case, tr, bs, n_return=case.W)
    bs.close()


def test_llama_full_size_every_sentence():
    """batch 64, W 4, V 128256 bf16 N(0,2.5) + Zipf bias: all 64 sentences checked at every one
    of the first 24 steps (the oracle runs in a process pool)."""
    case = hz.BeamCase("llama", 64, 4, 128256, 24, torch.bfloat16, eos=2, alpha=0.6, seed=1236, max_len=200)
    tr = hz.run_oracle_parallel(case)
    bs = hz.run_gpu_case(case, tr, check_every_step=True)
    hz.compare_finalize(case, tr, bs)
    bs.close()


def test_llama_full_size():
    """batch 64, W 4, V 128256 bf16 N(0,2.5) + Zipf bias, 200 steps (a sample checked every step)."""
    case = hz.BeamCase("llama", 64, 4, 128256, 200, torch.bfloat16, eos=2, alpha=0.6, seed=1236,
                       checked=[0, 21, 63])
    _run(case, every=True)


@pytest.mark.parametrize("B,W,V,dtype", [
    (B, W, V, dt) for B in (1, 32, 256) for W in (1, 4, 16) for V in (32000, 128256, 256000)
    for dt in (torch.float32, torch.bfloat16)])
def test_sweep_grid(B, W, V, dtype):
    """The large-vocabulary wide-beam grid, ~2% planted EOS hits per row and step."""
    big = B * W * V > 50_000_000
    steps = 4 if big else 12
    checked = [0] if B == 1 else [0, B // 3, 2 * B // 3, B - 1]
    case = hz.BeamCase("sweep", B, W, V, steps, dtype, eos=11, alpha=0.6, seed=B + W + V,
                       checked=checked)
    _run(case, every=not big)


@pytest.mark.parametrize("alpha,es", [(0.0, ob.ES_TRUE), (0.0, ob.ES_NEVER), (1.0, ob.ES_TRUE), (1.0, ob.ES_NEVER)])
@pytest.mark.parametrize("W,V,dtype", [
    (W, V, dt) for W in (1, 4, 16) for V in (32000, 128256, 256000) for dt in (torch.float32, torch.bfloat16)])
def test_sweep_corner_alpha_early_stopping(W, V, dtype, alpha, es):
    """Every (W, V, dtype) corner of the sweep under alpha in {0, 1} x early_stopping in
    {True, never}, 32 sentences with 4 checked at every step; the recipe's 50 steps where the
    oracle is quick (so that finished sets fill and the stopping rules decide), fewer above."""
    steps = 50 if W * V <= 600_000 else (12 if W * V <= 2_100_000 else 6)
    case = hz.BeamCase("sweep", 32, W, V, steps, dtype, eos=11, alpha=alpha, early_stopping=es,
                       seed=9000 + W * 7 + V % 997 + int(alpha * 3) + es * 11, checked=[0, 11, 22, 31])
    _run(case, every=True, parallel=True)


# ------------------------------------------------------------------------------------
# the two-pass coarse-selection ablation (bs_step_two_pass) against the same oracle
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("kind,B,W,V,T,dtype,eos,ld_pad", [
    ("tiny", 3, 2, 6, 8, torch.float32, 5, 0),
    ("sweep", 32, 4, 32000, 20, torch.bfloat16, 7, 0),
    ("sweep", 4, 16, 4096, 12, torch.float32, 3, 0),        # K = 32
    ("sweep", 5, 3, 1003, 12, torch.bfloat16, 2, 0),        # element path
    ("sweep", 2, 4, 4096, 10, torch.float32, 1, 5),         # row stride ld > V
    ("ramp", 2, 4, 32000, 4, torch.float32, 5, 0),          # many logits above the first bar
])
def test_two_pass_ablation_matches_oracle(kind, B, W, V, T, dtype, eos, ld_pad):
    case = hz.BeamCase(kind, B, W, V, T, dtype, eos=eos, alpha=0.6, seed=B * 13 + V % 101, ld_pad=ld_pad)
    tr = hz.run_oracle(case)
    bs = hz.run_gpu_case(case, tr, two_pass=True)
    hz.compare_finalize(case, tr, bs)
    bs.close()


def test_two_pass_ablation_llama_shape():
    case = hz.BeamCase("llama", 64, 4, 128256, 3, torch.bfloat16, eos=2, alpha=0.6, seed=1236, checked=[0, 17, 63])
    tr = hz.run_oracle(case)
    bs = hz.run_gpu_case(case, tr, two_pass=True)
    bs.close()


# ------------------------------------------------------------------------------------
# vocabulary shards: per-shard partials merged into the step (bs_step_shard / _merge_shards)
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("kind,B,W,V,T,dtype,eos,shards", [
    ("tiny", 3, 2, 6, 8, torch.float32, 5, [3]),
    ("sweep", 8, 4, 32000, 16, torch.bfloat16, 7, [10000]),
    ("sweep", 6, 4, 32000, 12, torch.bfloat16, 3, [7, 12345, 20001]),      # unaligned shards: element path
    ("sweep", 3, 16, 4096, 10, torch.float32, 11, [512, 1024, 2048, 3000]),  # K = 32
    ("sweep", 4, 3, 1003, 12, torch.float32, 2, [501]),
])
def test_vocab_shards_match_oracle(kind, B, W, V, T, dtype, eos, shards):
    case = hz.BeamCase(kind, B, W, V, T, dtype, eos=eos, alpha=0.6, seed=B * 17 + V % 103)
    tr = hz.run_oracle(case)
    bs = hz.run_gpu_case(case, tr, shards=shards)
    hz.compare_finalize(case, tr, bs)
    bs.close()


def test_vocab_shards_llama_shape():
    case = hz.BeamCase("llama", 64, 4, 128256, 2, torch.bfloat16, eos=2, alpha=0.6, seed=1236, checked=[3, 40])
    tr = hz.run_oracle(case)
    bs = hz.run_gpu_case(case, tr, shards=[32064, 64128, 96192])   # four shards of a 4-way vocab-parallel head
    bs.close()


def test_vocab_shards_limits():
    import verify_bs_step_gb300 as vbs
    bs = vbs.BeamSearch(2, 4, 64, eos=3, max_len=4, dtype=torch.float32)
    lg = torch.zeros(8, 64, device="cuda")
    with pytest.raises(vbs.VbsError):
        bs.shard_partial(lg[:, 60:64 + 0], 61)             # past V
    part = bs.shard_partial(lg, 0)
    with pytest.raises(vbs.VbsError) as e:
        bs.merge_shards(part.unsqueeze(0).repeat(33, 1))    # more shards than the merge holds (W 4: 32)
    assert e.value.status == vbs.EINVAL
    bs.close()


# ------------------------------------------------------------------------------------
# logits that are not finite: reported in the status word, the context stays usable
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("B,W,V,dtype", [
    (3, 2, 64, torch.float32),            # cluster kernel, element path
    (2, 4, 4096, torch.bfloat16),         # cluster kernel, bulk-copy path
    (4, 16, 512, torch.bfloat16),         # stream and merge kernels
])
@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_non_finite_logits_are_reported(B, W, V, dtype, bad):
    import verify_bs_step_gb300 as vbs
    bs = vbs.BeamSearch(B, W, V, eos=-1, max_len=4, dtype=dtype)
    g = torch.Generator().manual_seed(B * W + V)
    x = torch.randn(B * W, V, generator=g)
    x[0, 7] = bad                          # beam 0 of sentence 0: a row the first step reads
    bs.step(x.to(dtype).cuda())
    assert bs.status() == vbs.EINPUT
    bs.reset()
    bs.step(torch.randn(B * W, V, generator=g).to(dtype).cuda())
    assert bs.status() == 0
    bs.close()
