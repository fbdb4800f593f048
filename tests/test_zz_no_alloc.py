"""bs_expand_static, the entry point that allocates nothing, against bs_step.

Some callers cannot allocate device memory: code that runs inside an allocator
or a memory-pool callback, a host process whose device budget is fixed at
start-up, an embedding runtime that forbids cudaMalloc once it is serving.
bs_expand_static gives them one beam expansion whose scratch lives in a static
device array.  With no end-of-sequence token and no finished sentence, its
beams are exactly those bs_step keeps, so this file runs both on the same
seeded logits for two calls in a row (the second starting from the first's
scores) and compares parents and tokens exactly and scores within the tolerance
of the other beam tests; it also compares the two calls with the fp64 oracle
directly, and runs the largest problem the static array accepts (8192 rows at
W = 16) and one past it.  The file is named to be collected last.
"""

import numpy as np
import pytest
import torch

from tests import harness as hz

pytestmark = pytest.mark.gpu

CASES = [
    # kind, batch, W, V, dtype, ld_pad
    ("tbase", 3, 4, 1000, torch.float32, 0),
    ("llama", 64, 4, 128256, torch.bfloat16, 0),
    ("sweep", 5, 16, 777, torch.float32, 3),          # unaligned rows: the element-wise path
    ("sweep", 40, 1, 50000, torch.bfloat16, 0),
]


def _compare(bi_s, tok_s, sc_s, bi_r, tok_r, sc_r, t, what):
    bi_s, tok_s, sc_s = bi_s.cpu().numpy(), tok_s.cpu().numpy(), sc_s.cpu().numpy()
    bi_r, tok_r, sc_r = bi_r.cpu().numpy(), tok_r.cpu().numpy(), sc_r.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(bi_s, bi_r, err_msg=f"{what}: beam_idx, call {t}")
    np.testing.assert_array_equal(tok_s, tok_r, err_msg=f"{what}: tokens, call {t}")
    hz.check_scores(sc_s, sc_r, f"{what}: scores, call {t}")


@pytest.mark.parametrize("kind,B,W,V,dtype,ld_pad", CASES)
def test_static_scratch_matches_bs_step_on_two_calls(kind, B, W, V, dtype, ld_pad):
    import synth
    import verify_bs_step_gb300 as vbs

    dev = torch.device("cuda")
    case = hz.BeamCase(kind, B, W, V, 2, dtype, eos=-1, seed=77, ld_pad=ld_pad)
    bias = synth.zipf_bias(V, case.seed, dev) if kind == "llama" else None
    ref = vbs.BeamSearch(B, W, V, eos=-1, alpha=0.6, max_len=4, dtype=dtype, device=dev)
    scores = ref.scores.clone()                       # [0, -inf, ...] per sentence, as bs_reset leaves them
    out = torch.empty_like(scores)
    for t in (1, 2):
        logits = hz.step_logits(case, t, {}, dev, bias_dev=bias)
        view = logits[:, :V] if ld_pad else logits
        if t == 1:
            bi_s, tok_s, sc_s = vbs.bs_expand_static(view, scores, W, scores_out=out)
        else:
            bi_s, tok_s, sc_s = vbs.bs_expand_static(view, scores, W, scores_out=scores)   # in place
        bi_s, tok_s, sc_s = bi_s.clone(), tok_s.clone(), sc_s.clone()
        bi_r, tok_r, sc_r = ref.step(view)
        torch.cuda.synchronize()
        _compare(bi_s, tok_s, sc_s, bi_r, tok_r, sc_r, t, f"{kind} B{B} W{W} V{V}")
        scores = sc_s.clone()
    assert vbs.lib().vbs_stateless_status(vbs._stream(dev)) == 0
    assert ref.status() == 0
    ref.close()


@pytest.mark.parametrize("kind,B,W,V,dtype,ld_pad", [
    ("tiny", 3, 2, 6, torch.float32, 0),
    ("sweep", 16, 4, 32000, torch.bfloat16, 0),
    ("sweep", 5, 16, 777, torch.float32, 3),
    ("llama", 64, 4, 128256, torch.bfloat16, 0),
])
def test_static_scratch_matches_oracle_on_two_calls(kind, B, W, V, dtype, ld_pad):
    """The same two calls against the fp64 oracle (no end-of-sequence token): parents and
    tokens equal, scores within the relative bound; the oracle re-salts rows for its
    decision margins, and both sides read the same logits."""
    import synth
    import verify_bs_step_gb300 as vbs

    dev = torch.device("cuda")
    case = hz.BeamCase(kind, B, W, V, 2, dtype, eos=-1, seed=91, ld_pad=ld_pad,
                       checked=list(range(0, B, max(1, B // 8))))
    tr = hz.run_oracle(case)
    bias_dev = synth.zipf_bias(V, case.seed, dev) if kind == "llama" else None
    bias_cpu = synth.zipf_bias(V, case.seed) if kind == "llama" else None
    scores = torch.full((B, W), float("-inf"), device=dev)
    scores[:, 0] = 0.0
    scores = scores.reshape(-1).contiguous()
    for t in (1, 2):
        logits = hz.step_logits(case, t, tr.salts[t - 1], dev, bias_dev, bias_cpu)
        view = logits[:, :V] if ld_pad else logits
        bi, tok, sc = vbs.bs_expand_static(view, scores, W)
        torch.cuda.synchronize()
        hz.compare_step(case, tr, t, bi.cpu().numpy(), tok.cpu().numpy(), sc.cpu().numpy(), None)
        scores = sc.clone()
    assert vbs.lib().vbs_stateless_status(vbs._stream(dev)) == 0


def test_static_scratch_largest_accepted_problem():
    """8192 rows at W = 16 (the most partial keys the array holds) against bs_step, twice."""
    import verify_bs_step_gb300 as vbs

    dev = torch.device("cuda")
    B, W, V = 512, 16, 64
    case = hz.BeamCase("sweep", B, W, V, 2, torch.float32, eos=-1, seed=5)
    ref = vbs.BeamSearch(B, W, V, eos=-1, alpha=0.6, max_len=4, dtype=torch.float32, device=dev)
    scores = ref.scores.clone()
    for t in (1, 2):
        logits = hz.step_logits(case, t, {}, dev)
        bi_s, tok_s, sc_s = vbs.bs_expand_static(logits, scores, W)
        bi_s, tok_s, sc_s = bi_s.clone(), tok_s.clone(), sc_s.clone()
        bi_r, tok_r, sc_r = ref.step(logits)
        torch.cuda.synchronize()
        _compare(bi_s, tok_s, sc_s, bi_r, tok_r, sc_r, t, f"B{B} W{W} V{V}")
        scores = sc_s.clone()
    assert vbs.lib().vbs_stateless_status(vbs._stream(dev)) == 0
    assert ref.status() == 0
    ref.close()
    # one sentence more is past the row limit
    logits = torch.zeros((B + 1) * W, V, device=dev)
    with pytest.raises(vbs.VbsError) as e:
        vbs.bs_expand_static(logits, torch.zeros((B + 1) * W, device=dev), W)
    assert e.value.status == vbs.ESCRATCH


def test_static_scratch_checks_its_tensors():
    """Outputs of the wrong size, layout or device are refused before the library is called."""
    import verify_bs_step_gb300 as vbs

    dev = torch.device("cuda")
    logits = torch.zeros(8, 100, device=dev)
    scores = torch.zeros(8, device=dev)
    with pytest.raises(ValueError):
        vbs.bs_expand_static(logits, scores[:6], 4)
    with pytest.raises(ValueError):
        vbs.bs_expand_static(logits, torch.zeros(16, device=dev)[::2], 4)
    with pytest.raises(ValueError):
        vbs.bs_expand_static(logits, scores, 4, scores_out=torch.zeros(8))
    with pytest.raises(ValueError):
        vbs.bs_expand_static(logits, scores, 4, tokens=torch.zeros(7, dtype=torch.int32, device=dev))


def test_static_scratch_refuses_oversized_problems():
    import verify_bs_step_gb300 as vbs

    dev = torch.device("cuda")
    logits = torch.zeros(8200, 2, device=dev)
    scores = torch.zeros(8200, device=dev)
    with pytest.raises(vbs.VbsError) as e:
        vbs.bs_expand_static(logits, scores, 1)
    assert e.value.status == vbs.ESCRATCH
    assert vbs.lib().vbs_strerror(vbs.ESCRATCH).startswith(b"problem too large")
