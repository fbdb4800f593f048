"""bs_expand_static, the entry point that allocates nothing, against bs_step.

Some callers cannot allocate device memory: code that runs inside an allocator
or a memory-pool callback, a host process whose device budget is fixed at
start-up, an embedding runtime that forbids cudaMalloc once it is serving.
bs_expand_static gives them one beam expansion whose scratch lives in a static
device array.  With no end-of-sequence token and no finished sentence, its
beams are exactly those bs_step keeps, so this file runs both on the same
seeded logits for two calls in a row (the second starting from the first's
scores) and compares parents and tokens exactly and scores within the tolerance
of the other beam tests.  The file is named to be collected last.
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
    fin = np.isfinite(sc_r)
    assert (sc_s[~fin] == sc_r[~fin]).all(), f"{what}: non-finite scores, call {t}"
    err = np.abs(sc_s[fin].astype(np.float64) - sc_r[fin])
    assert (err <= hz.score_tol(sc_r[fin], t)).all(), f"{what}: scores, call {t}, max err {err.max()}"


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


def test_static_scratch_refuses_oversized_problems():
    import verify_bs_step_gb300 as vbs

    dev = torch.device("cuda")
    logits = torch.zeros(8200, 2, device=dev)
    scores = torch.zeros(8200, device=dev)
    with pytest.raises(vbs.VbsError) as e:
        vbs.bs_expand_static(logits, scores, 1)
    assert e.value.status == vbs.ESCRATCH
    assert vbs.lib().vbs_strerror(vbs.ESCRATCH).startswith(b"problem too large")
