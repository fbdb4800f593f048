"""Parity of blockwise-parallel-decoding predict / verify (CUDA, through the C ABI) with the oracle."""

import numpy as np
import pytest
import torch

import synth
from oracle import bpd as ob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from verify_bs_step_gb300 import _build
    _build.build()
    import verify_bs_step_gb300 as vbs
    return vbs.lib()


def _np(t):
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def test_figure_1(golden):
    import verify_bs_step_gb300 as vbs
    g = golden("bpd_figure1.json")
    vocab, k = g["vocab"], g["k"]
    V = len(vocab)
    props = torch.tensor([[vocab.index(t) for t in g["proposals"]]], dtype=torch.int32)
    heads = torch.full((1, k, k), vocab.index("<other>"))
    heads[0, 0, 0] = vocab.index(g["base_argmax_given_prefix"]["in"])
    heads[0, 1, 0] = vocab.index(g["base_argmax_given_prefix"]["in the"])
    logits = synth.planted_rows(heads, V, seed=5, salt=0, dtype=torch.float32)
    khat, nxt = vbs.bpd_verify(logits.cuda(), props.cuda())
    assert khat.item() == g["khat"]
    assert vocab[nxt[0, 0].item()] == "car"


@pytest.mark.parametrize("B,k,V,dtype,eos", [
    (37, 5, 1000, torch.bfloat16, -1),
    (37, 5, 1000, torch.float32, -1),
    (16, 8, 32000, torch.bfloat16, 3),
    (9, 1, 64, torch.float32, -1),         # k = 1: nothing to verify
    (11, 3, 77, torch.bfloat16, -1),       # V * 2 bytes not a multiple of 16: element path
    (5, 32, 4096, torch.bfloat16, -1),     # k = 32
])
def test_verify_matches_oracle(B, k, V, dtype, eos):
    import verify_bs_step_gb300 as vbs
    base, props, heads = synth.geometric_prefix_proposals(B, k, V, seed=B * k + V, step=0)
    if eos >= 0:
        props[::2, 2] = eos                      # an accepted EOS truncates khat
    logits = synth.planted_rows(heads, V, seed=B + k, salt=1, dtype=dtype)
    khat, nxt = vbs.bpd_verify(logits.cuda(), props.to(torch.int32).cuda(), eos)
    ekh, enx = ob.verify(_np(logits), props.numpy(), eos)
    np.testing.assert_array_equal(khat.cpu().numpy(), ekh)
    np.testing.assert_array_equal(nxt.cpu().numpy(), enx)


def test_ties_go_to_the_lower_token():
    import verify_bs_step_gb300 as vbs
    B, k, V = 4, 3, 512
    logits = torch.zeros(B, k, k, V)
    logits[..., 100] = 3.0
    logits[..., 7] = 3.0                         # a tie: token 7 wins
    logits[..., 300] = 3.0
    props = torch.tensor([[7, 7, 7], [7, 100, 7], [1, 7, 300], [7, 7, 2]], dtype=torch.int32)
    khat, nxt = vbs.bpd_verify(logits.cuda(), props.cuda())
    ekh, enx = ob.verify(logits.numpy(), props.numpy())
    assert khat.tolist() == ekh.tolist() == [3, 1, 2, 2]
    assert (nxt.cpu().numpy() == 7).all() and (enx == 7).all()
    p = vbs.bpd_propose(logits[:, 0].contiguous().cuda())
    assert (p.cpu().numpy() == ob.propose(logits[:, 0].numpy())).all()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_propose_matches_oracle(dtype):
    import verify_bs_step_gb300 as vbs
    x = synth.normal_rows(40 * 8, 32000, 2.0, seed=8, dtype=dtype).view(40, 8, 32000)
    got = vbs.bpd_propose(x.cuda())
    np.testing.assert_array_equal(got.cpu().numpy(), ob.propose(_np(x)))


def test_full_size_verify():
    """logits [256, 8, 8, 32000] bf16 (1.05 GB), geometric(0.7) agreement: every khat and proposal."""
    import verify_bs_step_gb300 as vbs
    B, k, V = 256, 8, 32000
    base, props, heads = synth.geometric_prefix_proposals(B, k, V, seed=4242, step=1)
    logits = synth.planted_rows(heads, V, seed=4242, salt=2, dtype=torch.bfloat16)
    khat, nxt = vbs.bpd_verify(logits.cuda(), props.to(torch.int32).cuda())
    ekh, enx = ob.verify(_np(logits), props.numpy())
    np.testing.assert_array_equal(khat.cpu().numpy(), ekh)
    np.testing.assert_array_equal(nxt.cpu().numpy(), enx)
    assert 2.7 < ekh.mean() < 3.6                 # E[khat] = 1 + sum_{n=1..7} 0.7^n = 3.14


def test_blockwise_decoding_on_gpu_reproduces_greedy():
    """The accepted tokens, iterated with the CUDA verify, equal greedy decoding token for token."""
    import verify_bs_step_gb300 as vbs
    B, k, V, length, seed, agree = 6, 4, 50, 40, 99, 0.7

    def truth_after(b, y):
        return synth.prefix_token(b, y, V, seed)

    greedy = [ob.greedy_decode(lambda y, b=b: truth_after(b, y), length) for b in range(B)]
    # predict for the first iteration: head 0 = base, heads >= 1 = proposals of the future
    heads0 = torch.zeros(B, k, dtype=torch.int64)
    for b in range(B):
        y = ()
        for h in range(k):
            t = truth_after(b, y)
            heads0[b, h] = t if h == 0 else synth.proposal_token(b, (), h, t, V, seed, agree)
            y = y + (t,)
    props = vbs.bpd_propose(synth.planted_rows(heads0, V, seed=seed, salt=0, dtype=torch.float32).cuda())
    out = [[] for _ in range(B)]
    it = 0
    while min(len(o) for o in out) < length:
        it += 1
        pr = props.cpu().numpy()
        heads = torch.zeros(B, k, k, dtype=torch.int64)
        for b in range(B):
            for p in range(k):
                ctx = tuple(out[b]) + tuple(int(v) for v in pr[b, :p + 1])
                y = ctx
                for h in range(k):
                    t = truth_after(b, y)
                    heads[b, p, h] = t if h == 0 else synth.proposal_token(b, ctx, h, t, V, seed, agree)
                    y = y + (t,)
        logits = synth.planted_rows(heads, V, seed=seed, salt=it, dtype=torch.bfloat16).cuda()
        khat, props = vbs.bpd_verify(logits, torch.from_numpy(pr).to(torch.int32).cuda())
        for b, n in enumerate(khat.tolist()):
            assert n >= 1
            out[b].extend(int(v) for v in pr[b, :n])
    for b in range(B):
        assert out[b][:length] == greedy[b]
    assert it < length                             # fewer iterations than greedy steps


@pytest.mark.parametrize("B,k", [(16384, 2), (16385, 2)])
def test_verify_on_both_sides_of_the_queue_limit(B, k):
    """Batches up to 16384 run the work-queue kernel, larger ones the one-CTA-per-element
    kernel; both must equal the oracle (a vectorised V = 64 keeps the rows small)."""
    import verify_bs_step_gb300 as vbs
    V = 64
    base, props, heads = synth.geometric_prefix_proposals(B, k, V, seed=B, step=0)
    logits = synth.planted_rows(heads, V, seed=B + 1, salt=2, dtype=torch.bfloat16)
    for _ in range(2):                            # twice: the queue's state resets between calls
        khat, nxt = vbs.bpd_verify(logits.cuda(), props.to(torch.int32).cuda())
        torch.cuda.synchronize()
    # the oracle on a sample of the batch (its loops are slow on 16k elements)
    pick = np.r_[0:64, B - 64:B]
    ekh, enx = ob.verify(_np(logits[pick]), props[pick].numpy())
    np.testing.assert_array_equal(khat.cpu().numpy()[pick], ekh)
    np.testing.assert_array_equal(nxt.cpu().numpy()[pick], enx)
    assert vbs.lib().vbs_stateless_status(vbs._stream()) == 0


# --- the relaxed verify tests of §5 (bpd_verify_approx) --------------------------------

_CRITERIA = [(0, 0, 1), (1, 2, 1), (1, 3, 1), (1, 1, 1), (2, 1, 1), (2, 2, 1), (2, 0, 1), (0, 0, 3), (1, 2, 4),
             (2, 1, 5)]


@pytest.mark.parametrize("B,k,V,dtype,eos", [
    (40, 5, 1000, torch.bfloat16, -1),
    (33, 6, 4096, torch.float32, 7),
    (17, 8, 32000, torch.bfloat16, -1),
    (13, 4, 77, torch.bfloat16, -1),        # element path
    (9, 3, 3001, torch.float32, 11),        # element path (V * 4 not a multiple of 16), EOS
])
def test_relaxed_verify_matches_oracle(B, k, V, dtype, eos):
    import verify_bs_step_gb300 as vbs
    logits, props = synth.near_miss_proposals(B, k, V, seed=B * 7 + k, step=V % 13, dtype=dtype)
    if eos >= 0:
        props[1::3, min(2, k - 1)] = eos
    lg, pr = logits.cuda(), props.to(torch.int32).cuda()
    x = _np(logits)
    for crit, param, ma in _CRITERIA:
        ma = min(ma, k)
        khat, nxt = vbs.bpd_verify(lg, pr, eos, criterion=crit, param=param, min_accept=ma)
        ekh, enx = ob.verify(x, props.numpy(), eos, crit, param, ma)
        np.testing.assert_array_equal(khat.cpu().numpy(), ekh, err_msg=f"khat {crit} {param} {ma}")
        np.testing.assert_array_equal(nxt.cpu().numpy(), enx, err_msg=f"next {crit} {param} {ma}")
    assert vbs.lib().vbs_stateless_status(vbs._stream()) == 0


def test_relaxed_verify_out_of_range_proposal_fails_topk():
    import verify_bs_step_gb300 as vbs
    B, k, V = 4, 3, 64
    logits, props = synth.near_miss_proposals(B, k, V, seed=2, step=0, dtype=torch.float32)
    props[:, 1] = torch.tensor([V, -1, V + 5, 0])
    khat, nxt = vbs.bpd_verify(logits.cuda(), props.to(torch.int32).cuda(), -1, criterion=vbs.BPD_TOPK, param=V)
    ekh, enx = ob.verify(_np(logits), props.numpy(), -1, ob.TOPK, V, 1)
    np.testing.assert_array_equal(khat.cpu().numpy(), ekh)
    np.testing.assert_array_equal(nxt.cpu().numpy(), enx)


@pytest.mark.parametrize("B", [16384, 16385])
def test_relaxed_verify_on_both_sides_of_the_queue_limit(B):
    import verify_bs_step_gb300 as vbs
    k, V = 3, 64
    logits, props = synth.near_miss_proposals(B, k, V, seed=B, step=1, dtype=torch.bfloat16)
    lg, pr = logits.cuda(), props.to(torch.int32).cuda()
    pick = np.r_[0:64, B - 64:B]
    x = _np(logits[pick])
    for crit, param, ma in ((1, 2, 1), (2, 1, 2)):
        khat, nxt = vbs.bpd_verify(lg, pr, -1, criterion=crit, param=param, min_accept=ma)
        ekh, enx = ob.verify(x, props[pick].numpy(), -1, crit, param, ma)
        np.testing.assert_array_equal(khat.cpu().numpy()[pick], ekh)
        np.testing.assert_array_equal(nxt.cpu().numpy()[pick], enx)


def test_relaxed_verify_rejects_bad_parameters():
    import verify_bs_step_gb300 as vbs
    logits, props = synth.near_miss_proposals(2, 3, 64, seed=1, step=0, dtype=torch.float32)
    lg, pr = logits.cuda(), props.to(torch.int32).cuda()
    for crit, param, ma in ((1, 0, 1), (2, -1, 1), (3, 0, 1), (0, 0, 0), (0, 0, 4)):
        with pytest.raises(vbs.VbsError) as e:
            vbs.bpd_verify(lg, pr, -1, criterion=crit, param=param, min_accept=ma)
        assert e.value.status == vbs.EINVAL
