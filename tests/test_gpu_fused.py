"""Parity of the fused beam step + paged KV remap (bs_step_paged, kv_paged_copy) with the oracle.

Each step: the new position's K/V is written for the live rows, then one
bs_step_paged call (the beam step, and the table remap on the beam_idx it
produces) and one kv_paged_copy.  The beam outputs are compared with the oracle's
beam search, and the cache with the oracle's naive gather driven by the oracle's
own beam_idx; the block accounting with the oracle's paged model.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import kv as ok
from tests import harness as hz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from verify_bs_step_gb300 import _build
    _build.build()
    import verify_bs_step_gb300 as vbs
    return vbs.lib()


def _run_fused(case: hz.BeamCase, L=2, H=2, D=8, P=5, blk=16):
    import verify_bs_step_gb300 as vbs
    tr = hz.run_oracle(case)
    B, W, R = case.B, case.W, case.R
    steps = len(tr.steps)
    S = -(-P // blk) + W * (-(-(steps + blk) // blk) + 2)
    MB = -(-(P + steps + 1) // blk) + 1
    bs = vbs.BeamSearch(B, W, case.V, eos=case.eos, alpha=case.alpha, early_stopping=case.early_stopping,
                        lp_kind=case.lp_kind, max_len=case.ML, bos=case.bos, pad=case.pad, dtype=case.dtype)
    pk = vbs.PagedKV(B, W, L, H, D, blocks_per_sentence=S, max_blocks=MB, block=blk, dtype=torch.float32)
    ref = ok.PagedKV(B, W, S, L, H, D, block=blk, dtype=np.float32)
    naive = np.zeros((L, 2, R, H, P + steps + 1, D), dtype=np.float32)
    rows = torch.arange(R)
    lead = torch.tensor([b * W for b in range(B)])
    pk.prefill(P)
    ref.prefill(P)
    table = pk.table()
    for pos in range(P):
        vals = synth.kv_token_values(pos, (rows // W) * W, L, H, D, seed=case.seed, dtype=torch.float32)
        naive[:, :, :, :, pos, :] = vals.numpy()
        pk.pool[table[lead, pos // blk].long(), :, :, :, pos % blk, :] = \
            vals[:, :, lead].permute(2, 0, 1, 3, 4).cuda()
        ref.write(pos, vals[:, :, lead].numpy(), rows=lead.tolist())
    pk.prepare(P)
    ref.prepare(P)
    for t in range(1, steps + 1):
        t_write = P + t - 1
        done_before = tr.done[t - 2] if t > 1 else np.zeros(B, dtype=bool)
        live = [r for r in range(R) if not done_before[r // W]]
        table = pk.table()
        vals = synth.kv_token_values(t_write, rows, L, H, D, seed=case.seed, dtype=torch.float32)
        lr = torch.tensor(live)
        pk.pool[table[lr, t_write // blk].long(), :, :, :, t_write % blk, :] = \
            vals[:, :, lr].permute(2, 0, 1, 3, 4).cuda()
        ref.write(t_write, vals[:, :, lr].numpy(), rows=live)
        for r in live:
            naive[:, :, r, :, t_write, :] = vals[:, :, r].numpy()

        logits = hz.step_logits(case, t, tr.salts[t - 1], "cuda")
        bi, tok, sc = bs.step_paged(logits, pk, t_write + 1)
        pk.copy()
        torch.cuda.synchronize()
        hz.compare_step(case, tr, t, bi.cpu().numpy(), tok.cpu().numpy(), sc.cpu().numpy(), bs.seqs.cpu().numpy())

        bi_ref = tr.steps[t - 1].beam_idx.astype(np.int32)        # every sentence is checked: global rows
        t_valid = t_write + 1
        naive = ok.reorder_naive(naive, naive, bi_ref, t_valid)
        ref.reorder(bi_ref, t_valid)
        assert pk.status() == 0 and bs.status() == 0
        rc, nb = pk.counts()
        assert int((rc > 0).sum()) == ref.blocks_in_use(), f"blocks in use, step {t}"
        tab = pk.table().cpu().numpy()
        nbh = nb.cpu().numpy()
        cnt = np.zeros(B * S, dtype=np.int64)
        for r in range(R):
            for i in range(nbh[r]):
                cnt[tab[r, i]] += 1
        np.testing.assert_array_equal(rc.cpu().numpy(), cnt, err_msg=f"reference counts, step {t}")
        table = pk.table()
        for r in live:
            pos = torch.arange(t_valid, device="cuda")
            view = pk.pool[table[r, pos // blk].long(), :, :, :, pos % blk, :]
            got = view.permute(1, 2, 3, 0, 4).cpu().numpy()
            np.testing.assert_array_equal(got, naive[:, :, r, :, :t_valid, :], err_msg=f"row {r} step {t}")
    bs.close()
    pk.close()


@pytest.mark.parametrize("B,W,V,dtype,T,eos", [
    (3, 4, 2048, torch.float32, 14, 7),      # clusters of 4 CTAs: the remap runs in the beam-step kernel
    (2, 3, 1001, torch.bfloat16, 12, 5),     # W = 3: clusters of 1 CTA, element path (V % 8 != 0)
    (40, 4, 512, torch.float32, 6, 3),       # 40 x 4 CTAs exceed the SMs: clusters of 2
    (2, 16, 1000, torch.float32, 6, 5),      # W.2W > 32: two-kernel step, separate remap launch
])
def test_fused_step_and_paged_remap(B, W, V, dtype, T, eos):
    case = hz.BeamCase("sweep", B, W, V, T, dtype, eos=eos, alpha=0.6, seed=B * 101 + W * 7 + V % 89)
    _run_fused(case)


def test_fused_llama_shape_two_steps():
    case = hz.BeamCase("llama", 64, 4, 128256, 2, torch.bfloat16, eos=2, alpha=0.6, seed=1236, checked=None)
    _run_fused(case, L=1, H=1, D=8, P=1000)


def test_fused_copies_must_run_before_the_next_remap():
    import verify_bs_step_gb300 as vbs
    bs = vbs.BeamSearch(2, 4, 64, eos=3, max_len=4, dtype=torch.float32)
    pk = vbs.PagedKV(2, 4, 1, 1, 8, blocks_per_sentence=8, max_blocks=4, block=16, dtype=torch.float32)
    pk.prefill(4)
    pk.prepare(4)
    logits = synth.normal_rows(8, 64, 2.0, seed=5).cuda()
    bs.step_paged(logits, pk, 5)
    for call in (lambda: bs.step_paged(logits, pk, 6), lambda: pk.reorder(bs.beam_idx, 6), lambda: pk.prepare(6)):
        with pytest.raises(vbs.VbsError) as e:
            call()
        assert e.value.status == vbs.ESTATE
    pk.copy()
    bs.step_paged(logits, pk, 6)
    pk.copy()
    assert pk.status() == 0 and bs.status() == 0
    bs.close()
    pk.close()


def test_fused_rejects_a_mismatched_cache():
    import verify_bs_step_gb300 as vbs
    bs = vbs.BeamSearch(2, 4, 64, eos=3, max_len=4, dtype=torch.float32)
    pk = vbs.PagedKV(3, 4, 1, 1, 8, blocks_per_sentence=8, max_blocks=4, block=16, dtype=torch.float32)
    pk.prefill(4)
    pk.prepare(4)
    logits = torch.zeros(8, 64, device="cuda")
    with pytest.raises(vbs.VbsError) as e:
        bs.step_paged(logits, pk, 5)
    assert e.value.status == vbs.EINVAL
    bs.close()
    pk.close()
