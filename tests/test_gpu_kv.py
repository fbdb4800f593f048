"""Parity of the KV reorder kernels (naive gather, paged table + copy-on-write) with the oracle."""

import numpy as np
import pytest
import torch

import synth
from oracle import kv as ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from verify_bs_step_gb300 import _build
    _build.build()
    import verify_bs_step_gb300 as vbs
    return vbs.lib()


def _beam_idx(rng, B, W, pad_sentences=()):
    bi = np.full(B * W, -1, dtype=np.int32)
    for b in range(B):
        if b not in pad_sentences:
            bi[b * W:(b + 1) * W] = b * W + np.sort(rng.integers(0, W, size=W))
    return bi


def _to_np(t):
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


@pytest.mark.parametrize("L,R,H,T,D,dtype,t_valid", [
    (2, 6, 3, 20, 8, torch.bfloat16, 13),     # 16-byte rows: bulk copies
    (1, 4, 2, 9, 4, torch.float32, 9),        # 16-byte rows, t_valid = t_max
    (2, 6, 2, 11, 3, torch.float32, 7),       # 12-byte rows: element copies
    (3, 5, 1, 8, 4, torch.bfloat16, 5),       # 8-byte rows: element copies
    (1, 3, 2, 40000, 16, torch.bfloat16, 39000),   # long rows: many bulk chunks per segment
])
def test_naive_matches_oracle(L, R, H, T, D, dtype, t_valid):
    import verify_bs_step_gb300 as vbs
    g = torch.Generator().manual_seed(L * 100 + R * 10 + T)
    src = (torch.randn(L, 2, R, H, T, D, generator=g) * 4).to(dtype)
    dst = (torch.randn(L, 2, R, H, T, D, generator=g) * 4).to(dtype)
    rng = np.random.default_rng(R + T)
    bi = rng.integers(-1, R, size=R).astype(np.int32)
    exp = ok.reorder_naive(_to_np(src), _to_np(dst), bi, t_valid)
    s, d = src.cuda(), dst.cuda()
    vbs.kv_reorder(s, d, torch.from_numpy(bi).cuda(), t_valid)
    assert vbs.lib().vbs_stateless_status(None) == 0
    np.testing.assert_array_equal(_to_np(d), exp)


def test_naive_tbase_full_size():
    """6 layers x 8 heads x 64 dims bf16, 512 rows, T_max 128, t_valid 64: sampled rows vs the oracle."""
    import verify_bs_step_gb300 as vbs
    L, R, H, T, D, W = 6, 512, 8, 128, 64, 4
    src = (torch.arange(L * 2 * R * H * T * D, device="cuda", dtype=torch.int64) % 251 - 125).to(torch.bfloat16)
    src = src.view(L, 2, R, H, T, D)
    dst = torch.full_like(src, 7.0)
    bi = _beam_idx(np.random.default_rng(3), R // W, W, pad_sentences=(5,))
    vbs.kv_reorder(src, dst, torch.from_numpy(bi).cuda(), 64)
    torch.cuda.synchronize()
    for r in (0, 1, 2, 3, 20, 21, 22, 23, 200, 511):
        got = _to_np(dst[:, :, r:r + 1])
        p = bi[r]
        srows = _to_np(src[:, :, p:p + 1]) if p >= 0 else None
        # the oracle on the sampled row (a one-row view of the same definition)
        exp = ok.reorder_naive(srows if p >= 0 else got, np.full_like(got, 7.0), [0 if p >= 0 else -1], 64)
        np.testing.assert_array_equal(got, exp)


def test_naive_llama_full_size():
    """32 layers x 8 heads x 128 dims bf16 (128 KiB/token), 256 rows, t_valid 1000: sampled rows."""
    import verify_bs_step_gb300 as vbs
    L, R, H, T, D, W = 32, 256, 8, 1200, 128, 4
    src = torch.empty(L, 2, R, H, T, D, dtype=torch.bfloat16, device="cuda")
    # each row's content identifies the row: value = row id mod 251 - 125, position-striped
    rowval = ((torch.arange(R, device="cuda") % 251) - 125).to(torch.bfloat16).view(1, 1, R, 1, 1, 1)
    src.copy_(rowval.expand_as(src))
    src[:, :, :, :, ::7, :] = 1.0
    dst = torch.zeros_like(src)
    bi = _beam_idx(np.random.default_rng(9), R // W, W)
    vbs.kv_reorder(src, dst, torch.from_numpy(bi).cuda(), 1000)
    torch.cuda.synchronize()
    for r in (0, 3, 100, 255):
        p = int(bi[r])
        got = dst[:, :, r].float()
        exp = src[:, :, p].float().clone()
        exp[:, :, :, 1000:] = 0.0
        assert torch.equal(got, exp), r
    del src, dst
    torch.cuda.empty_cache()


def _paged_decode(B, W, L, H, D, P, steps, dtype, seed, pad_after=None, check_every=1):
    """Drive the paged cache and the naive oracle through one decode; compare logical contents."""
    import verify_bs_step_gb300 as vbs
    R = B * W
    blk = 16
    S = -(-P // blk) + W * (-(-(steps + blk) // blk) + 2)
    MB = -(-(P + steps + 1) // blk) + 1
    pk = vbs.PagedKV(B, W, L, H, D, blocks_per_sentence=S, max_blocks=MB, block=blk, dtype=dtype)
    ref = ok.PagedKV(B, W, S, L, H, D, block=blk, dtype=np.float32)
    naive = np.zeros((L, 2, R, H, P + steps + 1, D), dtype=np.float32)
    rows = torch.arange(R)
    lead = torch.tensor([b * W for b in range(B)])
    pk.prefill(P)
    ref.prefill(P)
    table = pk.table()
    for pos in range(P):
        vals = synth.kv_token_values(pos, (rows // W) * W, L, H, D, seed=seed, dtype=torch.float32)
        naive[:, :, :, :, pos, :] = vals.numpy()
        blocks = table[lead, pos // blk].long()
        pk.pool[blocks, :, :, :, pos % blk, :] = vals[:, :, lead].permute(2, 0, 1, 3, 4).to(dtype).cuda()
        ref.write(pos, vals[:, :, lead].numpy(), rows=lead.tolist())
    pk.prepare(P)
    ref.prepare(P)
    rng = np.random.default_rng(seed)
    done = np.zeros(B, dtype=bool)
    for step in range(steps):
        t_write = P + step
        table = pk.table()
        live = [r for r in range(R) if not done[r // W]]
        vals = synth.kv_token_values(t_write, rows, L, H, D, seed=seed, dtype=torch.float32)
        lr = torch.tensor(live)
        blocks = table[lr, t_write // blk].long()
        pk.pool[blocks, :, :, :, t_write % blk, :] = vals[:, :, lr].permute(2, 0, 1, 3, 4).to(dtype).cuda()
        ref.write(t_write, vals[:, :, lr].numpy(), rows=live)
        for r in live:
            naive[:, :, r, :, t_write, :] = vals[:, :, r].numpy()
        if pad_after is not None and step == pad_after:
            done[0] = True
        bi = _beam_idx(rng, B, W, pad_sentences=[b for b in range(B) if done[b]])
        t_valid = t_write + 1
        naive = ok.reorder_naive(naive, naive, bi, t_valid)
        ref.reorder(bi, t_valid)
        pk.reorder(torch.from_numpy(bi).cuda(), t_valid)
        assert pk.status() == 0
        if step % check_every == 0 or step == steps - 1:
            table = pk.table()
            rc, nb = pk.counts()
            assert int((rc > 0).sum()) == ref.blocks_in_use()
            # reference counts equal the number of table entries naming each block
            tab = table.cpu().numpy()
            nbh = nb.cpu().numpy()
            cnt = np.zeros(B * S, dtype=np.int64)
            for r in range(R):
                for i in range(nbh[r]):
                    cnt[tab[r, i]] += 1
            np.testing.assert_array_equal(rc.cpu().numpy(), cnt)
            # the logical view through the table equals the naive cache
            for r in live:
                pos = torch.arange(t_valid, device="cuda")
                bl = table[r, pos // blk].long()
                view = pk.pool[bl, :, :, :, pos % blk, :]          # [t, L, 2, H, D]
                got = view.permute(1, 2, 3, 0, 4).float().cpu().numpy()
                np.testing.assert_array_equal(got, naive[:, :, r, :, :t_valid, :], err_msg=f"row {r} step {step}")
    assert ref.copied_slots >= 0
    pk.close()
    return ref


@pytest.mark.parametrize("P,steps", [(5, 20), (16, 18), (33, 40), (1000, 20)])
def test_paged_equals_naive(P, steps):
    _paged_decode(2, 3, 2, 2, 8, P, steps, torch.bfloat16, seed=P + steps)


def test_paged_fp32_with_a_finished_sentence():
    _paged_decode(3, 4, 1, 2, 4, 7, 25, torch.float32, seed=4, pad_after=6)


def test_paged_llama_full_size():
    """64 sentences x 4 rows, 32 layers x 8 heads x 128 dims bf16 (2 MiB blocks), P = 1000, 8 steps.

    Sampled rows: the writer of every slot comes from the naive oracle applied to
    writer ids; the slot must hold exactly what that writer stored.
    """
    import verify_bs_step_gb300 as vbs
    B, W, L, H, D, P, steps, blk, seed = 64, 4, 32, 8, 128, 1000, 8, 16, 77
    R = B * W
    S = -(-P // blk) + W * 3
    MB = -(-(P + steps + 1) // blk) + 1
    pk = vbs.PagedKV(B, W, L, H, D, blocks_per_sentence=S, max_blocks=MB, block=blk, dtype=torch.bfloat16)
    ref = ok.PagedKV(B, W, S, 1, 1, 1, block=blk)          # block accounting only
    rows = torch.arange(R, device="cuda")
    lead = torch.arange(0, R, W, device="cuda")
    writer = np.zeros((1, 1, R, 1, P + steps + 1, 1), dtype=np.int64)
    writer[0, 0, :, 0, :P, 0] = (np.arange(R) // W * W)[:, None]
    pk.prefill(P)
    ref.prefill(P)
    table = pk.table()
    for pos in range(P):
        vals = synth.kv_token_values(pos, lead, L, H, D, seed=seed, device="cuda")
        pk.pool[table[lead, pos // blk].long(), :, :, :, pos % blk, :] = vals.permute(2, 0, 1, 3, 4)
    pk.prepare(P)
    ref.prepare(P)
    rng = np.random.default_rng(seed)
    for step in range(steps):
        t_write = P + step
        table = pk.table()
        vals = synth.kv_token_values(t_write, rows, L, H, D, seed=seed, device="cuda")
        pk.pool[table[rows, t_write // blk].long(), :, :, :, t_write % blk, :] = vals.permute(2, 0, 1, 3, 4)
        writer[0, 0, :, 0, t_write, 0] = np.arange(R)
        bi = _beam_idx(rng, B, W)
        writer = ok.reorder_naive(writer, writer, bi, t_write + 1)
        ref.reorder(bi, t_write + 1)
        pk.reorder(torch.from_numpy(bi).cuda(), t_write + 1)
    assert pk.status() == 0
    t_valid = P + steps
    rc, _ = pk.counts()
    assert int((rc > 0).sum()) == ref.blocks_in_use()
    table = pk.table()
    for r in (0, 5, 130, 255):
        pos = torch.arange(t_valid, device="cuda")
        got = pk.pool[table[r, pos // blk].long(), :, :, :, pos % blk, :]          # [t, L, 2, H, D]
        for p_ in (0, 1, 17, 999, 1000, t_valid - 3, t_valid - 1):
            w = int(writer[0, 0, r, 0, p_, 0])
            exp = synth.kv_token_values(p_, torch.tensor([w]), L, H, D, seed=seed)[:, :, 0]
            assert torch.equal(got[p_].cpu(), exp), (r, p_)
    pk.close()


def test_paged_pool_exhaustion_is_reported():
    import verify_bs_step_gb300 as vbs
    # room for the prompt block and nothing else: the first exclusive tail cannot be made
    pk = vbs.PagedKV(1, 4, 1, 1, 8, blocks_per_sentence=2, max_blocks=4, block=16, dtype=torch.bfloat16)
    pk.prefill(8)
    assert pk.status() == vbs.OK
    pk.prepare(8)
    assert pk.status() == vbs.ENOMEM
    pk.close()
