"""Pins of the KV-reorder oracle: naive gather, paged table with copy-on-write."""

import numpy as np
import pytest
import torch

import synth
from oracle import kv as ok


def test_naive_reorder_by_hand():
    src = np.arange(1 * 2 * 3 * 1 * 4 * 2, dtype=np.float32).reshape(1, 2, 3, 1, 4, 2)
    dst = -np.ones_like(src)
    out = ok.reorder_naive(src, dst, [2, 2, -1], 3)
    assert (out[:, :, 0, :, :3] == src[:, :, 2, :, :3]).all()
    assert (out[:, :, 1, :, :3] == src[:, :, 2, :, :3]).all()     # a parent copied twice
    assert (out[:, :, 2] == -1).all()                              # pad row untouched
    assert (out[:, :, :, :, 3:] == -1).all()                       # beyond t_valid untouched


def test_bytes_per_token_and_prompt_sharing_accounting():
    # Llama-3-8B: 2 (K,V) x 8 KV heads x 128 dims x 32 layers numbers per token, bf16
    numbers = 2 * 8 * 128 * 32
    assert numbers == 65536 and numbers * 2 == 128 * 1024
    P, t, W = 1000, 200, 4
    tok = 128 * 1024
    assert W * (P + t) * tok == 600 * 2 ** 20
    assert (P + W * t) * tok == 225 * 2 ** 20
    # the paged model after a 200-step decode stays under the shared bound + block rounding
    kv = ok.PagedKV(1, W, blocks_per_sentence=200, L=1, H=1, D=1, block=16)
    kv.prefill(P)
    kv.prepare(P)
    rng = np.random.default_rng(0)
    for step in range(t):
        parents = np.sort(rng.integers(0, W, size=W))
        kv.reorder(parents, P + step + 1)
    used = kv.blocks_in_use() * 16 * tok
    assert used <= 225 * 2 ** 20 + (W + 1) * 16 * tok
    assert kv.check_refcounts()


def _simulate(B, W, P, steps, L=2, H=2, D=4, seed=3, pad_after=None):
    """Paged vs naive on the same random decode, with the model's writes."""
    S = -(-P // 16) + W * (-(-(steps + 16) // 16) + 2)
    kv = ok.PagedKV(B, W, S, L, H, D, block=16)
    R = B * W
    Tmax = P + steps + 1
    naive = np.zeros((L, 2, R, H, Tmax, D), dtype=np.float32)
    rows = torch.arange(R)
    kv.prefill(P)
    for pos in range(P):            # the prompt: written once per sentence (rows of a sentence agree)
        vals = synth.kv_token_values(pos, (rows // W) * W, L, H, D, seed=seed, dtype=torch.float32).numpy()
        naive[:, :, :, :, pos, :] = vals
        kv.write(pos, vals[:, :, ::W], rows=[b * W for b in range(B)])
    kv.prepare(P)
    rng = np.random.default_rng(seed)
    done = np.zeros(B, dtype=bool)
    for step in range(steps):
        t_valid = P + step
        # the model writes position t_valid for every live row
        vals = synth.kv_token_values(t_valid, rows, L, H, D, seed=seed, dtype=torch.float32).numpy()
        live_rows = [r for r in range(R) if not done[r // W]]
        kv.write(t_valid, vals[:, :, live_rows], rows=live_rows)
        for r in live_rows:
            naive[:, :, r, :, t_valid, :] = vals[:, :, r]
        t_valid += 1
        if pad_after is not None and step == pad_after:
            done[0] = True
        bi = np.full(R, -1)
        for b in range(B):
            if not done[b]:
                bi[b * W:(b + 1) * W] = b * W + np.sort(rng.integers(0, W, size=W))
        naive = ok.reorder_naive(naive, naive, bi, t_valid)
        kv.reorder(bi, t_valid)
        assert kv.check_refcounts()
        lg = kv.logical(t_valid)
        for r in range(R):
            if not done[r // W]:
                assert (lg[:, :, r] == naive[:, :, r, :, :t_valid]).all()
    return kv, naive


@pytest.mark.parametrize("P,steps", [(5, 20), (16, 18), (33, 40)])
def test_paged_equals_naive(P, steps):
    _simulate(2, 3, P, steps)


def test_paged_with_a_finished_sentence():
    _simulate(2, 3, 7, 12, pad_after=4)


def test_ancestry_invariant():
    # every slot holds the value its ancestor wrote at that position
    B, W, P, steps, L, H, D, seed = 1, 3, 4, 9, 1, 1, 2, 9
    kv, naive = _simulate(B, W, P, steps, L, H, D, seed)
    # rebuild each row's ancestry from the values: each slot must equal the value written
    # by some row at that position, and the rows a slot came from form a consistent chain
    for pos in range(P + steps):
        writers = synth.kv_token_values(pos, torch.arange(B * W), L, H, D, seed=seed,
                                        dtype=torch.float32).numpy()
        for r in range(B * W):
            hit = [w for w in range(B * W) if (writers[:, :, w] == naive[:, :, r, :, pos]).all()]
            if pos < P:
                hit = [0] if (writers[:, :, 0] == naive[:, :, r, :, pos]).all() else hit
            assert hit, (pos, r)


def test_cow_copies_only_filled_slots():
    kv = ok.PagedKV(1, 4, 80, 1, 1, 1, block=16)
    kv.prefill(1000)              # 63 blocks, the last one holds 8 positions
    kv.prepare(1000)              # three rows copy the 8 filled slots of the shared tail
    assert kv.copied_slots == 3 * 8
    assert kv.blocks_in_use() == 63 + 3
    kv2 = ok.PagedKV(1, 4, 80, 1, 1, 1, block=16)
    kv2.prefill(992)              # exactly 62 full blocks: every row starts a fresh block
    kv2.prepare(992)
    assert kv2.copied_slots == 0 and kv2.blocks_in_use() == 62 + 4
