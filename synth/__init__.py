"""Seeded synthetic inputs for the beam step, the KV reorder and blockwise verify.

This module is the one thing the oracle side and the CUDA side share: it draws
random numbers and plants structure (spikes, a Zipf bias, planted EOS hits,
planted argmaxes), and nothing else.  It holds none of the method's arithmetic:
no log-softmax, no score add, no selection, no length penalty.

Every draw is a pure function of integer coordinates (seed, step, sentence,
salt), so any sentence of any step can be regenerated on its own; that is what
lets the parity tests re-salt a single sentence and lets the bench build large
device rings without touching the host.

Workload recipes (all synthetic; the pages' WMT data and trained models are not
needed and not present):

* ``tiny``  fp32 N(0, 2).
* ``tbase`` bf16 N(0, 3) with one token per row raised by +8 at a uniformly drawn
  position.
* ``llama`` bf16 N(0, 2.5) plus a Zipf bias -ln(rank) over a seeded permutation
  of the vocabulary (a frequency skew).
* ``sweep`` fp32/bf16 N(0, 2); each row independently, with probability 0.02,
  gets its EOS logit set to the row maximum + U(0.5, 2) (a planted EOS hit).
"""

from __future__ import annotations

import torch

_MASK64 = (1 << 64) - 1

SIGMA = {"tiny": 2.0, "tbase": 3.0, "llama": 2.5, "sweep": 2.0, "bpd": 2.0, "ramp": 1.0}


def mix_seed(*coords: int) -> int:
    """Fold integer coordinates into one 63-bit seed (splitmix64 finaliser)."""
    z = 0x243F6A8885A308D3
    for c in coords:
        z = (z + (int(c) & _MASK64) + 0x9E3779B97F4A7C15) & _MASK64
        z ^= z >> 30
        z = (z * 0xBF58476D1CE4E5B9) & _MASK64
        z ^= z >> 27
        z = (z * 0x94D049BB133111EB) & _MASK64
        z ^= z >> 31
    return z & ((1 << 63) - 1)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def zipf_bias(V: int, seed: int, device="cpu") -> torch.Tensor:
    """-ln(rank) over a seeded permutation of the vocabulary, fp32 [V]."""
    g = _gen(mix_seed(seed, 0x5A1F), "cpu")
    rank = torch.randperm(V, generator=g).to(torch.float64) + 1.0
    return (-torch.log(rank)).to(torch.float32).to(device)


def beam_logits(kind: str, W: int, V: int, *, seed: int, step: int, sentence: int,
                salt: int = 0, dtype=torch.float32, eos: int = -1,
                bias: torch.Tensor | None = None, device="cpu") -> torch.Tensor:
    """Logits of one sentence's W rows at one step: a [W, V] tensor of ``dtype``.

    ``bias`` is the precomputed Zipf bias for ``kind == "llama"`` (see
    :func:`zipf_bias`); ``eos`` is the token planted by ``kind == "sweep"``.
    """
    g = _gen(mix_seed(seed, step, sentence, salt), device)
    x = torch.randn(W, V, generator=g, device=device, dtype=torch.float32) * SIGMA[kind]
    if kind == "tbase":
        pos = torch.randint(0, V, (W,), generator=g, device=device)
        x[torch.arange(W, device=device), pos] += 8.0
    elif kind == "llama":
        if bias is None:
            bias = zipf_bias(V, seed, device)
        x += bias.to(device)
    elif kind == "sweep":
        if eos >= 0:
            hit = torch.rand(W, generator=g, device=device) < 0.02
            lift = 0.5 + 1.5 * torch.rand(W, generator=g, device=device)
            rowmax = x.max(dim=1).values
            x[:, eos] = torch.where(hit, rowmax + lift, x[:, eos])
    elif kind == "ramp":
        # logits rising along the vocabulary (+12 over the row): each stretch of the row
        # beats everything before it, the worst order for a running top-k threshold
        x += torch.arange(V, device=device, dtype=torch.float32) * (12.0 / V)
    elif kind not in ("tiny",):
        raise ValueError(f"unknown logits kind {kind!r}")
    return x.to(dtype)


def batch_logits(kind: str, B: int, W: int, V: int, *, seed: int, step: int,
                 salts=None, dtype=torch.float32, eos: int = -1,
                 bias: torch.Tensor | None = None, device="cpu") -> torch.Tensor:
    """Logits of a whole batch at one step, [B*W, V]; sentence b uses salt salts[b]."""
    if kind == "llama" and bias is None:
        bias = zipf_bias(V, seed, device)
    parts = [beam_logits(kind, W, V, seed=seed, step=step, sentence=b,
                         salt=0 if salts is None else int(salts[b]), dtype=dtype,
                         eos=eos, bias=bias, device=device) for b in range(B)]
    return torch.cat(parts, dim=0)


def uniform_rows(R: int, V: int, lo: float, hi: float, *, seed: int, dtype=torch.float32,
                 device="cpu") -> torch.Tensor:
    g = _gen(mix_seed(seed, 0x0417), device)
    return (lo + (hi - lo) * torch.rand(R, V, generator=g, device=device)).to(dtype)


def normal_rows(R: int, V: int, sigma: float, *, seed: int, dtype=torch.float32,
                device="cpu") -> torch.Tensor:
    g = _gen(mix_seed(seed, 0x0D15), device)
    return (torch.randn(R, V, generator=g, device=device) * sigma).to(dtype)


# ----------------------------------------------------------------------------------
# KV cache contents
# ----------------------------------------------------------------------------------

def _hash32(x: torch.Tensor) -> torch.Tensor:
    """A 32-bit integer mixer on int64 tensors (values kept in [0, 2^32))."""
    m = 0xFFFFFFFF
    x = x & m
    x = (x ^ (x >> 16)) * 0x7FEB352D & m
    x = (x ^ (x >> 15)) * 0x846CA68B & m
    return x ^ (x >> 16)


def kv_token_values(pos: int, rows: torch.Tensor, L: int, H: int, D: int, *, seed: int,
                    dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """The K and V vectors that writer rows ``rows`` store at position ``pos``.

    Returns [L, 2, len(rows), H, D] of ``dtype``.  Every value is an integer in
    [-128, 127] (exact in bf16 and fp32) drawn from a hash of
    (seed, pos, writer row, layer, k/v, head, dim), so a cached slot names the
    step and the row that wrote it.
    """
    rows = rows.to(torch.int64).to(device)
    n = rows.numel()
    idx = torch.arange(L * 2 * H * D, device=device, dtype=torch.int64).view(L, 2, 1, H, D)
    key = (idx * 0x9E3779B1 + (rows.view(1, 1, n, 1, 1) + 1) * 0x85EBCA77
           + (pos + 1) * 0xC2B2AE3D + (seed & 0xFFFFFFFF) * 0x27D4EB2F)
    h = _hash32(_hash32(key))
    val = ((h >> 8) & 0xFF).to(torch.float32) - 128.0
    return val.to(dtype)


# ----------------------------------------------------------------------------------
# Blockwise parallel decoding: a deterministic synthetic "model"
# ----------------------------------------------------------------------------------

def prefix_token(b: int, prefix: tuple, V: int, seed: int) -> int:
    """The synthetic base model's greedy token after ``prefix`` for batch element b."""
    return mix_seed(seed, 0xB0, b, len(prefix), *prefix) % V


def proposal_token(b: int, prefix: tuple, head: int, truth: int, V: int, seed: int,
                   agree: float = 0.7) -> int:
    """Proposal head ``head`` (>= 1): agrees with ``truth`` with probability ``agree``."""
    h = mix_seed(seed, 0xA1, b, head, len(prefix), *prefix)
    if (h >> 11) / float(1 << 52) < agree:
        return truth
    alt = mix_seed(seed, 0xA2, b, head, len(prefix), *prefix) % V
    return alt if alt != truth else (alt + 1) % V


def planted_rows(argmax_tokens: torch.Tensor, V: int, *, seed: int, salt: int,
                 sigma: float = 2.0, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """Noise rows N(0, sigma) whose unique argmax is planted at ``argmax_tokens``.

    ``argmax_tokens`` is an int tensor of any shape S; the result has shape S + [V].
    The planted logit is the row's noise maximum + U(0.5, 2).
    """
    shape = tuple(argmax_tokens.shape)
    n = max(1, argmax_tokens.numel())
    g = _gen(mix_seed(seed, 0xBB, salt), device)
    x = torch.randn(n, V, generator=g, device=device) * sigma
    lift = 0.5 + 1.5 * torch.rand(n, generator=g, device=device)
    top = x.max(dim=1).values + lift
    tok = argmax_tokens.reshape(-1).to(torch.int64).to(device)
    x[torch.arange(n, device=device), tok] = top
    return x.to(dtype).reshape(*shape, V) if argmax_tokens.numel() else x[:0].to(dtype).reshape(*shape, V)


def near_miss_proposals(B: int, k: int, V: int, *, seed: int, step: int, sigma: float = 2.0,
                        dtype=torch.bfloat16, device="cpu"):
    """Verify-step inputs where proposals often miss the base model's argmax narrowly.

    Every row of logits [B, k, k, V] is N(0, sigma) noise; head 0's rows get three
    planted tokens above the noise (first, second and third, spaced by a third of a
    U(0.5, 2) lift), the other heads one planted argmax.  Proposal q >= 1 is, by a
    coin, head 0's first (40 %), second (15 %) or third (10 %) token at position q-1,
    its first token +-1 or +-2 (15 %, clipped to [0, V)), or uniform (20 %).
    Returns (logits, proposals int64 [B, k]).
    """
    g_ = _gen(mix_seed(seed, 0xD1, step), "cpu")
    x = torch.randn(B, k, k, V, generator=g_) * sigma
    lift = 0.5 + 1.5 * torch.rand(B, k, k, generator=g_)
    top = x.max(dim=-1).values + lift
    tok = torch.stack([torch.randperm(V, generator=g_)[:3] for _ in range(B * k * k)]).reshape(B, k, k, 3)
    for r in range(3):
        val = top - lift * (r / 3.0)
        keep = torch.ones(B, k, k, dtype=torch.bool) if r == 0 else torch.zeros(B, k, k, dtype=torch.bool)
        keep[:, :, 0] = True
        cur = x.gather(-1, tok[..., r:r + 1]).squeeze(-1)
        x.scatter_(-1, tok[..., r:r + 1], torch.where(keep, val, cur).unsqueeze(-1))
    props = torch.randint(0, V, (B, k), generator=g_)
    coin = torch.rand(B, k, generator=g_)
    shift = torch.tensor([-2, -1, 1, 2])[torch.randint(0, 4, (B, k), generator=g_)]
    first = tok[:, :, 0, 0]
    for q in range(1, k):
        c = coin[:, q]
        near = (first[:, q - 1] + shift[:, q]).clamp(0, V - 1)
        pick = torch.where(c < 0.40, first[:, q - 1],
               torch.where(c < 0.55, tok[:, q - 1, 0, 1],
               torch.where(c < 0.65, tok[:, q - 1, 0, 2],
               torch.where(c < 0.80, near, props[:, q]))))
        props[:, q] = pick
    return x.to(dtype).to(device), props.to(device)


def geometric_prefix_proposals(B: int, k: int, V: int, *, seed: int, step: int, p: float = 0.7,
                               device="cpu"):
    """Verify-step inputs with a planted agreement structure.

    For each batch element: the base model's argmax tokens g[b, 0..k-1] (head 0 at
    positions 0..k-1) and proposals whose first entry is free and whose entries
    1..k-1 equal g[b, pos-1] while a continue-coin with probability ``p`` keeps
    landing (a geometric prefix, capped at k).  Returns (g, proposals, heads) as
    int64 tensors where heads[b, pos, h] is the planted argmax of every
    (position, head) row, with heads[:, :, 0] == g.
    """
    g_ = _gen(mix_seed(seed, 0xC0, step), "cpu")
    base = torch.randint(0, V, (B, k), generator=g_)
    heads = torch.randint(0, V, (B, k, k), generator=g_)
    heads[:, :, 0] = base
    props = torch.randint(0, V, (B, k), generator=g_)
    coins = torch.rand(B, k, generator=g_)
    for b in range(B):
        agree = True
        for q in range(1, k):
            agree = agree and bool(coins[b, q] < p)
            if agree:
                props[b, q] = base[b, q - 1]
            elif props[b, q] == base[b, q - 1]:
                props[b, q] = (props[b, q] + 1) % V
    return base.to(device), props.to(device), heads.to(device)
