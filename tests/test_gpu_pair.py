"""Parity of the pair-of-SMs forward (tcgen05.mma.cta_group::2, head dim 128), which
takes contiguous, zigzag and Ulysses bf16 calls whose key walk spans at least 8192
keys: outputs and lse against the fp64 oracle on sampled query rows (every shard's
first and last rows, the rows around each 512-row quad edge and seeded uniform rows),
with ragged shards (not a multiple of the 512 rows a pair takes, nor of the 128-key
block), two batches, grouped key/value heads, zigzag shards, the ring trace, and
repeated calls bit for bit."""
import numpy as np
import pytest
import torch

import context_exact_attention_gb300 as cea
import oracle
from context_exact_attention_gb300.workloads import make_qkv, sample_rows
from helpers import assert_bf16_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _rows(L, P, n=96):
    Ls = L // P
    edges = set()
    for r in range(P):
        for e in range(0, Ls, 512):
            edges |= {r * Ls + x for x in (e - 1, e, e + 255, e + 256) if 0 <= x < Ls}
    return sorted(set(sample_rows(L, P, n, seed=3)) | edges)


def _check(q, k, v, out, lse, causal, L, P, what):
    rows = _rows(L, P)
    ref, lref = oracle.attention(q, k, v, causal=causal, rows=rows)
    assert_bf16_close(to_np(out[:, rows]), ref, f"{what} out")
    assert_bf16_close(to_np(lse[:, rows]), lref, f"{what} lse")


CASES = [
    # B, L, H, P: shards of 2048 (whole quads), 3000 (ragged quad), 4100 (ragged block),
    # then shards shorter than the four tiles a pair of CTAs takes
    (1, 8192, 2, 4),
    (2, 9000, 1, 3),
    (1, 8200, 2, 2),
    (1, 16384, 1, 1),
    (1, 8192, 1, 32),        # shards of 256: the odd CTA's two tiles lie past every shard
    (1, 8320, 1, 65),        # shards of one tile
]


@pytest.mark.parametrize("B,L,H,P", CASES)
@pytest.mark.parametrize("causal", [False, True])
def test_pair_forward_matches_oracle(B, L, H, P, causal):
    q, k, v = make_qkv(B, L, H, 128, seed=90 + L % 97, head_scale=True)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, lse = cea.ring_attn_fwd(qd, kd, vd, P=P, causal=causal)
    assert cea.check_status() == 0
    _check(q, k, v, out, lse, causal, L, P, f"B{B} L{L} H{H} P{P} causal={causal}")
    again, lagain = cea.ring_attn_fwd(qd, kd, vd, P=P, causal=causal)
    assert torch.equal(out, again) and torch.equal(lse, lagain)


def test_pair_forward_gqa_and_no_lse():
    """Four query heads over two key/value heads; the call without lse gives the same
    output bits."""
    B, L, H, Hkv, P = 1, 8192, 4, 2, 4
    q, _, _ = make_qkv(B, L, H, 128, seed=93)
    _, k, v = make_qkv(B, L, Hkv, 128, seed=94)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, lse = cea.ring_attn_fwd_gqa(qd, kd, vd, P=P, causal=True)
    _check(q, k, v, out, lse, True, L, P, "gqa")
    out2, none = cea.ring_attn_fwd_gqa(qd, kd, vd, P=P, causal=True, want_lse=False)
    assert none is None and cea.check_status() == 0
    assert torch.equal(out, out2)


@pytest.mark.parametrize("causal", [False, True])
def test_pair_forward_trace(causal):
    """The ring trace of the pair kernel: the K/V source of every (shard, ring step), -1
    where a causal step is skipped, as the oracle's ring schedule gives it (the schedule
    depends on P and causality only, so the oracle runs it on a small input)."""
    P, L = 4, 8192
    q, k, v = make_qkv(1, L, 1, 128, seed=95)
    out, lse, trace = cea.ring_attn_fwd_trace(*(t.to(DEV) for t in (q, k, v)), P=P,
                                              causal=causal)
    small = make_qkv(1, 16 * P, 1, 8, seed=95)
    _, _, tref = oracle.ring_attention(*small, P, causal=causal)
    assert np.array_equal(trace.cpu().numpy(), tref)
    _check(q, k, v, out, lse, causal, L, P, "trace call")


@pytest.mark.parametrize("seed", range(6))
def test_pair_forward_random_shapes(seed):
    """Seeded draws of batch, length (8192 to 12288 keys, any multiple of P), heads,
    grouped key/value heads, shard count and causal masking through the pair kernel, on
    sampled rows against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.choice([1, 2, 3, 4, 5, 8]))
    L = P * int(rng.integers(8192 // P + 1, 12288 // P + 1))
    Hkv = int(rng.choice([1, 2]))
    H = Hkv * int(rng.choice([1, 2]))
    B = int(rng.integers(1, 3))
    causal = bool(rng.integers(0, 2))
    q, _, _ = make_qkv(B, L, H, 128, seed=2000 + seed)
    _, k, v = make_qkv(B, L, Hkv, 128, seed=3000 + seed)
    out, lse = cea.ring_attn_fwd_gqa(*(t.to(DEV) for t in (q, k, v)), P=P, causal=causal)
    assert cea.check_status() == 0
    _check(q, k, v, out, lse, causal, L, P, f"B{B} L{L} H{H} Hkv{Hkv} P{P} causal={causal}")


@pytest.mark.parametrize("B,L,H,P", [
    (1, 8192, 2, 4),         # chunks of 1024 rows: two quads per chunk
    (1, 8960, 1, 7),         # chunks of 640 rows: a quad straddles the two chunks of a shard
    (2, 9216, 1, 3),
])
def test_pair_forward_zigzag(B, L, H, P):
    """Causal attention over the zigzag layout through the pair kernel: rows in zigzag
    order against the oracle on the position-ordered tensors (sampled rows), the ring trace
    (every shard meets every shard, its own first, each step passing on what the previous
    shard held)."""
    qg, kg, vg = make_qkv(B, L, H, 128, seed=96 + P)       # row = global position
    pos = torch.tensor(cea.zigzag_positions(L, P))
    q, k, v = (t[:, pos].contiguous() for t in (qg, kg, vg))
    out, lse, trace = cea.ring_attn_fwd_zigzag(*(t.to(DEV) for t in (q, k, v)), P=P, trace=True)
    assert cea.check_status() == 0
    rows = _rows(L, P)
    ref, lref = oracle.attention(qg, kg, vg, causal=True, rows=pos[rows].tolist())
    assert_bf16_close(to_np(out[:, rows]), ref, "zigzag out")
    assert_bf16_close(to_np(lse[:, rows]), lref, "zigzag lse")
    tr = trace.cpu().numpy()
    for r in range(P):
        assert sorted(tr[r].tolist()) == list(range(P)) and tr[r, 0] == r
        for t in range(1, P):
            assert tr[r, t] == tr[(r - 1) % P, t - 1]


def test_pair_forward_zigzag_grouped_heads():
    """Zigzag shards with four query heads over two key/value heads (the descriptor entry
    point), on sampled rows against the oracle on the position-ordered tensors."""
    B, L, H, Hkv, P = 1, 8192, 4, 2, 4
    qg, _, _ = make_qkv(B, L, H, 128, seed=97)
    _, kg, vg = make_qkv(B, L, Hkv, 128, seed=98)
    pos = torch.tensor(cea.zigzag_positions(L, P))
    q, k, v = (t[:, pos].contiguous().to(DEV) for t in (qg, kg, vg))
    out, lse = cea.ring_attn_fwd_ex(q, k, v, P=P, causal=True, layout="zigzag")
    assert cea.check_status() == 0
    rows = _rows(L, P)
    ref, lref = oracle.attention(qg, kg, vg, causal=True, rows=pos[rows].tolist())
    assert_bf16_close(to_np(out[:, rows]), ref, "zigzag gqa out")
    assert_bf16_close(to_np(lse[:, rows]), lref, "zigzag gqa lse")
