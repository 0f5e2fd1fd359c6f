"""Randomised parity sweep: seeded draws of the problem shape and options (batch, length,
heads, grouped key/value heads, head dim, shard count, causal masking, layout) through
every forward and backward entry point, each against the fp64 oracle.  Sizes stay small
(the oracle evaluates every element) but are drawn to land on ragged tiles, shard edges
and sequence boundaries."""
import numpy as np
import pytest
import torch

import context_exact_attention_gb300 as cea
import oracle
from context_exact_attention_gb300.workloads import make_qkv
from helpers import assert_bf16_close, assert_f32_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
U = 2.0 ** -9


def _draw(rng, layout):
    """(B, L, H, H_kv, D, P, causal) for a layout; zigzag needs chunks of 128 rows for bf16."""
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 3]))
    H = Hkv * int(rng.choice([1, 2, 3]))
    P = int(rng.choice([1, 2, 3, 4, 5, 8]))
    if layout == "zigzag":
        L = 2 * P * 128
        return 1, L, H, Hkv, D, P, True
    L = P * int(rng.integers(1, 400 // P + 2))
    B = 1 if layout == "packed" else int(rng.integers(1, 3))
    return B, L, H, Hkv, D, P, bool(rng.integers(0, 2))


def _lengths(rng, L):
    out = []
    while sum(out) < L:
        out.append(int(rng.integers(1, max(2, L // 2))))
    out[-1] -= sum(out) - L
    return [n for n in out if n > 0]


def _positions(layout, L, P):
    return np.array(cea.zigzag_positions(L, P)) if layout == "zigzag" else np.arange(L)


def _reference(layout, q, k, v, causal, cu, pos):
    """Oracle output and lse in the tensors' row order: per sequence for packed rows, in
    position order then permuted for zigzag rows."""
    if layout == "packed":
        o = np.empty(tuple(q.shape), np.float64)
        lse = np.empty(tuple(q.shape[:2]), np.float64)
        for a, b in zip(cu[:-1], cu[1:]):
            r, lr = oracle.attention(q[None, a:b], k[None, a:b], v[None, a:b], causal=causal)
            o[a:b], lse[a:b] = r[0], lr[0]
        return o, lse
    inv = np.argsort(pos)                          # row index of each position
    qg, kg, vg = (t[:, torch.as_tensor(inv)] for t in (q, k, v))
    r, lr = oracle.attention(qg, kg, vg, causal=causal)
    return r[:, pos], lr[:, pos]


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "packed"])
@pytest.mark.parametrize("draw", range(6))
def test_random_forward(layout, draw):
    rng = np.random.default_rng(1000 * draw + {"contiguous": 0, "zigzag": 1, "packed": 2}[layout])
    B, L, H, Hkv, D, P, causal = _draw(rng, layout)
    dtype = torch.bfloat16 if draw % 3 else torch.float32
    if dtype == torch.float32 and layout == "zigzag":
        L = 2 * P * int(rng.integers(1, 40))       # fp32 has no tile constraint
    q = make_qkv(B, L, H, D, seed=200 + draw, dtype=dtype)[0]
    _, k, v = make_qkv(B, L, Hkv, D, seed=300 + draw, dtype=dtype)
    cu = None
    if layout == "packed":
        q, k, v = q[0], k[0], v[0]
        lens = _lengths(rng, L)
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV) if cu else None
    out, lse = cea.ring_attn_fwd_ex(q.to(DEV), k.to(DEV), v.to(DEV), P=P, causal=causal,
                                    layout=layout, cu_seqlens=cu_d)
    assert cea.check_status() == 0
    ref, lref = _reference(layout, q, k, v, causal, cu, _positions(layout, L, P))
    check = assert_bf16_close if dtype == torch.bfloat16 else assert_f32_close
    check(to_np(out), ref, f"out {layout} B{B} L{L} H{H}/{Hkv} D{D} P{P} causal={causal}")
    check(to_np(lse), lref, "lse")


def _grad_scale(q, k, v, do, causal, G):
    """First-order rounding scale of each gradient element (term magnitudes; see
    tests/test_gpu_bwd.py), with the key/value heads repeated for their query heads and
    dk, dv summed back over each group."""
    q, k, v, do = (np.asarray(t.float().numpy(), np.float64) for t in (q, k, v, do))
    k, v = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    B, L, H, D = q.shape
    sq, sk, sv = np.zeros_like(q), np.zeros_like(q), np.zeros_like(q)
    c = 1.0 / np.sqrt(D)
    for b in range(B):
        for h in range(H):
            s = q[b, :, h] @ k[b, :, h].T * c
            if causal:
                s = np.where(np.tril(np.ones((L, L), bool)), s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            dp = do[b, :, h] @ v[b, :, h].T
            o = p @ v[b, :, h]
            ds = p * (dp - (do[b, :, h] * o).sum(axis=1, keepdims=True))
            w = np.abs(ds) + p * np.abs(do[b, :, h] * o).sum(axis=1, keepdims=True)
            sq[b, :, h] = w @ np.abs(k[b, :, h]) * c
            sk[b, :, h] = w.T @ np.abs(q[b, :, h]) * c
            sv[b, :, h] = p.T @ np.abs(do[b, :, h])
    Hk = H // G
    return sq, sk.reshape(B, L, Hk, G, D).sum(3), sv.reshape(B, L, Hk, G, D).sum(3)


def _close(got, ref, scale, what):
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert np.isfinite(got).all(), what
    assert (err <= 2 * U * (np.abs(ref) + scale) + 1e-6).all(), (what, float(err.max()))


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "packed"])
@pytest.mark.parametrize("draw", range(4))
def test_random_backward(layout, draw):
    rng = np.random.default_rng(5000 + 1000 * draw + {"contiguous": 0, "zigzag": 1, "packed": 2}[layout])
    B, L, H, Hkv, D, P, causal = _draw(rng, layout)
    G = H // Hkv
    q = make_qkv(B, L, H, D, seed=400 + draw, dtype=torch.bfloat16)[0]
    _, k, v = make_qkv(B, L, Hkv, D, seed=500 + draw, dtype=torch.bfloat16)
    do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(600 + draw)).to(torch.bfloat16)
    pos = _positions(layout, L, P)
    inv = torch.as_tensor(np.argsort(pos))
    cu = None
    if layout == "packed":
        lens = _lengths(rng, L)
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + n)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV) if cu else None
    view = (lambda t: t[0]) if layout == "packed" else (lambda t: t)
    qd, kd, vd, dod = (view(t).to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd_ex(qd, kd, vd, P=P, causal=causal, layout=layout, cu_seqlens=cu_d)
    dq, dk, dv = cea.ring_attn_bwd_ex(qd, kd, vd, out, lse, dod, P=P, causal=causal, layout=layout,
                                      cu_seqlens=cu_d)
    assert cea.check_status() == 0
    got = [to_np(t).reshape(B, L, -1, D) for t in (dq, dk, dv)]
    segs = list(zip(cu[:-1], cu[1:])) if cu else [(0, L)]
    for a, b in segs:
        # rows of the segment, in position order
        rows = inv[a:b] if layout != "packed" else torch.arange(a, b)
        seg = [t[:, rows] for t in (q, k, v, do)]
        refs = oracle.attention_bwd_gqa(*seg, causal=causal)
        scales = _grad_scale(*seg, causal, G)
        for name, g, r, sc in zip(("dq", "dk", "dv"), got, refs, scales):
            _close(g[:, rows.numpy()], r, sc, f"{name} {layout} B{B} L{L} H{H}/{Hkv} D{D} P{P} "
                                              f"causal={causal} rows {a}:{b}")


@pytest.mark.parametrize("draw,P,c", [(0, 1, 5), (1, 2, 3), (2, 3, 2), (3, 4, 2), (4, 1, 8)])
def test_random_zigzag_backward_multi_tile_chunks(draw, P, c):
    """Zigzag backward at head dim 128 with chunks of c 128-row tiles (odd counts leave a
    lone tile at the end of each chunk: the pair-of-SMs dQ forms its pairs inside a
    chunk), with seeded draws of the query and key/value head counts."""
    rng = np.random.default_rng(9000 + draw)
    B, L, D = 1, 2 * P * 128 * c, 128
    Hkv = int(rng.choice([1, 2]))
    H = Hkv * int(rng.choice([1, 2]))
    G = H // Hkv
    q = make_qkv(B, L, H, D, seed=700 + draw, dtype=torch.bfloat16)[0]
    _, k, v = make_qkv(B, L, Hkv, D, seed=800 + draw, dtype=torch.bfloat16)
    do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(900 + draw)).to(torch.bfloat16)
    pos = _positions("zigzag", L, P)
    inv = torch.as_tensor(np.argsort(pos))
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd_ex(qd, kd, vd, P=P, causal=True, layout="zigzag")
    dq, dk, dv = cea.ring_attn_bwd_ex(qd, kd, vd, out, lse, dod, P=P, causal=True, layout="zigzag")
    assert cea.check_status() == 0
    seg = [t[:, inv] for t in (q, k, v, do)]                  # position order
    refs = oracle.attention_bwd_gqa(*seg, causal=True)
    scales = _grad_scale(*seg, True, G)
    for name, g, r, sc in zip(("dq", "dk", "dv"), (dq, dk, dv), refs, scales):
        _close(to_np(g)[:, inv.numpy()], r, sc, f"{name} zigzag L{L} H{H}/{Hkv} P{P} chunk {c} tiles")
