"""Parity at the full sizes of the five workloads, in the launch configuration the
benchmark times: outputs compared with the fp64 oracle on sampled query rows (the first
and last row of every shard plus seeded uniform rows), element-wise merges and
bit-exact transposes over the whole tensors, and determinism over repeated calls."""
import numpy as np
import pytest
import torch

import context_exact_attention_gb300 as cea
import oracle
from context_exact_attention_gb300.workloads import (DIT, LM, LONG, ULYSSES, make_qkv,
                                                     make_workload_inputs, sample_rows)
from helpers import BF16_TOL, assert_bf16_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
U = 2.0 ** -9


def _check_rows(w, out, lse, q, k, v, n_rows):
    rows = sample_rows(w.L, w.P, n_rows, seed=1)
    ref, lref = oracle.attention(q, k, v, causal=w.causal, rows=rows)
    got = to_np(out[:, rows])
    assert_bf16_close(got, ref, f"{w.name} out")
    assert_bf16_close(to_np(lse[:, rows]), lref, f"{w.name} lse")


def _key_rows_close(q, k, v, do, dk, dv, key_rows, q_heads, kv_head, causal, what):
    """dk and dv of key/value head `kv_head` on the key rows `key_rows`, against the fp64
    oracle's key-row routine, element by element.  q, do: CPU [L, H, D]; k, v: CPU
    [L, H_kv, D]; dk, dv: the GPU's [L, H_kv, D] (fp64 numpy), rows in the same order as
    k.  `q_heads` are the query heads reading this key/value head: the reference is the
    sum of their per-head gradients (one head: plain attention).

    Bound: the first-order rounding bound of tests/test_gpu_bwd.py, 2u (|ref| + scale) +
    1e-6 with u = 2^-9, where the scale sums the magnitudes of each element's terms from
    the oracle's own fp64 quantities (P_ij from its lse, the Dvec error term from its
    output O): scale(dk_j) = sum_i (|dS_ij| + P_ij sum_d |dO_id O_id|) |q_i| / sqrt(D),
    scale(dv_j) = sum_i P_ij |dO_i|."""
    G = len(q_heads)
    qs, ds = q[None, :, q_heads], do[None, :, q_heads]
    ks, vs = k[None, :, [kv_head] * G], v[None, :, [kv_head] * G]
    rk, rv, lse, o = oracle.attention_bwd_dkdv_rows(qs, ks, vs, ds, key_rows, causal=causal,
                                                    stats=True)
    ref_k, ref_v = rk[0].sum(axis=1), rv[0].sum(axis=1)          # [n, D]
    qf, kf, vf, dof = (oracle.to_f64(t)[0] for t in (qs, ks, vs, ds))
    L, D = qf.shape[0], qf.shape[2]
    c = 1.0 / np.sqrt(D)
    sk, sv = np.zeros_like(ref_k), np.zeros_like(ref_v)
    for g in range(G):
        rowdot = (dof[:, g] * o[0, :, g]).sum(axis=-1)
        dvec_abs = np.abs(dof[:, g] * o[0, :, g]).sum(axis=-1)
        for ri, j in enumerate(key_rows):
            i0 = j if causal else 0
            p = np.exp(qf[i0:, g] @ kf[j, g] * c - lse[0, i0:, g])
            dsij = p * (dof[i0:, g] @ vf[j, g] - rowdot[i0:])
            sk[ri] += (np.abs(dsij) + p * dvec_abs[i0:]) @ np.abs(qf[i0:, g]) * c
            sv[ri] += p @ np.abs(dof[i0:, g])
    for name, got, ref, scale in (("dk", dk[key_rows, kv_head], ref_k, sk),
                                  ("dv", dv[key_rows, kv_head], ref_v, sv)):
        assert np.isfinite(got).all(), (what, name)
        err = np.abs(got - ref)
        worst = (err / (2 * U * (np.abs(ref) + scale) + 1e-6)).max()
        p3 = (err / (BF16_TOL + BF16_TOL * np.abs(ref))).max()
        print(f"{what} {name} key rows: worst/bound {worst:.3f}, p3 criterion ratio {p3:.3f}")
        assert worst <= 1.0, (what, name, worst)


def test_dit_full_attention_40_calls():
    """Non-causal B=1 H=24 L=4096 D=128 P=4, 40 calls (denoising steps): every call
    bit-identical to the first, and the result matches the oracle on 256 rows x 24 heads."""
    w = DIT
    q, k, v = make_workload_inputs(w, seed=0)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    first, lfirst = cea.ring_attn_fwd(qd, kd, vd, P=w.P, causal=False)
    out, lse = torch.empty_like(first), torch.empty_like(lfirst)
    for _ in range(w.repeats - 1):
        cea.ring_attn_fwd(qd, kd, vd, P=w.P, causal=False, out=out, lse=lse)
        assert torch.equal(out, first) and torch.equal(lse, lfirst)
    assert cea.check_status() == 0
    _check_rows(w, first, lfirst, q, k, v, 256)


def test_causal_lm_full_size():
    """Causal B=1 H=32 L=32768 D=128 P=8 with per-head score scales: 96 rows x 32 heads."""
    w = LM
    q, k, v = make_workload_inputs(w, seed=0)
    out, lse = cea.ring_attn_fwd(*(t.to(DEV) for t in (q, k, v)), P=w.P, causal=True)
    assert cea.check_status() == 0
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    _check_rows(w, out, lse, q, k, v, 96)


def test_long_context_full_size():
    """Causal B=1 H=8 L=131072 D=128 P=8: 512 sampled rows per head."""
    w = LONG
    q, k, v = make_workload_inputs(w, seed=0)
    out, lse = cea.ring_attn_fwd(*(t.to(DEV) for t in (q, k, v)), P=w.P, causal=True)
    assert cea.check_status() == 0
    assert torch.isfinite(out).all()
    _check_rows(w, out, lse, q, k, v, 512)


def test_ulysses_full_size():
    """B=2 L=8192 H=32 D=128 P=8: the three seq->head transposes are bit-exact against
    the oracle, the head->seq result of full attention per head group matches the
    oracle's attention of the global tensors on 64 rows x 64 (batch, head) pairs, and the
    fused one-kernel step gives the same bits."""
    w = ULYSSES
    q, k, v = make_workload_inputs(w, seed=0)
    Ls = w.L // w.P
    to_seq = lambda t: torch.stack([t[:, r * Ls:(r + 1) * Ls] for r in range(w.P)]).contiguous()
    qs, ks, vs = (to_seq(t) for t in (q, k, v))
    head = cea.ulysses_seq2head(qs.to(DEV), w.P)
    ref_head = oracle.seq2head(qs.view(torch.int16).numpy(), w.P)
    assert np.array_equal(head.cpu().view(torch.int16).numpy(), ref_head)
    o_seq = cea.ulysses_attention(qs.to(DEV), ks.to(DEV), vs.to(DEV), w.P)
    assert cea.check_status() == 0
    glob = torch.cat([o_seq[r] for r in range(w.P)], dim=1)      # [B, L, H, D]
    rows = sample_rows(w.L, w.P, 64, seed=1)
    ref, _ = oracle.attention(q, k, v, causal=False, rows=rows)
    assert_bf16_close(to_np(glob[:, rows]), ref, "ulysses out")
    back = cea.ulysses_head2seq(head, w.P)
    assert torch.equal(back.cpu(), qs)
    # the fused step (transposes folded into the attention's addressing): the same bits
    fused, _ = cea.ulysses_attention_fused(qs.to(DEV), ks.to(DEV), vs.to(DEV), w.P)
    assert cea.check_status() == 0
    assert torch.equal(fused, o_seq)


def test_merge_causal_lm_size():
    """Two partials of 1,048,576 rows x 128 (bf16 o, fp32 lse): the GPU merge against the
    oracle's, element by element over the whole tensors, and in place."""
    rows, D = LM.B * LM.L * LM.H, LM.D
    g = torch.Generator().manual_seed(3)
    oa = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    ob = torch.randn(rows, D, generator=g).to(torch.bfloat16)
    la = torch.randn(rows, generator=g) * 4
    lb = torch.randn(rows, generator=g) * 4
    ref, lref = oracle.merge(oa, la, ob, lb)
    oad, lad = oa.to(DEV), la.to(DEV)
    cea.attn_merge_partials(oad, lad, ob.to(DEV), lb.to(DEV), o_out=oad, lse_out=lad)
    assert_bf16_close(to_np(oad), ref, "merge o")
    assert_bf16_close(to_np(lad), lref, "merge lse")


def test_variants_at_causal_lm_size():
    """The causal-LM size (L=32768, D=128, P=8) through the grouped-head, zigzag and
    packed-sequence entry points, on sampled query rows."""
    w = LM
    rows = sample_rows(w.L, w.P, 48, seed=1)
    # grouped key/value heads: 16 query heads over 4 key/value heads
    q, _, _ = make_qkv(1, w.L, 16, w.D, seed=3, dtype=torch.bfloat16)
    _, k, v = make_qkv(1, w.L, 4, w.D, seed=4, dtype=torch.bfloat16)
    out, lse = cea.ring_attn_fwd_gqa(*(t.to(DEV) for t in (q, k, v)), P=w.P, causal=True)
    ref, lref = oracle.attention(q, k, v, causal=True, rows=rows)
    assert_bf16_close(to_np(out[:, rows]), ref, "gqa out")
    assert_bf16_close(to_np(lse[:, rows]), lref, "gqa lse")
    # zigzag: rows are in zigzag order, the oracle sees position order
    qg, kg, vg = make_qkv(1, w.L, 8, w.D, seed=5, dtype=torch.bfloat16)
    pos = torch.tensor(cea.zigzag_positions(w.L, w.P))
    out, lse = cea.ring_attn_fwd_zigzag(*(t[:, pos].contiguous().to(DEV) for t in (qg, kg, vg)),
                                        P=w.P)
    ref, lref = oracle.attention(qg, kg, vg, causal=True, rows=pos[rows].tolist())
    assert_bf16_close(to_np(out[:, rows]), ref, "zigzag out")
    assert_bf16_close(to_np(lse[:, rows]), lref, "zigzag lse")
    # packed sequences
    g = torch.Generator().manual_seed(6)
    lengths = []
    while sum(lengths) < w.L:
        lengths.append(int(torch.randint(1, 9000, (1,), generator=g)))
    lengths[-1] -= sum(lengths) - w.L
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    q, k, v = (t[0] for t in make_qkv(1, w.L, 8, w.D, seed=7, dtype=torch.bfloat16))
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, lse = cea.ring_attn_fwd_varlen(qd, kd, vd, cu_d, P=w.P, causal=True)
    # the heaviest-first schedule changes which CTA takes which unit, not the bits
    sched = cea.varlen_schedule(cu_d, w.L, w.P, True)
    out_s, lse_s = cea.ring_attn_fwd_varlen(qd, kd, vd, cu_d, P=w.P, causal=True, schedule=sched)
    assert cea.check_status() == 0
    assert torch.equal(out, out_s) and torch.equal(lse, lse_s)
    got, lg = to_np(out), to_np(lse)
    for a, b in zip(cu[:-1], cu[1:]):
        pick = [i - a for i in rows if a <= i < b]
        if not pick:
            continue
        ref, lref = oracle.attention(q[None, a:b], k[None, a:b], v[None, a:b], causal=True,
                                     rows=pick)
        assert_bf16_close(got[[a + i for i in pick]], ref[0], f"varlen rows in {a}:{b}")
        assert_bf16_close(lg[[a + i for i in pick]], lref[0], f"varlen lse in {a}:{b}")


def test_backward_at_causal_lm_size():
    """Backward at the causal-LM size (8 heads): identities that hold at any size -- the
    sum of dv over keys equals the sum of dout over queries, the sum of dk over keys is
    zero -- within the accumulated bf16 rounding, dq on sampled rows against the fp64
    chain rule for those rows (one query row needs only its own scores), and dk, dv on
    sampled key rows of two heads against the oracle's key-row routine."""
    w = LM
    H = 8
    q, k, v = make_qkv(1, w.L, H, w.D, seed=8, dtype=torch.bfloat16, head_scale=True)
    do = torch.randn(1, w.L, H, w.D, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd(qd, kd, vd, P=w.P, causal=True)
    dq, dk, dv = cea.ring_attn_bwd(qd, kd, vd, out, lse, dod, P=w.P, causal=True)
    assert cea.check_status() == 0
    u = 2.0 ** -9
    sdv = dv.double().sum(1).cpu().numpy()
    sdo = do.double().sum(1).numpy()
    bound = 4 * u * dv.double().abs().sum(1).cpu().numpy() + 1e-3
    assert (np.abs(sdv - sdo) <= bound).all()
    sdk = dk.double().sum(1).cpu().numpy()
    assert (np.abs(sdk) <= 4 * u * dk.double().abs().sum(1).cpu().numpy() + 1e-3).all()
    # sampled dq rows against the oracle; the error scale is the first-order rounding bound
    # of tests/test_gpu_bwd.py (term magnitudes of each element), from fp64 quantities
    rows = sample_rows(w.L, w.P, 24, seed=2)
    ref = oracle.attention_bwd_dq_rows(q, k, v, do, rows, causal=True)
    qf, kf, vf, dof = (t.double().numpy()[0] for t in (q, k, v, do))
    c = 1.0 / np.sqrt(w.D)
    for ri, i in enumerate(rows):
        for h in range(H):
            s = kf[:i + 1, h] @ qf[i, h] * c
            p = np.exp(s - s.max())
            p /= p.sum()
            dp = vf[:i + 1, h] @ dof[i, h]
            ds = p * (dp - (p * dp).sum())
            dvec_err = np.abs(dof[i, h] * (p @ vf[:i + 1, h])).sum()
            scale = (np.abs(ds) + p * dvec_err) @ np.abs(kf[:i + 1, h]) * c
            got = dq[0, i, h].double().cpu().numpy()
            r = ref[0, ri, h]
            assert (np.abs(got - r) <= 2 * u * (np.abs(r) + scale) + 1e-6).all(), (i, h)
    # dk, dv element-wise on sampled key rows (shard edges and seeded rows) of two heads
    key_rows = sample_rows(w.L, w.P, 24, seed=12)
    dkn, dvn = (t[0].double().cpu().numpy() for t in (dk, dv))
    for h in (1, 6):
        _key_rows_close(q[0], k[0], v[0], do[0], dkn, dvn, key_rows, [h], h, True, f"head {h}")


def test_grouped_backward_at_causal_lm_size():
    """Grouped backward at the causal-LM length (8 query heads over 2 key/value heads):
    sum of dv over keys per key/value head equals the sum of dout over queries and the
    group's query heads, sum of dk over keys is zero, dq on sampled rows matches the
    fp64 chain rule through the repeated heads, and dk, dv of one key/value head on
    sampled key rows match the oracle summed over the group's query heads."""
    w = LM
    H, Hkv = 8, 2
    G = H // Hkv
    q, _, _ = make_qkv(1, w.L, H, w.D, seed=50, dtype=torch.bfloat16, head_scale=True)
    _, k, v = make_qkv(1, w.L, Hkv, w.D, seed=51, dtype=torch.bfloat16)
    do = torch.randn(1, w.L, H, w.D, generator=torch.Generator().manual_seed(52)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd_gqa(qd, kd, vd, P=w.P, causal=True)
    dq, dk, dv = cea.ring_attn_bwd_gqa(qd, kd, vd, out, lse, dod, P=w.P, causal=True)
    assert cea.check_status() == 0
    u = 2.0 ** -9
    sdv = dv.double().sum(1).cpu().numpy()                                   # [1, Hkv, D]
    sdo = do.double().sum(1).numpy().reshape(1, Hkv, G, w.D).sum(axis=2)
    assert (np.abs(sdv - sdo) <= 4 * u * dv.double().abs().sum(1).cpu().numpy() + 1e-3).all()
    sdk = dk.double().sum(1).cpu().numpy()
    assert (np.abs(sdk) <= 4 * u * dk.double().abs().sum(1).cpu().numpy() + 1e-3).all()
    rows = sample_rows(w.L, w.P, 12, seed=3)
    kr, vr = k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2)
    ref = oracle.attention_bwd_dq_rows(q, kr, vr, do, rows, causal=True)
    got = to_np(dq[:, rows]).astype(np.float64)
    scale = np.abs(ref).max(axis=-1, keepdims=True)
    assert np.isfinite(got).all()
    # relative to each row's largest component: the first-order bound of the plain
    # backward's full-size test, taken conservatively per row
    assert (np.abs(got - ref) <= 4 * u * (np.abs(ref) + scale) + 1e-5).all()
    # dk, dv of key/value head 1 (the sum over its four query heads) on sampled key rows
    key_rows = sample_rows(w.L, w.P, 16, seed=13)
    dkn, dvn = (t[0].double().cpu().numpy() for t in (dk, dv))
    _key_rows_close(q[0], k[0], v[0], do[0], dkn, dvn, key_rows, list(range(G, 2 * G)), 1, True,
                    "grouped")


def _dq_row_bound(q, k, v, do, i, h, keys, D):
    """First-order rounding scale of dq[i, h] (term magnitudes, fp64), over the key rows
    `keys` that query row i sees."""
    c = 1.0 / np.sqrt(D)
    kk, vv = k[keys, h], v[keys, h]
    s = kk @ q[i, h] * c
    p = np.exp(s - s.max())
    p /= p.sum()
    dp = vv @ do[i, h]
    ds = p * (dp - (p * dp).sum())
    dvec_err = np.abs(do[i, h] * (p @ vv)).sum()
    return (np.abs(ds) + p * dvec_err) @ np.abs(kk) * c


def test_zigzag_backward_at_causal_lm_size():
    """Zigzag backward at the causal-LM size (8 heads): the sum identities over all rows,
    agreement with the contiguous layout's backward after the permutation, dq on sampled
    rows against the fp64 chain rule in position order, and dk, dv on sampled key rows
    of one head against the oracle's key-row routine in position order."""
    w = LM
    H = 8
    u = 2.0 ** -9
    qg, kg, vg = make_qkv(1, w.L, H, w.D, seed=60, dtype=torch.bfloat16, head_scale=True)
    dog = torch.randn(1, w.L, H, w.D, generator=torch.Generator().manual_seed(61)).to(torch.bfloat16)
    pos = torch.tensor(cea.zigzag_positions(w.L, w.P))
    q, k, v, do = (t[:, pos].contiguous().to(DEV) for t in (qg, kg, vg, dog))
    out, lse = cea.ring_attn_fwd_zigzag(q, k, v, P=w.P)
    dq, dk, dv = cea.ring_attn_bwd_zigzag(q, k, v, out, lse, do, P=w.P)
    assert cea.check_status() == 0
    sdv = dv.double().sum(1).cpu().numpy()
    assert (np.abs(sdv - dog.double().sum(1).numpy())
            <= 4 * u * dv.double().abs().sum(1).cpu().numpy() + 1e-3).all()
    assert (np.abs(dk.double().sum(1).cpu().numpy())
            <= 4 * u * dk.double().abs().sum(1).cpu().numpy() + 1e-3).all()
    # the contiguous layout's backward of the same problem, rows permuted
    gd = [t.to(DEV) for t in (qg, kg, vg, dog)]
    o2, l2 = cea.ring_attn_fwd(*gd[:3], P=w.P, causal=True)
    ref_layout = cea.ring_attn_bwd(*gd[:3], o2, l2, gd[3], P=w.P, causal=True)
    pd = pos.to(DEV)
    for name, a, z in zip(("dq", "dk", "dv"), ref_layout, (dq, dk, dv)):
        a, z = a[:, pd].double(), z.double()
        rel = float((a - z).norm() / a.norm())
        assert rel <= 4 * u, (name, rel)
    # sampled dq rows (zigzag row index -> position) against the oracle
    rows = sample_rows(w.L, w.P, 12, seed=4)
    prow = pos[rows].tolist()
    ref = oracle.attention_bwd_dq_rows(qg, kg, vg, dog, prow, causal=True)
    qf, kf, vf, dof = (t.double().numpy()[0] for t in (qg, kg, vg, dog))
    for ri, (i, pi) in enumerate(zip(rows, prow)):
        for h in range(H):
            scale = _dq_row_bound(qf, kf, vf, dof, pi, h, slice(0, pi + 1), w.D)
            got = dq[0, i, h].double().cpu().numpy()
            r = ref[0, ri, h]
            assert (np.abs(got - r) <= 2 * u * (np.abs(r) + scale) + 1e-6).all(), (i, h)
    # dk, dv on sampled key rows (zigzag row index -> position) of one head
    key_rows = sample_rows(w.L, w.P, 16, seed=14)
    order = np.argsort(pos.numpy())                 # position -> zigzag row
    dkn, dvn = (t[0, torch.from_numpy(order).to(DEV)].double().cpu().numpy() for t in (dk, dv))
    _key_rows_close(qg[0], kg[0], vg[0], dog[0], dkn, dvn, pos[key_rows].tolist(), [3], 3, True,
                    "zigzag head 3")


def test_packed_backward_at_causal_lm_size():
    """Packed-sequence backward at the causal-LM length (8 heads, lengths as in the
    forward's full-size test): per sequence, the sum of dv over its keys equals the sum
    of dout over its queries and the sum of dk is zero; dq on sampled rows and dk, dv on
    sampled key rows (each sequence's first and last among them) of every sequence
    against the fp64 chain rule of that sequence alone."""
    w = LM
    H = 8
    u = 2.0 ** -9
    g = torch.Generator().manual_seed(6)
    lengths = []
    while sum(lengths) < w.L:
        lengths.append(int(torch.randint(1, 9000, (1,), generator=g)))
    lengths[-1] -= sum(lengths) - w.L
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    q, k, v = (t[0] for t in make_qkv(1, w.L, H, w.D, seed=62, dtype=torch.bfloat16,
                                      head_scale=True))
    do = torch.randn(w.L, H, w.D, generator=torch.Generator().manual_seed(63)).to(torch.bfloat16)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd_varlen(qd, kd, vd, cu_d, P=w.P, causal=True)
    dq, dk, dv = cea.ring_attn_bwd_varlen(qd, kd, vd, out, lse, dod, cu_d, P=w.P, causal=True)
    sched = cea.varlen_schedule(cu_d, w.L, w.P, True)
    scheduled = cea.ring_attn_bwd_varlen(qd, kd, vd, out, lse, dod, cu_d, P=w.P, causal=True,
                                         schedule=sched)
    assert cea.check_status() == 0
    for a, b in zip((dq, dk, dv), scheduled):
        assert torch.equal(a, b)
    dqn, dkn, dvn = (t.double().cpu().numpy() for t in (dq, dk, dv))
    qf, kf, vf, dof = (t.double().numpy() for t in (q, k, v, do))
    rows = sample_rows(w.L, w.P, 24, seed=5)
    for a, b in zip(cu[:-1], cu[1:]):
        sdv, sdo = dvn[a:b].sum(0), dof[a:b].sum(0)
        assert (np.abs(sdv - sdo) <= 4 * u * np.abs(dvn[a:b]).sum(0) + 1e-3).all(), (a, b)
        assert (np.abs(dkn[a:b].sum(0)) <= 4 * u * np.abs(dkn[a:b]).sum(0) + 1e-3).all(), (a, b)
        pick = [i for i in rows if a <= i < b]
        if not pick:
            continue
        ref = oracle.attention_bwd_dq_rows(q[None, a:b], k[None, a:b], v[None, a:b],
                                           do[None, a:b], [i - a for i in pick], causal=True)
        for ri, i in enumerate(pick):
            for h in range(H):
                scale = _dq_row_bound(qf, kf, vf, dof, i, h, slice(a, i + 1), w.D)
                r = ref[0, ri, h]
                assert (np.abs(dqn[i, h] - r) <= 2 * u * (np.abs(r) + scale) + 1e-6).all(), (i, h)
    # dk, dv on sampled key rows of every sequence, two heads, that sequence alone
    key_rows = sample_rows(w.L, w.P, 32, seed=15)
    for a, b in zip(cu[:-1], cu[1:]):
        pick = [j - a for j in key_rows if a <= j < b] + [0, b - a - 1]
        pick = sorted(set(pick))
        for h in (2, 5):
            _key_rows_close(q[a:b], k[a:b], v[a:b], do[a:b], dkn[a:b], dvn[a:b], pick, [h], h,
                            True, f"sequence {a}:{b} head {h}")


def test_max_length_forward():
    """L = 2^20 (one head, D = 128, P = 8 shards of 131072, causal): positions, tile
    indices and row offsets far beyond the benchmark sizes in the kernels' index arithmetic;
    sampled rows (shard edges included) against the oracle."""
    B, L, H, D, P = 1, 1 << 20, 1, 128, 8
    q, k, v = make_qkv(B, L, H, D, seed=7, dtype=torch.bfloat16)
    out, lse = cea.ring_attn_fwd(*(t.to(DEV) for t in (q, k, v)), P=P, causal=True)
    assert cea.check_status() == 0
    rows = sample_rows(L, P, 48, seed=3)
    ref, lref = oracle.attention(q, k, v, causal=True, rows=rows)
    assert_bf16_close(to_np(out[:, rows]), ref, "out")
    assert_bf16_close(to_np(lse[:, rows]), lref, "lse")
