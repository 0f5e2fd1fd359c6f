"""GPU parity of the backward (dq, dk, dv) against the fp64 gradient oracle.

Tolerance.  A first-order rounding bound, element by element.  Every gradient
element is a sum of terms whose bf16 operands carry one rounding each (unit
roundoff u = 2^-9): dq_i = sum_j dS_ij k_j / sqrt(D) and dk_j = sum_i dS_ij q_i /
sqrt(D) with dS rounded; dv_j = sum_i P_ij dO_i with P rounded; and every dS_ij
of row i also carries the error of Dvec_i = dO_i . O_i computed from the bf16
output O, |dDvec_i| <= u sum_d |dO_id O_id|.  Accumulation is fp32 (negligible)
and the result is rounded to bf16 once.  So, with magnitudes taken from exact
fp64 quantities,
  |err(dq_id)| <= u |dq_id| + u sum_j (|dS_ij| + P_ij u^-1 |dDvec_i|) |k_jd| / sqrt(D)
and likewise for dk (sum over queries, q) and dv (sum_i P_ij |dO_id|).  The test
allows twice that, plus 1e-6.  Early causal query rows, which sum a few large
and cancelling terms, are where the term magnitudes matter: there an error of
several times the result's own rounding is still exact arithmetic on bf16
operands.  Norm-wise, ||got - ref|| <= 4u ||ref|| and cosine > 0.9999.

Beside the bound every check prints the bf16 criterion of the precision page
(|err| <= 5e-3 + 5e-3 |ref|, stated there for forward outputs) as the ratio
max |err| / (5e-3 + 5e-3 |ref|).  Without causal masking the gradients meet it,
and the plain, grouped-head and packed parity tests assert it; with causal
masking the early rows' cancellation takes some elements past it while the
first-order bound holds.
"""
import numpy as np
import pytest
import torch

import context_exact_attention_gb300 as cea
import oracle
from context_exact_attention_gb300.workloads import make_qkv
from helpers import BF16_TOL, cosine, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
U = 2.0 ** -9


def _term_scales(q, k, v, do, causal):
    """Magnitude sums of the terms behind each gradient element (see the module
    docstring), from fp64 copies of the inputs: an error scale, not a reference."""
    q, k, v, do = (np.asarray(t.float().numpy(), np.float64) for t in (q, k, v, do))
    B, L, H, D = q.shape
    sq, sk, sv = np.zeros_like(q), np.zeros_like(q), np.zeros_like(q)
    c = 1.0 / np.sqrt(D)
    for b in range(B):
        for h in range(H):
            qq, kk, vv, dd = q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h]
            s = qq @ kk.T * c
            if causal:
                s = np.where(np.tril(np.ones((L, L), bool)), s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            dp = dd @ vv.T
            o = p @ vv
            ds = p * (dp - (dd * o).sum(axis=1, keepdims=True))
            ddvec = np.abs(dd * o).sum(axis=1, keepdims=True)          # |dDvec_i| / u
            w = np.abs(ds) + p * ddvec
            sq[b, :, h] = w @ np.abs(kk) * c
            sk[b, :, h] = w.T @ np.abs(qq) * c
            sv[b, :, h] = p.T @ np.abs(dd)
    return sq, sk, sv


def _grad_close(got, ref, what, scale, p3_holds=False):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), what
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    worst = (err / (2 * U * (np.abs(ref) + scale) + 1e-6)).max()
    # the precision page's bf16 criterion (atol = rtol = 5e-3), reported beside the bound
    p3 = (err / (BF16_TOL + BF16_TOL * np.abs(ref))).max()
    print(f"{what}: rel_l2 {rel:.2e} cos {cosine(got, ref):.7f} worst/bound {worst:.3f} "
          f"p3 ratio {p3:.3f}")
    if p3_holds:
        # without causal masking no row sums a few large cancelling terms, and the
        # gradients also meet the page's forward criterion
        assert p3 <= 1.0, (what, p3)
    assert rel <= 4 * U, (what, rel)
    assert cosine(got, ref) > 0.9999, what
    assert worst <= 1.0, (what, worst)


CASES = [
    # B, L, H, D, P
    (1, 256, 2, 128, 1),
    (1, 512, 2, 128, 4),
    (2, 384, 2, 128, 2),     # shard of 192: ragged tiles on both sides
    (1, 192, 1, 64, 3),      # shard of 64
    (1, 640, 2, 64, 5),
    (1, 1024, 2, 128, 8),
    (1, 1280, 2, 128, 2),    # 5 tiles per shard: the last pair of query tiles has one
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%dL%dH%dD%dP%d" % c)
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_parity(case, causal):
    B, L, H, D, P = case
    q, k, v = make_qkv(B, L, H, D, seed=20, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(21)
    do = torch.randn(B, L, H, D, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd(qd, kd, vd, P=P, causal=causal)
    dq, dk, dv = cea.ring_attn_bwd(qd, kd, vd, out, lse, dod, P=P, causal=causal)
    assert cea.check_status() == 0
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=causal)
    sq, sk, sv = _term_scales(q, k, v, do, causal)
    _grad_close(to_np(dq), rq, "dq", sq, p3_holds=not causal)
    _grad_close(to_np(dk), rk, "dk", sk, p3_holds=not causal)
    _grad_close(to_np(dv), rv, "dv", sv, p3_holds=not causal)


def test_bwd_deterministic_and_spread_scores():
    """Per-head score scales up to 4: peaked softmax; two calls give identical bits."""
    B, L, H, D, P = 1, 1024, 4, 128, 4
    q, k, v = make_qkv(B, L, H, D, seed=22, dtype=torch.bfloat16, head_scale=True)
    do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(23)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd(qd, kd, vd, P=P, causal=True)
    first = cea.ring_attn_bwd(qd, kd, vd, out, lse, dod, P=P, causal=True)
    again = cea.ring_attn_bwd(qd, kd, vd, out, lse, dod, P=P, causal=True)
    for a, b in zip(first, again):
        assert torch.equal(a, b)
    ref = oracle.attention_bwd(q, k, v, do, causal=True)
    scales = _term_scales(q, k, v, do, True)
    for name, got, r, sc in zip(("dq", "dk", "dv"), first, ref, scales):
        _grad_close(to_np(got), r, name, sc)


def test_bwd_argument_errors():
    q, k, v = (t.to(DEV) for t in make_qkv(1, 256, 2, 128, seed=0, dtype=torch.bfloat16))
    out, lse = cea.ring_attn_fwd(q, k, v, P=2)
    lib = cea.load_library()
    assert lib.ring_attn_bwd_workspace_bytes(1, 256, 2) == 256 * 2 * 4
    small = torch.empty(10, dtype=torch.float32, device=DEV)
    with pytest.raises(cea.RingAttnError) as e:
        cea.ring_attn_bwd(q, k, v, out, lse, q.clone(), P=2, workspace=small)
    assert e.value.code == 1
    with pytest.raises(cea.RingAttnError) as e:
        cea.ring_attn_bwd(q, k, v, out, lse, q.clone(), P=3)
    assert e.value.code == 4


# ------------------------------------------------- grouped key/value heads --

GQA_CASES = [
    # B, L, H, H_kv, D, P
    (1, 512, 4, 2, 128, 4),
    (2, 384, 6, 3, 64, 2),      # shards of 192: ragged tiles
    (1, 256, 4, 1, 128, 1),     # one key/value head (multi-query)
    (1, 640, 8, 2, 64, 5),
]


@pytest.mark.parametrize("case", GQA_CASES, ids=lambda c: "B%dL%dH%dHkv%dD%dP%d" % c)
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_gqa_parity(case, causal):
    """dk, dv of each key/value head sum the gradients of its query heads: against the
    grouped fp64 oracle, with the rounding bound of each query head's terms summed over
    the group."""
    B, L, H, Hkv, D, P = case
    q, _, _ = make_qkv(B, L, H, D, seed=40, dtype=torch.bfloat16)
    _, k, v = make_qkv(B, L, Hkv, D, seed=41, dtype=torch.bfloat16)
    do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(42)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd_gqa(qd, kd, vd, P=P, causal=causal)
    dq, dk, dv = cea.ring_attn_bwd_gqa(qd, kd, vd, out, lse, dod, P=P, causal=causal)
    assert cea.check_status() == 0
    assert dk.shape == k.shape and dv.shape == v.shape
    rq, rk, rv = oracle.attention_bwd_gqa(q, k, v, do, causal=causal)
    G = H // Hkv
    kr, vr = k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2)
    sq, sk, sv = _term_scales(q, kr, vr, do, causal)
    sk = sk.reshape(B, L, Hkv, G, D).sum(axis=3)
    sv = sv.reshape(B, L, Hkv, G, D).sum(axis=3)
    _grad_close(to_np(dq), rq, "dq", sq, p3_holds=not causal)
    _grad_close(to_np(dk), rk, "dk", sk, p3_holds=not causal)
    _grad_close(to_np(dv), rv, "dv", sv, p3_holds=not causal)


def test_bwd_gqa_with_h_kv_equal_h_is_plain_backward():
    """H_kv = H through the grouped entry point gives the plain backward's bits."""
    B, L, H, D, P = 1, 512, 2, 128, 4
    q, k, v = (t.to(DEV) for t in make_qkv(B, L, H, D, seed=43, dtype=torch.bfloat16))
    do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(44)).to(torch.bfloat16).to(DEV)
    out, lse = cea.ring_attn_fwd(q, k, v, P=P, causal=True)
    a = cea.ring_attn_bwd(q, k, v, out, lse, do, P=P, causal=True)
    b = cea.ring_attn_bwd_gqa(q, k, v, out, lse, do, P=P, causal=True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_gqa_argument_errors():
    q, _, _ = (t.to(DEV) for t in make_qkv(1, 256, 6, 128, seed=0, dtype=torch.bfloat16))
    _, k, v = (t.to(DEV) for t in make_qkv(1, 256, 4, 128, seed=0, dtype=torch.bfloat16))
    out = torch.empty_like(q)
    lse = torch.empty(1, 256, 6, device=DEV)
    with pytest.raises(cea.RingAttnError) as e:
        cea.ring_attn_bwd_gqa(q, k, v, out, lse, torch.empty_like(q), P=2)
    assert e.value.code == 4          # 6 query heads over 4 key/value heads


# ---------------------------------------------------------------- zigzag layout --

ZIGZAG_CASES = [
    # B, L, H, D, P
    (1, 512, 2, 128, 2),
    (2, 1024, 2, 128, 4),
    (1, 768, 2, 64, 3),
    (1, 2048, 1, 128, 8),
    (1, 256, 2, 128, 1),
    # chunks of several tiles (head dim 128: dQ on pairs of SMs, a pair within a chunk):
    # 5 and 3 tiles (a lone tile ends each chunk), 4 tiles (whole pairs)
    (1, 2560, 2, 128, 2),
    (1, 1536, 2, 128, 2),
    (1, 4096, 1, 128, 4),
    (2, 2048, 1, 128, 2),
]


@pytest.mark.parametrize("case", ZIGZAG_CASES, ids=lambda c: "B%dL%dH%dD%dP%d" % c)
def test_bwd_zigzag_parity(case):
    """Causal backward of the position-ordered sequence, returned in zigzag row order:
    the oracle's gradients (and the error scales) are computed in position order and
    their rows permuted."""
    B, L, H, D, P = case
    qg, kg, vg = make_qkv(B, L, H, D, seed=80, dtype=torch.bfloat16)      # row = position
    dog = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(81)).to(torch.bfloat16)
    pos = torch.tensor(cea.zigzag_positions(L, P))
    q, k, v, do = (t[:, pos].contiguous().to(DEV) for t in (qg, kg, vg, dog))
    out, lse = cea.ring_attn_fwd_zigzag(q, k, v, P=P)
    dq, dk, dv = cea.ring_attn_bwd_zigzag(q, k, v, out, lse, do, P=P)
    assert cea.check_status() == 0
    rq, rk, rv = oracle.attention_bwd(qg, kg, vg, dog, causal=True)
    sq, sk, sv = _term_scales(qg, kg, vg, dog, True)
    pz = pos.numpy()
    _grad_close(to_np(dq), rq[:, pz], "dq", sq[:, pz])
    _grad_close(to_np(dk), rk[:, pz], "dk", sk[:, pz])
    _grad_close(to_np(dv), rv[:, pz], "dv", sv[:, pz])


def test_bwd_zigzag_matches_contiguous_layout():
    """The same causal problem through both layouts: gradients agree row for row after
    the zigzag permutation (to the rounding of two summation orders), and each layout
    is deterministic."""
    B, L, H, D, P = 1, 1024, 4, 128, 4
    qg, kg, vg = (t.to(DEV) for t in make_qkv(B, L, H, D, seed=82, dtype=torch.bfloat16,
                                              head_scale=True))
    dog = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(83)).to(torch.bfloat16)
    dog = dog.to(DEV)
    out, lse = cea.ring_attn_fwd(qg, kg, vg, P=P, causal=True)
    contig = cea.ring_attn_bwd(qg, kg, vg, out, lse, dog, P=P, causal=True)
    pos = torch.tensor(cea.zigzag_positions(L, P), device=DEV)
    q, k, v, do = (t[:, pos].contiguous() for t in (qg, kg, vg, dog))
    oz, lz = cea.ring_attn_fwd_zigzag(q, k, v, P=P)
    zig = cea.ring_attn_bwd_zigzag(q, k, v, oz, lz, do, P=P)
    again = cea.ring_attn_bwd_zigzag(q, k, v, oz, lz, do, P=P)
    assert cea.check_status() == 0
    for name, a, z, z2 in zip(("dq", "dk", "dv"), contig, zig, again):
        assert torch.equal(z, z2), name
        a = to_np(a)[:, pos.cpu().numpy()]
        z = to_np(z)
        rel = np.linalg.norm(a - z) / np.linalg.norm(a)
        assert rel <= 4 * U and cosine(a, z) > 0.9999, (name, rel)


def test_bwd_zigzag_argument_errors():
    q, k, v = (t.to(DEV) for t in make_qkv(1, 256, 1, 128, seed=0, dtype=torch.bfloat16))
    out, lse = cea.ring_attn_fwd(q, k, v, P=1)
    with pytest.raises(cea.RingAttnError) as e:
        cea.ring_attn_bwd_zigzag(q, k, v, out, lse, q.clone(), P=2)   # chunks of 64 rows
    assert e.value.code == 2
    q, k, v = (t.to(DEV) for t in make_qkv(1, 516, 1, 128, seed=0, dtype=torch.bfloat16))
    out, lse = cea.ring_attn_fwd(q, k, v, P=1)
    with pytest.raises(cea.RingAttnError) as e:
        cea.ring_attn_bwd_zigzag(q, k, v, out, lse, q.clone(), P=4)   # 516 % 8 != 0
    assert e.value.code == 4


# ---------------------------------------------------------------- packed sequences --

VARLEN_CASES = [
    # lengths, H, D, P
    ([37, 263, 1, 399, 324], 2, 128, 2),        # sequences cross the shard edge
    ([1024], 2, 128, 4),                        # one sequence = plain attention
    ([5, 600, 130, 7, 200, 1, 593, 512], 2, 64, 4),
    ([100, 412, 252, 300], 1, 128, 1),
    ([129, 127, 256, 1, 255, 256, 128], 2, 128, 3),  # boundaries one row off tile edges
]


def _packed_bwd_inputs(lengths, H, D, seed):
    L = sum(lengths)
    q, k, v = (t[0] for t in make_qkv(1, L, H, D, seed=seed, dtype=torch.bfloat16))
    do = torch.randn(L, H, D, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    return q, k, v, do, cu


@pytest.mark.parametrize("case", VARLEN_CASES, ids=lambda c: "n%d_H%d_D%d_P%d" % (len(c[0]), *c[1:]))
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_varlen_parity(case, causal):
    """Every sequence is its own attention problem: each gradient slice equals the fp64
    oracle's backward of that sequence alone."""
    lengths, H, D, P = case
    q, k, v, do, cu = _packed_bwd_inputs(lengths, H, D, seed=90)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd_varlen(qd, kd, vd, cu_d, P=P, causal=causal)
    dq, dk, dv = cea.ring_attn_bwd_varlen(qd, kd, vd, out, lse, dod, cu_d, P=P, causal=causal)
    assert cea.check_status() == 0
    got = [to_np(t) for t in (dq, dk, dv)]
    refs = [np.empty_like(g) for g in got]
    scales = [np.empty_like(g) for g in got]
    for a, b in zip(cu[:-1], cu[1:]):
        if a == b:
            continue
        seg = [t[None, a:b] for t in (q, k, v, do)]
        for i, (r, s) in enumerate(zip(oracle.attention_bwd(*seg, causal=causal),
                                       _term_scales(*seg, causal))):
            refs[i][a:b], scales[i][a:b] = r[0], s[0]
    for name, g, r, s in zip(("dq", "dk", "dv"), got, refs, scales):
        _grad_close(g, r, name, s, p3_holds=not causal)


def test_bwd_varlen_samples_do_not_see_each_other():
    """Replace one sequence's queries, keys, values and upstream gradient by other values:
    the other sequences' gradients keep their bits (masked pairs contribute exactly
    zero), the replaced sequence's change."""
    lengths = [300, 200, 524]
    q, k, v, do, cu = _packed_bwd_inputs(lengths, 2, 128, seed=92)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    for causal in (False, True):
        res = []
        for variant in range(2):
            tq, tk, tv, tdo = (t.clone() for t in (q, k, v, do))
            if variant:
                tq[300:500] *= 3.0
                tk[300:500] = 2.0
                tv[300:500] = 40.0
                tdo[300:500] = -tdo[300:500]
            qd, kd, vd, dod = (t.to(DEV) for t in (tq, tk, tv, tdo))
            out, lse = cea.ring_attn_fwd_varlen(qd, kd, vd, cu_d, P=4, causal=causal)
            res.append(cea.ring_attn_bwd_varlen(qd, kd, vd, out, lse, dod, cu_d, P=4,
                                                causal=causal))
        for a, b in zip(*res):
            assert torch.equal(a[:300], b[:300]) and torch.equal(a[500:], b[500:])
            assert not torch.equal(a[300:500], b[300:500])


def test_bwd_varlen_one_sequence_is_plain_backward():
    """A single packed sequence is the plain backward with P shards: identical bits."""
    L, H, D, P = 1024, 2, 128, 4
    q, k, v = (t.to(DEV) for t in make_qkv(1, L, H, D, seed=94, dtype=torch.bfloat16))
    do = torch.randn(1, L, H, D, generator=torch.Generator().manual_seed(95)).to(torch.bfloat16)
    do = do.to(DEV)
    cu_d = torch.tensor([0, L], dtype=torch.int32, device=DEV)
    for causal in (False, True):
        out, lse = cea.ring_attn_fwd(q, k, v, P=P, causal=causal)
        a = cea.ring_attn_bwd(q, k, v, out, lse, do, P=P, causal=causal)
        b = cea.ring_attn_bwd_varlen(q[0], k[0], v[0], out[0], lse[0], do[0], cu_d, P=P,
                                     causal=causal)
        for x, y in zip(a, b):
            assert torch.equal(x[0], y)


# ------------------------------------- combined options (ring_attn_bwd_ex) --

def _grouped_scales(q, k, v, do, causal, G):
    """Error scales of the grouped backward: the per-query-head scales of the repeated
    key/value heads, dk and dv summed over each group."""
    B, L, Hkv, D = k.shape
    sq, sk, sv = _term_scales(q, k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2),
                              do, causal)
    return sq, sk.reshape(B, L, Hkv, G, D).sum(axis=3), sv.reshape(B, L, Hkv, G, D).sum(axis=3)


@pytest.mark.parametrize("case", [(1, 1024, 4, 2, 128, 4), (2, 768, 6, 2, 64, 3),
                                  (1, 512, 4, 1, 128, 2), (1, 2048, 4, 2, 128, 2)],
                         ids=lambda c: "B%dL%dH%dHkv%dD%dP%d" % c)
def test_bwd_ex_zigzag_grouped_heads_parity(case):
    """Backward of grouped key/value heads over zigzag shards against the grouped fp64
    gradient oracle in position order, rows permuted."""
    B, L, H, Hkv, D, P = case
    G = H // Hkv
    qg, _, _ = make_qkv(B, L, H, D, seed=110, dtype=torch.bfloat16)
    _, kg, vg = make_qkv(B, L, Hkv, D, seed=111, dtype=torch.bfloat16)
    dog = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(112)).to(torch.bfloat16)
    pos = torch.tensor(cea.zigzag_positions(L, P))
    q, k, v, do = (t[:, pos].contiguous().to(DEV) for t in (qg, kg, vg, dog))
    out, lse = cea.ring_attn_fwd_ex(q, k, v, P=P, causal=True, layout="zigzag")
    dq, dk, dv = cea.ring_attn_bwd_ex(q, k, v, out, lse, do, P=P, causal=True, layout="zigzag")
    assert cea.check_status() == 0
    assert dk.shape == k.shape and dv.shape == v.shape
    rq, rk, rv = oracle.attention_bwd_gqa(qg, kg, vg, dog, causal=True)
    sq, sk, sv = _grouped_scales(qg, kg, vg, dog, True, G)
    pz = pos.numpy()
    _grad_close(to_np(dq), rq[:, pz], "dq", sq[:, pz])
    _grad_close(to_np(dk), rk[:, pz], "dk", sk[:, pz])
    _grad_close(to_np(dv), rv[:, pz], "dv", sv[:, pz])


@pytest.mark.parametrize("case", [([37, 263, 1, 399, 324], 4, 2, 128, 2),
                                  ([5, 600, 130, 7, 200, 1, 593, 512], 4, 1, 64, 4)],
                         ids=lambda c: "n%d_H%dHkv%d_P%d" % (len(c[0]), c[1], c[2], c[4]))
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_ex_packed_grouped_heads_parity(case, causal):
    """Backward of grouped key/value heads over packed sequences: each sequence against
    the grouped fp64 gradient oracle of that sequence alone."""
    lengths, H, Hkv, D, P = case
    G = H // Hkv
    L = sum(lengths)
    q = make_qkv(1, L, H, D, seed=113, dtype=torch.bfloat16)[0][0]
    _, k, v = (t[0] for t in make_qkv(1, L, Hkv, D, seed=114, dtype=torch.bfloat16))
    do = torch.randn(L, H, D, generator=torch.Generator().manual_seed(115)).to(torch.bfloat16)
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd_ex(qd, kd, vd, P=P, causal=causal, layout="packed",
                                    cu_seqlens=cu_d)
    dq, dk, dv = cea.ring_attn_bwd_ex(qd, kd, vd, out, lse, dod, P=P, causal=causal,
                                      layout="packed", cu_seqlens=cu_d)
    assert cea.check_status() == 0
    got = [to_np(t) for t in (dq, dk, dv)]
    refs = [np.empty_like(g) for g in got]
    scales = [np.empty_like(g) for g in got]
    for a, b in zip(cu[:-1], cu[1:]):
        seg = [t[None, a:b] for t in (q, k, v, do)]
        for i, (r, s) in enumerate(zip(oracle.attention_bwd_gqa(*seg, causal=causal),
                                       _grouped_scales(*seg, causal, G))):
            refs[i][a:b], scales[i][a:b] = r[0], s[0]
    for name, g, r, s in zip(("dq", "dk", "dv"), got, refs, scales):
        _grad_close(g, r, name, s)


def test_bwd_ex_matches_the_specialised_entry_points():
    """Same options as a specialised backward entry point: identical bits."""
    B, L, H, D, P = 1, 1024, 4, 128, 4
    q, k, v = (t.to(DEV) for t in make_qkv(B, L, H, D, seed=116, dtype=torch.bfloat16))
    do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(117)).to(torch.bfloat16)
    do = do.to(DEV)
    cu_d = torch.tensor([0, 300, 301, 1024], dtype=torch.int32, device=DEV)
    out, lse = cea.ring_attn_fwd(q, k, v, P=P, causal=True)
    oz, lz = cea.ring_attn_fwd_zigzag(q, k, v, P=P)
    ov, lv = cea.ring_attn_fwd_varlen(q[0], k[0], v[0], cu_d, P=P, causal=True)
    pairs = [
        (cea.ring_attn_bwd(q, k, v, out, lse, do, P=P, causal=True),
         cea.ring_attn_bwd_ex(q, k, v, out, lse, do, P=P, causal=True)),
        (cea.ring_attn_bwd_zigzag(q, k, v, oz, lz, do, P=P),
         cea.ring_attn_bwd_ex(q, k, v, oz, lz, do, P=P, causal=True, layout="zigzag")),
        (cea.ring_attn_bwd_varlen(q[0], k[0], v[0], ov, lv, do[0], cu_d, P=P, causal=True),
         cea.ring_attn_bwd_ex(q[0], k[0], v[0], ov, lv, do[0], P=P, causal=True, layout="packed",
                              cu_seqlens=cu_d)),
    ]
    assert cea.check_status() == 0
    for a, b in pairs:
        for x, y in zip(a, b):
            assert torch.equal(x, y)
