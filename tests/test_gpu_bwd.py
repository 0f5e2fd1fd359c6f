"""GPU parity of the backward (dq, dk, dv) against the fp64 gradient oracle.

Tolerance.  Each gradient element is an fp32-accumulated sum whose terms carry
one bf16 rounding of P or dS (unit roundoff u = 2^-9) plus the bf16 rounding of
the stored forward output inside Dvec, and the result is rounded to bf16 once
more; errors of independent terms add in quadrature while a gradient can cancel
to far below its terms (dk sums to zero over the keys).  So the bar is
norm-wise: ||got - ref|| <= 4u ||ref|| per tensor (u = 2^-9), cosine > 0.9999,
and element-wise |got - ref| <= 4u |ref| + 8u rms(ref).
"""
import numpy as np
import pytest
import torch

import context_exact_attention_gb300 as cea
import oracle
from context_exact_attention_gb300.workloads import make_qkv
from helpers import cosine, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
U = 2.0 ** -9


def _grad_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), what
    err = np.abs(got - ref)
    rms = np.sqrt((ref * ref).mean())
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    worst = (err / (4 * U * np.abs(ref) + 8 * U * rms)).max()
    print(f"{what}: rel_l2 {rel:.2e} cos {cosine(got, ref):.7f} worst/bound {worst:.3f}")
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
    _grad_close(to_np(dq), rq, "dq")
    _grad_close(to_np(dk), rk, "dk")
    _grad_close(to_np(dv), rv, "dv")


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
    for name, got, r in zip(("dq", "dk", "dv"), first, ref):
        _grad_close(to_np(got), r, name)


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
