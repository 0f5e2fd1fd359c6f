"""Degenerate sizes through the kernels, against the fp64 oracle: a single token, shards
of one row (L = P), odd shard counts with shards far smaller than a tile, and one row past
a tile boundary.  The tensor-map boxes are then larger than the tensors themselves; the
rows and keys outside the tensor must read as zero and never reach an output."""
import numpy as np
import pytest
import torch

import context_exact_attention_gb300 as cea
import oracle
from context_exact_attention_gb300.workloads import make_qkv
from helpers import assert_bf16_close, assert_f32_close, to_np
from test_gpu_bwd import _grad_close, _term_scales

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

FWD_CASES = [
    # B, L, H, D, P
    (1, 1, 1, 128, 1),       # one token: out = v_0
    (1, 8, 2, 128, 8),       # shards of one row
    (3, 7, 1, 64, 7),        # shards of one row, odd P, B > 1
    (2, 3, 2, 64, 1),
    (1, 129, 1, 128, 1),     # one row past a tile
    (1, 257, 2, 128, 1),     # one row past a query pair
]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: "B%dL%dH%dD%dP%d" % c)
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_degenerate_sizes(case, causal):
    B, L, H, D, P = case
    q, k, v = make_qkv(B, L, H, D, seed=31, dtype=torch.bfloat16)
    out, lse = cea.ring_attn_fwd(*(t.to(DEV) for t in (q, k, v)), P=P, causal=causal)
    assert cea.check_status() == 0
    ref, lref = oracle.attention(q, k, v, causal=causal)
    assert_bf16_close(to_np(out), ref, "out")
    assert_bf16_close(to_np(lse), lref, "lse")
    if L == 1:
        # a single visible key: the output is that key's value, rounded once
        assert torch.equal(out.cpu(), v)


@pytest.mark.parametrize("case", [(1, 1, 1, 64, 1), (1, 7, 2, 32, 7), (2, 5, 1, 128, 5)],
                         ids=lambda c: "B%dL%dH%dD%dP%d" % c)
@pytest.mark.parametrize("causal", [False, True])
def test_f32_degenerate_sizes(case, causal):
    B, L, H, D, P = case
    q, k, v = make_qkv(B, L, H, D, seed=32, dtype=torch.float32)
    out, lse = cea.ring_attn_fwd_f32(*(t.to(DEV) for t in (q, k, v)), P=P, causal=causal)
    assert cea.check_status() == 0
    ref, lref = oracle.attention(q, k, v, causal=causal)
    assert_f32_close(to_np(out), ref, "out")
    assert_f32_close(to_np(lse), lref, "lse")


@pytest.mark.parametrize("case", [(1, 8, 2, 128, 8), (2, 129, 1, 128, 1), (1, 7, 1, 64, 7)],
                         ids=lambda c: "B%dL%dH%dD%dP%d" % c)
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_degenerate_sizes(case, causal):
    B, L, H, D, P = case
    q, k, v = make_qkv(B, L, H, D, seed=33, dtype=torch.bfloat16)
    do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(34)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd(qd, kd, vd, P=P, causal=causal)
    dq, dk, dv = cea.ring_attn_bwd(qd, kd, vd, out, lse, dod, P=P, causal=causal)
    assert cea.check_status() == 0
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=causal)
    sq, sk, sv = _term_scales(q, k, v, do, causal)
    _grad_close(to_np(dq), rq, "dq", sq)
    _grad_close(to_np(dk), rk, "dk", sk)
    _grad_close(to_np(dv), rv, "dv", sv)


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_single_token(D):
    """One token: P = 1, so dv = dout exactly, and dq = dk = 0 in exact arithmetic (the
    kernel's dP - Dvec is the difference of two fp32 sums of the same bf16 products, so
    only rounding may remain, within the element-wise bound)."""
    q, k, v = make_qkv(2, 1, 3, D, seed=36, dtype=torch.bfloat16)
    do = torch.randn(2, 1, 3, D, generator=torch.Generator().manual_seed(37)).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = cea.ring_attn_fwd(qd, kd, vd, P=1, causal=True)
    dq, dk, dv = cea.ring_attn_bwd(qd, kd, vd, out, lse, dod, P=1, causal=True)
    assert cea.check_status() == 0
    assert torch.equal(dv.cpu(), do)
    sq, sk, _ = _term_scales(q, k, v, do, True)
    for got, scale in ((dq, sq), (dk, sk)):
        err = np.abs(to_np(got).astype(np.float64))
        assert (err <= 2 * 2.0 ** -9 * scale + 1e-6).all()


def test_host_entry_single_token():
    q, k, v = make_qkv(1, 1, 4, 128, seed=35, dtype=torch.bfloat16)
    out, lse = cea.ring_attn_fwd_host(q, k, v, P=1, causal=True, heads_per_group=2, device=DEV)
    torch.cuda.synchronize()
    assert torch.equal(out, v)
    ref_out, ref_lse = cea.ring_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), P=1, causal=True)
    assert torch.equal(lse, ref_lse.cpu())
