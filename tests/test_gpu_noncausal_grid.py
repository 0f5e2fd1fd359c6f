"""Forward calls without causal masking, which run on the static persistent grid (one CTA
per SM taking units round-robin): parity with the fp64 oracle on every row or on sampled
rows for fewer units than SMs, a ragged last wave, head dims 64 and 128, ragged shards,
grouped key/value heads, the ring trace and the fused Ulysses step, plus repeated calls
bit for bit."""
import pytest
import torch

import context_exact_attention_gb300 as cea
import oracle
from context_exact_attention_gb300.workloads import make_qkv, sample_rows
from helpers import assert_bf16_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("B,L,H,D,P", [
    (1, 2048, 2, 128, 2),      # 16 units of 16 blocks: fewer units than SMs
    (1, 1000, 3, 128, 4),      # shards of 250 rows: ragged tiles and key blocks
    (2, 4096, 5, 64, 4),       # 160 units: one whole wave, then a tail of 8 units
    (1, 8192, 1, 64, 1),       # 32 units of 64 blocks
    (1, 4096, 24, 128, 4),     # the DiT shape: 2.53 waves
])
def test_noncausal_grid_matches_oracle(B, L, H, D, P):
    q, k, v = make_qkv(B, L, H, D, seed=100 + H, head_scale=True)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, lse = cea.ring_attn_fwd(qd, kd, vd, P=P, causal=False)
    assert cea.check_status() == 0
    rows = None if B * L * H <= 16384 else sample_rows(L, P, 64, seed=2)
    ref, lref = oracle.attention(q, k, v, causal=False, rows=rows)
    got, lgot = (out, lse) if rows is None else (out[:, rows], lse[:, rows])
    assert_bf16_close(to_np(got), ref, "out")
    assert_bf16_close(to_np(lgot), lref, "lse")
    for _ in range(3):
        again, lagain = cea.ring_attn_fwd(qd, kd, vd, P=P, causal=False)
        assert torch.equal(out, again) and torch.equal(lse, lagain)


def test_noncausal_grid_gqa_and_trace():
    B, L, H, Hkv, D, P = 1, 2048, 4, 2, 128, 4
    q, _, _ = make_qkv(B, L, H, D, seed=110)
    _, k, v = make_qkv(B, L, Hkv, D, seed=111)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, lse = cea.ring_attn_fwd_gqa(qd, kd, vd, P=P, causal=False)
    ref, lref = oracle.attention(q, k, v, causal=False)
    assert_bf16_close(to_np(out), ref, "gqa out")
    assert_bf16_close(to_np(lse), lref, "gqa lse")
    q1, k1, v1 = make_qkv(1, L, 2, D, seed=112)
    o1, l1, trace = cea.ring_attn_fwd_trace(*(t.to(DEV) for t in (q1, k1, v1)), P=P,
                                            causal=False)
    _, _, tref = oracle.ring_attention(*make_qkv(1, 16 * P, 1, 8, seed=113), P, causal=False)
    assert torch.equal(trace.cpu(), torch.as_tensor(tref, dtype=trace.dtype))
    plain, lplain = cea.ring_attn_fwd(*(t.to(DEV) for t in (q1, k1, v1)), P=P, causal=False)
    assert torch.equal(o1, plain) and torch.equal(l1, lplain)


def test_noncausal_grid_fused_ulysses():
    """The fused Ulysses step (P = 4 shards of 512 rows, 8 heads): the same bits as the
    three-transpose pipeline, and the oracle's attention of the global tensors."""
    P, B, Ls, H, D = 4, 1, 512, 8, 128
    g = torch.Generator().manual_seed(114)
    qs, ks, vs = (torch.randn(P, B, Ls, H, D, generator=g).to(torch.bfloat16) for _ in range(3))
    qd, kd, vd = (t.to(DEV) for t in (qs, ks, vs))
    out, _ = cea.ulysses_attention_fused(qd, kd, vd, P, causal=False)
    assert torch.equal(out, cea.ulysses_attention(qd, kd, vd, P))
    glob = lambda t: t.permute(1, 0, 2, 3, 4).reshape(B, P * Ls, H, D)
    ref, lref = oracle.attention(glob(qs), glob(ks), glob(vs), causal=False)
    assert_bf16_close(to_np(glob(out.cpu())), ref, "fused out")
