"""The index-checked debug build (libringattn_debug.so) on the GPU.

In the debug build every global load and store that a kernel addresses by a
computed index is checked against its tensor's extent; a failed check is recorded
(ra_check_status returns 7) and the access is skipped, so these runs cannot touch
memory outside a buffer.  The tests route the Python binding through the debug
library and check that:
  - the check fires when it should (ra_probe_bounds_check, whose guarded write goes
    to a word of the library either way);
  - on well-formed inputs every entry point gives exactly the normal build's bits and
    no check fails;
  - with malformed sequence boundaries (decreasing, negative, past L, not starting at
    0, all zero, extreme values) the packed-sequence forward (bf16 and fp32), the
    schedule and the backward pass every check and finish without a timed-out wait --
    the in-bounds promise of the packed entry points.  Only then do the same calls run
    on the normal build, which must also finish cleanly.
"""
import ctypes

import pytest
import torch

import context_exact_attention_gb300 as cea
from context_exact_attention_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
RA_ERR_BOUNDS = 7


def _use(monkeypatch, lib):
    monkeypatch.setattr(cea, "_lib", lib)


def test_probe_reports_a_failed_check(monkeypatch):
    _use(monkeypatch, cea.load_debug_library(build_if_missing=True))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert cea.load_library().ra_probe_bounds_check(stream) == 0
    assert cea.check_status() == RA_ERR_BOUNDS
    assert cea.check_status() == 0            # read and cleared


def _bf16(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(torch.bfloat16).to(DEV)


def _every_entry_point():
    """One call of each entry point on small well-formed inputs (ragged tiles, several
    shards); returns every output tensor."""
    res = []
    B, L, H, D, P = 2, 1000, 4, 128, 4            # shards of 250 rows: ragged tiles
    q, k, v = (t.to(DEV) for t in make_qkv(B, L, H, D, seed=70, dtype=torch.bfloat16))
    do = _bf16(B, L, H, D, seed=71)
    for causal in (False, True):
        out, lse = cea.ring_attn_fwd(q, k, v, P=P, causal=causal)
        res += [out, lse, *cea.ring_attn_bwd(q, k, v, out, lse, do, P=P, causal=causal)]
    out, lse, tr = cea.ring_attn_fwd_trace(q, k, v, P=P, causal=True)
    res += [out, lse, tr]
    kk, vv = k[:, :, :2].contiguous(), v[:, :, :2].contiguous()
    out, lse = cea.ring_attn_fwd_gqa(q, kk, vv, P=P, causal=True)
    res += [out, lse, *cea.ring_attn_bwd_gqa(q, kk, vv, out, lse, do, P=P, causal=True)]
    # the pair-of-SMs forward (key walks of 8192 keys and more): ragged shards of 4100
    qx, kx, vx = (t.to(DEV) for t in make_qkv(1, 8200, 1, 128, seed=79, dtype=torch.bfloat16))
    for causal in (False, True):
        res += list(cea.ring_attn_fwd(qx, kx, vx, P=2, causal=causal))
    # zigzag: chunks of a multiple of 128 rows
    qz, kz, vz = (t.to(DEV) for t in make_qkv(1, 2048, 2, 64, seed=72, dtype=torch.bfloat16))
    dz = _bf16(1, 2048, 2, 64, seed=73)
    out, lse = cea.ring_attn_fwd_zigzag(qz, kz, vz, P=4)
    res += [out, lse, *cea.ring_attn_bwd_zigzag(qz, kz, vz, out, lse, dz, P=4)]
    # zigzag at head dim 128 with chunks of 5 tiles (pair-of-SMs dQ, a lone tile ending
    # each chunk), and the pair-of-SMs zigzag forward with a quad across a shard's chunks
    qz, kz, vz = (t.to(DEV) for t in make_qkv(1, 2560, 2, 128, seed=82, dtype=torch.bfloat16))
    dz = _bf16(1, 2560, 2, 128, seed=83)
    out, lse = cea.ring_attn_fwd_zigzag(qz, kz, vz, P=2)
    res += [out, lse, *cea.ring_attn_bwd_zigzag(qz, kz, vz, out, lse, dz, P=2)]
    qz, kz, vz = (t.to(DEV) for t in make_qkv(1, 8960, 1, 128, seed=84, dtype=torch.bfloat16))
    res += list(cea.ring_attn_fwd_zigzag(qz, kz, vz, P=7))
    # packed sequences, with and without the schedule
    Lp = 1024
    cu = torch.tensor([0, 5, 300, 301, 777, 1024], dtype=torch.int32, device=DEV)
    qp, kp, vp = (t[0].to(DEV) for t in make_qkv(1, Lp, 2, 128, seed=74, dtype=torch.bfloat16))
    dp = _bf16(Lp, 2, 128, seed=75)
    sched = cea.varlen_schedule(cu, Lp, 4, True)
    n_t = (Lp // 4 + 127) // 128
    res.append(sched[: 4 * ((n_t + 1) // 2) + 2 * 4 * n_t].clone())   # the three orders
    for s in (None, sched):
        out, lse = cea.ring_attn_fwd_varlen(qp, kp, vp, cu, P=4, causal=True, schedule=s)
        res += [out, lse, *cea.ring_attn_bwd_varlen(qp, kp, vp, out, lse, dp, cu, P=4,
                                                    causal=True, schedule=s)]
    # fp32 (contiguous and packed)
    qf, kf, vf = (t.float() for t in (qp, kp, vp))
    res += list(cea.ring_attn_fwd_f32(qf[None], kf[None], vf[None], P=4, causal=True))
    res += list(cea.ring_attn_fwd_varlen(qf, kf, vf, cu, P=4, causal=False))
    # Ulysses: both transposes (copy-engine path and, for D > 256, the vector path),
    # the fused step, and the merge in both element types
    for Dx in (128, 320):
        x = _bf16(4, 2, 256, 8, Dx, seed=76)
        y = cea.ulysses_seq2head(x, 4)
        res += [y, cea.ulysses_head2seq(y, 4)]
    qs, ks, vs = (_bf16(4, 1, 256, 8, 128, seed=77 + i) for i in range(3))
    res += list(cea.ulysses_attention_fused(qs, ks, vs, 4, causal=True, want_lse=True))
    g = torch.Generator().manual_seed(78)
    for dt in (torch.bfloat16, torch.float32):
        oa, ob = (torch.randn(777, 128, generator=g).to(dt).to(DEV) for _ in range(2))
        la, lb = (torch.randn(777, generator=g).to(DEV) for _ in range(2))
        res += list(cea.attn_merge_partials(oa, la, ob, lb))
    # the host-buffer forward (lse scattered on the device)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho = torch.empty(hq.shape, dtype=hq.dtype).pin_memory()
    hl = torch.empty((B, L, H), dtype=torch.float32).pin_memory()
    cea.ring_attn_fwd_host(hq, hk, hv, P=P, causal=True, out=ho, lse=hl, heads_per_group=2)
    torch.cuda.synchronize()
    res += [ho.clone(), hl.clone()]
    return res


def test_debug_build_gives_the_normal_bits_and_no_failed_check(monkeypatch):
    normal = _every_entry_point()
    assert cea.check_status() == 0
    _use(monkeypatch, cea.load_debug_library(build_if_missing=True))
    checked = _every_entry_point()
    assert cea.check_status() == 0            # no index check failed, no wait timed out
    assert len(normal) == len(checked)
    for i, (a, b) in enumerate(zip(normal, checked)):
        assert torch.equal(a, b), i


MALFORMED = {
    "decreasing": [0, 600, 300, 1024],
    "negative": [0, -50, 500, 1024],
    "past_L": [0, 700, 5000, 1024],
    "total_past_L": [0, 300, 2000],
    "first_not_zero": [300, 600, 1024],
    "all_zero": [0, 0, 0, 0],
    "extremes": [0, 2 ** 31 - 1, -2 ** 31, 1024],
}


def _packed_calls(cu, causal):
    L, H, D, P = 1024, 2, 128, 4
    q, k, v = (t[0].to(DEV) for t in make_qkv(1, L, H, D, seed=80, dtype=torch.bfloat16))
    do = _bf16(L, H, D, seed=81)
    res = []
    sched = cea.varlen_schedule(cu, L, P, causal)
    for s in (None, sched):
        out, lse = cea.ring_attn_fwd_varlen(q, k, v, cu, P=P, causal=causal, schedule=s)
        res += [out, lse]
        res += list(cea.ring_attn_bwd_varlen(q, k, v, out, lse, do, cu, P=P, causal=causal,
                                             schedule=s))
    res += list(cea.ring_attn_fwd_varlen(q.float(), k.float(), v.float(), cu, P=P,
                                         causal=causal))
    return res


@pytest.mark.parametrize("name", sorted(MALFORMED))
@pytest.mark.parametrize("causal", [False, True])
def test_malformed_boundaries_stay_in_bounds(monkeypatch, name, causal):
    cu = torch.tensor(MALFORMED[name], dtype=torch.int32, device=DEV)
    with monkeypatch.context() as m:
        _use(m, cea.load_debug_library(build_if_missing=True))
        _packed_calls(cu, causal)
        assert cea.check_status() == 0
    # every access was checked in range: the same calls on the normal build
    res = _packed_calls(cu, causal)
    assert cea.check_status() == 0
    if name == "first_not_zero" and causal:
        # rows before the first boundary see no key at all: 0 and -inf (bf16 and fp32)
        for out, lse in ((res[0], res[1]), (res[10], res[11])):
            assert torch.all(out[:300] == 0) and torch.all(lse[:300] == float("-inf"))
