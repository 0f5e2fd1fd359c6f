"""The packed-sequence schedule (ring_attn_varlen_schedule): the device writes the
heaviest-first unit orders a plain host restatement gives, and the packed forward and
backward return the same bits with and without it (the order only decides which CTA
takes which unit; every unit writes its own rows).  One case also goes to the oracle."""
import numpy as np
import pytest
import torch

import context_exact_attention_gb300 as cea
import oracle
from context_exact_attention_gb300.workloads import make_qkv
from helpers import assert_bf16_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROWS = 128
MAX_BINS = 4096


def _cu(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    return cu


def _host_schedule(cu, L, P, causal):
    """The three orders: per unit, the other side's 128-row tiles (each inside one shard)
    that hold a visible position; descending work, ties in ascending unit index."""
    Ls = L // P
    n_t = -(-Ls // ROWS)
    n_pair = -(-n_t // 2)
    cu = np.asarray(cu)

    def span(pos):
        g = int(np.searchsorted(cu[:-1], pos, side="right")) - 1
        return int(cu[g]), int(cu[g + 1]) - 1

    def tiles_in(lo, hi):
        lo, hi = max(lo, 0), min(hi, L - 1)
        n = 0
        for s in range(lo // Ls, hi // Ls + 1) if lo <= hi else ():
            a, b = max(lo, s * Ls) - s * Ls, min(hi, s * Ls + Ls - 1) - s * Ls
            n += b // ROWS - a // ROWS + 1
        return n

    max_work = P * n_t
    nb = min(max_work + 1, MAX_BINS)
    bin_of = (lambda w: w) if nb == max_work + 1 else (lambda w: w * nb // (max_work + 1))
    orders = []
    for kind in range(3):
        per = n_pair if kind == 0 else n_t
        rows = 2 * ROWS if kind == 0 else ROWS
        work = []
        for u in range(P * per):
            s, i = divmod(u, per)
            a = s * Ls + i * rows
            b = min(s * Ls + Ls - 1, a + rows - 1)
            (fa, _), (_, lb) = span(a), span(b)
            lo, hi = ((a if causal else fa), lb) if kind == 1 else (fa, (b if causal else lb))
            work.append(tiles_in(lo, hi))
        orders.append(sorted(range(len(work)), key=lambda u: (-bin_of(work[u]), u)))
    return orders


def _many(n, P, seed):
    """n sequences of 1..59 rows, the last one stretched so that P divides the total."""
    lengths = [int(x) for x in np.random.default_rng(seed).integers(1, 60, n)]
    lengths[-1] += -sum(lengths) % P
    return lengths


SCHED_CASES = [
    ([6755, 4302, 6383, 701, 4326, 4982, 5319], 8),     # the benchmark's length draw
    ([300, 1, 1000, 0, 747], 4),                         # ragged shards, an empty sequence
    ([2048] * 4, 2),
    ([5000], 5),                                         # one sequence
    ([17, 900, 83, 2000, 1, 1, 1, 93], 3),
    ([5, 7, 100, 200], 4),                               # shards shorter than one tile
    (_many(400, 8, 3), 8),                               # many short sequences
]


@pytest.mark.parametrize("case", SCHED_CASES, ids=lambda c: "n%d_P%d" % (len(c[0]), c[1]))
@pytest.mark.parametrize("causal", [False, True])
def test_schedule_matches_host_orders(case, causal):
    lengths, P = case
    cu = _cu(lengths)
    L = cu[-1]
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    sched = cea.varlen_schedule(cu_d, L, P, causal).cpu().numpy()
    got, off = [], 0
    for want in _host_schedule(cu, L, P, causal):
        got.append(sched[off:off + len(want)].tolist())
        off += len(want)
    for name, g, w in zip(("forward pairs", "backward keys", "backward queries"), got,
                          _host_schedule(cu, L, P, causal)):
        assert g == w, name
        assert sorted(g) == list(range(len(w))), name


def test_schedule_with_many_units_uses_the_global_scratch():
    """More units than the kernel keeps in shared memory (8192): the counts go through
    the scratch area of the schedule buffer."""
    lengths = [3000, 50000, 12345, 200, 131072 * 8 - 65545 + 1000]
    P = 1
    cu = _cu(lengths)
    L = cu[-1]
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    sched = cea.varlen_schedule(cu_d, L, P, True).cpu().numpy()
    want = _host_schedule(cu, L, P, True)
    n_f, n_b = len(want[0]), len(want[1])
    assert n_b > 8192
    assert sched[:n_f].tolist() == want[0]
    assert sched[n_f:n_f + n_b].tolist() == want[1]
    assert sched[n_f + n_b:n_f + 2 * n_b].tolist() == want[2]


BIT_CASES = [
    ([6755, 4302, 6383, 701, 4326, 4982, 5319], 4, 2, 128, 8),
    ([300, 1, 1000, 0, 747], 2, 2, 64, 4),
    ([129, 2000, 255, 1], 3, 1, 128, 5),
    ([5, 7, 100, 200], 2, 2, 128, 4),
    (_many(400, 8, 4), 2, 1, 64, 8),
]


@pytest.mark.parametrize("case", BIT_CASES, ids=lambda c: "n%d_H%d/%d_D%d_P%d" % (len(c[0]), *c[1:]))
@pytest.mark.parametrize("causal", [False, True])
def test_schedule_gives_the_same_bits(case, causal):
    lengths, H, Hkv, D, P = case
    cu = _cu(lengths)
    L = cu[-1]
    q = make_qkv(1, L, H, D, seed=31, dtype=torch.bfloat16)[0][0].to(DEV)
    _, k, v = (t[0].to(DEV) for t in make_qkv(1, L, Hkv, D, seed=32, dtype=torch.bfloat16))
    do = torch.randn(L, H, D, generator=torch.Generator().manual_seed(33)).to(torch.bfloat16).to(DEV)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    sched = cea.varlen_schedule(cu_d, L, P, causal)
    kw = dict(P=P, causal=causal, layout="packed", cu_seqlens=cu_d)
    o0, l0 = cea.ring_attn_fwd_ex(q, k, v, **kw)
    o1, l1 = cea.ring_attn_fwd_ex(q, k, v, schedule=sched, **kw)
    g0 = cea.ring_attn_bwd_ex(q, k, v, o0, l0, do, **kw)
    g1 = cea.ring_attn_bwd_ex(q, k, v, o0, l0, do, schedule=sched, **kw)
    assert cea.check_status() == 0
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    for a, b in zip(g0, g1):
        assert torch.equal(a, b)
    if Hkv == H:
        # the specialised packed entry points route a schedule the same way
        o2, l2 = cea.ring_attn_fwd_varlen(q, k, v, cu_d, P=P, causal=causal, schedule=sched)
        g2 = cea.ring_attn_bwd_varlen(q, k, v, o0, l0, do, cu_d, P=P, causal=causal,
                                      schedule=sched)
        assert torch.equal(o0, o2) and torch.equal(l0, l2)
        for a, b in zip(g0, g2):
            assert torch.equal(a, b)


def test_scheduled_forward_against_the_oracle():
    lengths, H, D, P = [700, 1, 1200, 147], 2, 128, 4
    cu = _cu(lengths)
    L = cu[-1]
    q, k, v = (t[0] for t in make_qkv(1, L, H, D, seed=41, dtype=torch.bfloat16))
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    sched = cea.varlen_schedule(cu_d, L, P, True)
    out, lse = cea.ring_attn_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu_d, P=P, causal=True,
                                        schedule=sched)
    assert cea.check_status() == 0
    ref = np.empty(tuple(q.shape), np.float64)
    lref = np.empty(tuple(q.shape[:2]), np.float64)
    for a, b in zip(cu[:-1], cu[1:]):
        r, lr = oracle.attention(q[None, a:b], k[None, a:b], v[None, a:b], causal=True)
        ref[a:b], lref[a:b] = r[0], lr[0]
    assert_bf16_close(to_np(out), ref, "out")
    assert_bf16_close(to_np(lse), lref, "lse")


def test_a_foreign_schedule_is_ignored_where_out_of_range():
    """Entries outside the unit range fall back to the position order: an all-(-1) or
    all-huge array gives the unscheduled result."""
    lengths, H, D, P = [1000, 24, 1024], 2, 64, 2
    cu = _cu(lengths)
    L = cu[-1]
    q, k, v = (t[0].to(DEV) for t in make_qkv(1, L, H, D, seed=51, dtype=torch.bfloat16))
    cu_d = torch.tensor(cu, dtype=torch.int32, device=DEV)
    n = cea.varlen_schedule(cu_d, L, P, True).numel()
    o0, l0 = cea.ring_attn_fwd_varlen(q, k, v, cu_d, P=P, causal=True)
    for fill in (-1, 1 << 30):
        bad = torch.full((n,), fill, dtype=torch.int32, device=DEV)
        o1, l1 = cea.ring_attn_fwd_varlen(q, k, v, cu_d, P=P, causal=True, schedule=bad)
        assert cea.check_status() == 0
        assert torch.equal(o0, o1) and torch.equal(l0, l1)
