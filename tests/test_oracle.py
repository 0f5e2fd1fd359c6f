"""Pins for the fp64 oracle: each test ties it to something other than itself.

The pins are values printed on the pages, closed forms, invariants of exact
softmax attention, special cases that reduce to library routines, and brute
force on tiny inputs.  Each was chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign or index, a transposed operand, a local instead
of a global causal index, a missing merge) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng


def _rand(shape, seed, scale=1.0):
    return rng(seed).standard_normal(shape) * scale


def _load_worked_example():
    rows = {"q": [], "k": [], "v": []}
    meta = {}
    with open(os.path.join(GOLDEN, "ring_attention_sim_4x2.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key in rows:
                rows[key].append([float(x) for x in vals])
            else:
                meta[key] = [float(x) for x in vals]
    q, k, v = (np.array(rows[n])[None, :, None, :] for n in "qkv")
    return q, k, v, meta


# -- values printed on the pages ------------------------------------------------

def test_worked_example_full_and_ring():
    """"序列并行与 Ring Attention", section 04: full[0] = ring[0] = [1.713718770, 1.717687378]."""
    q, k, v, meta = _load_worked_example()
    half_ulp_of_print = 0.5 * 10.0 ** (-meta["printed_decimals"][0])
    out, _ = oracle.attention(q, k, v)
    np.testing.assert_allclose(out[0, 0, 0], meta["full_row0"], rtol=0, atol=half_ulp_of_print)
    P = q.shape[1] // int(meta["kv_block"][0])
    ring, _, _ = oracle.ring_attention(q, k, v, P)
    np.testing.assert_allclose(ring[0, 0, 0], meta["ring_row0"], rtol=0, atol=half_ulp_of_print)
    assert np.abs(out - ring).max() < 1e-15


# -- closed forms -----------------------------------------------------------------

def test_zero_query_gives_column_mean():
    """All scores 0 -> uniform weights -> output is the mean of V, lse = ln(#keys)."""
    B, L, H, D = 2, 12, 3, 5
    q = np.zeros((B, L, H, D))
    k, v = _rand((B, L, H, D), 1), _rand((B, L, H, D), 2)
    out, lse = oracle.attention(q, k, v)
    np.testing.assert_allclose(out, np.broadcast_to(v.mean(axis=1, keepdims=True), out.shape),
                               rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(L), rtol=0, atol=1e-14)
    # causal: row i averages v[0..i], lse = ln(i + 1)
    outc, lsec = oracle.attention(q, k, v, causal=True)
    prefix_mean = np.cumsum(v, axis=1) / np.arange(1, L + 1)[None, :, None, None]
    np.testing.assert_allclose(outc, prefix_mean, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lsec, np.log(np.arange(1, L + 1))[None, :, None]
                               * np.ones((B, 1, H)), rtol=0, atol=1e-14)
    # the worked example's V has column mean [1.75, 1.5]
    _, _, vw, _ = _load_worked_example()
    ow, _ = oracle.attention(np.zeros_like(vw), vw, vw)
    np.testing.assert_allclose(ow[0, :, 0], [[1.75, 1.5]] * 4, rtol=0, atol=1e-15)


def test_single_key_and_causal_row0():
    """One visible key -> weight 1: the output is that key's value row exactly."""
    B, L, H, D = 1, 9, 2, 4
    q, k, v = _rand((B, L, H, D), 3), _rand((B, L, H, D), 4), _rand((B, L, H, D), 5)
    out, lse = oracle.attention(q, k, v, causal=True)
    np.testing.assert_array_equal(out[:, 0], v[:, 0])
    np.testing.assert_allclose(lse[:, 0], (q[:, 0] * k[:, 0]).sum(-1) / math.sqrt(D), atol=1e-15)


def test_two_keys_closed_form():
    """Two keys: o = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1 (independent closed form)."""
    q = np.array([0.3, -1.2, 2.0, 0.5])[None, None, None, :]
    k = np.array([[1.0, 0.5, -0.3, 2.0], [-0.7, 0.1, 0.9, -1.5]])[None, :, None, :]
    v = np.array([[2.0, -1.0, 0.5, 3.0], [-4.0, 1.0, 1.5, 0.25]])[None, :, None, :]
    s0 = float(q[0, 0, 0] @ k[0, 0, 0]) / 2.0
    s1 = float(q[0, 0, 0] @ k[0, 1, 0]) / 2.0
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = w0 * v[0, 0, 0] + (1.0 - w0) * v[0, 1, 0]
    out, lse = oracle.attention(q, k, v)
    np.testing.assert_allclose(out[0, 0, 0], expect, rtol=0, atol=1e-15)
    assert abs(lse[0, 0, 0] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-15


# -- library routines ---------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_matches_scipy_softmax(causal):
    """Per (b, h): softmax(q k^T / sqrt(D)) @ v with scipy's softmax and logsumexp."""
    B, L, H, D = 2, 17, 3, 8
    q, k, v = _rand((B, L, H, D), 6), _rand((B, L, H, D), 7), _rand((B, L, H, D), 8)
    out, lse = oracle.attention(q, k, v, causal=causal)
    for b in range(B):
        for h in range(H):
            s = q[b, :, h] @ k[b, :, h].T / math.sqrt(D)
            if causal:
                s = np.where(np.tril(np.ones((L, L), bool)), s, -np.inf)
            np.testing.assert_allclose(out[b, :, h], scipy.special.softmax(s, axis=1) @ v[b, :, h],
                                       rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse[b, :, h], scipy.special.logsumexp(s, axis=1),
                                       rtol=1e-13, atol=1e-13)


def test_sampled_rows_match_full():
    B, L, H, D = 1, 40, 2, 6
    q, k, v = _rand((B, L, H, D), 9), _rand((B, L, H, D), 10), _rand((B, L, H, D), 11)
    full, lfull = oracle.attention(q, k, v, causal=True)
    rows = [0, 7, 39, 20]
    part, lpart = oracle.attention(q, k, v, causal=True, rows=rows)
    np.testing.assert_array_equal(part, full[:, rows])
    np.testing.assert_array_equal(lpart, lfull[:, rows])


# -- invariants ----------------------------------------------------------------------

@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_recurrence_equals_full(P, causal):
    """Chunked/ring == one-shot to fp64 rounding (juejin page section 五 reports ~1e-16)."""
    B, L, H, D = 1, 48, 2, 8
    q, k, v = _rand((B, L, H, D), 12), _rand((B, L, H, D), 13), _rand((B, L, H, D), 14)
    full, lfull = oracle.attention(q, k, v, causal=causal)
    ring, lring, _ = oracle.ring_attention(q, k, v, P, causal=causal)
    assert np.abs(full - ring).max() < 1e-13
    assert np.abs(lfull - lring).max() < 1e-13


def test_key_value_permutation_invariance():
    """Non-causal attention is a set function of the (key, value) pairs."""
    B, L, H, D = 1, 33, 2, 7
    q, k, v = _rand((B, L, H, D), 15), _rand((B, L, H, D), 16), _rand((B, L, H, D), 17)
    perm = rng(18).permutation(L)
    a, la = oracle.attention(q, k, v)
    b, lb = oracle.attention(q, k[:, perm], v[:, perm])
    assert np.abs(a - b).max() < 1e-13 and np.abs(la - lb).max() < 1e-13
    # a slip that permutes only the keys must show
    c, _ = oracle.attention(q, k[:, perm], v)
    assert np.abs(a - c).max() > 1e-3


def test_key_shift_invariance_and_large_scores():
    """Adding one vector c to every key shifts each row's scores by q.c/sqrt(D): the
    output is unchanged and stays finite with scores near 1000 ("序列并行与 Ring
    Attention", section 09: add 1000 to the scores, the stable recurrence stays finite)."""
    B, L, H, D = 1, 24, 2, 8
    q, k, v = _rand((B, L, H, D), 19), _rand((B, L, H, D), 20), _rand((B, L, H, D), 21)
    q[..., 0] = np.abs(q[..., 0]) + 1.0
    c = np.zeros(D)
    c[0] = 1000.0 * math.sqrt(D) / 1.0
    base, lb = oracle.attention(q, k, v)
    shifted, ls = oracle.attention(q, k + c, v)
    assert np.isfinite(shifted).all() and np.isfinite(ls).all()
    assert np.abs(base - shifted).max() < 1e-9
    ring, _, _ = oracle.ring_attention(q, k + c, v, 4)
    assert np.abs(base - ring).max() < 1e-9
    np.testing.assert_allclose(ls - lb, (q @ c)[..., None].squeeze(-1) / math.sqrt(D), rtol=1e-12)


# -- causal mask: brute force and the global-index rule ---------------------------------

def test_causal_equals_prefix_attention():
    """Causal row i equals non-causal attention of q_i over keys 0..i (brute force)."""
    B, L, H, D = 1, 14, 2, 4
    q, k, v = _rand((B, L, H, D), 22), _rand((B, L, H, D), 23), _rand((B, L, H, D), 24)
    out, lse = oracle.attention(q, k, v, causal=True)
    for i in range(L):
        o_i, l_i = oracle.attention(q[:, i:i + 1], k[:, :i + 1], v[:, :i + 1])
        np.testing.assert_allclose(out[:, i], o_i[:, 0], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[:, i], l_i[:, 0], rtol=0, atol=1e-14)


def test_causal_query_slice_uses_global_positions():
    """A query slice starting at global position a, against all keys from position 0,
    reproduces rows a.. of the full causal result: the mask compares global positions."""
    B, L, H, D = 1, 20, 2, 4
    q, k, v = _rand((B, L, H, D), 46), _rand((B, L, H, D), 47), _rand((B, L, H, D), 48)
    full, lfull = oracle.attention(q, k, v, causal=True)
    a = 7
    part, lpart = oracle.attention(q[:, a:], k, v, causal=True, q_pos0=a, k_pos0=0)
    np.testing.assert_allclose(part, full[:, a:], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lpart, lfull[:, a:], rtol=0, atol=1e-15)
    # keys starting at global position a, one query at position L-1: sees keys a..L-1
    tail, _ = oracle.attention(q[:, L - 1:], k[:, a:], v[:, a:], causal=True,
                               q_pos0=L - 1, k_pos0=a)
    ref, _ = oracle.attention(q[:, L - 1:], k[:, a:], v[:, a:])
    np.testing.assert_allclose(tail, ref, rtol=0, atol=1e-15)


def test_local_index_mask_is_wrong():
    """Masking each shard with local (renumbered) positions must differ from the global rule
    ("序列并行与 Ring Attention", section 09 and section 6.5)."""
    B, L, H, D, P = 1, 32, 2, 4, 4
    q, k, v = _rand((B, L, H, D), 25), _rand((B, L, H, D), 26), _rand((B, L, H, D), 27)
    good, _, _ = oracle.ring_attention(q, k, v, P, causal=True)
    Ls = L // P
    bad = np.empty_like(good)
    for r in range(P):
        sl = slice(r * Ls, (r + 1) * Ls)
        # positions restart at 0 in every shard: the key block of shard r only
        o, _ = oracle.attention(q[:, sl], k[:, :(r + 1) * Ls], v[:, :(r + 1) * Ls], causal=True,
                                q_pos0=0, k_pos0=0)
        bad[:, sl] = o
    assert np.abs(good[:, Ls:] - bad[:, Ls:]).max() > 1e-2
    np.testing.assert_allclose(good[:, :Ls], bad[:, :Ls], atol=1e-14)


# -- did it communicate ----------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_ring_differs_from_local_only(causal):
    """For P > 1 every shard's output differs from local-only attention (juejin page, section
    二 step 4: max_err must be > 0); for P = 1 the two coincide."""
    B, L, H, D, P = 1, 32, 2, 8, 4
    q, k, v = _rand((B, L, H, D), 28), _rand((B, L, H, D), 29), _rand((B, L, H, D), 30)
    ring, _, _ = oracle.ring_attention(q, k, v, P, causal=causal)
    loc, _ = oracle.local_only(q, k, v, P, causal=causal)
    Ls = L // P
    first = 1 if causal else 0        # causal shard 0 sees only its own block
    for r in range(first, P):
        assert np.abs(ring[:, r * Ls:(r + 1) * Ls] - loc[:, r * Ls:(r + 1) * Ls]).max() > 1e-3
    if causal:
        assert np.abs(ring[:, :Ls] - loc[:, :Ls]).max() < 1e-14
    one, _, _ = oracle.ring_attention(q, k, v, 1, causal=causal)
    loc1, _ = oracle.local_only(q, k, v, 1, causal=causal)
    assert np.abs(one - loc1).max() < 1e-14


def test_poisoned_remote_block_changes_output():
    """Set shard s's K/V to 1e4 (juejin page, section 六): non-causal, every shard changes;
    causal, exactly the shards r >= s change."""
    B, L, H, D, P, s = 1, 32, 1, 4, 4, 2
    q, k, v = _rand((B, L, H, D), 31), _rand((B, L, H, D), 32), _rand((B, L, H, D), 33)
    Ls = L // P
    k2, v2 = k.copy(), v.copy()
    k2[:, s * Ls:(s + 1) * Ls] = 1e4 / math.sqrt(D) / 100.0
    v2[:, s * Ls:(s + 1) * Ls] = 1e4
    for causal in (False, True):
        a, _, _ = oracle.ring_attention(q, k, v, P, causal=causal)
        b, _, _ = oracle.ring_attention(q, k2, v2, P, causal=causal)
        for r in range(P):
            d = np.abs(a[:, r * Ls:(r + 1) * Ls] - b[:, r * Ls:(r + 1) * Ls]).max()
            assert (d > 1e-3) == (not causal or r >= s), (causal, r, d)


# -- schedule trace ----------------------------------------------------------------------

@pytest.mark.parametrize("P", [1, 2, 3, 5, 8])
def test_trace_properties(P):
    """Each shard meets every source exactly once, its own first, and at step t shard r
    holds what shard r-1 held at step t-1 (the ring pass).  Causal: exactly the sources
    0..r are visited; the rest are marked skipped."""
    L = 8 * P
    x = _rand((1, L, 1, 2), 34)
    _, _, tr = oracle.ring_attention(x, x, x, P)
    for r in range(P):
        assert sorted(tr[r].tolist()) == list(range(P))
        assert tr[r, 0] == r
        for t in range(1, P):
            assert tr[r, t] == tr[(r - 1) % P, t - 1]
    _, _, tc = oracle.ring_attention(x, x, x, P, causal=True)
    for r in range(P):
        visited = sorted(s for s in tc[r].tolist() if s >= 0)
        assert visited == list(range(r + 1))
        assert (tc[r] == -1).sum() == P - 1 - r
        assert tc[r, 0] == r


# -- merge ----------------------------------------------------------------------------------

def test_merge_of_disjoint_partials_equals_full():
    B, L, H, D = 2, 30, 2, 8
    q, k, v = _rand((B, L, H, D), 35), _rand((B, L, H, D), 36), _rand((B, L, H, D), 37)
    full, lfull = oracle.attention(q, k, v)
    cut = 11
    oa, la = oracle.attention(q, k[:, :cut], v[:, :cut])
    ob, lb = oracle.attention(q, k[:, cut:], v[:, cut:])
    om, lm = oracle.merge(oa, la, ob, lb)
    assert np.abs(om - full).max() < 1e-14 and np.abs(lm - lfull).max() < 1e-14
    # commutative
    om2, lm2 = oracle.merge(ob, lb, oa, la)
    assert np.abs(om - om2).max() < 1e-15 and np.abs(lm - lm2).max() < 1e-15


def test_merge_special_values():
    o = _rand((5, 4), 38)
    lse = _rand((5,), 39)
    ninf = np.full(5, -np.inf)
    om, lm = oracle.merge(o, lse, _rand((5, 4), 40), ninf)       # empty partial is neutral
    np.testing.assert_array_equal(lm, lse)
    np.testing.assert_allclose(om, o, rtol=0, atol=1e-15)
    om, lm = oracle.merge(o, lse, o, lse)                       # self-merge doubles the mass
    np.testing.assert_allclose(om, o, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lm, lse + math.log(2.0), rtol=0, atol=1e-15)
    om, lm = oracle.merge(o, ninf, o, ninf)                     # both empty
    assert np.all(om == 0) and np.all(lm == -np.inf)
    big = np.array([800.0, -800.0, 0.0, 700.0, 1e-300])         # no overflow in logaddexp
    om, lm = oracle.merge(o, big, o, big + 1.0)
    np.testing.assert_allclose(lm, np.logaddexp(big, big + 1.0), rtol=1e-15)


def test_wrong_merges_are_caught():
    """Mean of block outputs and last-block-only (juejin page, section 五) both miss the
    bf16 tolerance by a wide margin; only the LSE merge reproduces the full result."""
    B, L, H, D, n = 1, 128, 2, 32, 4
    q, k, v = _rand((B, L, H, D), 41), _rand((B, L, H, D), 42), _rand((B, L, H, D), 43)
    ref, _ = oracle.attention(q, k, v)
    per = L // n
    parts = [oracle.attention(q, k[:, i * per:(i + 1) * per], v[:, i * per:(i + 1) * per])
             for i in range(n)]
    mean_wrong = sum(p[0] for p in parts) / n
    last_wrong = parts[-1][0]
    o, l = parts[0]
    for p in parts[1:]:
        o, l = oracle.merge(o, l, p[0], p[1])
    tol = 5e-3 + 5e-3 * np.abs(ref)
    assert (np.abs(mean_wrong - ref) > tol).any()
    assert (np.abs(last_wrong - ref) > tol).any()
    assert np.abs(o - ref).max() < 1e-14


# -- Ulysses transposes -----------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [np.float32, np.uint16, np.float64])
def test_seq2head_matches_numpy_transpose_and_inverts(dtype):
    P, B, L, H, D = 4, 2, 16, 8, 3
    Ls, Hg = L // P, H // P
    x = (rng(44).integers(0, 60000, size=(P, B, Ls, H, D))).astype(dtype)
    y = oracle.seq2head(x, P)
    assert y.shape == (P, B, L, Hg, D)
    # library route: [r, b, l, g, hh, d] -> [g, b, r, l, hh, d]
    expect = x.reshape(P, B, Ls, P, Hg, D).transpose(3, 1, 0, 2, 4, 5).reshape(P, B, L, Hg, D)
    assert np.array_equal(y, expect)
    assert np.array_equal(oracle.head2seq(y, P), x)
    # all-to-all block invariant: block (r -> g) arrives whole, in order, in place
    for r in range(P):
        for g in range(P):
            assert np.array_equal(y[g, :, r * Ls:(r + 1) * Ls], x[r, :, :, g * Hg:(g + 1) * Hg])


def test_seq2head_for_one_batch_is_global_layout():
    """With B = 1 the P rank slices of [1, L/P, H, D] concatenate to the global [1, L, H, D];
    head group g of the result is the global tensor restricted to its heads."""
    P, L, H, D = 4, 32, 8, 2
    g_full = rng(45).standard_normal((1, L, H, D))
    seq = g_full.reshape(P, 1, L // P, H, D)
    head = oracle.seq2head(seq, P)
    for g in range(P):
        assert np.array_equal(head[g], g_full[:, :, g * (H // P):(g + 1) * (H // P)])


def test_divisibility_errors():
    with pytest.raises(ValueError):
        oracle.ring_attention(np.zeros((1, 10, 1, 2)), np.zeros((1, 10, 1, 2)),
                              np.zeros((1, 10, 1, 2)), 3)
    with pytest.raises(ValueError):
        oracle.seq2head(np.zeros((4, 1, 2, 6, 2)), 4)


# -- backward (gradients) ----------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    """dq, dk, dv are the gradient of the scalar sum(O * dO): central differences on a
    tiny problem (brute force, independent of the chain-rule code)."""
    B, L, H, D = 1, 5, 2, 3
    q, k, v, do = (_rand((B, L, H, D), 60 + i) for i in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=causal)

    def loss(q_, k_, v_):
        o, _ = oracle.attention(q_, k_, v_, causal=causal, threads=1)
        return float((o * do).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(**{k_ + "_": a for k_, a in args_p.items()})
                        - loss(**{k_ + "_": a for k_, a in args_m.items()})) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-7, err_msg=name)


def test_backward_matches_torch_autograd():
    """fp64 torch autograd of softmax(q k^T / sqrt(D)) v (a library route)."""
    torch = pytest.importorskip("torch")
    B, L, H, D = 2, 13, 3, 8
    q, k, v, do = (_rand((B, L, H, D), 70 + i) for i in range(4))
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
        s = torch.einsum("bihd,bjhd->bhij", tq, tk) / math.sqrt(D)
        if causal:
            s = s.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
        o = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), tv)
        o.backward(torch.tensor(do))
        dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=causal)
        np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_closed_forms(causal):
    """Rows of P sum to 1, so sum_j dV_j = sum_i dO_i; rows of dS sum to 0, so
    sum_j dK_j = 0; dO = 0 gives zero gradients."""
    B, L, H, D = 1, 11, 2, 4
    q, k, v, do = (_rand((B, L, H, D), 80 + i) for i in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=causal)
    np.testing.assert_allclose(dv.sum(axis=1), do.sum(axis=1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, rtol=0, atol=1e-12)
    z = oracle.attention_bwd(q, k, v, np.zeros_like(do), causal=causal)
    assert all(np.all(g == 0) for g in z)
    if causal:
        # the last key is visible to the last query only, so its dv is a multiple of dO
        # of that query (the multiple is that query's weight on it)
        cross = np.cross(dv[0, L - 1, 0, :3], do[0, L - 1, 0, :3])
        assert np.abs(cross).max() < 1e-12


# -- grouped key/value heads (GQA / MQA) ---------------------------------------------------------

@pytest.mark.parametrize("Hk", [1, 2, 3, 6])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_kv_heads_equal_repeated_heads(Hk, causal):
    """H query heads over Hk key/value heads equal ordinary attention with each key/value
    head repeated for its H/Hk consecutive query heads (numpy repeat); Hk = H is plain
    attention and Hk = 1 is multi-query attention."""
    B, L, H, D = 2, 19, 6, 5
    q = _rand((B, L, H, D), 90)
    k, v = _rand((B, L, Hk, D), 91), _rand((B, L, Hk, D), 92)
    got, lg = oracle.attention(q, k, v, causal=causal)
    rep = H // Hk
    ref, lr = oracle.attention(q, np.repeat(k, rep, axis=2), np.repeat(v, rep, axis=2),
                               causal=causal)
    assert np.abs(got - ref).max() < 1e-15 and np.abs(lg - lr).max() < 1e-15
    # each query head really uses its own group: scipy on head h with key head h // rep
    for h in (0, H - 1):
        s = q[0, :, h] @ k[0, :, h // rep].T / math.sqrt(D)
        if causal:
            s = np.where(np.tril(np.ones((L, L), bool)), s, -np.inf)
        np.testing.assert_allclose(got[0, :, h], scipy.special.softmax(s, 1) @ v[0, :, h // rep],
                                   rtol=1e-13, atol=1e-13)


def test_grouped_kv_heads_must_divide():
    with pytest.raises(ValueError):
        oracle.attention(np.zeros((1, 4, 6, 2)), np.zeros((1, 4, 4, 2)), np.zeros((1, 4, 4, 2)))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_dq_rows_match_full_backward(causal):
    """The per-row dq routine (for long sequences) reproduces the rows of the full
    backward, which the finite-difference and autograd pins tie down."""
    B, L, H, D = 2, 29, 2, 6
    q, k, v, do = (_rand((B, L, H, D), 100 + i) for i in range(4))
    dq, _, _ = oracle.attention_bwd(q, k, v, do, causal=causal)
    rows = [0, 1, 13, 28]
    part = oracle.attention_bwd_dq_rows(q, k, v, do, rows, causal=causal)
    np.testing.assert_allclose(part, dq[:, rows], rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_dkdv_rows_match_full_backward(causal):
    """The per-key-row dk, dv routine (for long sequences) reproduces the key rows of the
    full backward, which the finite-difference and autograd pins tie down, and its
    per-query pass reproduces the forward oracle."""
    B, L, H, D = 2, 29, 2, 6
    q, k, v, do = (_rand((B, L, H, D), 110 + i) for i in range(4))
    _, dk, dv = oracle.attention_bwd(q, k, v, do, causal=causal)
    rows = [0, 1, 13, 27, 28]
    pk, pv, lse, o = oracle.attention_bwd_dkdv_rows(q, k, v, do, rows, causal=causal,
                                                    stats=True)
    np.testing.assert_allclose(pk, dk[:, rows], rtol=0, atol=1e-14)
    np.testing.assert_allclose(pv, dv[:, rows], rtol=0, atol=1e-14)
    # the per-query pass is the naive forward: same output and lse as the forward oracle
    ref, lref = oracle.attention(q, k, v, causal=causal)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lref, rtol=0, atol=1e-14)


def test_backward_dkdv_rows_match_torch_autograd():
    """Key rows of fp64 torch autograd of softmax(q k^T / sqrt(D)) v (a library route,
    independent of both chain-rule routines), causal and not."""
    torch = pytest.importorskip("torch")
    B, L, H, D = 1, 41, 3, 8
    q, k, v, do = (_rand((B, L, H, D), 120 + i) for i in range(4))
    rows = [0, 7, 20, 39, 40]
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
        s = torch.einsum("bihd,bjhd->bhij", tq, tk) / math.sqrt(D)
        if causal:
            s = s.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
        o = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), tv)
        o.backward(torch.tensor(do))
        pk, pv = oracle.attention_bwd_dkdv_rows(q, k, v, do, rows, causal=causal)
        np.testing.assert_allclose(pk, tk.grad.numpy()[:, rows], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(pv, tv.grad.numpy()[:, rows], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_dkdv_rows_closed_forms(causal):
    """With every key row listed: the dv rows sum to the sum of dO over queries (rows of P
    sum to 1) and the dk rows sum to zero (rows of dS sum to 0); under causal masking the
    last key is seen by the last query alone, so its dv is that query's dO times its
    weight on it."""
    B, L, H, D = 1, 17, 2, 5
    q, k, v, do = (_rand((B, L, H, D), 130 + i) for i in range(4))
    pk, pv = oracle.attention_bwd_dkdv_rows(q, k, v, do, list(range(L)), causal=causal)
    np.testing.assert_allclose(pv.sum(axis=1), do.sum(axis=1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(pk.sum(axis=1), 0.0, rtol=0, atol=1e-12)
    if causal:
        cross = np.cross(pv[0, L - 1, 0, :3], do[0, L - 1, 0, :3])
        assert np.abs(cross).max() < 1e-12
        # and its weight is the last query's softmax weight on it, computed by scipy
        s = q[0, L - 1, 0] @ k[0, :, 0].T / math.sqrt(D)
        w = scipy.special.softmax(s)[L - 1]
        np.testing.assert_allclose(pv[0, L - 1, 0], w * do[0, L - 1, 0], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("Hk", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_backward_matches_finite_differences(Hk, causal):
    """Gradients with grouped key/value heads are the gradient of sum(O * dO) where O is
    the grouped forward oracle itself: central differences (independent of the repeat
    and sum inside attention_bwd_gqa)."""
    B, L, H, D = 1, 4, 4, 3
    q, do = _rand((B, L, H, D), 90), _rand((B, L, H, D), 91)
    k, v = _rand((B, L, Hk, D), 92), _rand((B, L, Hk, D), 93)
    dq, dk, dv = oracle.attention_bwd_gqa(q, k, v, do, causal=causal)
    assert dk.shape == k.shape and dv.shape == v.shape and dq.shape == q.shape

    def loss(q_, k_, v_):
        o, _ = oracle.attention(q_, k_, v_, causal=causal, threads=1)
        return float((o * do).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (loss(**{k_ + "_": a for k_, a in args_p.items()})
                        - loss(**{k_ + "_": a for k_, a in args_m.items()})) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-7, err_msg=name)


def test_grouped_backward_with_one_group_per_head_is_plain_backward():
    """Hk = H: every group has one query head, the plain backward."""
    B, L, H, D = 2, 9, 3, 4
    q, k, v, do = (_rand((B, L, H, D), 94 + i) for i in range(4))
    for causal in (False, True):
        a = oracle.attention_bwd_gqa(q, k, v, do, causal=causal)
        b = oracle.attention_bwd(q, k, v, do, causal=causal)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)
