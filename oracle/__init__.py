"""fp64 CPU oracle for exact context-parallel attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library in ``context_exact_attention_gb300`` and never imports it.

The arithmetic lives in ``attn_oracle.c`` (plain loops, double precision); this
module only compiles it with gcc and marshals numpy arrays.  What each routine
computes, and the passage it follows:

* :func:`attention` -- naive ``softmax(Q K^T / sqrt(D)) V`` with lse, optional
  causal rule ``j <= i`` on global positions ("序列并行与 Ring Attention",
  sections 3.1 and 3.4; the naive reference of the juejin ring-attention
  debugging page, section 三).
* :func:`ring_attention` -- the online-softmax recurrence (section 3.2) applied
  in ring order ``(r - t) mod P`` (section 3.3) with whole-shard causal skip
  (section 3.4); also returns the P x P schedule trace.
* :func:`local_only` -- each shard attending only to its own K/V: the
  "did it communicate" comparison of the juejin page, section 二 step 4.
* :func:`merge` -- the log-sum-exp ``combine`` of two partials (juejin page,
  section 四).
* :func:`seq2head` / :func:`head2seq` -- Ulysses all-to-all layout transposes
  (section 3.5), as byte copies.
* :func:`attention_bwd` -- gradients dQ, dK, dV of the attention output by the
  chain rule (the backward of sections 3.3 and 6.2, summed on one device).
* :func:`attention_bwd_dq_rows` / :func:`attention_bwd_dkdv_rows` -- the same
  gradients for chosen query rows (dq) or key rows (dk, dv) only, for long
  sequences: a query row needs only its own scores; a key row needs every query's
  softmax normaliser and row dot, computed first by the naive loops.

Every pin of these routines is in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``liboracle.so`` next to it (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            ip = ctypes.POINTER(ctypes.c_int)
            L = ctypes.c_long
            lib.oracle_attention.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, ctypes.c_int,
                                             L, L, lp, L, ctypes.c_int]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_attention_gqa.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, L,
                                                 ctypes.c_int, L, L, lp, L, ctypes.c_int]
            lib.oracle_attention_gqa.restype = ctypes.c_int
            lib.oracle_ring_attention.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, ctypes.c_int,
                                                  ip, ctypes.c_int]
            lib.oracle_ring_attention.restype = ctypes.c_int
            lib.oracle_merge.argtypes = [dp, dp, dp, dp, dp, dp, L, L]
            lib.oracle_merge.restype = ctypes.c_int
            lib.oracle_attention_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, L, L, L, L,
                                                 ctypes.c_int, ctypes.c_int]
            lib.oracle_attention_bwd.restype = ctypes.c_int
            lib.oracle_attention_bwd_dq_rows.argtypes = [dp, dp, dp, dp, dp, L, L, L, L,
                                                         ctypes.c_int, lp, L, ctypes.c_int]
            lib.oracle_attention_bwd_dq_rows.restype = ctypes.c_int
            lib.oracle_attention_bwd_dkdv_rows.argtypes = [dp, dp, dp, dp, dp, dp, L, L, L, L,
                                                           ctypes.c_int, lp, L, dp, dp,
                                                           ctypes.c_int]
            lib.oracle_attention_bwd_dkdv_rows.restype = ctypes.c_int
            for name in ("oracle_seq2head", "oracle_head2seq"):
                fn = getattr(lib, name)
                fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, L, L, L, L, L, L]
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def to_f64(x) -> np.ndarray:
    """Any array-like (numpy, or a CPU torch tensor of any float dtype) -> contiguous fp64 numpy.
    Arrays that already are contiguous fp64 are returned as they are (no copy)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    if isinstance(x, np.ndarray) and x.dtype == np.float64 and x.flags.c_contiguous:
        return x
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def attention(q, k, v, causal: bool = False, rows=None, q_pos0: int = 0, k_pos0: int = 0,
              threads: int | None = None):
    """Naive attention.  q: [B, Lq, H, D], k/v: [B, Lk, Hk, D] (any float type, computed in
    fp64).  Hk may be smaller than H (grouped key/value heads): H must be a multiple of
    Hk, and query head h reads key/value head h // (H // Hk).

    ``rows``: optional 1-D list of query rows to evaluate (the rest are not computed).
    Returns ``(out [B, n_rows, H, D], lse [B, n_rows, H])`` as fp64 numpy arrays.
    """
    lib = _load()
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, Lq, H, D = q.shape
    Lk, Hk = k.shape[1], k.shape[2]
    assert k.shape == (B, Lk, Hk, D) and v.shape == (B, Lk, Hk, D)
    if H % Hk:
        raise ValueError("query heads must be a multiple of key/value heads")
    if rows is None:
        n_rows, rows_p = Lq, None
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
        n_rows = rows_a.shape[0]
        rows_p = rows_a.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
    out = np.empty((B, n_rows, H, D), dtype=np.float64)
    lse = np.empty((B, n_rows, H), dtype=np.float64)
    rc = lib.oracle_attention_gqa(_dp(q), _dp(k), _dp(v), _dp(out), _dp(lse), B, Lq, Lk, H, Hk,
                                  D, int(bool(causal)), q_pos0, k_pos0, rows_p, n_rows,
                                  threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention failed ({rc})")
    return out, lse


def ring_attention(q, k, v, P: int, causal: bool = False, threads: int | None = None):
    """Ring-order blockwise recurrence over P equal virtual shards.

    Returns ``(out [B, L, H, D], lse [B, L, H], trace [P, P] int32)``.
    """
    lib = _load()
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, L, H, D = q.shape
    assert k.shape == q.shape and v.shape == q.shape
    out = np.empty_like(q)
    lse = np.empty((B, L, H), dtype=np.float64)
    trace = np.empty((P, P), dtype=np.int32)
    rc = lib.oracle_ring_attention(_dp(q), _dp(k), _dp(v), _dp(out), _dp(lse), B, L, H, D, P,
                                   int(bool(causal)),
                                   trace.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                   threads or default_threads())
    if rc == -2:
        raise ValueError("L must be divisible by P")
    if rc != 0:
        raise ValueError(f"oracle_ring_attention failed ({rc})")
    return out, lse, trace


def local_only(q, k, v, P: int, causal: bool = False, threads: int | None = None):
    """Each shard attends only to its own K/V block (no exchange between shards)."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, L, H, D = q.shape
    if L % P:
        raise ValueError("L must be divisible by P")
    Ls = L // P
    out = np.empty_like(q)
    lse = np.empty((B, L, H), dtype=np.float64)
    for r in range(P):
        sl = slice(r * Ls, (r + 1) * Ls)
        o, l = attention(q[:, sl], k[:, sl], v[:, sl], causal=causal, q_pos0=r * Ls,
                         k_pos0=r * Ls, threads=threads)
        out[:, sl], lse[:, sl] = o, l
    return out, lse


def attention_bwd(q, k, v, dout, causal: bool = False, threads: int | None = None):
    """Gradients (dq, dk, dv) of O = attention(q, k, v) for the upstream gradient dout.

    All [B, L, H, D]; small L only (two L x L matrices per (batch, head)).
    """
    lib = _load()
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    B, L, H, D = q.shape
    assert k.shape == q.shape and v.shape == q.shape and dout.shape == q.shape
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    rc = lib.oracle_attention_bwd(_dp(q), _dp(k), _dp(v), _dp(dout), _dp(dq), _dp(dk), _dp(dv),
                                  B, L, H, D, int(bool(causal)), threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd failed ({rc})")
    return dq, dk, dv


def attention_bwd_gqa(q, k, v, dout, causal: bool = False, threads: int | None = None):
    """Gradients with grouped key/value heads: q, dout [B, L, H, D]; k, v [B, L, Hk, D],
    query head h reading key/value head h // (H // Hk) (the forward oracle's rule).

    The grouped attention is ordinary attention on k, v with each key/value head repeated
    for its H // Hk query heads; the gradient of a repeated tensor is the sum of the
    gradients of its copies (chain rule of the copy), so dk, dv of head g sum the
    per-query-head gradients over the group.  Returns (dq [B,L,H,D], dk, dv [B,L,Hk,D])."""
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    B, L, H, D = q.shape
    Hk = k.shape[2]
    assert k.shape == (B, L, Hk, D) and v.shape == k.shape and dout.shape == q.shape
    if H % Hk:
        raise ValueError("query heads must be a multiple of key/value heads")
    G = H // Hk
    kr = np.ascontiguousarray(np.repeat(k, G, axis=2))
    vr = np.ascontiguousarray(np.repeat(v, G, axis=2))
    dq, dkr, dvr = attention_bwd(q, kr, vr, dout, causal=causal, threads=threads)
    dk = dkr.reshape(B, L, Hk, G, D).sum(axis=3)
    dv = dvr.reshape(B, L, Hk, G, D).sum(axis=3)
    return dq, dk, dv


def attention_bwd_dq_rows(q, k, v, dout, rows, causal: bool = False, threads: int | None = None):
    """dq of the listed query rows only (each row needs only its own scores): works at
    any sequence length.  Returns [B, len(rows), H, D]."""
    lib = _load()
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    B, L, H, D = q.shape
    rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    out = np.empty((B, rows_a.shape[0], H, D), dtype=np.float64)
    rc = lib.oracle_attention_bwd_dq_rows(_dp(q), _dp(k), _dp(v), _dp(dout), _dp(out), B, L, H, D,
                                          int(bool(causal)),
                                          rows_a.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                                          rows_a.shape[0], threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd_dq_rows failed ({rc})")
    return out


def attention_bwd_dkdv_rows(q, k, v, dout, rows, causal: bool = False,
                            threads: int | None = None, stats: bool = False):
    """dk and dv of the listed key rows only: dk_j and dv_j sum over every query that sees
    key j, so the routine first evaluates the naive forward of every query row (its lse
    and output O_i, whence the row dot dO_i . O_i), one pass over all query/key pairs,
    then the listed key rows.  Works at any sequence length.  Returns (dk, dv), each
    [B, len(rows), H, D]; with stats=True also the per-query lse [B, L, H] and output
    O [B, L, H, D] it computed on the way."""
    lib = _load()
    q, k, v, dout = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    B, L, H, D = q.shape
    assert k.shape == q.shape and v.shape == q.shape and dout.shape == q.shape
    rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    dk = np.empty((B, rows_a.shape[0], H, D), dtype=np.float64)
    dv = np.empty_like(dk)
    lse = np.empty((B, L, H), dtype=np.float64) if stats else None
    o = np.empty((B, L, H, D), dtype=np.float64) if stats else None
    null = ctypes.POINTER(ctypes.c_double)()
    rc = lib.oracle_attention_bwd_dkdv_rows(_dp(q), _dp(k), _dp(v), _dp(dout), _dp(dk), _dp(dv),
                                            B, L, H, D, int(bool(causal)),
                                            rows_a.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                                            rows_a.shape[0], _dp(lse) if stats else null,
                                            _dp(o) if stats else null,
                                            threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attention_bwd_dkdv_rows failed ({rc})")
    return (dk, dv, lse, o) if stats else (dk, dv)


def merge(o_a, lse_a, o_b, lse_b):
    """LSE combine of two partials.  o_*: [..., D], lse_*: [...] (same leading shape)."""
    lib = _load()
    o_a, o_b = to_f64(o_a), to_f64(o_b)
    lse_a, lse_b = to_f64(lse_a), to_f64(lse_b)
    lead = o_a.shape[:-1]
    D = o_a.shape[-1]
    rows = int(np.prod(lead)) if lead else 1
    assert o_b.shape == o_a.shape and lse_a.shape == lead and lse_b.shape == lead
    o = np.empty_like(o_a)
    lse = np.empty(lead, dtype=np.float64)
    rc = lib.oracle_merge(_dp(o_a), _dp(lse_a), _dp(o_b), _dp(lse_b), _dp(o), _dp(lse), rows, D)
    if rc != 0:
        raise ValueError(f"oracle_merge failed ({rc})")
    return o, lse


def _permute(name, x: np.ndarray, B, L, H, D, P, out_shape):
    lib = _load()
    x = np.ascontiguousarray(x)
    out = np.empty(out_shape, dtype=x.dtype)
    rc = getattr(lib, name)(x.ctypes.data, out.ctypes.data, B, L, H, D, P, x.dtype.itemsize)
    if rc == -2:
        raise ValueError("L and H must be divisible by P")
    if rc != 0:
        raise ValueError(f"{name} failed ({rc})")
    return out


def seq2head(x: np.ndarray, P: int) -> np.ndarray:
    """[P, B, L/P, H, D] sequence-sharded -> [P, B, L, H/P, D] head-sharded (any dtype, bit copy)."""
    Pp, B, Ls, H, D = x.shape
    assert Pp == P
    if H % P:
        raise ValueError("H must be divisible by P")
    return _permute("oracle_seq2head", x, B, Ls * P, H, D, P, (P, B, Ls * P, H // P, D))


def head2seq(x: np.ndarray, P: int) -> np.ndarray:
    """[P, B, L, H/P, D] head-sharded -> [P, B, L/P, H, D] sequence-sharded (bit copy)."""
    Pp, B, L, Hg, D = x.shape
    assert Pp == P
    if L % P:
        raise ValueError("L must be divisible by P")
    return _permute("oracle_head2seq", x, B, L, Hg * P, D, P, (P, B, L // P, Hg * P, D))
