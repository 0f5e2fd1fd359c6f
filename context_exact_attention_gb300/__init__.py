"""Exact context-parallel attention on one GB300: thin Python binding of libringattn.so.

Every function here only checks tensor properties, allocates outputs with
torch when the caller passes none, and forwards raw device pointers to the C
ABI declared in ``include/ring_attn.h``.  All arithmetic runs in the library's
CUDA kernels; there is no fallback of any kind, and calling into a missing or
unbuilt library raises.

Layout: q, k, v, out are contiguous [B, L, H, D]; lse is fp32 [B, L, H].
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import workloads  # noqa: F401  (seeded inputs; no attention arithmetic)

__all__ = [
    "RingAttnError", "library_path", "load_library", "ring_attn_fwd", "ring_attn_fwd_f32",
    "ring_attn_fwd_trace", "attn_merge_partials", "ulysses_seq2head", "ulysses_head2seq",
    "ulysses_attention", "ring_attn_bwd", "ring_attn_fwd_gqa", "ring_attn_fwd_zigzag",
    "zigzag_positions", "ring_attn_fwd_varlen", "varlen_padded_length", "check_status",
    "probe_wait_timeout", "ring_attn_fwd_host", "host_workspace_bytes", "ring_attn_bwd_gqa",
    "ring_attn_bwd_zigzag", "ring_attn_bwd_varlen", "ring_attn_fwd_ex", "ring_attn_bwd_ex",
    "ulysses_attention_fused", "varlen_schedule", "EXPORTED_SYMBOLS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libringattn.so")
_DEBUG_LIB_PATH = os.path.join(_PKG, "libringattn_debug.so")
_lock = threading.Lock()
_lib = None
_debug_lib = None

RA_BF16, RA_F32 = 0, 1
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "misaligned",
           4: "not divisible", 5: "CUDA error", 6: "device-side wait timed out",
           7: "index check of the debug build failed"}

EXPORTED_SYMBOLS = (
    "ring_attn_fwd", "ring_attn_fwd_f32", "ring_attn_fwd_trace", "attn_merge_partials",
    "ulysses_seq2head", "ulysses_head2seq", "ra_check_status", "ra_status_string",
    "ra_probe_wait_timeout", "ring_attn_bwd", "ring_attn_bwd_workspace_bytes",
    "ring_attn_bwd_noalloc", "ring_attn_fwd_gqa", "ring_attn_fwd_zigzag",
    "ring_attn_fwd_varlen", "ring_attn_fwd_host", "ring_attn_fwd_host_workspace_bytes",
    "ring_attn_bwd_gqa", "ring_attn_bwd_zigzag", "ring_attn_bwd_varlen", "ring_attn_fwd_ex",
    "ring_attn_bwd_ex", "ulysses_attention_fused", "ring_attn_varlen_schedule",
    "ring_attn_varlen_schedule_bytes", "ra_padded_length", "ra_probe_bounds_check",
)


LAYOUTS = {"contiguous": 0, "zigzag": 1, "packed": 2}


class AttnDesc(ctypes.Structure):
    """Mirror of ra_attn_desc (include/ring_attn.h)."""
    _fields_ = [("B", ctypes.c_int), ("L", ctypes.c_int), ("H", ctypes.c_int),
                ("H_kv", ctypes.c_int), ("D", ctypes.c_int), ("P", ctypes.c_int),
                ("causal", ctypes.c_int), ("layout", ctypes.c_int),
                ("cu_seqlens", ctypes.c_void_p), ("n_seqs", ctypes.c_int),
                ("dtype", ctypes.c_int), ("schedule", ctypes.c_void_p)]


class RingAttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {_STATUS.get(code, 'unknown')} (status {code})")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load_library(build_if_missing: bool = False):
    """Load libringattn.so (ctypes).  Raises if it is absent and not built here."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = _open(_LIB_PATH, build_if_missing, debug_bounds=False)
        return _lib


def load_debug_library(build_if_missing: bool = False):
    """Load libringattn_debug.so: the same entry points compiled with an index check on
    every global load and store of the kernels (a failed check is skipped and reported
    by ra_check_status as status 7).  For tests and debugging, not for speed."""
    global _debug_lib
    with _lock:
        if _debug_lib is None:
            _debug_lib = _open(_DEBUG_LIB_PATH, build_if_missing, debug_bounds=True)
        return _debug_lib


def _open(path, build_if_missing, debug_bounds):
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(
                f"{path} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        from . import _build
        _build.build(debug_bounds=debug_bounds)
    lib = ctypes.CDLL(path)
    vp, i, ll, f_p = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_void_p
    sigs = {
        "ring_attn_fwd": [vp, vp, vp, vp, f_p, i, i, i, i, i, i, vp],
        "ring_attn_fwd_f32": [vp, vp, vp, vp, f_p, i, i, i, i, i, i, vp],
        "ring_attn_fwd_trace": [vp, vp, vp, vp, f_p, i, i, i, i, i, i, i, vp, vp],
        "attn_merge_partials": [vp, vp, vp, vp, vp, vp, ll, i, i, vp],
        "ulysses_seq2head": [vp, vp, i, i, i, i, i, i, vp],
        "ulysses_head2seq": [vp, vp, i, i, i, i, i, i, vp],
        "ra_check_status": [vp],
        "ra_probe_wait_timeout": [ctypes.c_ulonglong, vp],
        "ra_probe_bounds_check": [vp],
        "ring_attn_bwd": [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_ulonglong,
                          i, i, i, i, i, i, vp],
        "ring_attn_bwd_noalloc": [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp],
        "ring_attn_bwd_gqa": [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_ulonglong,
                              i, i, i, i, i, i, i, vp],
        "ring_attn_bwd_zigzag": [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_ulonglong,
                                 i, i, i, i, i, vp],
        "ring_attn_bwd_varlen": [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_ulonglong,
                                 vp, i, i, i, i, i, i, vp],
        "ring_attn_fwd_ex": [vp, vp, vp, vp, vp, f_p, vp, vp],
        "ulysses_attention_fused": [vp, vp, vp, vp, f_p, i, i, i, i, i, i, i, vp],
        "ring_attn_bwd_ex": [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                             ctypes.c_ulonglong, vp],
        "ring_attn_fwd_gqa": [vp, vp, vp, vp, f_p, i, i, i, i, i, i, i, i, vp],
        "ring_attn_fwd_zigzag": [vp, vp, vp, vp, f_p, i, i, i, i, i, i, vp, vp],
        "ring_attn_fwd_varlen": [vp, vp, vp, vp, f_p, vp, i, i, i, i, i, i, i, vp, vp],
        "ring_attn_fwd_host": [vp, vp, vp, vp, f_p, vp, ctypes.c_ulonglong, i, i, i, i, i, i,
                               i, vp],
        "ring_attn_varlen_schedule": [vp, i, i, i, i, vp, ctypes.c_ulonglong, vp],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.ring_attn_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.ring_attn_fwd_host_workspace_bytes.restype = ctypes.c_ulonglong
    lib.ring_attn_bwd_workspace_bytes.argtypes = [i, i, i]
    lib.ring_attn_bwd_workspace_bytes.restype = ctypes.c_ulonglong
    lib.ring_attn_varlen_schedule_bytes.argtypes = [i, i]
    lib.ring_attn_varlen_schedule_bytes.restype = ctypes.c_ulonglong
    lib.ra_status_string.argtypes = [ctypes.c_int]
    lib.ra_status_string.restype = ctypes.c_char_p
    lib.ra_padded_length.argtypes = [ctypes.c_longlong, i, i]
    lib.ra_padded_length.restype = ctypes.c_longlong
    return lib


def _call(name, *args):
    rc = getattr(load_library(), name)(*args)
    if rc != 0:
        raise RingAttnError(name, rc)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check_qkv(q, k, v, dtype, grouped=False):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, L, H, D] tensor")
    if grouped:
        if k.shape != v.shape or k.shape[0] != q.shape[0] or k.shape[1] != q.shape[1] \
                or k.shape[3] != q.shape[3]:
            raise ValueError("k, v must be [B, L, H_kv, D] matching q's B, L, D")
    elif not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v must have the same shape")


def _attn(name, q, k, v, P, causal, out, lse, want_lse, dtype, stream, trace=None):
    _check_qkv(q, k, v, dtype)
    B, L, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, L, H), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, L, H)
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [B, L, H] tensor")
    if trace is None:
        _call(name, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L, H, D, P,
              int(bool(causal)), _stream(stream))
    else:
        _call(name, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L, H, D, P,
              int(bool(causal)), RA_BF16 if dtype == torch.bfloat16 else RA_F32, _ptr(trace),
              _stream(stream))
    return out, lse


def ring_attn_fwd(q, k, v, P: int = 1, causal: bool = False, out=None, lse=None,
                  want_lse: bool = True, stream=None):
    """bf16 ring attention forward over P virtual shards.  Returns (out, lse)."""
    return _attn("ring_attn_fwd", q, k, v, P, causal, out, lse, want_lse, torch.bfloat16, stream)


def host_workspace_bytes(B: int, L: int, H: int, D: int, heads_per_group: int) -> int:
    """Device workspace bytes ring_attn_fwd_host needs (0 for invalid sizes)."""
    return int(load_library().ring_attn_fwd_host_workspace_bytes(B, L, H, D, heads_per_group))


def ring_attn_fwd_host(q, k, v, P: int = 1, causal: bool = False, out=None, lse=None,
                       want_lse: bool = True, heads_per_group: int | None = None,
                       workspace=None, device=None, stream=None):
    """ring_attn_fwd on HOST bf16 [B, L, H, D] tensors (pin them for overlap): the
    library copies head groups in, runs the attention and copies the results back,
    overlapping the three.  Returns host (out, lse) once the work is enqueued on
    `stream`; synchronize the stream before reading them."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 [B, L, H, D] host tensor")
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v must have the same shape")
    B, L, H, D = q.shape
    if heads_per_group is None:
        heads_per_group = next(g for g in (4, 2, 1) if H % g == 0)
    dev = torch.device(device) if device is not None else torch.device(
        "cuda", torch.cuda.current_device())
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin)
    if lse is None and want_lse:
        lse = torch.empty((B, L, H), dtype=torch.float32, pin_memory=pin)
    if out.is_cuda or (lse is not None and lse.is_cuda):
        raise ValueError("out and lse must be host tensors")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, L, H)
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [B, L, H] tensor")
    need = host_workspace_bytes(B, L, H, D, heads_per_group)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if not workspace.is_cuda:
        raise ValueError("workspace must be a device tensor")
    _call("ring_attn_fwd_host", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace),
          ctypes.c_ulonglong(workspace.numel() * workspace.element_size()), B, L, H, D, P,
          int(bool(causal)), int(heads_per_group), _stream(stream))
    return out, lse


def ring_attn_fwd_f32(q, k, v, P: int = 1, causal: bool = False, out=None, lse=None,
                      want_lse: bool = True, stream=None):
    """fp32 ring attention forward (SIMT path).  Returns (out, lse)."""
    return _attn("ring_attn_fwd_f32", q, k, v, P, causal, out, lse, want_lse, torch.float32,
                 stream)


def ring_attn_fwd_gqa(q, k, v, P: int = 1, causal: bool = False, out=None, lse=None,
                      want_lse: bool = True, stream=None):
    """Ring attention forward with grouped key/value heads: q [B, L, H, D], k and v
    [B, L, H_kv, D] (bf16 or fp32), query head h reading key/value head h // (H // H_kv).
    Returns (out, lse)."""
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q must be bf16 or fp32")
    _check_qkv(q, k, v, dtype, grouped=True)
    B, L, H, D = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, L, H), dtype=torch.float32, device=q.device)
    _call("ring_attn_fwd_gqa", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L, H, Hkv, D,
          P, int(bool(causal)), RA_BF16 if dtype == torch.bfloat16 else RA_F32, _stream(stream))
    return out, lse


def zigzag_positions(L: int, P: int):
    """Global position of every row of the zigzag layout (shard r holds chunks r and
    2P-1-r of 2P chunks): a list of L ints.  Index bookkeeping only."""
    c = L // (2 * P)
    pos = []
    for r in range(P):
        pos.extend(range(r * c, (r + 1) * c))
        pos.extend(range((2 * P - 1 - r) * c, (2 * P - r) * c))
    return pos


def ring_attn_fwd_zigzag(q, k, v, P: int = 1, out=None, lse=None, want_lse: bool = True,
                         trace: bool = False, stream=None):
    """Causal ring attention over the zigzag shard layout (rows in zigzag order, see
    zigzag_positions).  bf16 or fp32.  Returns (out, lse) or (out, lse, trace)."""
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q must be bf16 or fp32")
    _check_qkv(q, k, v, dtype)
    B, L, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, L, H), dtype=torch.float32, device=q.device)
    tr = torch.full((P, P), -7, dtype=torch.int32, device=q.device) if trace else None
    _call("ring_attn_fwd_zigzag", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L, H, D, P,
          RA_BF16 if dtype == torch.bfloat16 else RA_F32, _ptr(tr), _stream(stream))
    return (out, lse, tr) if trace else (out, lse)


def varlen_padded_length(total: int, P: int, multiple: int = 1) -> int:
    """Smallest length >= total that P shards of a multiple of `multiple` rows divide:
    ceil(total / (P * multiple)) * P * multiple (the Ulysses guideline page's
    padded_seq_len rule, e.g. 3000 tokens, 4 shards, multiple 8 -> 3008), computed by
    the library's ra_padded_length."""
    n = load_library().ra_padded_length(int(total), int(P), int(multiple))
    if n < 0:
        raise ValueError(f"no padded length for total={total}, P={P}, multiple={multiple}")
    return int(n)


def ring_attn_fwd_varlen(q, k, v, cu_seqlens, P: int = 1, causal: bool = False, out=None,
                         lse=None, want_lse: bool = True, trace: bool = False, stream=None,
                         schedule=None):
    """Ring attention over packed sequences.  q, k, v: [L, H, D] (bf16 or fp32);
    cu_seqlens: int32 CUDA tensor [n_seqs + 1] of sequence starts ending with L;
    schedule: None, or varlen_schedule(cu_seqlens, L, P, causal) (same results, heaviest
    work units first; passed through ring_attn_fwd_ex).  Returns (out, lse) or
    (out, lse, trace)."""
    if schedule is not None:
        return ring_attn_fwd_ex(q, k, v, P=P, causal=causal, layout="packed",
                                cu_seqlens=cu_seqlens, out=out, lse=lse, want_lse=want_lse,
                                trace=trace, stream=stream, schedule=schedule)
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q must be bf16 or fp32")
    if q.dim() != 3:
        raise ValueError("packed q, k, v are [L, H, D]")
    _check_qkv(q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), dtype)
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    L, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((L, H), dtype=torch.float32, device=q.device)
    tr = torch.full((P, P), -7, dtype=torch.int32, device=q.device) if trace else None
    _call("ring_attn_fwd_varlen", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
          _ptr(cu_seqlens), cu_seqlens.numel() - 1, L, H, D, P, int(bool(causal)),
          RA_BF16 if dtype == torch.bfloat16 else RA_F32, _ptr(tr), _stream(stream))
    return (out, lse, tr) if trace else (out, lse)


def ring_attn_fwd_trace(q, k, v, P: int = 1, causal: bool = False, stream=None):
    """Attention forward that also returns the [P, P] schedule trace (source shard per
    (shard, step), -1 where skipped).  Returns (out, lse, trace)."""
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q must be bf16 or fp32")
    trace = torch.full((P, P), -7, dtype=torch.int32, device=q.device)
    out, lse = _attn("ring_attn_fwd_trace", q, k, v, P, causal, None, None, True, dtype, stream,
                     trace=trace)
    return out, lse, trace


def attn_merge_partials(o_a, lse_a, o_b, lse_b, o_out=None, lse_out=None, stream=None):
    """LSE merge of two partials: o_*: [..., D] (bf16 or fp32), lse_*: [...] fp32."""
    for t in (o_a, o_b, lse_a, lse_b):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("merge inputs must be contiguous CUDA tensors")
    if o_a.dtype not in (torch.bfloat16, torch.float32) or o_b.dtype != o_a.dtype:
        raise ValueError("o_a, o_b must both be bf16 or both fp32")
    if lse_a.dtype != torch.float32 or lse_b.dtype != torch.float32:
        raise ValueError("lse tensors must be fp32")
    if o_a.shape != o_b.shape or lse_a.shape != o_a.shape[:-1] or lse_b.shape != lse_a.shape:
        raise ValueError("shape mismatch")
    D = o_a.shape[-1]
    rows = o_a.numel() // D
    if o_out is None:
        o_out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    _call("attn_merge_partials", _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o_out),
          _ptr(lse_out), rows, D, RA_BF16 if o_a.dtype == torch.bfloat16 else RA_F32,
          _stream(stream))
    return o_out, lse_out


def _permute(name, x, P, out_shape, B, L, H, D, out, stream):
    if not x.is_cuda or not x.is_contiguous() or x.element_size() not in (2, 4):
        raise ValueError("x must be a contiguous CUDA tensor of 2- or 4-byte elements")
    if out is None:
        out = torch.empty(out_shape, dtype=x.dtype, device=x.device)
    _call(name, _ptr(x), _ptr(out), B, L, H, D, P, x.element_size(), _stream(stream))
    return out


def ulysses_seq2head(x, P: int, out=None, stream=None):
    """[P, B, L/P, H, D] sequence-sharded -> [P, B, L, H/P, D] head-sharded (bit copy)."""
    Pp, B, Ls, H, D = x.shape
    if Pp != P or H % P:
        raise ValueError("x must be [P, B, L/P, H, D] with H divisible by P")
    return _permute("ulysses_seq2head", x, P, (P, B, Ls * P, H // P, D), B, Ls * P, H, D, out,
                    stream)


def ulysses_head2seq(x, P: int, out=None, stream=None):
    """[P, B, L, H/P, D] head-sharded -> [P, B, L/P, H, D] sequence-sharded (bit copy)."""
    Pp, B, L, Hg, D = x.shape
    if Pp != P or L % P:
        raise ValueError("x must be [P, B, L, H/P, D] with L divisible by P")
    return _permute("ulysses_head2seq", x, P, (P, B, L // P, Hg * P, D), B, L, Hg * P, D, out,
                    stream)


def ulysses_attention(q_seq, k_seq, v_seq, P: int, stream=None, buffers=None):
    """Ulysses path: seq->head transpose of q, k, v; full non-causal attention per head
    group (the head-sharded buffer is a [P*B, L, H/P, D] batch); head->seq transpose of
    the output.  Inputs [P, B, L/P, H, D] bf16 (k, v may have H_kv < H heads, with
    H_kv divisible by P as well).  Returns the output in the same layout."""
    Pp, B, Ls, H, D = q_seq.shape
    Hkv = k_seq.shape[3]
    L, Hg, Hkg = Ls * P, H // P, Hkv // P
    if Hkv % P:
        raise ValueError("key/value heads must be divisible by P for the Ulysses transpose")
    if buffers is None:
        buffers = {n: torch.empty((P, B, L, Hkg if n in ("k", "v") else Hg, D), dtype=q_seq.dtype,
                                  device=q_seq.device) for n in ("q", "k", "v", "o")}
    qh = ulysses_seq2head(q_seq, P, out=buffers["q"], stream=stream)
    kh = ulysses_seq2head(k_seq, P, out=buffers["k"], stream=stream)
    vh = ulysses_seq2head(v_seq, P, out=buffers["v"], stream=stream)
    shape, kv_shape = (P * B, L, Hg, D), (P * B, L, Hkg, D)
    if Hkv == H:
        ring_attn_fwd(qh.view(shape), kh.view(shape), vh.view(shape), P=1, causal=False,
                      out=buffers["o"].view(shape), want_lse=False, stream=stream)
    else:
        ring_attn_fwd_gqa(qh.view(shape), kh.view(kv_shape), vh.view(kv_shape), P=1,
                          causal=False, out=buffers["o"].view(shape), want_lse=False,
                          stream=stream)
    return ulysses_head2seq(buffers["o"], P, stream=stream)


def ulysses_attention_fused(q_seq, k_seq, v_seq, P: int, causal: bool = False, out=None,
                            lse=None, want_lse: bool = False, stream=None):
    """The Ulysses step on sequence-sharded bf16 buffers q_seq [P, B, L/P, H, D] and
    k_seq, v_seq [P, B, L/P, H_kv, D] in one kernel (the transposes folded into the tensor
    maps' addressing).  Returns (out [P, B, L/P, H, D], lse [P, B, L/P, H] or None), the
    same bits as ulysses_attention."""
    for name, t in (("q_seq", q_seq), ("k_seq", k_seq), ("v_seq", v_seq)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 5 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [P, B, L/P, H, D]")
    Pp, B, Ls, H, D = q_seq.shape
    if Pp != P or k_seq.shape != v_seq.shape or k_seq.shape[:3] != q_seq.shape[:3] \
            or k_seq.shape[4] != D:
        raise ValueError("q_seq, k_seq, v_seq must share P, B, L/P and D")
    if out is None:
        out = torch.empty_like(q_seq)
    if lse is None and want_lse:
        lse = torch.empty(q_seq.shape[:4], dtype=torch.float32, device=q_seq.device)
    _call("ulysses_attention_fused", _ptr(q_seq), _ptr(k_seq), _ptr(v_seq), _ptr(out), _ptr(lse),
          B, Ls * P, H, k_seq.shape[3], D, P, int(bool(causal)), _stream(stream))
    return out, lse


def ring_attn_bwd(q, k, v, out, lse, dout, P: int = 1, causal: bool = False, dq=None, dk=None,
                  dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of ring_attn_fwd for the upstream gradient dout (bf16).

    out and lse are the forward's results for the same q, k, v, P, causal.  The
    workspace (fp32, one value per query row) is allocated with torch if not given."""
    _check_qkv(q, k, v, torch.bfloat16)
    for name, t in (("out", out), ("dout", dout)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    B, L, H, D = q.shape
    if lse is None or lse.dtype != torch.float32 or tuple(lse.shape) != (B, L, H):
        raise ValueError("lse must be the forward's fp32 [B, L, H] tensor")
    lib = load_library()
    need = lib.ring_attn_bwd_workspace_bytes(B, L, H)
    if workspace is None:
        workspace = torch.empty(max(1, need // 4), dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _call("ring_attn_bwd", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
          _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(), B, L,
          H, D, P, int(bool(causal)), _stream(stream))
    return dq, dk, dv


def ring_attn_bwd_gqa(q, k, v, out, lse, dout, P: int = 1, causal: bool = False, dq=None,
                      dk=None, dv=None, workspace=None, stream=None):
    """Gradients of ring_attn_fwd_gqa: q, out, dout [B, L, H, D]; k, v [B, L, H_kv, D];
    returns dq like q and dk, dv like k (summed over each key/value head's query heads)."""
    _check_qkv(q, k, v, torch.bfloat16, grouped=True)
    for name, t in (("out", out), ("dout", dout)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    B, L, H, D = q.shape
    Hkv = k.shape[2]
    if lse is None or lse.dtype != torch.float32 or tuple(lse.shape) != (B, L, H):
        raise ValueError("lse must be the forward's fp32 [B, L, H] tensor")
    lib = load_library()
    need = lib.ring_attn_bwd_workspace_bytes(B, L, H)
    if workspace is None:
        workspace = torch.empty(max(1, need // 4), dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _call("ring_attn_bwd_gqa", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
          _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
          workspace.numel() * workspace.element_size(), B, L, H, Hkv, D, P, int(bool(causal)),
          _stream(stream))
    return dq, dk, dv


def _bwd_outputs(q, k, v, out, lse, dout, lse_shape, dq, dk, dv, workspace, rows):
    for name, t in (("out", out), ("dout", dout)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    if lse is None or lse.dtype != torch.float32 or tuple(lse.shape) != lse_shape:
        raise ValueError(f"lse must be the forward's fp32 {list(lse_shape)} tensor")
    if workspace is None:
        workspace = torch.empty(max(1, rows), dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    return dq, dk, dv, workspace


def ring_attn_bwd_zigzag(q, k, v, out, lse, dout, P: int = 1, dq=None, dk=None, dv=None,
                         workspace=None, stream=None):
    """Gradients of ring_attn_fwd_zigzag (bf16, causal): every tensor in the zigzag row
    order of the forward (see zigzag_positions); returns (dq, dk, dv) in that order."""
    _check_qkv(q, k, v, torch.bfloat16)
    B, L, H, D = q.shape
    dq, dk, dv, workspace = _bwd_outputs(q, k, v, out, lse, dout, (B, L, H), dq, dk, dv,
                                         workspace, B * L * H)
    _call("ring_attn_bwd_zigzag", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
          _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
          workspace.numel() * workspace.element_size(), B, L, H, D, P, _stream(stream))
    return dq, dk, dv


def ring_attn_bwd_varlen(q, k, v, out, lse, dout, cu_seqlens, P: int = 1, causal: bool = False,
                         dq=None, dk=None, dv=None, workspace=None, stream=None, schedule=None):
    """Gradients of ring_attn_fwd_varlen (bf16): q, k, v, out, dout [L, H, D], lse [L, H],
    cu_seqlens the forward's int32 CUDA tensor; schedule as ring_attn_fwd_varlen.
    Returns (dq, dk, dv), each [L, H, D]."""
    if schedule is not None:
        return ring_attn_bwd_ex(q, k, v, out, lse, dout, P=P, causal=causal, layout="packed",
                                cu_seqlens=cu_seqlens, dq=dq, dk=dk, dv=dv, workspace=workspace,
                                stream=stream, schedule=schedule)
    if q.dim() != 3:
        raise ValueError("packed q, k, v are [L, H, D]")
    _check_qkv(q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), torch.bfloat16)
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    L, H, D = q.shape
    dq, dk, dv, workspace = _bwd_outputs(q, k, v, out, lse, dout, (L, H), dq, dk, dv, workspace,
                                         L * H)
    _call("ring_attn_bwd_varlen", _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
          _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _ptr(cu_seqlens), cu_seqlens.numel() - 1,
          L, H, D, P, int(bool(causal)), _stream(stream))
    return dq, dk, dv


def _desc(q, k, P, causal, layout, cu_seqlens, schedule=None):
    """Descriptor and the [B, L, H, D] view of q for ring_attn_fwd_ex / ring_attn_bwd_ex."""
    if layout not in LAYOUTS:
        raise ValueError(f"layout must be one of {sorted(LAYOUTS)}")
    packed = layout == "packed"
    if schedule is not None:
        if not packed:
            raise ValueError("schedule belongs to the packed layout only")
        if schedule.dtype != torch.int32 or not schedule.is_cuda or not schedule.is_contiguous():
            raise ValueError("schedule must be the int32 CUDA tensor varlen_schedule returns")
    if packed:
        if q.dim() != 3 or k.dim() != 3:
            raise ValueError("packed q, k, v are [L, H, D] / [L, H_kv, D]")
        if (cu_seqlens is None or cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda
                or cu_seqlens.dim() != 1):
            raise ValueError("packed layout needs cu_seqlens, a 1-D int32 CUDA tensor")
        B, (L, H, D) = 1, q.shape
    else:
        if cu_seqlens is not None:
            raise ValueError("cu_seqlens belongs to the packed layout only")
        B, L, H, D = q.shape
    d = AttnDesc(B=B, L=L, H=H, H_kv=k.shape[-2], D=D, P=P, causal=int(bool(causal)),
                 layout=LAYOUTS[layout], cu_seqlens=cu_seqlens.data_ptr() if packed else None,
                 n_seqs=cu_seqlens.numel() - 1 if packed else 0,
                 dtype=RA_BF16 if q.dtype == torch.bfloat16 else RA_F32,
                 schedule=schedule.data_ptr() if schedule is not None else None)
    if schedule is not None and schedule.numel() * 4 < _schedule_bytes(L, P):
        raise ValueError("schedule is too short for this L and P")
    return d, (B, L, H, D)


def _schedule_bytes(L: int, P: int) -> int:
    return int(load_library().ring_attn_varlen_schedule_bytes(L, P))


def varlen_schedule(cu_seqlens, L: int, P: int = 1, causal: bool = False, stream=None):
    """Heaviest-first unit orders for the packed layout (ring_attn_varlen_schedule): an
    int32 CUDA tensor to pass as schedule= to the packed forward and backward with the
    same cu_seqlens, L and P.  Written asynchronously on `stream`."""
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    nbytes = _schedule_bytes(L, P)
    if nbytes == 0:
        raise ValueError("L and P must be positive with L % P == 0")
    sched = torch.empty(nbytes // 4, dtype=torch.int32, device=cu_seqlens.device)
    _call("ring_attn_varlen_schedule", _ptr(cu_seqlens), cu_seqlens.numel() - 1, L, P,
          int(bool(causal)), _ptr(sched), nbytes, _stream(stream))
    return sched


def ring_attn_fwd_ex(q, k, v, P: int = 1, causal: bool = False, layout: str = "contiguous",
                     cu_seqlens=None, out=None, lse=None, want_lse: bool = True,
                     trace: bool = False, stream=None, schedule=None):
    """The forward for any combination of options: grouped key/value heads (k, v with
    fewer heads than q) with the contiguous, zigzag or packed layout.  q, k, v: [B, L, H, D]
    / [B, L, H_kv, D], or [L, H, D] / [L, H_kv, D] for layout="packed" (with cu_seqlens).
    bf16 or fp32.  Returns (out, lse) or (out, lse, trace); lse is [B, L, H] or [L, H]."""
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q must be bf16 or fp32")
    d, (B, L, H, D) = _desc(q, k, P, causal, layout, cu_seqlens, schedule)
    view = (lambda t: t.unsqueeze(0)) if layout == "packed" else (lambda t: t)
    _check_qkv(view(q), view(k), view(v), dtype, grouped=True)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    tr = torch.full((P, P), -7, dtype=torch.int32, device=q.device) if trace else None
    _call("ring_attn_fwd_ex", ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
          _ptr(tr), _stream(stream))
    return (out, lse, tr) if trace else (out, lse)


def ring_attn_bwd_ex(q, k, v, out, lse, dout, P: int = 1, causal: bool = False,
                     layout: str = "contiguous", cu_seqlens=None, dq=None, dk=None, dv=None,
                     workspace=None, stream=None, schedule=None):
    """Gradients of ring_attn_fwd_ex (bf16) for the same options: returns (dq, dk, dv),
    dq shaped like q and dk, dv like k (summed over each key/value head's query heads)."""
    d, (B, L, H, D) = _desc(q, k, P, causal, layout, cu_seqlens, schedule)
    view = (lambda t: t.unsqueeze(0)) if layout == "packed" else (lambda t: t)
    _check_qkv(view(q), view(k), view(v), torch.bfloat16, grouped=True)
    dq, dk, dv, workspace = _bwd_outputs(q, k, v, out, lse, dout, tuple(q.shape[:-1]), dq, dk,
                                         dv, workspace, B * L * H)
    _call("ring_attn_bwd_ex", ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
          _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream(stream))
    return dq, dk, dv


def check_status(stream=None) -> int:
    """Synchronise the stream and read/clear the device status word; returns the status code."""
    return getattr(load_library(), "ra_check_status")(_stream(stream))


def probe_wait_timeout(timeout_ns: int = 1_000_000, stream=None):
    _call("ra_probe_wait_timeout", ctypes.c_ulonglong(timeout_ns), _stream(stream))
