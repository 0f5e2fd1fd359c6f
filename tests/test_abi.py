"""Host-side checks of the C ABI that need no GPU: the library builds, loads, and
exports every function that include/ring_attn.h declares."""
import ctypes
import os
import re

import pytest

import context_exact_attention_gb300 as cea
from context_exact_attention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ring_attn.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w \t*]*?[ \t*](\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return cea.load_library()


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(cea.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(cea.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_debug_library_exports_every_declared_symbol():
    """The index-checked debug build has the same entry points."""
    dbg = cea.load_debug_library(build_if_missing=True)
    for name in declared_functions():
        assert hasattr(dbg, name), name


def test_bounds_probe_is_refused_by_the_normal_build(lib):
    """The normal build has no index checks: the probe launches nothing."""
    assert lib.ra_probe_bounds_check(ctypes.c_void_p(0)) == 2     # RA_ERR_UNSUPPORTED


def test_status_strings(lib):
    for code in range(8):
        s = lib.ra_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.ra_status_string(99) == b"unknown status"


def test_argument_errors_are_caught_before_any_cuda_call(lib):
    """Validation runs on the host before the runtime is touched, so these codes come
    back even without a GPU."""
    fake = ctypes.c_void_p(1 << 20)            # 16-byte aligned, never dereferenced
    odd = ctypes.c_void_p((1 << 20) + 8)
    null = ctypes.c_void_p(0)
    s = ctypes.c_void_p(0)
    # null pointer
    assert lib.ring_attn_fwd(null, fake, fake, fake, null, 1, 256, 2, 128, 4, 0, s) == 1
    # L not divisible by P
    assert lib.ring_attn_fwd(fake, fake, fake, ctypes.c_void_p(1 << 40), null, 1, 250, 2, 128, 4, 0, s) == 4
    # misaligned
    assert lib.ring_attn_fwd(odd, fake, fake, ctypes.c_void_p(1 << 40), null, 1, 256, 2, 128, 4, 0, s) == 3
    # unsupported head dim for bf16
    assert lib.ring_attn_fwd(fake, fake, fake, ctypes.c_void_p(1 << 40), null, 1, 256, 2, 96, 4, 0, s) == 2
    # out overlapping q
    assert lib.ring_attn_fwd(fake, fake, fake, fake, null, 1, 256, 2, 128, 4, 0, s) == 1
    # permutes: H not divisible by P, and in == out
    assert lib.ulysses_seq2head(fake, ctypes.c_void_p(1 << 40), 1, 64, 6, 128, 4, 2, s) == 4
    assert lib.ulysses_seq2head(fake, fake, 1, 64, 8, 128, 4, 2, s) == 1
    assert lib.ulysses_seq2head(fake, ctypes.c_void_p(1 << 40), 1, 64, 8, 128, 4, 3, s) == 2
    # merge: zero rows is a no-op, partial overlap rejected, bad D
    assert lib.attn_merge_partials(null, null, null, null, null, null, 0, 128, 0, s) == 0
    assert lib.attn_merge_partials(fake, fake, fake, fake, ctypes.c_void_p((1 << 20) + 16), fake,
                                   10, 128, 0, s) == 1
    assert lib.attn_merge_partials(fake, fake, fake, fake, fake, fake, 10, 4, 0, s) == 2
    assert lib.ra_probe_wait_timeout(0, s) == 1


def test_zigzag_positions_layout_and_balance():
    """Shard r of the zigzag layout holds chunks r and 2P-1-r; every shard then has the
    same number of visible causal (query, key) pairs, while contiguous shards grow
    with r ("序列并行与 Ring Attention", section 3.4)."""
    for L, P in ((16, 2), (48, 3), (64, 4)):
        pos = cea.zigzag_positions(L, P)
        assert sorted(pos) == list(range(L))
        c, Ls = L // (2 * P), L // P
        for r in range(P):
            shard = pos[r * Ls:(r + 1) * Ls]
            assert shard[:c] == list(range(r * c, (r + 1) * c))
            assert shard[c:] == list(range((2 * P - 1 - r) * c, (2 * P - r) * c))
        work_zig = [sum(p + 1 for p in pos[r * Ls:(r + 1) * Ls]) for r in range(P)]
        work_contig = [sum(p + 1 for p in range(r * Ls, (r + 1) * Ls)) for r in range(P)]
        assert len(set(work_zig)) == 1
        assert work_contig == sorted(work_contig) and work_contig[0] < work_contig[-1]


def test_varlen_padded_length_rule():
    """ceil(total / (P * multiple)) * P * multiple: the Ulysses guideline page's example
    of 3000 tokens over 4 shards padded to 3008 (multiple 8), and no-ops when divisible."""
    assert cea.varlen_padded_length(3000, 4, 8) == 3008
    assert cea.varlen_padded_length(3008, 4, 8) == 3008
    assert cea.varlen_padded_length(1, 8) == 8
    for total in range(1, 200):
        for P in (1, 3, 4):
            n = cea.varlen_padded_length(total, P, 2)
            assert n >= total and n % (2 * P) == 0 and n - total < 2 * P


def test_padded_length_through_the_c_abi(lib):
    """ra_padded_length called through ctypes: the guideline page's example, exact
    multiples, zero, the largest length the kernels take, and the refused arguments."""
    f = lib.ra_padded_length
    f.argtypes = [ctypes.c_longlong, ctypes.c_int, ctypes.c_int]
    f.restype = ctypes.c_longlong
    assert f(3000, 4, 8) == 3008
    assert f(3008, 4, 8) == 3008
    assert f(0, 4, 8) == 0
    assert f(32768, 8, 128) == 32768 and f(32769, 8, 128) == 33792
    assert f(2 ** 31 - 1, 1, 1) == 2 ** 31 - 1
    assert f(2 ** 31 - 1, 2, 1) == -1                  # would be 2^31: beyond int
    assert f(2 ** 40, 1, 1) == -1
    assert f(-1, 4, 8) == -1 and f(10, 0, 8) == -1 and f(10, 4, 0) == -1
    for total in range(0, 300, 7):
        for P, m in ((1, 1), (3, 5), (8, 16)):
            n = f(total, P, m)
            assert n >= total and n % (P * m) == 0 and n - total < P * m


def test_host_entry_argument_errors(lib):
    """ring_attn_fwd_host checks its arguments on the host before touching the runtime."""
    fake = ctypes.c_void_p(1 << 20)
    out = ctypes.c_void_p(1 << 40)
    ws = ctypes.c_void_p(1 << 44)
    null = ctypes.c_void_p(0)
    s = ctypes.c_void_p(0)
    B, L, H, D, P = 1, 256, 8, 128, 4
    need = lib.ring_attn_fwd_host_workspace_bytes(B, L, H, D, 2)
    big = ctypes.c_ulonglong(need)
    f = lib.ring_attn_fwd_host
    # group size must divide H
    assert f(fake, fake, fake, out, null, ws, big, B, L, H, D, P, 1, 3, s) == 4
    assert f(fake, fake, fake, out, null, ws, big, B, L, H, D, P, 1, 0, s) == 1
    assert f(fake, fake, fake, out, null, ws, big, B, L, H, D, P, 1, 9, s) == 1
    # short or misaligned workspace, missing pointers
    assert f(fake, fake, fake, out, null, ws, ctypes.c_ulonglong(need - 1), B, L, H, D, P, 1, 2, s) == 1
    assert f(fake, fake, fake, out, null, ctypes.c_void_p((1 << 44) + 16), big, B, L, H, D, P, 1, 2, s) == 3
    assert f(fake, fake, fake, out, null, null, big, B, L, H, D, P, 1, 2, s) == 1
    # head dim, shard divisibility, output overlapping an input
    assert f(fake, fake, fake, out, null, ws, big, B, L, H, 96, P, 1, 2, s) == 2
    assert f(fake, fake, fake, out, null, ws, ctypes.c_ulonglong(1 << 30), B, 250, H, D, P, 1, 2, s) == 4
    assert f(fake, fake, fake, fake, null, ws, big, B, L, H, D, P, 1, 2, s) == 1


def test_host_workspace_size():
    """Three slots of (q, k, v, out, lse) for one head group plus the full lse, each
    rounded up to 256 bytes; 0 for sizes that cannot be grouped."""
    lib = cea.load_library()
    r = lambda x: (x + 255) // 256 * 256
    for (B, L, H, D, g) in [(1, 256, 8, 128, 2), (2, 1000, 6, 64, 3), (1, 32768, 32, 128, 4)]:
        rows = B * L
        slot = 4 * r(rows * g * D * 2) + r(rows * g * 4)
        assert lib.ring_attn_fwd_host_workspace_bytes(B, L, H, D, g) == 3 * slot + r(rows * H * 4)
    assert lib.ring_attn_fwd_host_workspace_bytes(1, 256, 8, 128, 3) == 0
    assert lib.ring_attn_fwd_host_workspace_bytes(1, 256, 8, 128, 16) == 0


def test_descriptor_layout_and_argument_errors(lib):
    """The ctypes mirror of ra_attn_desc has the C layout (eight ints, the boundary
    pointer, two ints, the schedule pointer: 56 bytes), and the general entry points
    reject bad descriptors on the host before touching the runtime."""
    assert ctypes.sizeof(cea.AttnDesc) == 56
    assert cea.AttnDesc.cu_seqlens.offset == 32 and cea.AttnDesc.dtype.offset == 44
    assert cea.AttnDesc.schedule.offset == 48
    fake = ctypes.c_void_p(1 << 20)
    out = ctypes.c_void_p(1 << 40)
    ws = ctypes.c_void_p(1 << 44)
    null = ctypes.c_void_p(0)
    s = ctypes.c_void_p(0)

    def desc(**kw):
        d = dict(B=1, L=1024, H=4, H_kv=2, D=128, P=4, causal=1, layout=1, cu_seqlens=None,
                 n_seqs=0, dtype=0, schedule=None)
        d.update(kw)
        return ctypes.byref(cea.AttnDesc(**d))

    fwd = lambda d: lib.ring_attn_fwd_ex(d, fake, fake, fake, out, null, null, s)
    bwd = lambda d: lib.ring_attn_bwd_ex(d, fake, fake, fake, fake, fake, fake, out, out, out, ws,
                                         ctypes.c_ulonglong(1 << 20), s)
    assert lib.ring_attn_fwd_ex(None, fake, fake, fake, out, null, null, s) == 1
    assert fwd(desc(layout=3)) == 1                         # unknown layout
    assert fwd(desc(causal=0)) == 2                         # zigzag is causal only
    assert fwd(desc(L=1020)) == 4                           # L % 2P
    assert fwd(desc(L=512)) == 2                            # chunks of 64 rows (bf16)
    assert fwd(desc(H_kv=3)) == 4                           # H % H_kv
    assert fwd(desc(layout=0, cu_seqlens=1 << 20)) == 1     # boundaries without packed layout
    assert fwd(desc(layout=2)) == 1                         # packed without boundaries
    assert fwd(desc(layout=2, cu_seqlens=1 << 20, n_seqs=3, B=2)) == 1
    assert fwd(desc(layout=2, cu_seqlens=(1 << 20) + 2, n_seqs=3)) == 3
    assert fwd(desc(layout=0, schedule=1 << 36)) == 1       # schedule without packed layout
    assert fwd(desc(layout=1, schedule=1 << 36)) == 1
    assert fwd(desc(layout=2, cu_seqlens=1 << 20, n_seqs=3, schedule=(1 << 36) + 2)) == 3
    assert bwd(desc(layout=2, cu_seqlens=1 << 20, n_seqs=3, schedule=(1 << 36) + 2)) == 3
    # a schedule overlapping the output
    assert fwd(desc(layout=2, cu_seqlens=1 << 20, n_seqs=3, H_kv=4, schedule=1 << 40)) == 1
    assert bwd(desc(dtype=1)) == 2                          # backward is bf16 only
    assert bwd(desc(causal=0)) == 2
    assert bwd(desc(H_kv=0)) == 1


def test_varlen_schedule_size_and_argument_errors(lib):
    """ring_attn_varlen_schedule_bytes counts three unit orders (forward tile pairs,
    backward key tiles, backward query tiles), a scratch of the same size and eight
    work counters of the persistent kernels, and ring_attn_varlen_schedule rejects bad
    arguments before launching anything."""
    def n_units(L, P):
        n_t = -(-(L // P) // 128)
        return n_t, -(-n_t // 2)
    for L, P in ((32768, 8), (1000, 4), (1, 1), (4096, 1), (300, 3)):
        n_t, n_pair = n_units(L, P)
        assert lib.ring_attn_varlen_schedule_bytes(L, P) == 8 * P * (n_pair + 2 * n_t) + 4 * 8
    assert lib.ring_attn_varlen_schedule_bytes(1000, 3) == 0
    assert lib.ring_attn_varlen_schedule_bytes(0, 1) == 0
    assert lib.ring_attn_varlen_schedule_bytes(4, 8) == 0
    cu = ctypes.c_void_p(1 << 20)
    sched = ctypes.c_void_p(1 << 30)
    s = ctypes.c_void_p(0)
    nb = lib.ring_attn_varlen_schedule_bytes(4096, 4)
    call = lambda *a: lib.ring_attn_varlen_schedule(*a, s)
    assert call(None, 3, 4096, 4, 1, sched, nb) == 1
    assert call(cu, 3, 4096, 4, 1, None, nb) == 1
    assert call(cu, 0, 4096, 4, 1, sched, nb) == 1
    assert call(cu, 3, 4096, 4, 1, sched, nb - 4) == 1       # short schedule
    assert call(cu, 3, 4098, 4, 1, sched, nb) == 4           # L % P
    assert call(cu, 3, 4096, 4, 1, ctypes.c_void_p((1 << 30) + 2), nb) == 3
    assert call(cu, 3, 4096, 4, 1, ctypes.c_void_p((1 << 20) - 8), nb) == 1   # overlaps cu
