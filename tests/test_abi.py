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


def test_status_strings(lib):
    for code in range(7):
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
