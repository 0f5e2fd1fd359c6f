"""ring_attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Plugins that only receive tensors, runtimes that keep all device memory in their
own pool, and servers that forbid allocation after warm-up cannot hand the
backward a workspace.  This entry point uses an array built into the library
instead.  The test calls it through the C ABI.  Before each checked call it makes
one call of the same shape whose upstream gradient is all NaN, which leaves NaN in
every row of the shared array that the checked call will use: the checked call
must still give exactly the bits of the workspace-taking ring_attn_bwd on the same
inputs (so it writes each row before reading it), and that backward is itself
checked against the fp64 oracle elsewhere.  Two shapes run back to back.  A call
made after the first one must leave the device's free memory unchanged, and a
problem larger than the array is refused.  This file is collected last.
"""
import ctypes

import pytest
import torch

import context_exact_attention_gb300 as cea
from context_exact_attention_gb300.workloads import make_qkv
from helpers import assert_bf16_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, q, k, v, out, lse, do, grads, B, L, H, D, P, causal, stream):
    return lib.ring_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(do),
                                     _ptr(grads[0]), _ptr(grads[1]), _ptr(grads[2]), B, L, H, D, P,
                                     int(causal), stream)


def test_noalloc_backward_matches_workspace_backward_twice():
    lib = cea.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    shapes = [(1, 1024, 4, 128, 4, True, 40), (2, 768, 2, 64, 3, False, 41)]
    for B, L, H, D, P, causal, seed in shapes:
        q, k, v = (t.to(DEV) for t in make_qkv(B, L, H, D, seed=seed, dtype=torch.bfloat16))
        do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(seed + 100))
        do = do.to(torch.bfloat16).to(DEV)
        out, lse = cea.ring_attn_fwd(q, k, v, P=P, causal=causal)
        ref = cea.ring_attn_bwd(q, k, v, out, lse, do, P=P, causal=causal)
        # same shape, NaN upstream gradient: every row of the array it uses becomes NaN
        poison = [torch.empty_like(q) for _ in range(3)]
        rc = _noalloc(lib, q, k, v, out, lse, torch.full_like(do, float("nan")), poison,
                      B, L, H, D, P, causal, stream)
        assert rc == 0, lib.ra_status_string(rc)
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = _noalloc(lib, q, k, v, out, lse, do, got, B, L, H, D, P, causal, stream)
        assert rc == 0, lib.ra_status_string(rc)
        assert cea.check_status() == 0
        assert torch.isnan(poison[0]).any()       # the poisoning call did read NaN rows
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert_bf16_close(to_np(g), to_np(r), name)
            assert torch.equal(g, r), name   # same kernels, deterministic: identical bits


def test_noalloc_backward_allocates_nothing_after_its_first_call():
    """Once the library's module is loaded on the device (by a first call), a call does
    not change the device's free memory."""
    lib = cea.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, L, H, D, P = 1, 512, 2, 128, 2
    q, k, v = (t.to(DEV) for t in make_qkv(B, L, H, D, seed=42, dtype=torch.bfloat16))
    do = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(43))
    do = do.to(torch.bfloat16).to(DEV)
    out, lse = cea.ring_attn_fwd(q, k, v, P=P, causal=True)
    grads = [torch.empty_like(q) for _ in range(3)]
    assert _noalloc(lib, q, k, v, out, lse, do, grads, B, L, H, D, P, True, stream) == 0
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    assert _noalloc(lib, q, k, v, out, lse, do, grads, B, L, H, D, P, True, stream) == 0
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert cea.check_status() == 0
    assert free_after == free_before


def test_noalloc_backward_refuses_problems_larger_than_its_array():
    lib = cea.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(16, dtype=torch.float32, device=DEV)
    rows_limit = 1048576
    L = rows_limit // 8 + 1               # B * L * H just above the limit with H = 8
    rc = lib.ring_attn_bwd_noalloc(_ptr(t), _ptr(t), _ptr(t), _ptr(t), _ptr(lse), _ptr(t), _ptr(t),
                                   _ptr(t), _ptr(t), 1, L, 8, 128, 1, 0, stream)
    assert rc == 1                        # RA_ERR_INVALID_ARG, nothing launched
    assert cea.check_status() == 0
