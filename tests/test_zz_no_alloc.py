"""ring_attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Plugins that only receive tensors, runtimes that keep all device memory in their
own pool, and servers that forbid allocation after warm-up cannot hand the
backward a workspace.  This entry point uses an array built into the library
instead.  The test calls it through the C ABI, twice in a row on different inputs
(the second call must not be disturbed by what the first left in the shared
array), and checks every gradient against the workspace-taking ring_attn_bwd on
the same inputs, within the bf16 tolerance the other tests use.  It also checks
that a problem larger than the array is refused.  This file is collected last.
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
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        rc = lib.ring_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(do),
                                       _ptr(got[0]), _ptr(got[1]), _ptr(got[2]), B, L, H, D, P,
                                       int(causal), stream)
        assert rc == 0, lib.ra_status_string(rc)
        assert cea.check_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert_bf16_close(to_np(g), to_np(r), name)
            assert torch.equal(g, r), name   # same kernels, deterministic: identical bits


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
