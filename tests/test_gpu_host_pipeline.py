"""ring_attn_fwd_host: host tensors in, host tensors out, copies overlapped with the
attention.  Its results must be bit-identical to ring_attn_fwd on the same values on
the device (each head goes through the same kernel), and ring_attn_fwd itself is
checked against the fp64 oracle elsewhere; one case here also goes to the oracle."""
import pytest
import torch

import context_exact_attention_gb300 as cea
import oracle
from context_exact_attention_gb300.workloads import make_qkv
from helpers import assert_bf16_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _device_ref(q, k, v, P, causal):
    out, lse = cea.ring_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), P=P, causal=causal)
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("B,L,H,D,P,causal,group,pinned", [
    (1, 1024, 8, 128, 4, True, 2, True),
    (1, 1024, 8, 128, 4, False, 4, True),
    (2, 640, 6, 64, 5, True, 3, True),
    (1, 512, 4, 128, 1, True, 1, False),
    (1, 768, 8, 128, 3, True, 8, True),
])
def test_host_entry_matches_device_entry(B, L, H, D, P, causal, group, pinned):
    q, k, v = make_qkv(B, L, H, D, seed=11, dtype=torch.bfloat16)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    stream = torch.cuda.current_stream(DEV)
    out, lse = cea.ring_attn_fwd_host(q, k, v, P=P, causal=causal, heads_per_group=group,
                                      device=DEV, stream=stream)
    stream.synchronize()
    assert cea.check_status() == 0
    ref_out, ref_lse = _device_ref(q, k, v, P, causal)
    assert torch.equal(out, ref_out)
    assert torch.equal(lse, ref_lse)


def test_host_entry_against_oracle_and_repeat():
    """Non-trivial sizes against the fp64 oracle, and a second call into the same output
    buffers (slots reused across calls) gives the same bits."""
    B, L, H, D, P = 1, 2048, 8, 128, 4
    q, k, v = (t.pin_memory() for t in make_qkv(B, L, H, D, seed=12, dtype=torch.bfloat16))
    ws = torch.empty(cea.host_workspace_bytes(B, L, H, D, 2), dtype=torch.uint8, device=DEV)
    out, lse = cea.ring_attn_fwd_host(q, k, v, P=P, causal=True, heads_per_group=2,
                                      workspace=ws, device=DEV)
    torch.cuda.synchronize()
    first_out, first_lse = out.clone(), lse.clone()
    cea.ring_attn_fwd_host(q, k, v, P=P, causal=True, heads_per_group=2, workspace=ws,
                           out=out, lse=lse, device=DEV)
    torch.cuda.synchronize()
    assert torch.equal(out, first_out) and torch.equal(lse, first_lse)
    rows = [0, 1, 511, 512, 1023, 1500, 2047]
    ref, lref = oracle.attention(q, k, v, causal=True, rows=rows)
    assert_bf16_close(to_np(out[:, rows]), ref, "host entry out")
    assert_bf16_close(to_np(lse[:, rows]), lref, "host entry lse")


def test_host_entry_without_lse_and_errors():
    q, k, v = make_qkv(1, 256, 4, 128, seed=13, dtype=torch.bfloat16)
    out, lse = cea.ring_attn_fwd_host(q, k, v, P=2, causal=True, want_lse=False,
                                      heads_per_group=2, device=DEV)
    torch.cuda.synchronize()
    assert lse is None
    ref_out, _ = _device_ref(q, k, v, 2, True)
    assert torch.equal(out, ref_out)
    with pytest.raises(cea.RingAttnError):
        cea.ring_attn_fwd_host(q, k, v, P=2, causal=True, heads_per_group=3, device=DEV)
    small = torch.empty(1024, dtype=torch.uint8, device=DEV)
    with pytest.raises(cea.RingAttnError):
        cea.ring_attn_fwd_host(q, k, v, P=2, causal=True, heads_per_group=2, workspace=small,
                               device=DEV)
