"""GPU test of kda_bwd_noalloc, the backward on the library's static scratch (no caller
workspace, nothing allocated per call).  Kept in a file collected last: the first call
on a device reserves the 128 MiB static scratch for the rest of the process."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_noalloc_equals_workspace_call():
    """The same kernel on the static scratch gives the workspace call's gradients bit for bit,
    for a batched and a packed problem.  (The refusal of an oversize problem happens before
    any CUDA call and is tested on the CPU, in test_capi.py.)"""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(2, 500, 3, seed=9101, device="cuda", init="normal")
    do = torch.randn(2, 500, 3, 128, generator=torch.Generator(device="cuda").manual_seed(9102), device="cuda")
    dSf = torch.randn(2, 3, 128, 128, generator=torch.Generator(device="cuda").manual_seed(9103), device="cuda")
    ref = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], dSf, chunk=1)
    got = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], dSf, no_alloc=True)
    torch.cuda.synchronize()
    for name in ref:
        assert torch.equal(ref[name], got[name]), name

    xv = synth.varlen_inputs([300, 0, 129], 2, seed=9104, device="cuda")
    dov = torch.randn(429, 2, 128, generator=torch.Generator(device="cuda").manual_seed(9105), device="cuda")
    refv = kda.kda_bwd(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], dov, xv["init_states"],
                       cu_seqlens=xv["cu_seqlens"], chunk=1)
    gotv = kda.kda_bwd(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], dov, xv["init_states"],
                       cu_seqlens=xv["cu_seqlens"], no_alloc=True)
    torch.cuda.synchronize()
    for name in refv:
        assert torch.equal(refv[name], gotv[name]), name
    assert kda.kda_get_device_status() == 0
