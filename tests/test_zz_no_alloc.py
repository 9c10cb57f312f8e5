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


def test_noalloc_at_the_scratch_limit():
    """A packed problem whose scratch is exactly KDA_NOALLOC_SCRATCH_BYTES (110 sequences, one head:
    a 64 KB checkpoint per 64 tokens and per sequence, plus 16 per-sequence recomputation states)
    runs on the static array up to its last byte and matches the workspace call bit for bit; one
    more checkpoint's worth of tokens is refused before anything is launched."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import binding, synth

    lengths = [103] * 108 + [102] * 2  # 11,328 tokens: 11,328 / 64 + 110 + 1 + 16 x 110 = 2048 states
    t_total = sum(lengths)
    assert binding.kda_workspace_size(binding.KDA_OP_BWD, 110, t_total, 1) == binding.KDA_NOALLOC_SCRATCH_BYTES
    xv = synth.varlen_inputs(lengths, 1, seed=9106, device="cuda")
    do = torch.randn(t_total, 1, 128, generator=torch.Generator(device="cuda").manual_seed(9107), device="cuda")
    args = (xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], do, xv["init_states"])
    ref = kda.kda_bwd(*args, cu_seqlens=xv["cu_seqlens"], chunk=1)
    got = kda.kda_bwd(*args, cu_seqlens=xv["cu_seqlens"], no_alloc=True)
    torch.cuda.synchronize()
    for name in ref:
        assert torch.equal(ref[name], got[name]), name
    assert kda.kda_get_device_status() == 0

    longer = [103] * 108 + [102] + [166]  # 64 more tokens: one more checkpoint slot
    assert binding.kda_workspace_size(binding.KDA_OP_BWD, 110, sum(longer), 1) > binding.KDA_NOALLOC_SCRATCH_BYTES
    xl = synth.varlen_inputs(longer, 1, seed=9108, device="cuda")
    dol = torch.zeros(sum(longer), 1, 128, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_bwd(xl["q"], xl["k"], xl["v"], xl["log_alpha"], xl["beta"], dol, xl["init_states"],
                    cu_seqlens=xl["cu_seqlens"], no_alloc=True)
    assert e.value.code == binding.KDA_ERR_SCRATCH_TOO_SMALL
