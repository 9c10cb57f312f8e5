"""GPU test of kda_chunk_fwd_host, the prefill streamed from host memory in segments: its
results equal kda_chunk_fwd's on the device, bit for bit (segments start at chunk
boundaries), for pinned and pageable host buffers, several segment sizes and ragged ends."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,segment", [(1000, 256), (1000, 64), (333, 0), (64, 64), (0, 128)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_host_streamed_equals_device_call(T, segment, out_dtype):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, H = 2, 3
    x = synth.prefill_inputs(B, T, H, seed=2024 + T, device="cuda", init="normal")
    out_d, fin_d = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                                     out_dtype=out_dtype)
    hx = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "log_alpha", "beta")}
    out_h, fin_h = kda.kda_chunk_fwd_host(hx["q"], hx["k"], hx["v"], hx["log_alpha"], hx["beta"], x["init_state"],
                                          out_dtype=out_dtype, segment_tokens=segment)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(fin_h, fin_d.cpu())
    assert kda.kda_get_device_status() == 0


def test_host_streamed_pageable_and_zero_state():
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    x = synth.prefill_inputs(1, 700, 2, seed=2100, device="cuda")
    out_d, fin_d = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None)
    hx = {n: x[n].cpu() for n in ("q", "k", "v", "log_alpha", "beta")}  # pageable
    out = torch.empty(1, 700, 2, 128)
    fin = torch.empty(1, 2, 128, 128)
    kda.kda_chunk_fwd_host(hx["q"], hx["k"], hx["v"], hx["log_alpha"], hx["beta"], None, out, fin,
                           segment_tokens=192)
    torch.cuda.synchronize()
    assert torch.equal(out, out_d.cpu()) and torch.equal(fin, fin_d.cpu())
