"""Failure detection on the GPU, without faulting or hanging it: the bounded mbarrier wait
that every kernel uses gives up on a barrier nothing arrives at, reports KDA_ERR_TIMEOUT in
the device status word, and the kernel returns; the context stays usable."""
import time

import numpy as np
import pytest
import torch

from kda_testutil import assert_close, batch_heads, np64
from oracle import oracle

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_context_survives():
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import binding, synth

    assert kda.kda_get_device_status() == 0
    t0 = time.time()
    binding.kda_selftest_bounded_wait()
    st = kda.kda_get_device_status()  # waits for the stream
    dt = time.time() - t0
    assert st == binding.KDA_ERR_TIMEOUT, kda.kda_status_string(st)
    assert 0.2 < dt < 60, dt
    assert kda.kda_get_device_status() == 0  # read and cleared

    x = synth.prefill_inputs(1, 200, 2, seed=31337, device="cuda", init="normal")
    out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"])
    torch.cuda.synchronize()
    pairs = [(0, 0), (0, 1)]
    ro, rs = oracle.recurrent(batch_heads(x["q"], pairs), batch_heads(x["k"], pairs), batch_heads(x["v"], pairs),
                              batch_heads(x["log_alpha"], pairs), batch_heads(x["beta"], pairs),
                              np.stack([np64(x["init_state"][b, h]) for b, h in pairs]))
    assert_close(batch_heads(out, pairs), ro, "prefill after the timeout")
    assert_close(np.stack([np64(fin[b, h]) for b, h in pairs]), rs, "state after the timeout")
    assert kda.kda_get_device_status() == 0
