"""GPU parity of kda_decode_step against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

from kda_testutil import assert_close, np64
from oracle import oracle

pytestmark = pytest.mark.gpu


def _oracle_steps(d, pairs, steps):
    """Oracle over `steps` tokens for the listed (b,h) pairs, starting from d['state']."""
    col = lambda t, b, h: np64(t[:steps, b, h])
    q = np.stack([col(d["q"], b, h) for b, h in pairs])
    k = np.stack([col(d["k"], b, h) for b, h in pairs])
    v = np.stack([col(d["v"], b, h) for b, h in pairs])
    la = np.stack([col(d["log_alpha"], b, h) for b, h in pairs])
    be = np.stack([col(d["beta"], b, h) for b, h in pairs])
    S0 = np.stack([np64(d["state"][b, h]) for b, h in pairs])
    return oracle.recurrent(q, k, v, la, be, S0)


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_small(in_dtype, out_dtype):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, H, steps = 5, 3, 6
    d = synth.decode_inputs(B, H, seed=101, steps=steps, device="cuda", in_dtype=in_dtype)
    state = d["state"].clone()
    outs = []
    for s in range(steps):
        outs.append(kda.kda_decode_step(d["q"][s], d["k"][s], d["v"][s], d["log_alpha"][s], d["beta"][s], state,
                                        out_dtype=out_dtype))
    torch.cuda.synchronize()
    pairs = [(b, h) for b in range(B) for h in range(H)]
    ro, rs = _oracle_steps(d, pairs, steps)
    got_o = np.stack([np.stack([np64(outs[s][b, h]) for s in range(steps)]) for b, h in pairs])
    assert_close(got_o, ro, "decode outputs")
    assert_close(np.stack([np64(state[b, h]) for b, h in pairs]), rs, "decode state")
    assert kda.kda_get_device_status() == 0


def test_decode_full_size_sampled():
    """256 sessions x 96 heads, 64 successive steps with the state updated in place (the
    batched-decode workload); sampled (session, head) pairs are checked against the oracle."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    Bs, H, steps = 256, 96, 64
    d = synth.decode_inputs(Bs, H, seed=synth.SEED_BASE + 3, steps=steps, device="cuda")
    state = d["state"].clone()
    pairs = [(0, 0), (255, 95), (17, 40), (128, 3), (200, 77), (63, 64)]
    outs = torch.empty(steps, len(pairs), 128, device="cuda")
    for s in range(steps):
        o = kda.kda_decode_step(d["q"][s], d["k"][s], d["v"][s], d["log_alpha"][s], d["beta"][s], state)
        for i, (b, h) in enumerate(pairs):
            outs[s, i] = o[b, h]
    torch.cuda.synchronize()
    ro, rs = _oracle_steps(d, pairs, steps)
    assert_close(np64(outs).transpose(1, 0, 2), ro, "decode outputs")
    assert_close(np.stack([np64(state[b, h]) for b, h in pairs]), rs, "decode state")


def test_decode_empty_is_noop():
    import kda_recurrent_state_gb300 as kda

    z = torch.empty(0, 4, 128, device="cuda", dtype=torch.bfloat16)
    st = torch.empty(0, 4, 128, 128, device="cuda")
    out = kda.kda_decode_step(z, z, z, z.float(), torch.empty(0, 4, device="cuda"), st)
    assert out.shape == (0, 4, 128)
