"""Out-of-bounds writes, without a sanitizer: every output of an entry point is a view into
a larger buffer whose guard regions (before and after it) hold a sentinel; after the call
the guards must be unchanged.  Sizes are ragged so that tail chunks and partial blocks are
exercised."""
import pytest
import torch

pytestmark = pytest.mark.gpu
GUARD = 4096  # elements on each side (a multiple of 16 bytes for every dtype used)


def guarded(shape, dtype, fill=float("nan")):
    n = 1
    for d in shape:
        n *= d
    buf = torch.full((GUARD + n + GUARD,), fill, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(*shape)


def guards_intact(buf):
    g = torch.cat([buf[:GUARD], buf[-GUARD:]])
    return bool(torch.isnan(g.float()).all())


@pytest.mark.parametrize("chunk", [64, 1])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_outputs_stay_in_bounds(chunk, out_dtype):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    B, T, H = 2, 333, 3
    x = synth.prefill_inputs(B, T, H, seed=1201, device="cuda", init="normal")
    ob, out = guarded((B, T, H, 128), out_dtype)
    fb, fin = guarded((B, H, 128, 128), torch.float32)
    kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"], out, fin, chunk=chunk)
    torch.cuda.synchronize()
    assert guards_intact(ob) and guards_intact(fb)
    assert not torch.isnan(out.float()).any() and not torch.isnan(fin).any()


@pytest.mark.parametrize("chunk", [64, 1])
def test_varlen_snapshots_stay_in_bounds(chunk):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths, H = [130, 0, 64, 257], 2
    xv = synth.varlen_inputs(lengths, H, seed=1202, device="cuda")
    Tt = sum(lengths)
    off = kda.kda_snapshot_offsets(xv["cu_seqlens"].cpu(), 64)
    n_snap = int(off[-1])
    ob, out = guarded((Tt, H, 128), torch.float32)
    fb, fin = guarded((len(lengths), H, 128, 128), torch.float32)
    sb, snaps = guarded((n_snap, H, 128, 128), torch.float32)
    kda.kda_varlen_fwd(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], xv["cu_seqlens"], xv["init_states"],
                       chunk=chunk, snapshot_interval=64, out=out, final_states=fin, snapshots=snaps)
    torch.cuda.synchronize()
    assert guards_intact(ob) and guards_intact(fb) and guards_intact(sb)
    assert not torch.isnan(snaps).any()


@pytest.mark.parametrize("bf16state", [False, True])
def test_decode_stays_in_bounds(bf16state):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    Bs, H = 7, 3
    d = synth.decode_inputs(Bs, H, seed=1203, steps=1, device="cuda")
    sdt = torch.bfloat16 if bf16state else torch.float32
    stb, state = guarded((Bs, H, 128, 128), sdt)
    state.copy_(d["state"].to(sdt))
    ob, out = guarded((Bs, H, 128), torch.float32)
    step = kda.kda_decode_step_bf16state if bf16state else kda.kda_decode_step
    step(d["q"][0], d["k"][0], d["v"][0], d["log_alpha"][0], d["beta"][0], state, out)
    torch.cuda.synchronize()
    assert guards_intact(stb) and guards_intact(ob)


def test_pool_and_backward_stay_in_bounds():
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    lengths, H = [200, 65], 2
    xv = synth.varlen_inputs(lengths, H, seed=1204, device="cuda")
    pb, pool = guarded((4, H, 128, 128), torch.bfloat16)
    pool[0] = xv["init_states"][0].to(torch.bfloat16)
    assert int(kda.kda_snapshot_offsets([0, 200, 265], 64)[-1]) == 4  # 3 + 1 snapshot slots to give
    kda.kda_varlen_fwd_pool(xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], xv["cu_seqlens"], pool,
                            torch.tensor([0, -1], device="cuda"), torch.tensor([1, 2, 3, -1], device="cuda"),
                            snapshot_interval=64)
    torch.cuda.synchronize()
    assert guards_intact(pb)

    x = synth.prefill_inputs(1, 77, 2, seed=1205, device="cuda", init="normal")
    do = torch.randn(1, 77, 2, 128, device="cuda")
    lib = kda.binding.lib()
    P = kda.binding._ptr
    for chunk in (1, 64):  # token-serial kda_bwd, chunked kda_chunk_bwd
        g = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"], chunk=chunk)
        bufs = {name: guarded(tuple(t.shape), torch.float32) for name, t in g.items()}
        need = kda.kda_workspace_size(kda.KDA_OP_CHUNK_BWD, 1, 77, 2, chunk=chunk)
        wb, ws = guarded((need // 4,), torch.float32)
        head = (P(x["q"]), P(x["k"]), P(x["v"]), P(x["log_alpha"]), 0, P(x["beta"]), P(x["init_state"]), P(do),
                None, None, 1, 77, 2, 128, 128)
        grads = (P(bufs["dq"][1]), P(bufs["dk"][1]), P(bufs["dv"][1]), P(bufs["dlog_alpha"][1]), P(bufs["dbeta"][1]),
                 P(bufs["d_init"][1]), 0)
        if chunk == 1:
            rc = lib.kda_bwd(*head, *grads, P(ws), need, kda.binding._stream(None))
        else:
            rc = lib.kda_chunk_bwd(*head, chunk, *grads, P(ws), need, kda.binding._stream(None))
        torch.cuda.synchronize()
        assert rc == 0
        for name, (b, v) in bufs.items():
            assert guards_intact(b), (chunk, name)
            assert torch.equal(v, g[name]), (chunk, name)
        assert guards_intact(wb), chunk
