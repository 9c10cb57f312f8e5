"""Seeded random cases across every entry point: shapes, lengths, dtypes, gates, chunk sizes,
snapshot intervals and pool dtypes drawn from a fixed generator, each checked against the
fp64 oracle (sampled heads), plus the bit-exact invariants (a packed sequence equals the
same sequence run alone; the host-streamed prefill equals the device one).

Numerical bar: the workloads' rel-L2 <= 2e-3 and max-abs <= 1e-2 (for gradients, of their
largest magnitude).  One reading is added for inputs outside the workloads: on the chunked
path the operands are fp16, and when an output is nearly cancelled (a single token whose q.k
is close to 0, so o = beta (q.k) v is small) their rounding gives a large relative error at a
tiny absolute one.  Only there, for an output whose reference has an L2 norm below
CANCEL_NORM (a token's 128 outputs with |q.k| below about 0.02, against a typical 0.09), the
relative bar is replaced by max-abs <= 1e-3, ten times tighter than the absolute bar; every
other chunked result must meet the relative bar.  A gradient that is identically zero in the
oracle has no relative error at all; there the absolute bar alone applies."""
import random

import numpy as np
import pytest
import torch

from kda_testutil import MAX_ABS, REL_L2, batch_heads, errors, np64, packed_heads

pytestmark = pytest.mark.gpu
CASES = 40  # per kind
CANCEL_ABS = 1e-3
CANCEL_NORM = 0.1  # L2 norm of a nearly cancelled output (see the module docstring)


def _close(got, ref, chunk, grad=False):
    rel, mx = errors(got, ref)
    scale = max(1.0, float(np.abs(ref).max())) if grad else 1.0
    if mx > MAX_ABS * scale:
        return False, rel, mx
    if rel <= REL_L2:
        return True, rel, mx
    if grad:  # gradients that vanish identically (oracle exact zeros): the absolute bar applies
        return float(np.abs(ref).max()) == 0.0 or (chunk == 64 and mx <= CANCEL_ABS * scale), rel, mx
    cancelled = float(np.linalg.norm(np.asarray(ref, dtype=np.float64))) < CANCEL_NORM
    return chunk == 64 and cancelled and mx <= CANCEL_ABS, rel, mx


def _check(name, got, ref, case, chunk, grad=False):
    ok, rel, mx = _close(got, ref, chunk, grad)
    assert ok, f"{name}: rel-L2 {rel:.3e}, max-abs {mx:.3e}, |ref| {np.linalg.norm(ref):.3e}, case {case}"


def _batched_case(rng, kind):
    B, H = rng.choice([1, 2]), rng.choice([1, 2, 3, 5])
    T = rng.choice([1, 2, 63, 64, 65, 127, 128, 129, rng.randrange(1, 1500)])
    dt = rng.choice([torch.bfloat16, torch.float32])
    return dict(kind=kind, B=B, T=T, H=H, dt=dt, chunk=rng.choice([64, 64, 1]), gate=rng.choice(["config", "slow"]),
                init=rng.choice(["zero", "normal"]), seed=rng.randrange(10**6), pair=(rng.randrange(B), rng.randrange(H)))


def _oracle_fwd(x, la, pair, S0):
    from oracle import oracle

    p = [pair]
    return oracle.recurrent(batch_heads(x["q"], p), batch_heads(x["k"], p), batch_heads(x["v"], p), batch_heads(la, p),
                            batch_heads(x["beta"], p), S0)


@pytest.mark.parametrize("kind", ["chunk", "gdn", "deltanet", "host", "bwd"])
def test_random_batched(kind):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth

    rng = random.Random(f"batched-{kind}")
    for _ in range(CASES):
        c = _batched_case(rng, kind)
        B, T, H, pair = c["B"], c["T"], c["H"], c["pair"]
        if kind == "bwd":
            T = c["T"] = min(T, 800)
            c["init"] = "normal"
        x = synth.prefill_inputs(B, T, H, seed=c["seed"], device="cuda", init=c["init"], in_dtype=c["dt"],
                                 gate=c["gate"])
        S0 = None if x["init_state"] is None else np64(x["init_state"][pair[0], pair[1]])[None]
        if kind == "chunk":
            out, fin = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"],
                                         chunk=c["chunk"])
            ro, rs = _oracle_fwd(x, x["log_alpha"], pair, S0)
        elif kind in ("gdn", "deltanet"):
            la_h = None if kind == "deltanet" else synth.head_gates((B, T), H, seed=c["seed"] + 1, device="cuda",
                                                                  gate=c["gate"])
            out, fin = kda.kda_gdn_chunk_fwd(x["q"], x["k"], x["v"], la_h, x["beta"], x["init_state"],
                                             chunk=c["chunk"])
            la = torch.zeros_like(x["log_alpha"]) if la_h is None else la_h.unsqueeze(-1).expand(B, T, H, 128)
            ro, rs = _oracle_fwd(x, la, pair, S0)
        elif kind == "host":
            seg = rng.choice([0, 64, 128, 192, 4096])
            out_d, fin_d = kda.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["init_state"])
            hx = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "log_alpha", "beta")}
            out_h, fin_h = kda.kda_chunk_fwd_host(hx["q"], hx["k"], hx["v"], hx["log_alpha"], hx["beta"],
                                                  x["init_state"], segment_tokens=seg)
            torch.cuda.synchronize()
            assert torch.equal(out_h, out_d.cpu()) and torch.equal(fin_h, fin_d.cpu()), (c, seg)
            continue
        else:
            from oracle import oracle

            do = torch.randn(B, T, H, 128, device="cuda", generator=torch.Generator(device="cuda").manual_seed(c["seed"]))
            g = kda.kda_bwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], do, x["init_state"])
            p = [pair]
            ref = oracle.recurrent_bwd(batch_heads(x["q"], p), batch_heads(x["k"], p), batch_heads(x["v"], p),
                                       batch_heads(x["log_alpha"], p), batch_heads(x["beta"], p), S0,
                                       batch_heads(do, p))
            for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta"):
                _check(name, batch_heads(g[name], p), ref[name], c, 1, grad=True)
            _check("d_init", np64(g["d_init"][pair[0], pair[1]])[None], ref["dS0"], c, 1, grad=True)
            assert kda.kda_get_device_status() == 0, c
            continue
        torch.cuda.synchronize()
        _check("out", batch_heads(out, [pair]), ro, c, c["chunk"])
        _check("final state", np64(fin[pair[0], pair[1]])[None], rs, c, c["chunk"])
        assert kda.kda_get_device_status() == 0, c


@pytest.mark.parametrize("kind", ["varlen", "pool"])
def test_random_packed(kind):
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth
    from oracle import oracle

    rng = random.Random(f"packed-{kind}")
    for _ in range(CASES):
        N, H = rng.randrange(1, 12), rng.choice([1, 2, 3, 5])
        lengths = [rng.choice([0, 1, 63, 64, 65, rng.randrange(0, 700)]) for _ in range(N)]
        chunk, iv = rng.choice([64, 64, 1]), rng.choice([0, 64, 128, 256])
        dt, gate, seed = rng.choice([torch.bfloat16, torch.float32]), rng.choice(["config", "slow"]), rng.randrange(10**6)
        c = dict(kind=kind, lengths=lengths, H=H, chunk=chunk, iv=iv, dt=dt, gate=gate, seed=seed)
        xv = synth.varlen_inputs(lengths, H, seed=seed, device="cuda", in_dtype=dt, gate=gate)
        args = (xv["q"], xv["k"], xv["v"], xv["log_alpha"], xv["beta"], xv["cu_seqlens"])
        snaps = None
        if kind == "varlen":
            out, fin, snaps = kda.kda_varlen_fwd(*args, xv["init_states"], chunk=chunk, snapshot_interval=iv)
            init = xv["init_states"]
        else:
            nsnap = int(kda.kda_snapshot_offsets(xv["cu_seqlens"].cpu(), iv)[-1]) if iv else 0
            pdt = rng.choice([torch.float32, torch.bfloat16])
            c["pool"] = pdt
            pool = torch.zeros(N + nsnap, H, 128, 128, dtype=pdt, device="cuda")
            pool[:N] = xv["init_states"].to(pdt)
            snap_slots = torch.arange(N, N + nsnap, device="cuda") if iv else None
            out, fin = kda.kda_varlen_fwd_pool(*args, pool, torch.arange(N, device="cuda"), snap_slots, chunk=chunk,
                                               snapshot_interval=iv)
            init = pool[:N].float()  # the states the sequences resumed from, as stored
            if iv and nsnap:
                snaps = pool[N:].float()
        torch.cuda.synchronize()
        assert kda.kda_get_device_status() == 0, c
        cu = xv["cu_seqlens"].tolist()
        offs = kda.kda_snapshot_offsets(cu, iv).tolist() if iv else None
        for s in rng.sample(range(N), min(N, 3)):
            a, b = cu[s], cu[s + 1]
            one = lambda t: t[a:b].unsqueeze(0).contiguous()  # noqa: E731
            o1, f1 = kda.kda_chunk_fwd(one(xv["q"]), one(xv["k"]), one(xv["v"]), one(xv["log_alpha"]),
                                       one(xv["beta"]), init[s:s + 1].contiguous(), chunk=chunk)
            assert torch.equal(out[a:b], o1[0]) and torch.equal(fin[s], f1[0]), (c, s)
            if snaps is not None and offs[s + 1] > offs[s]:
                # the last snapshot of a sequence is its state after token m*iv: compare with a run of that prefix
                m = offs[s + 1] - offs[s]
                e = a + m * iv
                pre = lambda t: t[a:e].unsqueeze(0).contiguous()  # noqa: E731
                _, fp = kda.kda_chunk_fwd(pre(xv["q"]), pre(xv["k"]), pre(xv["v"]), pre(xv["log_alpha"]),
                                          pre(xv["beta"]), init[s:s + 1].contiguous(), chunk=chunk)
                want = fp[0] if c.get("pool") != torch.bfloat16 else fp[0].to(torch.bfloat16).float()
                assert torch.equal(snaps[offs[s + 1] - 1], want), (c, s)
            if b > a:
                h = rng.randrange(H)
                ro, _ = oracle.recurrent(packed_heads(xv["q"], a, b, [h]), packed_heads(xv["k"], a, b, [h]),
                                         packed_heads(xv["v"], a, b, [h]), packed_heads(xv["log_alpha"], a, b, [h]),
                                         packed_heads(xv["beta"], a, b, [h]), np64(init[s, h])[None])
                _check("out", packed_heads(out, a, b, [h]), ro, dict(c, seq=s, len=b - a), chunk)


def test_random_decode():
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth
    from oracle import oracle

    rng = random.Random("decode")
    for _ in range(CASES):
        Bs, H, steps = rng.randrange(1, 40), rng.choice([1, 2, 3, 7]), rng.randrange(1, 6)
        dt, gate, seed = rng.choice([torch.bfloat16, torch.float32]), rng.choice(["config", "slow"]), rng.randrange(10**6)
        bf16 = rng.random() < 0.3
        c = dict(Bs=Bs, H=H, steps=steps, dt=dt, gate=gate, seed=seed, bf16state=bf16)
        d = synth.decode_inputs(Bs, H, seed=seed, steps=steps, device="cuda", in_dtype=dt, gate=gate)
        b, h = rng.randrange(Bs), rng.randrange(H)
        state = d["state"].to(torch.bfloat16) if bf16 else d["state"].clone()
        S0 = np64(state[b, h].float())[None]
        step = kda.kda_decode_step_bf16state if bf16 else kda.kda_decode_step
        outs = [step(d["q"][t], d["k"][t], d["v"][t], d["log_alpha"][t], d["beta"][t], state) for t in range(steps)]
        torch.cuda.synchronize()
        assert kda.kda_get_device_status() == 0, c
        seq = lambda t: np.stack([np64(t[s][b, h]) for s in range(steps)])[None]  # noqa: E731
        fn = oracle.recurrent_bf16state if bf16 else oracle.recurrent
        ro, rs = fn(seq(d["q"]), seq(d["k"]), seq(d["v"]), seq(d["log_alpha"]), seq(d["beta"]), S0)
        _check("out", np.stack([np64(o[b, h]) for o in outs])[None], ro, c, 1)
        _check("state", np64(state[b, h].float())[None], rs, c, 1)


@pytest.mark.parametrize("units", ["few", "many"])
def test_random_bwd_packed(units):
    """The chunked backward on random packed batches (empty and one-token sequences, every gate
    layout, both input dtypes, with and without a final-state cotangent): a sampled (sequence,
    head) against the oracle, and empty sequences passing d_final through.  A gradient that is
    identically zero in the oracle (dlog alpha of a one-token sequence from a zero state: the
    output does not depend on that gate) has no relative error, so there the absolute bar applies.
    "few": at most 18 (sequence, head) units, the serial passes' warp-level form with split value
    columns; "many": 40 to 128 units, their tcgen05 form (one CTA per unit) on a 152-SM GPU."""
    import kda_recurrent_state_gb300 as kda
    from kda_recurrent_state_gb300 import synth
    from oracle import oracle

    rng = random.Random("bwd-packed" if units == "few" else "bwd-packed-many")
    for _ in range(CASES):
        if units == "few":
            N, H = rng.randrange(1, 7), rng.choice([1, 2, 3])
        else:
            N, H = rng.randrange(5, 9), rng.choice([8, 12, 16])
        lengths = [rng.choice([0, 1, 2, 63, 64, 65, 128, rng.randrange(0, 700)]) for _ in range(N)]
        dt, gl, gate = rng.choice([torch.bfloat16, torch.float32]), rng.choice(["config", "slow"]), rng.choice([0, 0, 1, 2])
        seed = rng.randrange(10**6)
        c = dict(lengths=lengths, H=H, dt=dt, gl=gl, gate=gate, seed=seed)
        xv = synth.varlen_inputs(lengths, H, seed=seed, device="cuda", in_dtype=dt, gate=gl)
        Tt = xv["q"].shape[0]
        la = {0: xv["log_alpha"], 1: synth.head_gates((Tt,), H, seed=seed + 1, device="cuda", gate=gl), 2: None}[gate]
        gen = torch.Generator(device="cuda").manual_seed(seed + 2)
        do = torch.randn(Tt, H, 128, generator=gen, device="cuda")
        dSf = torch.randn(N, H, 128, 128, generator=gen, device="cuda") if rng.random() < 0.5 else None
        g = kda.kda_bwd(xv["q"], xv["k"], xv["v"], la, xv["beta"], do, xv["init_states"], dSf, gate=gate,
                        cu_seqlens=xv["cu_seqlens"], chunk=64)
        torch.cuda.synchronize()
        assert kda.kda_get_device_status() == 0, c
        cu = xv["cu_seqlens"].tolist()
        for s in range(N):
            if cu[s] == cu[s + 1]:
                want = dSf[s] if dSf is not None else torch.zeros_like(g["d_init"][s])
                assert torch.equal(g["d_init"][s], want), (c, s)
        s = rng.choice([i for i in range(N) if cu[i + 1] > cu[i]] or [None])
        if s is None:
            continue
        a, b, h = cu[s], cu[s + 1], rng.randrange(H)
        la_full = (torch.zeros(Tt, H, 128, device="cuda") if gate == 2
                   else la.unsqueeze(-1).expand(Tt, H, 128) if gate == 1 else la)
        ref = oracle.recurrent_bwd(packed_heads(xv["q"], a, b, [h]), packed_heads(xv["k"], a, b, [h]),
                                   packed_heads(xv["v"], a, b, [h]), packed_heads(la_full, a, b, [h]),
                                   packed_heads(xv["beta"], a, b, [h]), np64(xv["init_states"][s, h])[None],
                                   packed_heads(do, a, b, [h]), None if dSf is None else np64(dSf[s, h])[None])
        pairs = [("dq", ref["dq"]), ("dk", ref["dk"]), ("dv", ref["dv"]), ("dbeta", ref["dbeta"])]
        if gate != 2:
            pairs.append(("dlog_alpha", ref["dlog_alpha"] if gate == 0 else ref["dlog_alpha"].sum(-1)))
        for name, r in pairs:
            got = packed_heads(g[name], a, b, [h])
            if not np.any(r):  # identically zero: the absolute bar
                assert float(np.abs(got).max()) <= MAX_ABS, (name, c, s)
            else:
                _check(name, got, r, dict(c, seq=s, head=h), 1, grad=True)
        _check("d_init", np64(g["d_init"][s, h])[None], ref["dS0"], dict(c, seq=s, head=h), 1, grad=True)
