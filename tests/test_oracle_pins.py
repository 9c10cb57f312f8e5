"""Pins for the fp64 oracle, against facts the pages and the mathematics fix.

None of these re-types the oracle's own loop.  Each check is one of:
  * a value the pages print or an example they describe (tests/golden/),
  * a closed form (pure decay when beta = 0; identity when alpha = 1, beta = 0),
  * the textbook matrix form of the update, built as explicit dk x dk
    matrices (I - beta k k^T) Diag(alpha) and multiplied with numpy,
  * the transition product A_t ... A_{j+1} of the "Kimi K3" article
    (lshu.cn/news/263999), §五, as an explicit matrix product,
  * reductions to DeltaNet (alpha = 1) and Gated DeltaNet (scalar alpha), §三-§四,
  * structural invariants (linearity, split-and-resume, snapshots, contraction),
  * agreement of the two independent formulations: per-token recurrence and the
    chunked WY rewrite of §六.
The last test plants plausible mistakes in the oracle (compiled variants) and
checks that at least one pin catches each.
"""
import os

import numpy as np
import pytest

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            key, rhs = line.split("=", 1)
            vals[key.strip()] = np.array([float(x) for x in rhs.split()])
    return vals


def _inputs(rng, n, T, dk, dv, gate="config", beta=None):
    q = rng.standard_normal((n, T, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((n, T, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((n, T, dv))
    lo, hi = (0.001, 0.1) if gate == "config" else (1e-5, 1e-3)
    la = -rng.uniform(lo, hi, (n, T, dk))
    b = 1 / (1 + np.exp(-rng.standard_normal((n, T)))) if beta is None else np.full((n, T), float(beta))
    # round to fp32 once, so what the oracle sees (fp32 inputs) is what numpy sees
    f = lambda x: x.astype(np.float32).astype(np.float64)
    return f(q), f(k), f(v), f(la), f(b)


def _matrix_form(q, k, v, la, beta, S0):
    """Textbook form, explicit matrices: S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T; o_t = S_t^T q_t."""
    T, dk = q.shape
    S = S0.copy()
    outs = []
    for t in range(T):
        A = (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(la[t]))
        S = A @ S + beta[t] * np.outer(k[t], v[t])
        outs.append(S.T @ q[t])
    return np.array(outs), S


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# --------------------------------------------------------------------------- pins
def pin_matrix_form(lib):
    rng = np.random.default_rng(1)
    for dk, dv, T in [(4, 3, 7), (8, 8, 20), (16, 5, 33)]:
        q, k, v, la, b = _inputs(rng, 2, T, dk, dv)
        S0 = 0.3 * rng.standard_normal((2, dk, dv))
        out, Sf = oracle.recurrent(q, k, v, la, b, S0, lib=lib)
        for h in range(2):
            o_ref, S_ref = _matrix_form(q[h], k[h], v[h], la[h], b[h], S0[h])
            assert rel(out[h], o_ref) < 1e-13, rel(out[h], o_ref)
            assert rel(Sf[h], S_ref) < 1e-13


def pin_identity(lib):
    """alpha = 1, beta = 0: the state is unchanged (bit-exact) and o_t = S0^T q_t."""
    rng = np.random.default_rng(2)
    q, k, v, _, _ = _inputs(rng, 2, 9, 8, 6)
    la = np.zeros_like(q)
    b = np.zeros(q.shape[:2])
    S0 = rng.standard_normal((2, 8, 6))
    out, Sf = oracle.recurrent(q, k, v, la, b, S0, lib=lib)
    assert np.array_equal(Sf, S0)
    for h in range(2):
        assert rel(out[h], q[h] @ S0[h]) < 1e-14


def pin_pure_decay(lib):
    """beta = 0: S_T = Diag(exp(sum_t log alpha_t)) S0, and o_t reads the decayed S0."""
    rng = np.random.default_rng(3)
    q, k, v, la, _ = _inputs(rng, 1, 40, 8, 5)
    b = np.zeros(q.shape[:2])
    S0 = rng.standard_normal((1, 8, 5))
    out, Sf = oracle.recurrent(q, k, v, la, b, S0, lib=lib)
    g = np.cumsum(la[0], axis=0)
    assert rel(Sf[0], np.exp(g[-1])[:, None] * S0[0]) < 1e-13
    o_ref = np.stack([(np.exp(g[t])[:, None] * S0[0]).T @ q[0, t] for t in range(40)])
    assert rel(out[0], o_ref) < 1e-13


def pin_overwrite_example(lib):
    """The pages' overwrite example: the later write under the same key wins, exactly."""
    gd = _golden("overwrite_example.txt")
    key, v1, v2 = gd["key"], gd["value_1"], gd["value_2"]
    q = np.stack([key, key])[None]
    v = np.stack([v1, v2])[None]
    la = np.zeros_like(q)
    b = np.ones((1, 2))
    out, Sf = oracle.recurrent(q, q, v, la, b, None, lib=lib)
    assert np.array_equal(out[0, 1], gd["read_delta"])
    assert not np.allclose(out[0, 1], gd["read_additive"])
    rng = np.random.default_rng(4)
    vv = rng.standard_normal((2, 16)).astype(np.float32).astype(np.float64)
    # an exactly unit key with several nonzero channels: the latest value, exactly
    kk = np.zeros(16)
    kk[[1, 5, 6, 11]] = [0.5, -0.5, 0.5, 0.5]
    out, _ = oracle.recurrent(np.stack([kk, kk])[None], np.stack([kk, kk])[None], vv[None],
                              np.zeros((1, 2, 16)), np.ones((1, 2)), None, lib=lib)
    assert np.array_equal(out[0, 1], vv[1])
    # a random key with |k|^2 = n2 != 1: closed form n2 * (v2 + (1 - n2) v1)
    kk = rng.standard_normal(16)
    kk = (kk / np.linalg.norm(kk)).astype(np.float32).astype(np.float64)
    n2 = kk @ kk
    out, _ = oracle.recurrent(np.stack([kk, kk])[None], np.stack([kk, kk])[None], vv[None],
                              np.zeros((1, 2, 16)), np.ones((1, 2)), None, lib=lib)
    assert np.abs(out[0, 1] - n2 * (vv[1] + (1 - n2) * vv[0])).max() < 1e-14


def pin_orthonormal_retrieval(lib):
    """alpha = 1, beta = 1 and orthonormal keys: every stored value is read back by its key."""
    rng = np.random.default_rng(5)
    for exact, dk, n_keys in [(True, 8, 8), (False, 16, 12)]:
        keys = np.eye(dk)[:n_keys] if exact else np.linalg.qr(rng.standard_normal((dk, dk)))[0].T[:n_keys]
        vals = rng.standard_normal((n_keys, 6))
        # write all pairs, then read each key with beta = 0 (read-only steps)
        kin = np.concatenate([keys, keys])[None]
        vin = np.concatenate([vals, np.zeros_like(vals)])[None]
        b = np.concatenate([np.ones(n_keys), np.zeros(n_keys)])[None]
        out, _ = oracle.recurrent(kin, kin, vin, np.zeros_like(kin), b, None, lib=lib)
        got = out[0, n_keys:]
        if exact:
            assert np.array_equal(got, vals)
        else:
            assert np.abs(got - vals).max() < 1e-13


def pin_transition_product(lib):
    """Affine in S0 with the transition product of §五: S_T(S0) - S_T(0) = A_T ... A_1 S0."""
    rng = np.random.default_rng(6)
    q, k, v, la, b = _inputs(rng, 1, 25, 8, 4)
    S0 = rng.standard_normal((1, 8, 4))
    _, S1 = oracle.recurrent(q, k, v, la, b, S0, lib=lib)
    _, Sz = oracle.recurrent(q, k, v, la, b, None, lib=lib)
    Phi = np.eye(8)
    for t in range(25):
        Phi = (np.eye(8) - b[0, t] * np.outer(k[0, t], k[0, t])) @ np.diag(np.exp(la[0, t])) @ Phi
    assert rel(S1[0] - Sz[0], Phi @ S0[0]) < 1e-12


def pin_reductions(lib):
    """alpha = 1 gives DeltaNet; a scalar alpha gives Gated DeltaNet, S = a (I - b k k^T) S + b k v^T."""
    rng = np.random.default_rng(7)
    q, k, v, la, b = _inputs(rng, 1, 30, 8, 5)
    S0 = rng.standard_normal((1, 8, 5))
    # DeltaNet
    out, Sf = oracle.recurrent(q, k, v, np.zeros_like(la), b, S0, lib=lib)
    S = S0[0].copy()
    for t in range(30):
        S = (np.eye(8) - b[0, t] * np.outer(k[0, t], k[0, t])) @ S + b[0, t] * np.outer(k[0, t], v[0, t])
        assert rel(out[0, t], S.T @ q[0, t]) < 1e-13
    # Gated DeltaNet: the gate outside the bracket (the per-head placement)
    la_s = np.repeat(la[:, :, :1], 8, axis=2)
    out, Sf = oracle.recurrent(q, k, v, la_s, b, S0, lib=lib)
    S = S0[0].copy()
    for t in range(30):
        a = np.exp(la_s[0, t, 0])
        S = a * (np.eye(8) - b[0, t] * np.outer(k[0, t], k[0, t])) @ S + b[0, t] * np.outer(k[0, t], v[0, t])
    assert rel(Sf[0], S) < 1e-13


def pin_recurrent_equals_chunked(lib):
    rng = np.random.default_rng(8)
    for T in (1, 63, 64, 65, 200):
        for C in (1, 4, 64):
            for gate in ("config", "slow"):
                q, k, v, la, b = _inputs(rng, 2, T, 16, 8, gate=gate)
                S0 = 0.5 * rng.standard_normal((2, 16, 8))
                o1, s1 = oracle.recurrent(q, k, v, la, b, S0, lib=lib)
                o2, s2 = oracle.chunked(q, k, v, la, b, S0, chunk=C, lib=lib)
                assert rel(o2, o1) < 1e-12, (T, C, gate, rel(o2, o1))
                assert rel(s2, s1) < 1e-12


def pin_linearity(lib):
    rng = np.random.default_rng(9)
    q, k, v, la, b = _inputs(rng, 1, 50, 8, 6)
    v2 = rng.standard_normal(v.shape).astype(np.float32).astype(np.float64)
    o1, s1 = oracle.recurrent(q, k, v, la, b, None, lib=lib)
    o2, s2 = oracle.recurrent(q, k, v2, la, b, None, lib=lib)
    o3, s3 = oracle.recurrent(q, k, v + v2, la, b, None, lib=lib)
    assert rel(o3, o1 + o2) < 1e-13 and rel(s3, s1 + s2) < 1e-13
    o4, s4 = oracle.recurrent(q, k, 2 * v, la, b, None, lib=lib)
    assert np.array_equal(o4, 2 * o1) and np.array_equal(s4, 2 * s1)


def pin_split_resume_and_snapshots(lib):
    rng = np.random.default_rng(10)
    q, k, v, la, b = _inputs(rng, 2, 96, 8, 6)
    S0 = rng.standard_normal((2, 8, 6))
    o, s, snaps = oracle.recurrent(q, k, v, la, b, S0, snap_interval=32, lib=lib)
    oa, sa = oracle.recurrent(q[:, :40], k[:, :40], v[:, :40], la[:, :40], b[:, :40], S0, lib=lib)
    ob, sb = oracle.recurrent(q[:, 40:], k[:, 40:], v[:, 40:], la[:, 40:], b[:, 40:], sa, lib=lib)
    assert np.array_equal(np.concatenate([oa, ob], axis=1), o) and np.array_equal(sb, s)
    assert snaps.shape == (2, 3, 8, 6)
    for m in range(1, 4):
        _, sm = oracle.recurrent(q[:, :32 * m], k[:, :32 * m], v[:, :32 * m], la[:, :32 * m], b[:, :32 * m],
                                 S0, lib=lib)
        assert np.array_equal(snaps[:, m - 1], sm)
    assert np.array_equal(snaps[:, -1], s)
    _, sc, snc = oracle.chunked(q, k, v, la, b, S0, chunk=16, snap_interval=32, lib=lib)
    assert rel(snc, snaps) < 1e-12


def pin_contraction(lib):
    """||k|| = 1, beta in [0,1], alpha <= 1: ||S_t||_2 <= ||S_{t-1}||_2 + beta_t ||v_t||."""
    rng = np.random.default_rng(11)
    q, k, v, la, b = _inputs(rng, 1, 60, 8, 5)
    S0 = rng.standard_normal((1, 8, 5))
    _, _, snaps = oracle.recurrent(q, k, v, la, b, S0, snap_interval=1, lib=lib)
    prev = np.linalg.norm(S0[0], 2)
    for t in range(60):
        cur = np.linalg.norm(snaps[0, t], 2)
        assert cur <= prev + b[0, t] * np.linalg.norm(v[0, t]) + 1e-12
        prev = cur


PINS = [pin_matrix_form, pin_identity, pin_pure_decay, pin_overwrite_example, pin_orthonormal_retrieval,
        pin_transition_product, pin_reductions, pin_recurrent_equals_chunked, pin_linearity,
        pin_split_resume_and_snapshots, pin_contraction]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_state_bytes_independent_of_T(oracle_lib):
    """The state is dk x dv per head whatever T is; the K3 session state is 217,055,232 bytes."""
    gd = _golden("state_bytes.txt")
    rng = np.random.default_rng(12)
    shapes = set()
    for T in (1, 7, 130):
        q, k, v, la, b = _inputs(rng, 1, T, 128, 128)
        _, Sf = oracle.recurrent(q, k, v, la, b, None, lib=oracle_lib)
        shapes.add(Sf.shape[1:])
    assert shapes == {(128, 128)}
    per_head = shapes.pop()
    total = int(gd["layers"][0]) * int(gd["heads"][0]) * per_head[0] * per_head[1] * int(gd["bytes_per_element"][0])
    assert total == int(gd["state_bytes"][0]) == 217_055_232


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5])
def test_planted_mistakes_are_caught(mutant, tmp_path):
    """Each planted mistake (no decay; prediction from the undecayed state; sign of the
    error; query/key swapped in the read; read before the write) fails at least one pin."""
    lib = oracle.load(oracle.build(str(tmp_path / f"mutant{mutant}.so"), mutant=mutant))
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"


# --------------------------------------------------------------------------- bf16-stored state
def test_round_bf16_matches_torch():
    """The oracle's bf16 rounding equals torch's fp32 -> bf16 conversion (round to nearest,
    ties to even) on fp32 values: random magnitudes, exact ties, subnormals, values near
    the largest bf16 and beyond it."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    x = rng.standard_normal(20000) * np.exp2(rng.uniform(-140, 127, 20000))
    ties = (1.0 + (2 * rng.integers(0, 128, 2000) + 1) * 2.0 ** -8) * np.exp2(rng.integers(-120, 120, 2000))
    special = np.array([0.0, -0.0, 1.0, 3.3895313892515355e38, 3.3961e38, -3.3961e38, 2.0 ** -133, 2.0 ** -134,
                        3 * 2.0 ** -135, 1e-45, 2.0 ** -126 * (1 - 2.0 ** -9)])
    x32 = np.concatenate([x, ties, -ties, special]).astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x32.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16state_overwrite_reads_before_rounding():
    """alpha = 1, beta = 1, unit key e_1: the step overwrites row 1 of the state with v.
    The read o = S^T e_1 returns v exactly (taken before the state is rounded); the stored
    row is v rounded to bf16, the other rows (bf16 values) are unchanged."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(22)
    dk, dv = 8, 5
    S0 = torch.from_numpy(rng.standard_normal((1, dk, dv)).astype(np.float32)).to(torch.bfloat16).double().numpy()
    v = (1.0 + rng.integers(1, 2 ** 20, (1, 1, dv)) * 2.0 ** -21).astype(np.float32).astype(np.float64)
    e1 = np.zeros((1, 1, dk))
    e1[0, 0, 1] = 1.0
    out, S = oracle.recurrent_bf16state(e1, e1, v, np.zeros((1, 1, dk)), np.ones((1, 1)), S0)
    np.testing.assert_array_equal(out[0, 0], v[0, 0])
    want_row = torch.from_numpy(v[0, 0].astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(S[0, 1], want_row)
    rest = [i for i in range(dk) if i != 1]
    np.testing.assert_array_equal(S[0, rest], S0[0, rest])


def test_bf16state_equals_fp64_when_exact():
    """Orthonormal basis keys, alpha = 1, beta = 1 and bf16-valued v: every state stays
    exactly representable in bf16, so the rounding variant equals the fp64 recurrence."""
    rng = np.random.default_rng(23)
    dk, dv, T = 8, 6, 12
    idx = rng.integers(0, dk, T)
    k = np.zeros((1, T, dk))
    k[0, np.arange(T), idx] = 1.0
    q = np.zeros((1, T, dk))
    q[0, np.arange(T), rng.integers(0, dk, T)] = 1.0
    v = (rng.integers(-127, 128, (1, T, dv)) / 16.0)
    la = np.zeros((1, T, dk))
    b = np.ones((1, T))
    o1, S1 = oracle.recurrent(q, k, v, la, b)
    o2, S2 = oracle.recurrent_bf16state(q, k, v, la, b)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)


def test_bf16state_error_bounded():
    """With general inputs the stored state differs from the fp64 recurrence by no more than
    bf16 rounding can explain: relative error of the final state well below 2^-6 over 64 steps."""
    rng = np.random.default_rng(24)
    q, k, v, la, b = _inputs(rng, 2, 64, 16, 8)
    o1, S1 = oracle.recurrent(q, k, v, la, b)
    o2, S2 = oracle.recurrent_bf16state(q, k, v, la, b)
    assert 0 < rel(S2, S1) < 2.0 ** -6
    assert 0 < rel(o2, o1) < 2.0 ** -6


# --------------------------------------------------------------------------- backward
def _loss_fd(lib, args, do, dSf, h=1e-6):
    """Central finite differences of L = <do, o> + <dSf, S_T> through the forward oracle."""
    def L(a):
        o, Sf = oracle.recurrent(a["q"], a["k"], a["v"], a["la"], a["b"], a["S0"], lib=lib)
        return float((o * do).sum() + (Sf * dSf).sum())
    fd = {}
    for name, x in args.items():
        g = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            a = dict(args)
            xp = x.copy(); xp[idx] += h; a[name] = xp; Lp = L(a)
            xm = x.copy(); xm[idx] -= h; a[name] = xm; Lm = L(a)
            g[idx] = (Lp - Lm) / (2 * h)
        fd[name] = g
    return fd


BWD_NAMES = {"q": "dq", "k": "dk", "v": "dv", "la": "dlog_alpha", "b": "dbeta", "S0": "dS0"}


def pin_bwd_finite_differences(lib):
    """Every gradient of the reverse sweep equals central finite differences of the forward
    oracle (an independent computation: no derivative is written down)."""
    rng = np.random.default_rng(31)
    for T, dSf_on in ((7, True), (4, False)):
        q, k, v, la, b = _inputs(rng, 2, T, 5, 4, gate="slow")
        la = la * 300  # decays of order e^-0.15 per token, so the gate gradient is not tiny
        S0 = rng.standard_normal((2, 5, 4))
        do = rng.standard_normal((2, T, 4))
        dSf = rng.standard_normal((2, 5, 4)) if dSf_on else np.zeros((2, 5, 4))
        g = oracle.recurrent_bwd(q, k, v, la, b, S0, do, dSf if dSf_on else None, lib=lib)
        fd = _loss_fd(lib, {"q": q, "k": k, "v": v, "la": la, "b": b, "S0": S0}, do, dSf)
        for name, want in fd.items():
            got = g[BWD_NAMES[name]]
            err = np.abs(got - want).max()
            assert err <= 1e-6 * max(1.0, np.abs(want).max()), (name, T, err)


def pin_bwd_closed_form_no_write(lib):
    """alpha = 1, beta = 0: the state never changes (S_t = S0), so o_t = S0^T q_t and
    dq_t = S0 do_t, dS0 = dS_T + sum_t q_t do_t^T, dk = dv = 0,
    dlog_alpha_t = rowsum(G_t * S0) with G_t = dS_T + sum_{t' >= t} q_t' do_t'^T, and
    dbeta_t = (G_t^T k_t) . (v_t - S0^T k_t)."""
    rng = np.random.default_rng(32)
    T, dk, dv = 6, 5, 4
    q, k, v, _, _ = _inputs(rng, 1, T, dk, dv)
    la, b = np.zeros((1, T, dk)), np.zeros((1, T))
    S0, do, dSf = rng.standard_normal((1, dk, dv)), rng.standard_normal((1, T, dv)), rng.standard_normal((1, dk, dv))
    g = oracle.recurrent_bwd(q, k, v, la, b, S0, do, dSf, lib=lib)
    np.testing.assert_allclose(g["dq"][0], do[0] @ S0[0].T, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dS0"][0], dSf[0] + q[0].T @ do[0], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(g["dk"], 0.0)
    np.testing.assert_array_equal(g["dv"], 0.0)
    for t in range(T):
        G = dSf[0] + q[0, t:].T @ do[0, t:]
        np.testing.assert_allclose(g["dlog_alpha"][0, t], (G * S0[0]).sum(axis=1), rtol=0, atol=1e-12)
        np.testing.assert_allclose(g["dbeta"][0, t], (G.T @ k[0, t]) @ (v[0, t] - S0[0].T @ k[0, t]), rtol=0,
                                   atol=1e-12)


def pin_bwd_first_gate_from_zero_state(lib):
    """From a zero initial state the first token's gate multiplies nothing (S_1 = beta_1 k_1 v_1^T),
    so no output depends on it and its gradient is exactly zero; from a non-zero state it is not.
    Later tokens' gate gradients are non-zero either way."""
    rng = np.random.default_rng(33)
    q, k, v, la, b = _inputs(rng, 1, 5, 6, 4)
    do, dSf = rng.standard_normal((1, 5, 4)), rng.standard_normal((1, 6, 4))
    g0 = oracle.recurrent_bwd(q, k, v, la, b, np.zeros((1, 6, 4)), do, dSf, lib=lib)
    np.testing.assert_array_equal(g0["dlog_alpha"][0, 0], 0.0)
    assert np.all(np.abs(g0["dlog_alpha"][0, 1:]).max(axis=-1) > 0)
    g1 = oracle.recurrent_bwd(q, k, v, la, b, rng.standard_normal((1, 6, 4)), do, dSf, lib=lib)
    assert np.abs(g1["dlog_alpha"][0, 0]).max() > 0


BWD_PINS = [pin_bwd_finite_differences, pin_bwd_closed_form_no_write, pin_bwd_first_gate_from_zero_state]


@pytest.mark.parametrize("pin", BWD_PINS, ids=[p.__name__ for p in BWD_PINS])
def test_bwd_pin(pin, oracle_lib):
    pin(oracle_lib)


@pytest.mark.parametrize("mutant", [6, 7])
def test_bwd_planted_mistakes_are_caught(mutant, tmp_path):
    """Dropping the prediction's key-gradient term (6) or the decay on the carried state
    gradient (7) fails the finite-difference pin."""
    lib = oracle.load(oracle.build(str(tmp_path / f"mutant{mutant}.so"), mutant=mutant))
    with pytest.raises(AssertionError):
        pin_bwd_finite_differences(lib)
