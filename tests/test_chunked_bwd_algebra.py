"""The chunked backward's algebra, written out in fp64 numpy and checked against the oracle's
token-serial reverse mode (no GPU).

The GPU's chunked backward (kda_chunk_bwd, chunk = 64) evaluates, per chunk, the reverse mode
of the WY form of the "Kimi K3" article (lshu.cn/news/263999) §六.2 with the decays factored
about row 31 of the chunk:
    Q~ = q e^{g-ref}, K~ = k e^{g-ref}, K^ = k e^{ref-g},   T = (I + strict_lower(diag(beta) K~ K^^T))^-1
    U' = T diag(beta) V,  W~ = T diag(beta) K~,  P = lower_incl(Q~ K^^T),  X = Diag(e^ref) S_0
    U = U' - W~ X,  O = Q~ X + P U,  S_C = Diag(e^{g_C - ref}) (X + K^^T U)
This file takes the same steps in the same order: the chunk-start states forward, the state
gradients backward (dS_n = Diag(e^ref)(dD - W~^T (K^ dD) + Q~^T dO - W~^T (P^T dO))), then each
chunk's input gradients.  The adjoint of ref is never formed: the outputs do not depend on it.
Agreement to rounding with the oracle, at ragged lengths, pins the derivation the kernel follows."""
import numpy as np
import pytest

from oracle import oracle

C = 64


def _pad(x, L):
    return np.concatenate([x, np.zeros((C - L,) + x.shape[1:])]) if L < C else x


def _local(q, k, v, la, beta):
    L = q.shape[0]
    q, k, v, la, beta = (_pad(x, L) for x in (q, k, v, la, beta))
    g = np.cumsum(la, axis=0)
    ref = g[31]
    E, F = np.exp(g - ref), np.exp(ref - g)
    Qt, Kt, Kh = q * E, k * E, k * F
    G = Kt @ Kh.T
    T = np.linalg.inv(np.eye(C) + np.tril(beta[:, None] * G, -1))
    Bv, Bk = beta[:, None] * v, beta[:, None] * Kt
    return dict(L=L, v=v, beta=beta, E=E, F=F, Qt=Qt, Kt=Kt, Kh=Kh, G=G, T=T, Bv=Bv, Bk=Bk, Up=T @ Bv, Wt=T @ Bk,
                P=np.tril(Qt @ Kh.T), eref=np.exp(ref), egc=np.exp(g[-1] - ref))


def chunked_bwd(q, k, v, la, beta, S0, dO, dST):
    """Gradients of L = <dO, O> + <dST, S_T> for one head, by chunks."""
    T_, d = q.shape
    n = (T_ + C - 1) // C
    loc = [_local(*(x[i * C:(i + 1) * C] for x in (q, k, v, la, beta))) for i in range(n)]
    dOs = [_pad(dO[i * C:(i + 1) * C], loc[i]["L"]) for i in range(n)]
    S = [S0]
    for c in loc:  # chunk-start states
        X = c["eref"][:, None] * S[-1]
        S.append(c["egc"][:, None] * (X + c["Kh"].T @ (c["Up"] - c["Wt"] @ X)))
    dS = [None] * (n + 1)
    dS[n] = dST
    for i in range(n - 1, -1, -1):  # gradients of the chunk-end states
        c, dOi = loc[i], dOs[i]
        dD = c["egc"][:, None] * dS[i + 1]
        E = c["Qt"].T @ dOi - c["Wt"].T @ (c["P"].T @ dOi)
        dS[i] = c["eref"][:, None] * (dD - c["Wt"].T @ (c["Kh"] @ dD) + E)
    out = {name: [] for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta")}
    for i, c in enumerate(loc):  # each chunk's input gradients
        dOi, X = dOs[i], c["eref"][:, None] * S[i]
        U = c["Up"] - c["Wt"] @ X
        dD = c["egc"][:, None] * dS[i + 1]
        dgc = (S[i + 1] * dS[i + 1]).sum(axis=1)
        dU = c["Kh"] @ dD + c["P"].T @ dOi
        dP = np.tril(dOi @ U.T)
        dWt = -dU @ X.T
        dQt = dOi @ X.T + dP @ c["Kh"]
        dKh = U @ dD.T + dP.T @ c["Qt"]
        dT = dU @ c["Bv"].T + dWt @ c["Bk"].T
        dBv, dBk = c["T"].T @ dU, c["T"].T @ dWt
        dA = np.tril(-c["T"].T @ dT @ c["T"].T, -1)
        dbeta = (dBv * c["v"]).sum(1) + (dBk * c["Kt"]).sum(1) + (dA * c["G"]).sum(1)
        M = c["beta"][:, None] * dA
        dKt = c["beta"][:, None] * dBk + M @ c["Kh"]
        dKh = dKh + M.T @ c["Kt"]
        dlogE = dQt * c["Qt"] + dKt * c["Kt"] - dKh * c["Kh"]
        dlogE[-1] += dgc
        L = c["L"]
        out["dq"].append((dQt * c["E"])[:L])
        out["dk"].append((dKt * c["E"] + dKh * c["F"])[:L])
        out["dv"].append((c["beta"][:, None] * dBv)[:L])
        out["dlog_alpha"].append(np.cumsum(dlogE[::-1], axis=0)[::-1][:L])
        out["dbeta"].append(dbeta[:L])
    res = {name: np.concatenate(parts) for name, parts in out.items()}
    res["dS0"] = dS[0]
    return res


@pytest.mark.parametrize("T", [1, 5, 64, 65, 200])
def test_chunked_algebra_equals_token_serial_reverse_mode(T):
    rng = np.random.default_rng(100 + T)
    d = 128
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)  # noqa: E731
    q, k = unit(rng.standard_normal((T, d))), unit(rng.standard_normal((T, d)))
    v = rng.standard_normal((T, d))
    la = -rng.uniform(0.001, 0.1, (T, d))
    beta = 1 / (1 + np.exp(-rng.standard_normal(T)))
    S0, dO, dST = 0.02 * rng.standard_normal((d, d)), rng.standard_normal((T, d)), rng.standard_normal((d, d))
    ref = oracle.recurrent_bwd(q[None], k[None], v[None], la[None], beta[None], S0[None], dO[None], dST[None])
    got = chunked_bwd(q, k, v, la, beta, S0, dO, dST)
    for name in ("dq", "dk", "dv", "dlog_alpha", "dbeta", "dS0"):
        r = ref[name][0]
        assert np.linalg.norm(got[name] - r) <= 1e-12 * np.linalg.norm(r), name
