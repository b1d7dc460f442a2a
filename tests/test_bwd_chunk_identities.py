"""The chunked (WY) reverse-mode equations the backward kernels evaluate, written out in
fp64 numpy, equal the oracle's token-by-token reverse mode: the derivation is checked on
the CPU independently of the GPU (varlen sequences, partial chunks padded with zero
tokens, chunk-start states from the token recurrence).  Chunk length 8 keeps it small;
the equations do not depend on it."""
import numpy as np

import oracle

C = 8


def _chunked_backward(q, k, v, g, b, cu, s0, do, dfin, sc):
    T, H, dk = k.shape
    dv = v.shape[2]
    N = len(cu) - 1
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "dg": np.zeros_like(g),
           "dbeta": np.zeros_like(b), "d_init": np.zeros((N, H, dk, dv))}
    for n in range(N):
        bos, eos = cu[n], cu[n + 1]
        for h in range(H):
            # chunk-start states by the token recurrence (the forward pass's checkpoints)
            S, ck = s0[n, h].copy(), []
            for t in range(bos, eos):
                if (t - bos) % C == 0:
                    ck.append(S.copy())
                S = np.exp(g[t, h])[:, None] * S
                u = b[t, h] * (v[t, h] - S.T @ k[t, h])
                S = S + np.outer(k[t, h], u)
            dS = dfin[n, h].copy()
            for c in range((eos - bos + C - 1) // C - 1, -1, -1):
                t0 = bos + c * C
                L = min(C, eos - t0)

                def pad(x):
                    return np.concatenate([x, np.zeros((C - L,) + x.shape[1:])]) if L < C else x

                K, Q, V = pad(k[t0:t0 + L, h]), pad(q[t0:t0 + L, h]), pad(v[t0:t0 + L, h])
                Gl, beta, dO = pad(g[t0:t0 + L, h]), pad(b[t0:t0 + L, h]), pad(do[t0:t0 + L, h])
                Sc = ck[c]
                A = np.exp(np.cumsum(Gl, 0))
                AC = A[-1]
                Kb, Kt, Qb = K * A, K / A, sc * Q * A
                Kh = Kt * AC
                Mr = Kb @ Kt.T
                T_ = np.linalg.inv(np.eye(C) + np.tril(beta[:, None] * Mr, -1))
                Tp = T_ * beta[None, :]
                P = np.tril(Qb @ Kt.T)
                R = V - Kb @ Sc
                U = Tp @ R
                dU = Kh @ dS + P.T @ dO
                dP = np.tril(dO @ U.T)
                dR = Tp.T @ dU
                dTp = dU @ R.T
                dQb = dO @ Sc.T + dP @ Kt
                dKh = U @ dS.T
                dKb = -dR @ Sc.T
                dKt = dP.T @ Qb
                dbeta = (dTp * T_).sum(0)
                dM = np.tril(-(T_.T @ (dTp * beta[None, :]) @ T_.T), -1)
                dbeta += (dM * Mr).sum(1)
                dMr = dM * beta[:, None]
                dKb += dMr @ Kt
                dKt += dMr.T @ Kb
                dlac = (dS * Sc).sum(1) * AC + (dKh * Kh).sum(0)
                dla = dKb * Kb - dKt * Kt + dQb * Qb - dKh * Kh
                dgc = np.cumsum(dla[::-1], 0)[::-1] + dlac
                out["dq"][t0:t0 + L, h] = (sc * dQb * A)[:L]
                out["dk"][t0:t0 + L, h] = (dKb * A + dKt / A + dKh * AC / A)[:L]
                out["dv"][t0:t0 + L, h] = dR[:L]
                out["dg"][t0:t0 + L, h] = dgc[:L]
                out["dbeta"][t0:t0 + L, h] = dbeta[:L]
                dS = AC[:, None] * dS + Qb.T @ dO - Kb.T @ dR
            out["d_init"][n, h] = dS
    return out


def test_chunked_backward_equals_token_reverse_mode():
    rng = np.random.default_rng(12)
    lens, H, dk, dv = [1, 7, 8, 9, 0, 20], 2, 5, 3
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    N = len(lens)
    k = rng.standard_normal((T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q, v = rng.standard_normal((T, H, dk)), rng.standard_normal((T, H, dv))
    g = -np.log1p(np.exp(-(rng.standard_normal((T, H, dk)) + 2.0)))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    s0 = rng.standard_normal((N, H, dk, dv)) * 0.1
    do, dfin = rng.standard_normal((T, H, dv)), rng.standard_normal((N, H, dk, dv)) * 0.1
    got = _chunked_backward(q, k, v, g, b, cu, s0, do, dfin, 0.6)
    ref = oracle.backward(q, k, v, g, b, cu, s0, do, dfin, scale=0.6)
    for key in ref:
        err = np.abs(got[key] - ref[key]).max() / max(1e-30, np.abs(ref[key]).max())
        assert err < 1e-12, (key, err)
