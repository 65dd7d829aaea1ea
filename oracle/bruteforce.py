"""Dense float64 numpy formulation of the verify decode, for tiny shapes.

TEST INFRASTRUCTURE ONLY.  A second, independently written statement of the
same definition as ``kda_oracle.c`` ("[KDA] Fuse causal conv1d into MTP
verify decode", cuLA pull request 107, description section), phrased in
matrix form: the conv as a sliding-window contraction, softplus through
``logaddexp``, and the recurrence with explicit matrices

    S <- diag(exp g) @ S ;  S <- S + beta * outer(k, v - S.T @ k) ;  o = K^-1/2 S.T @ q

It is used to cross-check the C oracle on small inputs; it is slow and
allocates freely.
"""

from __future__ import annotations

import numpy as np
from numpy.lib.stride_tricks import sliding_window_view


def _np(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def verify_dense(inputs, gate: str, eps: float = 1e-6):
    x = _np(inputs["mixed_qkv"])          # [N, T, dim]
    w = _np(inputs["conv_w"])             # [dim, W]
    cs = _np(inputs["conv_state"])        # [N, dim, W-1]
    a = _np(inputs["a"])                  # [N, T, HV, K]
    b = _np(inputs["b"])                  # [N, T, HV]
    S0 = _np(inputs["S0"])                # [N, HV, K, V]
    N, T, dim = x.shape
    W = w.shape[1]
    HV, K = a.shape[2], a.shape[3]
    V = S0.shape[3]
    H = (dim - HV * V) // (2 * K)
    G = HV // H

    # [N, dim, T+W-1]: old state then the new tokens along time.
    xext = np.concatenate([cs, np.transpose(x, (0, 2, 1))], axis=2)
    win = sliding_window_view(xext, W, axis=2)        # [N, dim, T, W]
    pre = np.einsum("nctj,cj->nct", win, w)
    y = pre / (1.0 + np.exp(-pre))                    # SiLU
    snaps = np.stack([xext[:, :, t + 1:t + W] for t in range(T)], axis=1)  # [N,T,dim,W-1]
    cs_new = xext[:, :, T:T + W - 1]

    yq = y[:, :H * K, :].reshape(N, H, K, T)
    yk = y[:, H * K:2 * H * K, :].reshape(N, H, K, T)
    yv = y[:, 2 * H * K:, :].reshape(N, HV, V, T)

    if gate == "softplus":
        A_log = _np(inputs["A_log"])
        dt_bias = _np(inputs["dt_bias"])
        z = a + dt_bias[None, None]
        sp = np.where(z > 20.0, z, np.logaddexp(0.0, np.minimum(z, 20.0)))
        g = -np.exp(A_log)[None, None, :, None] * sp
    else:
        g = np.minimum(a, 0.0)
    beta = 1.0 / (1.0 + np.exp(-b))

    o = np.zeros((N, T, HV, V))
    inter = np.zeros((N, T, HV, K, V))
    scale = K ** -0.5
    for n in range(N):
        for hv in range(HV):
            h = hv // G
            S = S0[n, hv].copy()
            for t in range(T):
                q = yq[n, h, :, t]
                k = yk[n, h, :, t]
                q = q / np.sqrt(q @ q + eps)
                k = k / np.sqrt(k @ k + eps)
                v = yv[n, hv, :, t]
                S = np.diag(np.exp(g[n, t, hv])) @ S
                S = S + beta[n, t, hv] * np.outer(k, v - S.T @ k)
                o[n, t, hv] = scale * (S.T @ q)
                inter[n, t, hv] = S
    return {"o": o, "inter_ssm": inter, "conv_snapshots": snaps, "conv_state": cs_new}
