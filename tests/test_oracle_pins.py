"""Pins of the CPU oracle against facts fixed by the definition itself.

The definition is the one on "[KDA] Fuse causal conv1d into MTP verify
decode" (cuLA pull request 107): causal conv1d + SiLU, q/k L2 norm,
gate/beta, the gated delta rule S <- diag(exp g) S, S <- S + beta k (v -
S^T k)^T, o = K^-1/2 S^T q, with per-token state and conv-window snapshots.
Each test names the fact it pins; together they are chosen so that a dropped
term, a wrong sign, a transposed operand, a swapped channel block, a wrong
head map or an off-by-one conv tap fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.bruteforce import verify_dense
from linear_attention_speculative_gb300 import workloads as wk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- scalar functions ------------------------------------------------------

def test_softplus_closed_values():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    # just below the threshold: log(1+e^20) = 20 + log(1+e^-20)
    assert oracle.softplus(20.0) == pytest.approx(20.0 + math.exp(-20.0), rel=1e-15)
    # linear branch above 20 (exact identity), and no overflow at 100 / 1000
    assert oracle.softplus(20.5) == 20.5
    assert oracle.softplus(100.0) == 100.0
    assert oracle.softplus(1000.0) == 1000.0
    # far negative: log1p(e^x) ~ e^x
    assert oracle.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-12)
    # softplus(x) - softplus(-x) = x
    for x in (-3.0, -0.25, 0.7, 5.0, 19.0):
        assert oracle.softplus(x) - oracle.softplus(-x) == pytest.approx(x, abs=1e-13)


def test_sigmoid_and_silu_identities():
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.sigmoid(40.0) == 1.0  # beta saturates to exactly 1 in fp64
    for x in (-7.0, -1.0, 0.3, 2.5):
        assert oracle.sigmoid(x) + oracle.sigmoid(-x) == pytest.approx(1.0, abs=1e-15)
        # silu(y) - silu(-y) = y * (sigmoid(y) + sigmoid(-y)) = y
        assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, abs=1e-14)
        assert oracle.silu(x) == pytest.approx(x * oracle.sigmoid(x), rel=1e-15)
    assert oracle.silu(0.0) == 0.0


def test_gates():
    # softplus gate: A_log = 0, a + dt_bias = 0 -> g = -ln 2 exactly
    assert oracle.gate_softplus(0.0, 0.3, -0.3) == pytest.approx(-math.log(2.0), rel=1e-15)
    # A_log = ln 3 scales by -3; linear branch above 20
    assert oracle.gate_softplus(math.log(3.0), 30.0, -5.0) == pytest.approx(-75.0, rel=1e-14)
    # the gate is a decay: g <= 0 always
    for a in (-40.0, -1.0, 0.0, 1.0, 25.0, 100.0):
        assert oracle.gate_softplus(0.5, a, 0.1) <= 0.0
    # safe gate clamps to <= 0 and is the identity below 0
    assert oracle.gate_safe(-3.25) == -3.25
    assert oracle.gate_safe(2.0) == 0.0
    assert oracle.gate_safe(0.0) == 0.0


# ---- conv ----------------------------------------------------------------

def test_conv_identity_tap_selects_newest_input():
    T, W = 5, 4
    xext = np.arange(1, T + W) * 0.25 - 1.0
    w = np.zeros(W); w[W - 1] = 1.0
    y = oracle.causal_conv1d_silu(xext, w, T)
    expect = [oracle.silu(v) for v in xext[W - 1:]]
    np.testing.assert_array_equal(y, expect)


def test_conv_oldest_tap_reads_the_state():
    T, W = 3, 4
    xext = np.array([0.5, -1.5, 2.0, 3.0, -4.0, 1.0])
    w = np.zeros(W); w[0] = 1.0
    y = oracle.causal_conv1d_silu(xext, w, T)
    np.testing.assert_array_equal(y, [oracle.silu(v) for v in xext[:T]])


def test_conv_matches_library_correlation():
    rng = np.random.default_rng(7)
    T, W = 6, 4
    xext = rng.standard_normal(T + W - 1)
    w = rng.standard_normal(W)
    pre = np.correlate(xext, w, mode="valid")  # sum_j w[j] x[t+j]
    expect = pre / (1.0 + np.exp(-pre))
    np.testing.assert_allclose(oracle.causal_conv1d_silu(xext, w, T), expect, rtol=1e-14, atol=1e-15)


# ---- L2 norm -------------------------------------------------------------

def test_l2norm():
    x = np.array([3.0, 4.0])
    y = oracle.l2norm(x, 0.0)
    np.testing.assert_allclose(y, [0.6, 0.8], rtol=1e-15)
    # with eps inside the root: |y|^2 = s / (s + eps)
    rng = np.random.default_rng(3)
    x = rng.standard_normal(128)
    s = float(x @ x)
    y = oracle.l2norm(x, 1e-6)
    assert float(y @ y) == pytest.approx(s / (s + 1e-6), rel=1e-14)
    np.testing.assert_allclose(y / np.linalg.norm(y), x / np.linalg.norm(x), rtol=1e-14)
    # zero input stays zero (eps > 0 avoids 0/0)
    np.testing.assert_array_equal(oracle.l2norm(np.zeros(8), 1e-6), np.zeros(8))


# ---- one recurrence token ------------------------------------------------

def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *rest = line.split()
            vals[key] = np.array([float(r) for r in rest])
    return vals


def test_delta_rule_hand_worked_2x2():
    gv = _read_golden("delta_rule_2x2.txt")
    S, o = oracle.delta_rule_step(gv["S0"].reshape(2, 2), np.log(gv["expg"]), gv["k"], gv["v"],
                                  float(gv["beta"][0]), gv["q"], float(gv["scale"][0]))
    np.testing.assert_allclose(S.ravel(), gv["S_out"], rtol=1e-14)
    np.testing.assert_allclose(o, gv["o_out"], rtol=1e-14)


def test_delta_rule_unit_key_full_beta_stores_v():
    # beta = 1, |k| = 1, g = 0  =>  S^T k = v after the update
    rng = np.random.default_rng(11)
    K, V = 16, 12
    S0 = rng.standard_normal((K, V))
    k = rng.standard_normal(K); k /= np.linalg.norm(k)
    v = rng.standard_normal(V)
    S, _ = oracle.delta_rule_step(S0, np.zeros(K), k, v, 1.0, rng.standard_normal(K), 1.0)
    np.testing.assert_allclose(S.T @ k, v, rtol=1e-12, atol=1e-12)


def test_delta_rule_zero_beta_zero_gate_keeps_state():
    rng = np.random.default_rng(12)
    K, V = 8, 8
    S0 = rng.standard_normal((K, V))
    q = rng.standard_normal(K)
    S, o = oracle.delta_rule_step(S0, np.zeros(K), rng.standard_normal(K),
                                  rng.standard_normal(V), 0.0, q, 0.5)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, 0.5 * S0.T @ q, rtol=1e-14)


def test_delta_rule_zero_beta_is_pure_decay():
    rng = np.random.default_rng(13)
    K, V = 8, 5
    S0 = rng.standard_normal((K, V))
    g = -rng.uniform(0, 3, K)
    S, _ = oracle.delta_rule_step(S0, g, rng.standard_normal(K), rng.standard_normal(V), 0.0,
                                  np.zeros(K), 1.0)
    np.testing.assert_allclose(S, np.exp(g)[:, None] * S0, rtol=1e-15)


def test_delta_rule_closed_form_from_zero_state():
    # S0 = 0 => S = beta k v^T, o = scale * beta (k . q) v   (any gate)
    rng = np.random.default_rng(14)
    K, V = 8, 6
    k, q, v = rng.standard_normal(K), rng.standard_normal(K), rng.standard_normal(V)
    beta, scale = 0.3, 0.25
    S, o = oracle.delta_rule_step(np.zeros((K, V)), -rng.uniform(0, 1, K), k, v, beta, q, scale)
    np.testing.assert_allclose(S, beta * np.outer(k, v), rtol=1e-14)
    np.testing.assert_allclose(o, scale * beta * float(k @ q) * v, rtol=1e-13)


# ---- the whole call --------------------------------------------------------

def _tiny(N=2, T=3, H=2, HV=2, K=8, V=8, gate="softplus", seed=5):
    wl = wk.custom(N, T, H, HV, K, V, act="f32", gate=gate, seed=seed, s0_std=0.3)
    return wl, wk.make_inputs(wl)


@pytest.mark.parametrize("gate", ["softplus", "safe"])
@pytest.mark.parametrize("shape", [(2, 1, 1, 1, 4, 4), (2, 3, 2, 2, 8, 4), (1, 5, 1, 3, 4, 8),
                                   (3, 2, 2, 4, 8, 8), (1, 4, 2, 2, 4, 4)])
def test_oracle_matches_dense_bruteforce(gate, shape):
    wl, inp = _tiny(*shape, gate=gate, seed=sum(shape))
    got = oracle.verify(inp, gate)
    ref = verify_dense(inp, gate)
    for key in ("o", "inter_ssm"):
        np.testing.assert_allclose(got[key], ref[key], rtol=1e-12, atol=1e-12)
    for key in ("conv_snapshots", "conv_state"):
        np.testing.assert_array_equal(got[key], ref[key])


def test_oracle_matches_dense_bruteforce_tiny_fp32_workload():
    inp = wk.make_inputs(wk.TINY)
    got = oracle.verify(inp, wk.TINY.gate)
    ref = verify_dense(inp, wk.TINY.gate)
    for key in ("o", "inter_ssm"):
        np.testing.assert_allclose(got[key], ref[key], rtol=1e-12, atol=1e-12)
    for key in ("conv_snapshots", "conv_state"):
        np.testing.assert_array_equal(got[key], ref[key])


@pytest.mark.parametrize("gate", ["softplus", "safe"])
@pytest.mark.parametrize("T", [1, 2, 3, 5])
def test_chain_of_single_token_calls_equals_one_call(gate, T):
    # one T-token call == T chained T=1 calls (S0 <- last snapshot, conv_state <- rolled state)
    wl, inp = _tiny(N=2, T=T, H=1, HV=2, K=8, V=4, gate=gate, seed=40 + T)
    full = oracle.verify(inp, gate)
    S = inp["S0"].double()
    cs = inp["conv_state"].double()
    for t in range(T):
        step = dict(inp)
        step["mixed_qkv"] = inp["mixed_qkv"][:, t:t + 1]
        step["a"] = inp["a"][:, t:t + 1]
        step["b"] = inp["b"][:, t:t + 1]
        step["S0"] = S
        step["conv_state"] = cs
        out = oracle.verify(step, gate)
        np.testing.assert_array_equal(out["o"][:, 0], full["o"][:, t])
        np.testing.assert_array_equal(out["inter_ssm"][:, 0], full["inter_ssm"][:, t])
        np.testing.assert_array_equal(out["conv_snapshots"][:, 0], full["conv_snapshots"][:, t])
        S = torch.from_numpy(out["inter_ssm"][:, 0])
        cs = torch.from_numpy(out["conv_state"])
    np.testing.assert_array_equal(cs.numpy(), full["conv_state"])


def test_conv_snapshots_and_rolled_state_are_raw_windows():
    wl, inp = _tiny(N=2, T=4, H=1, HV=1, K=4, V=4, seed=9)
    out = oracle.verify(inp, "softplus")
    cs = inp["conv_state"].double().numpy()
    x = inp["mixed_qkv"].double().numpy()
    for n in range(2):
        xext = np.concatenate([cs[n], x[n].T], axis=1)  # [dim, T+3]
        for t in range(4):
            np.testing.assert_array_equal(out["conv_snapshots"][n, t], xext[:, t + 1:t + 4])
        np.testing.assert_array_equal(out["conv_state"][n], xext[:, 4:7])
    # the rolled state is the last snapshot
    np.testing.assert_array_equal(out["conv_state"], out["conv_snapshots"][:, -1])


def test_short_verify_keeps_old_state_in_window():
    # T = 1 < W-1: the rolled state keeps two old values and the new token
    wl, inp = _tiny(N=1, T=1, H=1, HV=1, K=4, V=4, seed=10)
    out = oracle.verify(inp, "softplus")
    cs = inp["conv_state"].double().numpy()[0]
    x = inp["mixed_qkv"].double().numpy()[0, 0]
    np.testing.assert_array_equal(out["conv_state"][0][:, :2], cs[:, 1:])
    np.testing.assert_array_equal(out["conv_state"][0][:, 2], x)


def test_channel_order_q_k_v_and_closed_form_first_token():
    # identity conv (tap W-1 = 1), S0 = 0, T = 1: S = beta k^ v^T, o = K^-1/2 beta (k^.q^) v
    # with q^, k^ the L2-normalised SiLU of the q and k channel blocks.  Distinct
    # values per block make a swapped q|k|v order fail.
    K = V = 4
    wl, inp = _tiny(N=1, T=1, H=1, HV=1, K=K, V=V, gate="safe", seed=17)
    w = torch.zeros_like(inp["conv_w"]); w[:, 3] = 1.0
    inp["conv_w"] = w
    inp["S0"] = torch.zeros_like(inp["S0"])
    xq = np.array([1.0, -2.0, 0.5, 3.0]); xk = np.array([-1.0, 0.25, 2.0, 1.5])
    xv = np.array([0.125, -0.75, 1.25, 2.5])  # exact in fp32
    inp["mixed_qkv"] = torch.tensor(np.concatenate([xq, xk, xv])[None, None], dtype=torch.float32)
    inp["b"] = torch.tensor([[[0.375]]])
    out = oracle.verify(inp, "safe")
    silu = np.vectorize(oracle.silu)
    q, k, v = silu(xq), silu(xk), silu(xv)
    q = q / math.sqrt(q @ q + 1e-6); k = k / math.sqrt(k @ k + 1e-6)
    beta = oracle.sigmoid(0.375)
    np.testing.assert_allclose(out["inter_ssm"][0, 0, 0], beta * np.outer(k, v), rtol=1e-13)
    np.testing.assert_allclose(out["o"][0, 0, 0], 0.5 * beta * float(k @ q) * v, rtol=1e-12)


def test_zero_conv_weights_leave_only_the_decay():
    # conv_w = 0 => q = k = v = 0 => o = 0 and S_t = diag(exp(sum_{tau<=t} g_tau)) S0.
    # Softplus gate with A_log = 0 and a + dt_bias = 0 gives g = -ln 2: S_t = 2^-(t+1) S0.
    T = 3
    wl, inp = _tiny(N=1, T=T, H=1, HV=2, K=4, V=4, seed=21)
    inp["conv_w"] = torch.zeros_like(inp["conv_w"])
    inp["A_log"] = torch.zeros_like(inp["A_log"])
    inp["a"] = -inp["dt_bias"][None, None].expand_as(inp["a"]).clone()
    out = oracle.verify(inp, "softplus")
    np.testing.assert_array_equal(out["o"], 0.0)
    S0 = inp["S0"].double().numpy()
    for t in range(T):
        np.testing.assert_allclose(out["inter_ssm"][0, t], 0.5 ** (t + 1) * S0[0], rtol=1e-14)


def test_safe_gate_decay_accumulates():
    T = 4
    wl, inp = _tiny(N=1, T=T, H=1, HV=1, K=4, V=4, gate="safe", seed=22)
    inp["conv_w"] = torch.zeros_like(inp["conv_w"])
    out = oracle.verify(inp, "safe")
    a = np.minimum(inp["a"].double().numpy()[0, :, 0], 0.0)  # [T, K]
    S0 = inp["S0"].double().numpy()[0, 0]
    for t in range(T):
        np.testing.assert_allclose(out["inter_ssm"][0, t, 0],
                                   np.exp(a[:t + 1].sum(0))[:, None] * S0, rtol=1e-13)


def test_gva_equals_duplicated_qk_heads():
    # HV = H*G sharing q/k head hv // G  ==  an H'=HV problem whose q/k head j is
    # a copy of the shared head j // G (channels, conv weights and conv state).
    H, G, K, V, T, N = 2, 2, 4, 4, 3, 2
    HV = H * G
    wl, inp = _tiny(N=N, T=T, H=H, HV=HV, K=K, V=V, seed=31)
    out = oracle.verify(inp, "softplus")

    def dup_qk(t, axis):
        # channel axis `axis` holds q (H*K) | k (H*K) | v (HV*V)
        q, k, v = torch.split(t, [H * K, H * K, HV * V], dim=axis)
        rep = lambda z: torch.repeat_interleave(z.unflatten(axis, (H, K)), G, dim=axis).flatten(axis, axis + 1)
        return torch.cat([rep(q), rep(k), v], dim=axis)

    mha = dict(inp)
    mha["mixed_qkv"] = dup_qk(inp["mixed_qkv"], 2)
    mha["conv_state"] = dup_qk(inp["conv_state"], 1)
    mha["conv_w"] = dup_qk(inp["conv_w"], 0)
    out2 = oracle.verify(mha, "softplus")
    np.testing.assert_array_equal(out["o"], out2["o"])
    np.testing.assert_array_equal(out["inter_ssm"], out2["inter_ssm"])


def test_rejects_bad_shapes():
    wl, inp = _tiny(N=1, T=2, H=2, HV=2, K=4, V=4)
    bad = dict(inp)
    bad["a"] = inp["a"][:, :, :1].contiguous()  # HV = 1 < H = 2
    with pytest.raises(ValueError):
        oracle.verify(bad, "softplus")


def test_frozen_tiny_fp32_values():
    # regression anchor written by tests/golden/make_golden.py (calls only oracle/)
    path = os.path.join(GOLDEN, "tiny_fp32_oracle.txt")
    stored = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, idx, val = line.split()
            stored[(key, tuple(int(i) for i in idx.split(",")))] = float(val)
    out = oracle.verify(wk.make_inputs(wk.TINY), wk.TINY.gate)
    for (key, idx), val in stored.items():
        assert out[key][idx] == pytest.approx(val, rel=1e-12, abs=1e-15), (key, idx)


# ---- commit after verify ----------------------------------------------------

@pytest.mark.parametrize("gate", ["softplus", "safe"])
def test_commit_equals_verify_of_the_accepted_prefix(gate):
    # verify T tokens, then accept a of them == verify only the first a tokens
    T = 4
    wl, inp = _tiny(N=4, T=T, H=1, HV=2, K=8, V=4, gate=gate, seed=61)
    full = oracle.verify(inp, gate)
    acc = [1, 2, 3, 4]
    com = oracle.commit(acc, full["inter_ssm"], full["conv_snapshots"])
    for n, a in enumerate(acc):
        pre = dict(inp)
        for key in ("mixed_qkv", "a", "b"):
            pre[key] = inp[key][n:n + 1, :a]
        for key in ("conv_state", "S0"):
            pre[key] = inp[key][n:n + 1]
        ref = oracle.verify(pre, gate)
        np.testing.assert_array_equal(com["S"][n], ref["inter_ssm"][0, a - 1])
        np.testing.assert_array_equal(com["conv_state"][n], ref["conv_state"][0])


def test_commit_of_every_token_is_the_rolled_state():
    wl, inp = _tiny(N=2, T=3, H=1, HV=1, K=4, V=4, seed=62)
    full = oracle.verify(inp, "softplus")
    com = oracle.commit([3, 3], full["inter_ssm"], full["conv_snapshots"])
    np.testing.assert_array_equal(com["conv_state"], full["conv_state"])
    np.testing.assert_array_equal(com["S"], full["inter_ssm"][:, -1])


def test_commit_rejects_out_of_range_counts():
    wl, inp = _tiny(N=2, T=3, H=1, HV=1, K=4, V=4, seed=63)
    full = oracle.verify(inp, "softplus")
    for bad in ([0, 1], [1, 4], [-1, 2]):
        with pytest.raises(ValueError):
            oracle.commit(bad, full["inter_ssm"], full["conv_snapshots"])
