"""The seeded input generator: shapes, dtypes, determinism, planted values."""
import torch

from linear_attention_speculative_gb300 import workloads as wk


def test_shapes_and_dtypes():
    for wl in wk.WORKLOADS.values():
        if wl.shape.N * wl.shape.HV > 1024:
            continue  # keep the CPU suite fast; LARGE is drawn in the GPU tests
        s = wl.shape
        inp = wk.make_inputs(wl)
        assert inp["mixed_qkv"].shape == (s.N, s.T, s.dim)
        assert inp["mixed_qkv"].dtype == s.torch_act
        assert inp["conv_state"].shape == (s.N, s.dim, s.W - 1)
        assert inp["conv_w"].shape == (s.dim, s.W)
        assert inp["a"].shape == (s.N, s.T, s.HV, s.K)
        assert inp["b"].shape == (s.N, s.T, s.HV)
        assert inp["S0"].shape == (s.N, s.HV, s.K, s.V) and inp["S0"].dtype == torch.float32
        if wl.gate == wk.GATE_SOFTPLUS:
            assert inp["A_log"].shape == (s.HV,) and inp["dt_bias"].shape == (s.HV, s.K)
        else:
            assert inp["A_log"] is None and inp["dt_bias"] is None
            assert float(inp["a"].float().max()) <= 0.0


def test_deterministic():
    a = wk.make_inputs(wk.DECODE)
    b = wk.make_inputs(wk.DECODE)
    for k in a:
        assert torch.equal(a[k], b[k])


def test_planted_softplus_overflow_values():
    wl = wk.custom(8, 4, 2, 2, 128, 128)
    wl = wk.Workload(wl.name, wl.shape, wl.gate, wl.seed, wl.s0_std, ("normal", 4.0), (25.0, 100.0))
    a = wk.make_inputs(wl)["a"].float().view(-1)
    assert float(a[0]) == 25.0 and float(a[2048]) == 100.0 and float(a[4096]) == 25.0


def test_sweep_has_150_points():
    pts = list(wk.sweep())
    assert len(pts) == 150
    assert len({p.seed for p in pts}) == 150


def test_algorithmic_bytes_large():
    s = wk.LARGE.shape
    # S0 read + 4 snapshots written dominate: 5 * 4 * N*HV*K*V
    state = 5 * 4 * s.N * s.HV * s.K * s.V
    assert s.algorithmic_bytes() > state
    assert state / s.algorithmic_bytes() > 0.94
