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


def _tensor_bytes(wl):
    """Bytes of the tensors one verify call reads and writes, counted from the
    generated inputs and the outputs: every input read once, conv_state read
    and written, every output written once."""
    inp = wk.make_inputs(wl)
    out = wk.empty_outputs(wl)
    read = sum(v.numel() * v.element_size() for v in inp.values() if v is not None)
    cs = inp["conv_state"]
    written = sum(v.numel() * v.element_size() for v in out.values()) + cs.numel() * cs.element_size()
    return read, written


def test_algorithmic_bytes_equal_the_tensors_a_call_touches():
    for wl in (wk.TINY, wk.DECODE, wk.custom(3, 5, 2, 8, 64, 128, gate="safe", seed=1),
               wk.custom(2, 3, 1, 2, 32, 64, act="f32", seed=2)):
        read, written = _tensor_bytes(wl)
        assert wl.shape.algorithmic_bytes(wl.gate) == read + written, wl.name


def test_algorithmic_bytes_of_the_large_batch():
    # the figure the large-batch roofline divides by: 589,480,064 B read
    # (S0 536.9 MB, inputs 52.6 MB) and 2,250,244,096 B written
    s = wk.LARGE.shape
    S = 4 * s.N * s.HV * s.K * s.V
    read = S + 2 * (s.N * s.T * s.dim + s.N * s.dim * 3 + s.dim * 4 + s.N * s.T * s.HV * s.K
                    + s.N * s.T * s.HV) + 4 * s.HV * (1 + s.K)
    written = s.T * S + 2 * (s.N * s.T * s.HV * s.V + s.N * s.T * s.dim * 3 + s.N * s.dim * 3)
    assert (read, written) == (589_480_064, 2_250_244_096)
    assert s.algorithmic_bytes(wk.LARGE.gate) == read + written == 2_839_724_160
