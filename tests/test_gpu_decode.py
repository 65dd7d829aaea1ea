"""GPU parity of kda_conv_decode (plain decode: no snapshots, state updated
in place).  Every test compares the decode with the CPU oracle's verify of
the same inputs (the state it leaves against the oracle's last state
snapshot, o within the tolerance, the rolled conv_state bit for bit), and
also checks that it equals the GPU verify bit for bit: its state the verify's
last snapshot, its o and conv_state the verify's, and T single-token decodes
one T-token verify."""
import pytest
import torch

import oracle
from linear_attention_speculative_gb300 import workloads as wk
from parity_util import assert_decode_parity, plan_built, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from linear_attention_speculative_gb300 import kda
    kda.lib()


def _decode(kda, inp, gate, plan=None, idx=None):
    o = torch.empty((inp["mixed_qkv"].shape[0], inp["mixed_qkv"].shape[1], inp["a"].shape[2],
                     inp["S0"].shape[3]), dtype=inp["mixed_qkv"].dtype, device="cuda")
    shape = kda.shape_of(inp["mixed_qkv"], inp["a"], inp["S0"][: inp["mixed_qkv"].shape[0]])
    ws = kda.alloc_workspace(shape, "cuda")
    kda.conv_decode(inp["mixed_qkv"], inp["conv_w"], inp["conv_state"], inp["A_log"], inp["dt_bias"],
                    inp["a"], inp["b"], inp["S0"], gate, o, ws, plan=plan, idx=idx, shape=shape)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("plan", [None, "item:128", "item:32", "item:16:0:-1", "smem:128", "smem:64",
                                  "item:32:0:0:kernel", "smem:64:0:0:kernel", "smem:128:0:0:counter",
                                  "item:64", "smem:32", "item:128:0:0:cluster", "item:32:0:0:cluster",
                                  "item:64:0:0:cluster"])
@pytest.mark.parametrize("case", [(5, 4, 2, 4, 128, 128, "bf16", "softplus"),
                                  (3, 1, 2, 2, 128, 128, "bf16", "safe"),
                                  (4, 3, 1, 2, 64, 64, "f32", "softplus"),
                                  (3, 2, 1, 2, 256, 128, "bf16", "softplus")],
                         ids=lambda c: "N{}_T{}_H{}_HV{}_K{}_V{}_{}_{}".format(*c))
def test_decode_equals_last_verify_snapshot(case, plan):
    from linear_attention_speculative_gb300 import kda
    N, T, H, HV, K, V, act, gate = case
    if not plan_built(plan, K, V, decode=True, G=HV // H):
        pytest.skip("no such kernel for this shape")
    wl = wk.custom(N, T, H, HV, K, V, act=act, gate=gate, seed=91 + T)
    inp_cpu = wk.make_inputs(wl)
    orc = oracle.verify(inp_cpu, gate)
    inp = to_device(inp_cpu)
    ver = dict(inp, conv_state=inp["conv_state"].clone())
    ref = kda.run(ver, gate)
    dec = dict(inp, conv_state=inp["conv_state"].clone(), S0=inp["S0"].clone())
    o = _decode(kda, dec, gate, plan)
    assert_decode_parity(o, dec["S0"], dec["conv_state"], orc)
    assert torch.equal(dec["S0"], ref["inter_ssm"][:, -1])
    assert torch.equal(o, ref["o"])
    assert torch.equal(dec["conv_state"], ver["conv_state"])


def test_single_token_decodes_chain_to_one_verify():
    from linear_attention_speculative_gb300 import kda
    T = 4
    wl = wk.custom(6, T, 2, 4, 128, 128, seed=95)
    inp_cpu = wk.make_inputs(wl)
    orc = oracle.verify(inp_cpu, wl.gate)
    inp = to_device(inp_cpu)
    ver = dict(inp, conv_state=inp["conv_state"].clone())
    ref = kda.run(ver, wl.gate)
    st = dict(inp, conv_state=inp["conv_state"].clone(), S0=inp["S0"].clone())
    for t in range(T):
        step = dict(st)
        for key in ("mixed_qkv", "a", "b"):
            step[key] = inp[key][:, t:t + 1].contiguous()
        o = _decode(kda, step, wl.gate)
        # token t of the chain against token t of the oracle's one call
        assert_decode_parity(o, st["S0"], None, orc, t=t)
        assert torch.equal(o[:, 0], ref["o"][:, t])
        assert torch.equal(st["S0"], ref["inter_ssm"][:, t])
    assert_decode_parity(o, st["S0"], st["conv_state"], orc, t=T - 1)
    assert torch.equal(st["conv_state"], ver["conv_state"])


def test_decode_over_state_pools():
    from linear_attention_speculative_gb300 import kda
    wl = wk.custom(5, 2, 2, 2, 128, 128, seed=96)
    inp_cpu = wk.make_inputs(wl)
    inp = to_device(inp_cpu)
    N = 5
    slot_s = torch.tensor([7, 0, -1, 3, 5], dtype=torch.int32, device="cuda")
    slot_c = torch.tensor([1, 4, 2, 0, 6], dtype=torch.int32, device="cuda")
    S_pool = torch.randn((8, 2, 128, 128), device="cuda")
    cs_pool = torch.randn((7, inp["conv_state"].shape[1], 3), device="cuda").to(torch.bfloat16)
    for n in range(N):
        if slot_s[n] >= 0:
            S_pool[slot_s[n]] = inp["S0"][n]
        cs_pool[slot_c[n]] = inp["conv_state"][n]
    S_before, cs_before = S_pool.clone(), cs_pool.clone()
    idx = kda.state_indices(slot_s, slot_c, None, 8, 7, 0)
    dec = dict(inp, conv_state=cs_pool, S0=S_pool)
    shape = kda.shape_of(inp["mixed_qkv"], inp["a"], inp["S0"])
    ws = kda.alloc_workspace(shape, "cuda")
    o = torch.full((N, 2, 2, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    kda.conv_decode(inp["mixed_qkv"], inp["conv_w"], cs_pool, inp["A_log"], inp["dt_bias"], inp["a"],
                    inp["b"], S_pool, wl.gate, o, ws, idx=idx, shape=shape)
    ver = dict(inp, conv_state=inp["conv_state"].clone())
    ref = kda.run(ver, wl.gate)
    torch.cuda.synchronize()
    live = [0, 1, 3, 4]
    orc = oracle.verify(inp_cpu, wl.gate, seqs=live)
    assert_decode_parity(o[live], torch.stack([S_pool[int(slot_s[n])] for n in live]),
                         torch.stack([cs_pool[int(slot_c[n])] for n in live]), orc)
    for n in live:
        assert torch.equal(S_pool[slot_s[n]], ref["inter_ssm"][n, -1])
        assert torch.equal(cs_pool[slot_c[n]], ver["conv_state"][n])
        assert torch.equal(o[n], ref["o"][n])
    assert bool((o[2] == 5.0).all())                      # padding sequence untouched
    assert torch.equal(cs_pool[slot_c[2]], cs_before[slot_c[2]])
    for sl in (1, 2, 4, 6):                               # unused state slots untouched
        assert torch.equal(S_pool[sl], S_before[sl])


def test_decode_rejects_persistent_plans():
    from linear_attention_speculative_gb300 import kda
    wl = wk.custom(2, 1, 2, 2, 128, 128, seed=97)
    inp = to_device(wk.make_inputs(wl))
    with pytest.raises(kda.KdaError) as e:
        _decode(kda, inp, wl.gate, plan="pipe:64")
    assert e.value.code == -8


def _random_decode_cases(seed=2027):
    # KDA_RANDOM_CASES sets how many (default 24); the first 24 are always the same
    import os
    import numpy as np
    n = int(os.environ.get("KDA_RANDOM_CASES", "24"))
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        K = int(rng.choice([32, 64, 128, 256]))
        V = int(rng.choice([32, 64, 128, 256]))
        H = int(rng.integers(1, 4))
        HV = H * int(rng.choice([1, 2, 3, 4]))
        T = int(rng.integers(1, 9))
        N = int(rng.integers(1, 7))
        act = str(rng.choice(["bf16", "f32"]))
        gate = str(rng.choice(["softplus", "safe"]))
        plans = [None] + [p for p in ("item:16", "item:32", "item:64", "item:128", "smem:32", "smem:64",
                                      "smem:128", "item:64:0:0:kernel", "item:32:0:0:counter")
                          if plan_built(p, K, V, decode=True, T=T, act=act, G=HV // H)]
        plan = plans[int(rng.integers(0, len(plans)))]
        cases.append((N, T, H, HV, K, V, act, gate, plan, 3000 + len(cases)))
    return cases


@pytest.mark.parametrize("case", _random_decode_cases(),
                         ids=lambda c: "N{}_T{}_H{}_HV{}_K{}_V{}_{}_{}_{}".format(*c[:9]))
def test_random_decode_shapes_and_plans(case):
    # the decode of random shapes and plans against the oracle's verify of the
    # same inputs (its state after the last token, o, the rolled conv_state)
    from linear_attention_speculative_gb300 import kda
    N, T, H, HV, K, V, act, gate, plan, seed = case
    wl = wk.custom(N, T, H, HV, K, V, act=act, gate=gate, seed=seed)
    inp_cpu = wk.make_inputs(wl)
    orc = oracle.verify(inp_cpu, gate)
    dec = to_device(inp_cpu)
    o = _decode(kda, dec, gate, plan)
    assert_decode_parity(o, dec["S0"], dec["conv_state"], orc)
