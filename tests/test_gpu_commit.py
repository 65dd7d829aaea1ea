"""GPU parity of kda_commit (accept the first acc[n] verified tokens).

Pure copies, so the check is bit-exact: against the CPU oracle's commit, and
against the identity that a T-token verify followed by commit(a) equals a
verify of the first a tokens alone."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_speculative_gb300 import workloads as wk
from parity_util import assert_parity, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from linear_attention_speculative_gb300 import kda
    kda.lib()


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_commit_matches_oracle_and_reports_bad_counts(act):
    from linear_attention_speculative_gb300 import kda
    T = 4
    wl = wk.custom(9, T, 2, 4, 128, 64, act=act, seed=71)
    inp = to_device(wk.make_inputs(wl))
    out = kda.run(dict(inp, conv_state=inp["conv_state"].clone()), wl.gate)
    acc = torch.tensor([1, 2, 3, 4, 4, 0, 5, -1, 2], dtype=torch.int32, device="cuda")
    S = torch.full_like(inp["S0"], 7.0)
    cs = torch.full_like(inp["conv_state"], 3.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.commit(acc, out["inter_ssm"], out["conv_snapshots"], S, cs, status=status)
    torch.cuda.synchronize()
    good = [i for i, a in enumerate(acc.tolist()) if 1 <= a <= T]
    bad = [i for i in range(9) if i not in good]
    ref = oracle.commit([acc.tolist()[i] for i in good], out["inter_ssm"][good].cpu(),
                        out["conv_snapshots"][good].cpu())
    np.testing.assert_array_equal(S[good].double().cpu().numpy(), ref["S"])
    np.testing.assert_array_equal(cs[good].double().cpu().numpy(), ref["conv_state"])
    assert bool((S[bad] == 7.0).all()) and bool((cs[bad] == 3.0).all())  # untouched
    assert int(status.item()) == kda.STATUS_BAD_ACCEPT


@pytest.mark.parametrize("gate", ["softplus", "safe"])
def test_verify_then_commit_equals_verify_of_the_prefix(gate):
    from linear_attention_speculative_gb300 import kda
    T = 5
    wl = wk.custom(5, T, 2, 4, 128, 128, gate=gate, seed=72)
    inp = to_device(wk.make_inputs(wl))
    full = kda.run(dict(inp, conv_state=inp["conv_state"].clone()), gate)
    acc = torch.tensor([1, 2, 3, 4, 5], dtype=torch.int32, device="cuda")
    S = torch.empty_like(inp["S0"])
    cs = torch.empty_like(inp["conv_state"])
    kda.commit(acc, full["inter_ssm"], full["conv_snapshots"], S, cs)
    for n, a in enumerate(acc.tolist()):
        pre = dict(inp)
        for key in ("mixed_qkv", "a", "b"):
            pre[key] = inp[key][n:n + 1, :a].contiguous()
        pre["S0"] = inp["S0"][n:n + 1].contiguous()
        pre["conv_state"] = inp["conv_state"][n:n + 1].clone()
        ref = kda.run(pre, gate)
        torch.cuda.synchronize()
        assert torch.equal(S[n], ref["inter_ssm"][0, a - 1])
        assert torch.equal(cs[n], pre["conv_state"][0])


def test_commit_in_place_into_the_verified_state():
    # the usual chain: verify reads S0, commit writes the accepted state back into S0
    from linear_attention_speculative_gb300 import kda
    wl = wk.custom(4, 3, 2, 2, 128, 128, seed=73)
    inp = to_device(wk.make_inputs(wl))
    out = kda.run(inp, wl.gate)
    acc = torch.tensor([3, 1, 2, 3], dtype=torch.int32, device="cuda")
    kda.commit(acc, out["inter_ssm"], out["conv_snapshots"], inp["S0"], inp["conv_state"])
    torch.cuda.synchronize()
    for n, a in enumerate(acc.tolist()):
        assert torch.equal(inp["S0"][n], out["inter_ssm"][n, a - 1])
        assert torch.equal(inp["conv_state"][n], out["conv_snapshots"][n, a - 1])


def _random_commit_cases(seed=2029):
    # KDA_RANDOM_CASES sets how many (default 24); the first 24 are always the same
    import os
    n = int(os.environ.get("KDA_RANDOM_CASES", "24"))
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        K = int(rng.choice([32, 64, 128, 256]))
        V = int(rng.choice([32, 64, 128, 256]))
        H = int(rng.integers(1, 4))
        HV = H * int(rng.choice([1, 2, 3, 4]))
        T = int(rng.integers(1, 17))
        N = int(rng.integers(1, 9))
        act = str(rng.choice(["bf16", "f32"]))
        acc = [int(rng.integers(1, T + 1)) for _ in range(N)]
        cases.append((N, T, H, HV, K, V, act, tuple(acc), 7000 + i))
    return cases


@pytest.mark.parametrize("case", _random_commit_cases(),
                         ids=lambda c: "N{}_T{}_H{}_HV{}_K{}_V{}_{}".format(*c[:7]))
def test_random_commit_matches_the_oracle(case):
    # random shapes and accepted counts: the committed state and conv_state
    # bit for bit against the oracle's commit of the same snapshots
    from linear_attention_speculative_gb300 import kda
    N, T, H, HV, K, V, act, acc_l, seed = case
    wl = wk.custom(N, T, H, HV, K, V, act=act, seed=seed)
    inp = to_device(wk.make_inputs(wl))
    out = kda.run(dict(inp, conv_state=inp["conv_state"].clone()), wl.gate)
    acc = torch.tensor(acc_l, dtype=torch.int32, device="cuda")
    S = torch.full_like(inp["S0"], 7.0)
    cs = torch.full_like(inp["conv_state"], 3.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.commit(acc, out["inter_ssm"], out["conv_snapshots"], S, cs, status=status)
    torch.cuda.synchronize()
    ref = oracle.commit(list(acc_l), out["inter_ssm"].cpu(), out["conv_snapshots"].cpu())
    np.testing.assert_array_equal(S.double().cpu().numpy(), ref["S"])
    np.testing.assert_array_equal(cs.double().cpu().numpy(), ref["conv_state"])
    assert int(status.item()) == 0


@pytest.mark.parametrize("plan", [None, "item:64:0:0:cluster", "item:128:0:0:kernel", "smem:128"])
def test_verify_commit_loop_without_a_sync(plan):
    """A serving loop: verify, commit, verify, commit ... queued back to back
    on one stream with nothing between them and no synchronisation.  Both
    kernels are launched as programmatic dependents of the kernel before
    them, so each commit must see its verify's snapshots and each verify the
    state and conv_state the commit before it wrote: every verify is checked
    against the oracle run on the state that commit left (taken from the
    previous verify's own snapshots), and the final state bit for bit."""
    from linear_attention_speculative_gb300 import kda
    N, T, H, HV, steps = 24, 3, 4, 8, 4
    cpu = [wk.make_inputs(wk.custom(N, T, H, HV, 128, 128, seed=130 + i)) for i in range(steps)]
    dev = [to_device(c) for c in cpu]
    S = dev[0]["S0"].clone()
    cs = dev[0]["conv_state"].clone()
    rng = np.random.default_rng(5)
    accs = [torch.tensor(rng.integers(1, T + 1, N), dtype=torch.int32, device="cuda") for _ in range(steps)]
    shape = kda.shape_of(dev[0]["mixed_qkv"], dev[0]["a"], S)
    ws = kda.alloc_workspace(shape, "cuda")
    outs = [{k: v.cuda() for k, v in wk.empty_outputs(wk.custom(N, T, H, HV, 128, 128)).items()}
            for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        x, o = dev[i], outs[i]
        kda.conv_verify(x["mixed_qkv"], x["conv_w"], cs, x["A_log"], x["dt_bias"], x["a"], x["b"], S,
                        "softplus", o["o"], o["inter_ssm"], o["conv_snapshots"], ws, shape=shape, plan=plan,
                        validate=False)
        kda.commit(accs[i], o["inter_ssm"], o["conv_snapshots"], S, cs, shape=shape, validate=False)
    torch.cuda.synchronize()
    for i in range(steps):
        inp = dict(cpu[i])
        if i > 0:  # the state the previous commit left: the previous verify's accepted snapshot
            a = accs[i - 1].long().cpu()
            prev = outs[i - 1]
            inp["S0"] = prev["inter_ssm"].cpu()[torch.arange(N), a - 1].contiguous()
            inp["conv_state"] = prev["conv_snapshots"].cpu()[torch.arange(N), a - 1].contiguous()
        orc = oracle.verify(inp, "softplus")
        # the conv_state each verify rolled is overwritten by its commit, so the
        # rolled windows are checked through the snapshots (bit-exact) instead
        np.testing.assert_array_equal(outs[i]["conv_snapshots"].double().cpu().numpy(), orc["conv_snapshots"])
        got = {"o": outs[i]["o"], "inter_ssm": outs[i]["inter_ssm"],
               "conv_snapshots": outs[i]["conv_snapshots"]}
        assert_parity(got, torch.from_numpy(orc["conv_state"]), orc)
    a = accs[-1].long().cpu()
    assert torch.equal(S.cpu(), outs[-1]["inter_ssm"].cpu()[torch.arange(N), a - 1])
    assert torch.equal(cs.cpu(), outs[-1]["conv_snapshots"].cpu()[torch.arange(N), a - 1])
