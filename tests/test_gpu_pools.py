"""GPU parity of the state-pool entry points (kda_conv_verify_indexed,
kda_commit_indexed): slots of the S0, conv_state and snapshot pools are
given per sequence, negative slots are padding.  The indexed call must equal,
bit for bit, the dense call on the gathered inputs, touch no other slot, and
match the CPU oracle."""
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


def _pools(wl, seed, pad=(2, 5), extra=(5, 3, 4)):
    """Dense inputs plus pools holding them at shuffled slots (padding rows
    get slot -1) and sentinel-filled output pools."""
    g = torch.Generator().manual_seed(seed)
    s = wl.shape
    inp = wk.make_inputs(wl)
    PS, PC, PI = s.N + extra[0], s.N + extra[1], s.N + extra[2]
    slot_s = torch.randperm(PS, generator=g)[:s.N].to(torch.int32)
    slot_c = torch.randperm(PC, generator=g)[:s.N].to(torch.int32)
    slot_i = torch.randperm(PI, generator=g)[:s.N].to(torch.int32)
    for n in pad:
        slot_s[n] = -1
    S_pool = torch.randn((PS, s.HV, s.K, s.V), generator=g)
    cs_pool = torch.randn((PC, s.dim, 3), generator=g).to(s.torch_act)
    live = [n for n in range(s.N) if n not in pad]
    for n in live:
        S_pool[slot_s[n]] = inp["S0"][n]
        cs_pool[slot_c[n]] = inp["conv_state"][n]
    return inp, live, dict(slot_s=slot_s, slot_c=slot_c, slot_i=slot_i, S_pool=S_pool,
                           cs_pool=cs_pool, PS=PS, PC=PC, PI=PI)


def _run_indexed(kda, wl, inp, pl, plan=None):
    s = wl.shape
    dev = to_device(inp)
    shape = kda.shape_of(dev["mixed_qkv"], dev["a"], dev["S0"])
    slot = {k: pl[k].cuda() for k in ("slot_s", "slot_c", "slot_i")}
    idx = kda.state_indices(slot["slot_s"], slot["slot_c"], slot["slot_i"], pl["PS"], pl["PC"], pl["PI"])
    S_pool = pl["S_pool"].cuda()
    cs_pool = pl["cs_pool"].cuda()
    o = torch.full((s.N, s.T, s.HV, s.V), 5.0, dtype=s.torch_act, device="cuda")
    inter = torch.full((pl["PI"], s.T, s.HV, s.K, s.V), 9.0, device="cuda")
    snaps = torch.full((pl["PI"], s.T, s.dim, 3), 7.0, dtype=s.torch_act, device="cuda")
    ws = kda.alloc_workspace(shape, "cuda")
    kda.conv_verify_indexed(shape, idx, dev["mixed_qkv"], dev["conv_w"], cs_pool, dev["A_log"],
                            dev["dt_bias"], dev["a"], dev["b"], S_pool, wl.gate, o, inter, snaps, ws,
                            plan=plan)
    torch.cuda.synchronize()
    return dict(o=o, inter=inter, snaps=snaps, S_pool=S_pool, cs_pool=cs_pool, ws=ws, shape=shape,
                idx=idx, slot=slot)


@pytest.mark.parametrize("plan", [None, "item:128", "item:32", "pipe:64", "pipe:128:0:0:counter",
                                  "pipe:128:0:0:kernel", "split:32", "split:128",
                                  "item:128:0:0:kernel", "item:32:0:0:counter", "smem:64:0:0:kernel",
                                  "item:128:0:0:cluster", "item:64:0:0:cluster"])
def test_indexed_equals_dense_on_gathered_inputs(plan):
    from linear_attention_speculative_gb300 import kda
    wl = wk.custom(8, 3, 2, 4, 128, 128, seed=81)
    inp, live, pl = _pools(wl, seed=1)
    got = _run_indexed(kda, wl, inp, pl, plan)
    # dense call on the live sequences
    sub = {k: (v[live] if v is not None and k in ("mixed_qkv", "conv_state", "a", "b", "S0") else v)
           for k, v in inp.items()}
    dsub = to_device(sub)
    ref = kda.run(dsub, wl.gate)
    torch.cuda.synchronize()
    si = pl["slot_i"].long()
    for j, n in enumerate(live):
        assert torch.equal(got["o"][n], ref["o"][j])
        assert torch.equal(got["inter"][si[n]], ref["inter_ssm"][j])
        assert torch.equal(got["snaps"][si[n]], ref["conv_snapshots"][j])
        assert torch.equal(got["cs_pool"][pl["slot_c"][n].long()], dsub["conv_state"][j])
    # padding sequences and unused slots are untouched
    pad = [n for n in range(wl.shape.N) if n not in live]
    for n in pad:
        assert bool((got["o"][n] == 5.0).all())
    used_i = {int(si[n]) for n in live}
    for slot in range(pl["PI"]):
        if slot not in used_i:
            assert bool((got["inter"][slot] == 9.0).all()) and bool((got["snaps"][slot] == 7.0).all())
    used_c = {int(pl["slot_c"][n]) for n in live}
    for slot in range(pl["PC"]):
        if slot not in used_c:
            assert torch.equal(got["cs_pool"][slot].cpu(), pl["cs_pool"][slot])
    assert torch.equal(got["S_pool"].cpu(), pl["S_pool"])  # S0 pool is read only
    assert kda.read_status(got["shape"], got["ws"]) == 0


@pytest.mark.parametrize("plan", [None, "pipe:64", "split:64", "item:64:0:0:cluster"])
def test_indexed_matches_the_oracle(plan):
    from linear_attention_speculative_gb300 import kda
    wl = wk.custom(6, 4, 2, 2, 128, 128, gate="safe", seed=82)
    inp, live, pl = _pools(wl, seed=2, pad=(1,))
    got = _run_indexed(kda, wl, inp, pl, plan)
    ref = oracle.verify(inp, wl.gate, seqs=live, threads=4)
    si = pl["slot_i"].long()
    out = {"o": got["o"][live], "inter_ssm": got["inter"][si[live]],
           "conv_snapshots": got["snaps"][si[live]]}
    cs = got["cs_pool"][pl["slot_c"].long()[live]]
    assert_parity(out, cs, ref)


@pytest.mark.parametrize("plan", [None, "item:128:0:0:counter", "item:128:0:0:kernel", "pipe:128",
                                  "split:128", "item:128:0:0:cluster"])
def test_out_of_range_slot_skips_and_reports(plan):
    from linear_attention_speculative_gb300 import kda
    wl = wk.custom(4, 2, 2, 2, 128, 128, seed=83)  # two v-heads read each q/k head
    inp, live, pl = _pools(wl, seed=3, pad=())
    pl["slot_i"][2] = pl["PI"] + 7  # beyond the snapshot pool
    got = _run_indexed(kda, wl, inp, pl, plan)
    assert bool((got["o"][2] == 5.0).all())
    # the skipped sequence's conv_state slot is not rolled, by either q/k roll
    c2 = int(pl["slot_c"][2])
    assert torch.equal(got["cs_pool"][c2].cpu(), pl["cs_pool"][c2])
    assert kda.read_status(got["shape"], got["ws"]) == kda.STATUS_BAD_INDEX


def test_commit_indexed_rolls_back_into_pool_slots():
    from linear_attention_speculative_gb300 import kda
    wl = wk.custom(8, 4, 2, 4, 128, 64, seed=84)
    inp, live, pl = _pools(wl, seed=4)
    got = _run_indexed(kda, wl, inp, pl)
    acc = torch.tensor([1, 2, 3, 4, 4, 3, 2, 1], dtype=torch.int32, device="cuda")
    S_before = got["S_pool"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.commit_indexed(got["shape"], got["idx"], acc, got["inter"], got["snaps"], got["S_pool"],
                       got["cs_pool"], status=status)
    torch.cuda.synchronize()
    ss, sc, si = (pl[k].long() for k in ("slot_s", "slot_c", "slot_i"))
    for n in live:
        a = int(acc[n])
        assert torch.equal(got["S_pool"][ss[n]], got["inter"][si[n], a - 1])
        assert torch.equal(got["cs_pool"][sc[n]], got["snaps"][si[n], a - 1])
    untouched = [sl for sl in range(pl["PS"]) if sl not in {int(ss[n]) for n in live}]
    assert torch.equal(got["S_pool"][untouched], S_before[untouched])
    assert int(status.item()) == 0


def _random_pool_cases(seed=2028):
    # KDA_RANDOM_CASES sets how many (default 24); the first 24 are always the same
    import os
    n = int(os.environ.get("KDA_RANDOM_CASES", "24"))
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        K = int(rng.choice([32, 64, 128]))
        V = int(rng.choice([32, 64, 128]))
        H = int(rng.integers(1, 3))
        HV = H * int(rng.choice([1, 2, 4]))
        T = int(rng.integers(1, 7))
        N = int(rng.integers(2, 7))
        gate = str(rng.choice(["softplus", "safe"]))
        from parity_util import plan_built
        plans = [None] + [p for p in ("item:32", "item:64", "item:128", "smem:64", "smem:128", "pipe:64",
                                      "pipe:128", "split:32", "split:64", "split:128")
                          if plan_built(p, K, V, T=T, G=HV // H)]
        plan = plans[int(rng.integers(0, len(plans)))]
        n_pad = int(rng.integers(0, N))  # padding sequences among the N
        pad = tuple(sorted(rng.choice(N, size=n_pad, replace=False).tolist())) if n_pad else ()
        cases.append((N, T, H, HV, K, V, gate, plan, pad, 5000 + len(cases)))
    return cases


@pytest.mark.parametrize("case", _random_pool_cases(),
                         ids=lambda c: "N{}_T{}_H{}_HV{}_K{}_V{}_{}_{}_pad{}".format(*c[:7], c[7], len(c[8])))
def test_random_pools_match_the_oracle(case):
    # random shapes, plans and slot maps (shuffled slots, padding sequences):
    # the live sequences' outputs in their pool slots against the oracle
    from linear_attention_speculative_gb300 import kda
    N, T, H, HV, K, V, gate, plan, pad, seed = case
    wl = wk.custom(N, T, H, HV, K, V, gate=gate, seed=seed)
    inp, live, pl = _pools(wl, seed=seed, pad=pad)
    got = _run_indexed(kda, wl, inp, pl, plan)
    si = pl["slot_i"].long()
    if live:
        ref = oracle.verify(inp, wl.gate, seqs=live, threads=4)
        out = {"o": got["o"][live], "inter_ssm": got["inter"][si[live]],
               "conv_snapshots": got["snaps"][si[live]]}
        assert_parity(out, got["cs_pool"][pl["slot_c"].long()[live]], ref)
    for n in pad:
        assert bool((got["o"][n] == 5.0).all())
    assert torch.equal(got["S_pool"].cpu(), pl["S_pool"])  # the state pool is read only
    assert kda.read_status(got["shape"], got["ws"]) == 0
