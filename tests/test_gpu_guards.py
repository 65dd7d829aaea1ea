"""Out-of-bounds write fences (GPU).

Every buffer a call writes (o, inter_ssm, conv_snapshots, conv_state, the
workspace, the decode state, the commit outputs) is placed inside a larger
allocation whose guard zones before and after it hold a sentinel pattern.
After the call the guards must be untouched: any write outside a buffer's
extent by any kernel, plan, pool mapping or shape shows up here.  This stands
in for a memory checker run.
"""
import pytest
import torch

from linear_attention_speculative_gb300 import workloads as wk
from parity_util import to_device

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side (keeps 16-byte alignment)
SENTINEL = 0x5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from linear_attention_speculative_gb300 import kda
    kda.lib()


class Fenced:
    """A tensor view with sentinel guard zones on both sides."""

    def __init__(self, shape, dtype, fill=None):
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self) -> bool:
        return bool((self.raw[:GUARD] == SENTINEL).all()) and bool((self.raw[-GUARD:] == SENTINEL).all())


def _verify_fenced(kda, wl, plan=None, pools=False):
    s = wl.shape
    inp = to_device(wk.make_inputs(wl))
    extra = 3 if pools else 0
    cs = Fenced((s.N + extra, s.dim, 3), s.torch_act)
    cs.t[: s.N].copy_(inp["conv_state"])
    o = Fenced((s.N, s.T, s.HV, s.V), s.torch_act)
    inter = Fenced((s.N + extra, s.T, s.HV, s.K, s.V), torch.float32)
    snaps = Fenced((s.N + extra, s.T, s.dim, 3), s.torch_act)
    shape = kda.shape_of(inp["mixed_qkv"], inp["a"], inp["S0"])
    ws = Fenced((kda.workspace_bytes(shape),), torch.uint8, fill=torch.zeros(kda.workspace_bytes(shape),
                                                                               dtype=torch.uint8))
    if pools:
        S_pool = torch.cat([inp["S0"], torch.zeros((extra, s.HV, s.K, s.V), device="cuda")])
        perm = torch.randperm(s.N + extra, generator=torch.Generator().manual_seed(5))[: s.N]
        slot = perm.to(torch.int32).cuda()
        idx = kda.state_indices(torch.arange(s.N, dtype=torch.int32, device="cuda"), slot, slot,
                                s.N + extra, s.N + extra, s.N + extra)
        kda.conv_verify_indexed(shape, idx, inp["mixed_qkv"], inp["conv_w"], cs.t, inp["A_log"],
                                inp["dt_bias"], inp["a"], inp["b"], S_pool, wl.gate, o.t, inter.t,
                                snaps.t, ws.t, plan=plan)
    else:
        kda.conv_verify(inp["mixed_qkv"], inp["conv_w"], cs.t, inp["A_log"], inp["dt_bias"],
                        inp["a"], inp["b"], inp["S0"], wl.gate, o.t, inter.t, snaps.t, ws.t,
                        shape=shape, plan=plan)
    torch.cuda.synchronize()
    return dict(cs=cs, o=o, inter=inter, snaps=snaps, ws=ws, shape=shape, inp=inp)


CASES = [
    (wk.custom(5, 3, 2, 4, 128, 128, seed=401), ("item:128", "item:16", "smem:128", "pipe:64",
                                                 "pipe:128:2", "split:32", "split:128", "item:128:0:0:kernel",
                                                 "smem:128:0:0:kernel", "item:64:0:0:counter",
                                                 "item:128:0:0:cluster", "item:64:0:0:cluster")),
    (wk.custom(3, 2, 1, 2, 256, 256, seed=402), ("smem:64", "smem:32", "item:64", "item:16",
                                                 "item:64:0:0:kernel", "item:64:0:0:cluster")),
    (wk.custom(4, 16, 2, 2, 32, 32, act="f32", seed=403), ("item:32", "item:16")),
    (wk.custom(4, 16, 2, 2, 32, 64, act="f32", seed=406), ("pipe:64", "pipe:64:1:0:counter")),
    (wk.custom(6, 1, 3, 6, 64, 128, gate="safe", seed=404), ("item:64", "smem:64", "pipe:64", "split:64",
                                                              "item:64:0:0:kernel")),
]


@pytest.mark.parametrize("wl,plans", CASES, ids=lambda c: c.name if hasattr(c, "name") else "")
def test_verify_writes_stay_inside_their_buffers(wl, plans):
    from linear_attention_speculative_gb300 import kda
    for plan in plans:
        for pools in (False, True):
            f = _verify_fenced(kda, wl, plan, pools)
            for name in ("cs", "o", "inter", "snaps", "ws"):
                assert f[name].intact(), (plan, pools, name)


def test_decode_and_commit_writes_stay_inside_their_buffers():
    from linear_attention_speculative_gb300 import kda
    wl = wk.custom(5, 3, 2, 4, 128, 128, seed=405)
    f = _verify_fenced(kda, wl)
    s = wl.shape
    # commit into fenced state / conv_state
    S = Fenced((s.N, s.HV, s.K, s.V), torch.float32)
    cs = Fenced((s.N, s.dim, 3), s.torch_act)
    acc = torch.tensor([1, 2, 3, 3, 1], dtype=torch.int32, device="cuda")
    kda.commit(acc, f["inter"].t, f["snaps"].t, S.t, cs.t)
    torch.cuda.synchronize()
    assert S.intact() and cs.intact()
    # decode with a fenced in/out state and outputs
    inp = f["inp"]
    for plan in ("item:128", "smem:128", "item:32"):
        Sd = Fenced((s.N, s.HV, s.K, s.V), torch.float32, fill=inp["S0"])
        csd = Fenced((s.N, s.dim, 3), s.torch_act, fill=wk.make_inputs(wl)["conv_state"].cuda())
        o = Fenced((s.N, s.T, s.HV, s.V), s.torch_act)
        ws = kda.alloc_workspace(f["shape"], "cuda")
        kda.conv_decode(inp["mixed_qkv"], inp["conv_w"], csd.t, inp["A_log"], inp["dt_bias"],
                        inp["a"], inp["b"], Sd.t, wl.gate, o.t, ws, plan=plan, shape=f["shape"])
        torch.cuda.synchronize()
        assert Sd.intact() and csd.intact() and o.intact(), plan
