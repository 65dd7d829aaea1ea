"""The Python entry points check every tensor against the shape the call
implies before any library call (CPU: the tensors below never reach a GPU)."""
import pytest
import torch

from linear_attention_speculative_gb300 import kda
from linear_attention_speculative_gb300 import workloads as wk


def _call(inp, out, **over):
    args = dict(inp, **{k: v for k, v in out.items()})
    args.update(over)
    shape = kda.make_shape(2, 3, 2, 4, 32, 32, "bf16")
    kda.conv_verify(args["mixed_qkv"], args["conv_w"], args["conv_state"], args["A_log"],
                    args["dt_bias"], args["a"], args["b"], args["S0"], "softplus", args["o"],
                    args["inter_ssm"], args["conv_snapshots"], torch.zeros(256, dtype=torch.uint8),
                    shape=shape)


def _tensors():
    wl = wk.custom(2, 3, 2, 4, 32, 32, seed=5)
    return wk.make_inputs(wl), wk.empty_outputs(wl)


def test_right_shapes_on_the_host_are_refused_as_host_tensors():
    inp, out = _tensors()
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        _call(inp, out)


@pytest.mark.parametrize("name,bad,msg", [
    ("o", lambda t: t[:, :2].contiguous(), "o must have shape"),
    ("inter_ssm", lambda t: t[:1].contiguous(), "inter_ssm must have shape"),
    ("conv_snapshots", lambda t: t.float(), "conv_snapshots must be torch.float32|conv_snapshots must be torch.bfloat16"),
    ("S0", lambda t: t.transpose(2, 3), "S0 must be contiguous"),
    ("conv_w", lambda t: t[:, :3].contiguous(), "conv_w must have shape"),
    ("a", lambda t: t.to(torch.float32), "a must be torch.bfloat16"),
    ("A_log", lambda t: None, "A_log is required"),
])
def test_wrong_tensors_are_named(name, bad, msg):
    inp, out = _tensors()
    src = inp if name in inp else out
    with pytest.raises(ValueError, match=msg):
        _call(inp, out, **{name: bad(src[name])})


def test_commit_checks_accepted_and_pools():
    wl = wk.custom(2, 3, 2, 4, 32, 32, seed=6)
    out = wk.empty_outputs(wl)
    S = torch.empty(2, 4, 32, 32)
    cs = torch.empty(2, 2 * 2 * 32 + 4 * 32, 3, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="accepted must be torch.int32"):
        kda.commit(torch.ones(2, dtype=torch.int64), out["inter_ssm"], out["conv_snapshots"], S, cs)
    with pytest.raises(ValueError, match="S must have shape"):
        kda.commit(torch.ones(2, dtype=torch.int32), out["inter_ssm"], out["conv_snapshots"], S[:1], cs)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        kda.commit(torch.ones(2, dtype=torch.int32), out["inter_ssm"], out["conv_snapshots"], S, cs)
