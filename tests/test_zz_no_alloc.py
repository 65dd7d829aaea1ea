"""The allocation-free entry point, kda_conv_verify_noalloc.

It serves callers that cannot allocate device memory (a plugin handed only
its input and output buffers, a serving loop whose memory pool is fixed after
start-up, code that must not call cudaMalloc): its scratch is a fixed array
inside the library instead of a caller-supplied workspace.  These tests call
it through the C ABI and compare it with the regular entry point.  The file
is named to be collected last, so a run that stops at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from linear_attention_speculative_gb300 import _build
from linear_attention_speculative_gb300 import workloads as wk
from parity_util import TOL, max_rel_err, max_rel_err_rounded, to_device


def _lib():
    _build.build()
    from linear_attention_speculative_gb300 import kda
    return kda, kda.lib()


def _noalloc(L, kda, shape, inp, gate, out, conv_state, stream):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    gm = kda.GATE_SOFTPLUS if gate == "softplus" else kda.GATE_SAFE
    return L.kda_conv_verify_noalloc(
        ctypes.byref(shape), p(inp["mixed_qkv"]), p(inp["conv_w"]), p(conv_state),
        p(inp["A_log"]), p(inp["dt_bias"]), p(inp["a"]), p(inp["b"]), p(inp["S0"]), gm,
        p(out["o"]), p(out["inter_ssm"]), p(out["conv_snapshots"]),
        ctypes.c_void_p(stream.cuda_stream) if stream is not None else None)


def test_rejects_shapes_beyond_the_built_in_scratch():
    # N*H counters beyond the array: refused on the host before any CUDA call
    kda, L = _lib()
    s = kda.make_shape(70000, 1, 1, 1, 32, 32)
    assert kda.workspace_bytes(s) > kda.NOALLOC_MAX_SCRATCH_BYTES
    fake = {k: type("P", (), {"data_ptr": (lambda self, a=0x7f0000000000 + i * (1 << 30): a)})()
            for i, k in enumerate(("mixed_qkv", "conv_w", "A_log", "dt_bias", "a", "b", "S0"))}
    out = {k: type("P", (), {"data_ptr": (lambda self, a=0x7e0000000000 + i * (1 << 34): a)})()
           for i, k in enumerate(("o", "inter_ssm", "conv_snapshots"))}
    cs = type("P", (), {"data_ptr": lambda self: 0x7d0000000000})()
    assert _noalloc(L, kda, s, fake, "softplus", out, cs, None) == -10
    assert "scratch" in kda.strerror(-10)


def test_empty_batch_is_checked_like_the_regular_entry_point():
    # N == 0 launches nothing; the shape and gate mode are still checked, with
    # the same codes as kda_conv_verify (no CUDA call is made either way)
    kda, L = _lib()
    s = kda.make_shape(0, 2, 2, 2)
    none = {k: None for k in ("mixed_qkv", "conv_w", "A_log", "dt_bias", "a", "b", "S0",
                              "o", "inter_ssm", "conv_snapshots")}
    assert _noalloc(L, kda, s, none, "softplus", none, None, None) == 0
    gm_bad = kda.KdaShape(0, 2, 2, 2, 128, 128, 4, kda.BF16)
    rc = L.kda_conv_verify_noalloc(ctypes.byref(gm_bad), *([None] * 8), 7, None, None, None, None)
    assert rc == -7
    rc_regular = L.kda_conv_verify(ctypes.byref(gm_bad), *([None] * 8), 7, None, None, None, None, 0,
                                   None)
    assert rc == rc_regular
    bad_shape = kda.make_shape(0, 0, 2, 2)  # T = 0
    assert _noalloc(L, kda, bad_shape, none, "softplus", none, None, None) == -2


def test_status_reader_rejects_bad_arguments_on_the_host():
    kda, L = _lib()
    st = ctypes.c_int(0)
    assert L.kda_noalloc_read_status(None, ctypes.byref(st), None) == -1
    assert L.kda_noalloc_read_status(ctypes.byref(kda.make_shape(4, 1, 1, 1)), None, None) == -1
    assert L.kda_noalloc_read_status(ctypes.byref(kda.make_shape(70000, 1, 1, 1, 32, 32)),
                                     ctypes.byref(st), None) == -10


# Several v-heads per q/k head in each.  The first small launch rolls the
# shared q/k conv_state in a thread-block cluster of a group's items, the second
# (groups of 16 items, too many for one cluster) with the arrival counters kept
# in the scratch array; the large one uses the separate roll kernel.  The
# scratch always holds the status word.
NOALLOC_CASES = [wk.custom(8, 4, 2, 8, 128, 128, gate="safe", seed=901),
                 wk.custom(4, 4, 2, 16, 128, 128, seed=902), wk.GVA]


@pytest.mark.gpu
@pytest.mark.parametrize("wl", NOALLOC_CASES, ids=lambda w: w.name)
def test_noalloc_matches_the_regular_entry_point_on_two_calls_in_a_row(wl):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kda, L = _lib()
    inp = to_device(wk.make_inputs(wl))
    shape = kda.shape_of(inp["mixed_qkv"], inp["a"], inp["S0"])
    assert kda.workspace_bytes(shape) <= kda.NOALLOC_MAX_SCRATCH_BYTES
    cs0 = inp["conv_state"].clone()
    ref_cs = cs0.clone()
    ref = kda.run(dict(inp, conv_state=ref_cs), wl.gate)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    for call in range(2):
        cs = cs0.clone()
        out = {k: torch.full_like(v, float("nan")) if v.is_floating_point() else torch.empty_like(v)
               for k, v in ref.items()}
        rc = _noalloc(L, kda, shape, inp, wl.gate, out, cs, stream)
        assert rc == 0, kda.strerror(rc)
        # a clean call leaves no status bit (no bounded wait gave up)
        assert kda.noalloc_read_status(shape, stream) == 0, f"call {call}: device status"
        torch.cuda.synchronize()
        o = out["o"].double().cpu().numpy()
        y = ref["o"].double().cpu().numpy()
        assert max_rel_err_rounded(o, y, out["o"].dtype) <= TOL, f"call {call}: o"
        assert max_rel_err(out["inter_ssm"].cpu().numpy(), ref["inter_ssm"].cpu().numpy()) <= TOL
        assert torch.equal(out["conv_snapshots"], ref["conv_snapshots"]), f"call {call}"
        assert torch.equal(cs, ref_cs), f"call {call}: rolled conv_state"
