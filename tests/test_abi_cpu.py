"""The C ABI on the host: the library loads, exports every declared symbol,
rejects bad arguments before touching the GPU, and plans launches.

No test here launches a kernel: argument checks run before any CUDA call, and
the pointers below are fake addresses that are never dereferenced."""

import ctypes
import os
import re

import pytest

from linear_attention_speculative_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda_verify.h")


@pytest.fixture(scope="module")
def kda():
    _build.build()
    from linear_attention_speculative_gb300 import kda as mod
    mod.lib()
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(kda_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("kda_conv_verify", "kda_workspace_bytes", "kda_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(kda):
    L = ctypes.CDLL(_build.LIB_PATH)
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in kda_verify.h but not exported"
    assert set(kda.EXPORTED) <= set(declared_functions())


def test_version_and_strerror(kda):
    assert kda.lib().kda_version() == 0x000100
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -1234):
        assert isinstance(kda.strerror(code), str) and kda.strerror(code)


def test_workspace_bytes(kda):
    s = kda.make_shape(256, 4, 32, 32)
    ws = kda.workspace_bytes(s)
    assert ws % 256 == 0 and ws >= (256 * 32 + 1) * 4
    assert kda.lib().kda_workspace_bytes(None) == 0


# ---- the dispatcher (host logic only) --------------------------------------

def test_plan_auto_uses_one_item_per_cta(kda):
    # whole states per 8-warp CTA, one item per CTA
    p = kda.make_plan(kda.make_shape(256, 4, 32, 32), 152)
    assert p.variant == kda.VARIANT_ONE_ITEM
    assert p.bv == 128 and p.warps == 8 and p.items == 256 * 32 and p.grid == p.items
    # single-token calls, one v-head per q/k head, from 8 units per SM: state
    # kept in shared memory (3 CTAs per SM)
    p2 = kda.make_plan(kda.make_shape(512, 1, 32, 32), 152)
    assert p2.variant == kda.VARIANT_ONE_ITEM_SMEM and p2.bv == 128 and p2.items == 512 * 32
    assert p2.ctas_per_sm == 3
    assert kda.plan_label(kda.make_plan(kda.make_shape(76, 1, 16, 16), 152)) == "smem:128"  # 8 per SM
    assert kda.plan_label(kda.make_plan(kda.make_shape(75, 1, 16, 16), 152)) == "item:128"
    for shape in ((512, 2, 32, 32), (512, 3, 16, 16), (8, 1, 16, 16), (32, 1, 16, 16), (128, 3, 16, 16),
                  (16, 4, 16, 16), (512, 4, 32, 64), (512, 3, 32, 64), (3, 4, 16, 32)):
        assert kda.plan_label(kda.make_plan(kda.make_shape(*shape), 152)) == "item:128", shape
    # several v-heads per q/k head: 64-column items up to T = 2 and at most
    # half a unit per SM
    for shape in ((512, 1, 32, 64), (512, 2, 32, 64), (32, 2, 16, 32), (8, 1, 16, 32), (1, 4, 16, 32),
                  (2, 4, 16, 32), (1, 8, 32, 64)):
        p = kda.make_plan(kda.make_shape(*shape), 152)
        assert kda.plan_label(p) == "item:64" and p.warps == 4, shape
    # K = 256 and V = 64: the widest one-item tile (64 columns)
    assert kda.plan_label(kda.make_plan(kda.make_shape(1, 4, 1, 2, K=256, V=256), 152)) == "item:64"
    assert kda.plan_label(kda.make_plan(kda.make_shape(512, 1, 8, 16, K=256, V=256), 152)) == "item:64"
    assert kda.plan_label(kda.make_plan(kda.make_shape(1, 4, 1, 2, K=64, V=64), 152)) == "item:64"
    # L2 prefetch 3/8 of a wave of resident CTAs ahead; plans may set or disable it
    p4 = kda.make_plan(kda.make_shape(256, 4, 32, 32), 152)
    assert p4.prefetch == 152 * p4.ctas_per_sm * 3 // 8 > 0
    assert kda.resolve_plan(kda.make_shape(256, 4, 32, 32), 152, "item:128:0:40").prefetch == 40
    assert kda.resolve_plan(kda.make_shape(256, 4, 32, 32), 152, "item:128:0:-1").prefetch == 0


def test_decode_plan(kda):
    # kda_conv_decode's dispatcher: the shared-memory state for single tokens
    # from 8 units per SM; with several v-heads per q/k head 64-column items
    # for one or two tokens; else 128 columns
    def label(*shape, variant="auto", **dims):
        return kda.plan_label(kda.make_plan(kda.make_shape(*shape, **dims), 152, variant, decode=True))
    assert label(512, 1, 32, 64) == "smem:128" and label(76, 1, 16, 16) == "smem:128"
    assert label(75, 1, 16, 16) == "item:128" and label(8, 1, 16, 16) == "item:128"
    assert label(152, 2, 16, 16) == "item:128" and label(512, 2, 16, 16) == "item:128"
    assert label(38, 2, 16, 32) == "item:64" and label(37, 2, 16, 32) == "item:64"
    assert label(32, 1, 16, 32) == "item:64" and label(8, 2, 16, 32) == "item:64"
    assert label(8, 3, 16, 32) == "item:128" and label(512, 2, 32, 64) == "item:64"
    assert label(1, 2, 16, 32) == "item:64" and label(1, 3, 32, 64) == "item:128"
    assert label(1, 4, 16, 32) == "item:128" and label(1, 8, 32, 64) == "item:128"
    for T in (3, 4):
        assert label(512, T, 32, 64) == "item:128"
    assert label(64, 1, 8, 16, K=256, V=256) == "item:64"  # fewer than 8 units per SM
    # the other head dims: the shared-memory state for single tokens from 8
    # units per SM where it is built (not at K = V = 32)
    assert label(128, 1, 16, 16, K=256, V=256) == "smem:64"
    assert label(512, 1, 16, 32, K=64, V=64) == "smem:64"
    assert label(512, 1, 16, 32, K=32, V=32) == "item:32"
    assert label(512, 2, 16, 32, K=64, V=64) == "item:64"
    assert label(8, 1, 16, 16, variant="one_item_smem") == "smem:128"
    for bad in ("pipelined", "split"):
        with pytest.raises(kda.KdaError) as e:
            kda.make_plan(kda.make_shape(8, 1, 16, 16), 152, bad, decode=True)
        assert e.value.code == -8


def test_plan_picks_the_qk_roll(kda):
    # one reader per q/k group: rolled inside the verify kernel, one launch
    p = kda.make_plan(kda.make_shape(256, 4, 32, 32), 152)
    assert p.qk_roll == kda.QK_ROLL_COUNTER and p.launches == 1
    # four readers (two v-heads x two 64-column tiles), many waves: the
    # separate roll kernel
    p = kda.make_plan(kda.make_shape(512, 1, 32, 64), 152)
    assert kda.plan_label(p) == "item:64"
    assert p.qk_roll == kda.QK_ROLL_KERNEL and p.launches == 2
    # four readers (two v-heads x two 64-column tiles), a fraction of a wave:
    # one cluster per group, one launch
    p = kda.make_plan(kda.make_shape(2, 1, 16, 32), 152)
    assert kda.plan_label(p) == "item:64"
    assert p.qk_roll == kda.QK_ROLL_CLUSTER and p.launches == 1
    # the same below 4 waves for the plain decode; a group of more than 8
    # items (G = 16) cannot be one portable cluster: the counter
    p = kda.make_plan(kda.make_shape(8, 1, 8, 32), 152, decode=True)  # 4 v-heads x 2 tiles
    assert kda.plan_label(p) == "item:64" and p.qk_roll == kda.QK_ROLL_CLUSTER
    p = kda.make_plan(kda.make_shape(8, 1, 4, 32), 152, decode=True)  # 8 v-heads x 2 tiles
    assert p.qk_roll == kda.QK_ROLL_COUNTER
    p = kda.make_plan(kda.make_shape(2, 4, 2, 32), 152)
    assert p.qk_roll == kda.QK_ROLL_COUNTER and p.launches == 1
    # the pipelined variant: the same choice by items per resident CTA
    p = kda.make_plan(kda.make_shape(512, 4, 32, 64), 152, "pipelined")
    assert p.qk_roll == kda.QK_ROLL_KERNEL and p.launches == 2
    p = kda.make_plan(kda.make_shape(2, 4, 16, 32), 152, "pipelined")
    assert p.qk_roll == kda.QK_ROLL_COUNTER and p.launches == 1


def test_resolve_plan_fills_derived_fields(kda):
    s = kda.make_shape(512, 1, 32, 64)
    p = kda.resolve_plan(s, 152, "smem:128:0:0:counter")
    assert p.qk_roll == kda.QK_ROLL_COUNTER and p.launches == 1 and p.ctas_per_sm == 3
    p = kda.resolve_plan(s, 152, "item:64")
    assert p.qk_roll == kda.QK_ROLL_KERNEL and p.launches == 2 and p.items == 512 * 64 * 2
    with pytest.raises(kda.KdaError):
        kda.resolve_plan(s, 152, "pipe:64", decode=True)


def test_cluster_roll_plans(kda):
    # the items of a q/k group as one cluster: one launch, one-item kernels only,
    # at most 8 items per group
    s = kda.make_shape(64, 4, 8, 32)  # G = 4
    p = kda.resolve_plan(s, 152, "item:128:0:0:cluster")
    assert p.qk_roll == kda.QK_ROLL_CLUSTER and p.launches == 1 and p.grid == 64 * 32
    p = kda.resolve_plan(s, 152, "item:64:0:0:cluster")  # 4 v-heads x 2 tiles = 8
    assert p.qk_roll == kda.QK_ROLL_CLUSTER and p.launches == 1
    p = kda.resolve_plan(s, 152, "item:128:0:0:cluster", decode=True)
    assert p.qk_roll == kda.QK_ROLL_CLUSTER and p.launches == 1
    # built for the register-state kernel at 4 or 8 warps, groups of <= 8 items
    for bad in ("item:32:0:0:cluster",   # 2 warps (and 16 items per group)
                "smem:128:0:0:cluster", "pipe:128:0:0:cluster", "split:128:0:0:cluster"):
        with pytest.raises(kda.KdaError):
            kda.resolve_plan(s, 152, bad)
    s2 = kda.make_shape(4, 2, 2, 4, K=256, V=256)  # 4 warps = 32 columns at K = 256
    assert kda.resolve_plan(s2, 152, "item:64:0:0:cluster").qk_roll == kda.QK_ROLL_CLUSTER  # 2 x 4
    with pytest.raises(kda.KdaError):
        kda.resolve_plan(s2, 152, "item:32:0:0:cluster")  # 2 x 8 items
    # one item per group: nothing is shared, the request is moot
    p = kda.resolve_plan(kda.make_shape(4, 4, 8, 8), 152, "item:128:0:0:cluster")
    assert p.qk_roll == kda.QK_ROLL_COUNTER and p.launches == 1
    # the grid is a whole number of clusters
    for N, H, HV, bv in ((3, 2, 6, 64), (5, 1, 4, 128), (1, 3, 3, 64), (7, 2, 8, 128)):
        p = kda.resolve_plan(kda.make_shape(N, 2, H, HV), 152, f"item:{bv}:0:0:cluster")
        assert p.grid % ((HV // H) * (128 // bv)) == 0


def test_plan_strings_carry_the_qk_roll(kda):
    assert kda.parse_plan("item:64").qk_roll == kda.QK_ROLL_AUTO
    assert kda.parse_plan("item:64:0:0:kernel").qk_roll == kda.QK_ROLL_KERNEL
    assert kda.parse_plan("item:64:0:0:cluster").qk_roll == kda.QK_ROLL_CLUSTER
    assert kda.parse_plan("smem:128:0:-1:counter").qk_roll == kda.QK_ROLL_COUNTER
    with pytest.raises(KeyError):
        kda.parse_plan("item:64:0:0:sometimes")
    # fewer units than SMs at K = 256 (no pipelined kernel): whole states per CTA
    p1 = kda.make_plan(kda.make_shape(1, 4, 16, 16, K=256, V=256), 152)
    assert p1.variant == kda.VARIANT_ONE_ITEM and p1.bv == 64 and p1.warps == 8
    assert p1.items == 64 and p1.grid == 64


def test_plan_split_variant(kda):
    # two launches (prep kernel + recurrence kernel), one item per CTA, the
    # recurrence kernel with the one-item kernel's resources
    s = kda.make_shape(64, 4, 8, 32)
    p = kda.resolve_plan(s, 152, "split:128")
    assert p.variant == kda.VARIANT_SPLIT and p.launches == 2 and p.qk_roll == 0
    assert p.items == 64 * 32 and p.grid == p.items and p.ctas_per_sm == 2 and p.warps == 8
    p32 = kda.resolve_plan(s, 152, "split:32")
    assert p32.items == 64 * 32 * 4 and p32.warps == 2 and p32.ctas_per_sm == 8
    assert kda.plan_label(kda.make_plan(s, 152, "split")) == "split:128"
    # the stage must fit the item's slice of the last snapshot: at K = 128 a
    # 32-column item holds up to T = 7
    assert kda.resolve_plan(kda.make_shape(4, 7, 2, 2), 152, "split:32").launches == 2
    for bad, shape in (("split:32", (4, 8, 2, 2)), ("split:16", (4, 2, 2, 2)),
                       ("split:64", (4, 2, 2, 2, 256, 256))):
        with pytest.raises(kda.KdaError) as e:
            kda.resolve_plan(kda.make_shape(*shape), 152, bad)
        assert e.value.code == -8, bad
    with pytest.raises(kda.KdaError):  # no plain-decode form
        kda.resolve_plan(s, 152, "split:128", decode=True)
    # the dispatcher no longer picks it: the one-item kernels measured faster
    for shape in ((8, 1, 16, 32), (8, 1, 32, 64), (32, 1, 16, 32)):
        assert kda.make_plan(kda.make_shape(*shape), 152).variant == kda.VARIANT_ONE_ITEM


def test_plan_small_batches_use_one_item_kernels(kda):
    # small batches run one item per CTA too (the pipelined kernel, whose
    # producer warps stage inputs by bulk copies, measured slower at every
    # point of the sweep); it stays available by name.  At most half a unit
    # per SM: 64-column tiles, whatever the head layout (the plain decode
    # keeps 128 columns from three tokens on)
    for T in (1, 2, 4, 8):
        assert kda.plan_label(kda.make_plan(kda.make_shape(1, T, 16, 16), 152)) == "item:64"
        assert kda.plan_label(kda.make_plan(kda.make_shape(1, T, 16, 16), 152, "pipelined")) == "pipe:128"
    assert kda.plan_label(kda.make_plan(kda.make_shape(1, 4, 16, 16), 152, decode=True)) == "item:128"
    assert kda.plan_label(kda.make_plan(kda.make_shape(2, 4, 32, 32), 152)) == "item:64"
    assert kda.plan_label(kda.make_plan(kda.make_shape(3, 4, 32, 32), 152)) == "item:128"
    assert kda.plan_label(kda.make_plan(kda.make_shape(8, 4, 16, 16), 152)) == "item:128"
    assert kda.plan_label(kda.make_plan(kda.make_shape(1, 4, 16, 32), 152)) == "item:64"


def test_plan_pipelined_is_persistent(kda):
    p = kda.make_plan(kda.make_shape(256, 4, 32, 32), 152, "pipelined")
    assert p.variant == kda.VARIANT_PIPELINED and kda.plan_label(p) == "pipe:128"
    assert p.bv == 128 and p.warps == 8 and p.items == 256 * 32
    assert p.ctas_per_sm == 1 and p.grid == 152 and p.prefetch == 0  # inputs requested one item ahead
    p64 = kda.resolve_plan(kda.make_shape(256, 4, 32, 32), 152, "pipe:64")
    assert p64.warps == 4 and p64.ctas_per_sm == 2 and p64.grid == 304
    tiny = kda.make_plan(kda.make_shape(1, 2, 1, 1), 152, "pipelined")
    assert tiny.grid == tiny.items == 1  # never more CTAs than items


def test_plan_small_heads(kda):
    s = kda.make_shape(8, 2, 2, 4, K=64, V=32)
    with pytest.raises(kda.KdaError) as e:  # the pipelined kernel needs V >= 64
        kda.make_plan(s, 152, "pipelined")
    assert e.value.code == -8
    small = kda.make_plan(s, 152, "one_item")
    assert small.variant == kda.VARIANT_ONE_ITEM and small.bv in (16, 32)
    p = kda.make_plan(kda.make_shape(8, 2, 2, 4, K=64, V=64), 152, "pipelined")
    assert p.variant == kda.VARIANT_PIPELINED and p.bv == 64 and p.warps == 4


@pytest.mark.parametrize("bad", [dict(T=0), dict(T=17), dict(W=3), dict(K=96), dict(V=512),
                                 dict(H=3, HV=4), dict(HV=1, H=2)])
def test_plan_rejects_bad_shapes(kda, bad):
    args = dict(N=2, T=2, H=2, HV=2, K=32, V=32, W=4)
    args.update(bad)
    s = kda.KdaShape(args["N"], args["T"], args["H"], args["HV"], args["K"], args["V"],
                     args["W"], kda.BF16)
    with pytest.raises(kda.KdaError) as e:
        kda.make_plan(s, 152)
    assert e.value.code == -2


# ---- argument validation with fake (never dereferenced) pointers -----------

def _fake_args(kda, **over):
    base = 0x7f0000000000
    names = ["mixed_qkv", "conv_w", "conv_state", "A_log", "dt_bias", "a", "b", "S0", "o",
             "inter_ssm", "conv_snapshots", "workspace"]
    ptrs = {n: base + i * (1 << 24) for i, n in enumerate(names)}
    ptrs.update(over)
    return ptrs


def _call_plan(kda, shape, ptrs, plan, gate=0, ws_bytes=1 << 20):
    L = kda.lib()
    v = lambda n: ctypes.c_void_p(ptrs[n]) if ptrs[n] is not None else None
    return L.kda_conv_verify_plan(
        ctypes.byref(shape), v("mixed_qkv"), v("conv_w"), v("conv_state"), v("A_log"),
        v("dt_bias"), v("a"), v("b"), v("S0"), gate, v("o"), v("inter_ssm"),
        v("conv_snapshots"), v("workspace"), ws_bytes, ctypes.byref(plan), None)


def test_rejects_invalid_plans(kda):
    s = kda.make_shape(2, 2, 2, 2, 32, 64)
    for spec in ("item:8", "item:128", "item:48", "pipe:16", "pipe:32", "pipe:128"):
        assert _call_plan(kda, s, _fake_args(kda), kda.parse_plan(spec)) == -8, spec
    bad = kda.KdaPlan()
    bad.variant, bad.bv = 0, 32  # AUTO is not a concrete plan
    assert _call_plan(kda, s, _fake_args(kda), bad) == -8
    # a NULL plan is rejected before anything else is looked at
    args = [ctypes.byref(s)] + [None] * 8 + [0] + [None] * 4 + [0]
    assert kda.lib().kda_conv_verify_plan(*args, None, None) == -1


def _call(kda, shape, ptrs, gate=0, ws_bytes=1 << 20, variant=0):
    L = kda.lib()
    v = lambda n: ctypes.c_void_p(ptrs[n]) if ptrs[n] is not None else None
    return L.kda_conv_verify_variant(
        ctypes.byref(shape), v("mixed_qkv"), v("conv_w"), v("conv_state"), v("A_log"),
        v("dt_bias"), v("a"), v("b"), v("S0"), gate, v("o"), v("inter_ssm"),
        v("conv_snapshots"), v("workspace"), ws_bytes, variant, None)


def test_rejects_null_pointers(kda):
    s = kda.make_shape(2, 2, 2, 2, 32, 32)
    for name in ("mixed_qkv", "conv_w", "conv_state", "a", "b", "S0", "o", "inter_ssm",
                 "conv_snapshots"):
        assert _call(kda, s, _fake_args(kda, **{name: None})) == -1, name
    assert _call(kda, s, _fake_args(kda, workspace=None)) == -6
    # softplus needs A_log and dt_bias; the safe gate does not
    assert _call(kda, s, _fake_args(kda, A_log=None)) == -7
    assert _call(kda, s, _fake_args(kda, A_log=None, dt_bias=None), gate=1) not in (-1, -7)


def test_rejects_misaligned_pointers(kda):
    s = kda.make_shape(2, 2, 2, 2, 32, 32)
    for name in ("mixed_qkv", "S0", "inter_ssm", "conv_state", "o", "a"):
        ptrs = _fake_args(kda)
        ptrs[name] += 8
        assert _call(kda, s, ptrs) == -4, name


def test_rejects_aliasing(kda):
    s = kda.make_shape(2, 2, 2, 2, 32, 32)
    ptrs = _fake_args(kda)
    ptrs["inter_ssm"] = ptrs["S0"] + 4096  # output inside an input
    assert _call(kda, s, ptrs) == -5
    ptrs = _fake_args(kda)
    ptrs["o"] = ptrs["conv_snapshots"]     # two outputs on one buffer
    assert _call(kda, s, ptrs) == -5
    ptrs = _fake_args(kda)
    ptrs["conv_state"] = ptrs["mixed_qkv"] + 64  # in-place buffer inside an input
    assert _call(kda, s, ptrs) == -5


def test_rejects_small_workspace_bad_gate_and_variant(kda):
    s = kda.make_shape(64, 2, 8, 8, 32, 32)
    assert _call(kda, s, _fake_args(kda), ws_bytes=16) == -6
    assert _call(kda, s, _fake_args(kda), gate=7) == -7
    assert _call(kda, s, _fake_args(kda), variant=9) == -8


def test_empty_batch_is_a_noop(kda):
    s = kda.make_shape(0, 2, 2, 2, 32, 32)
    nulls = {n: None for n in _fake_args(kda)}
    assert _call(kda, s, nulls) == 0


def test_valid_arguments_reach_the_device_query(kda):
    # Everything valid: on a machine without a GPU the call stops at the first
    # CUDA query and reports its error (a positive cudaError_t), no crash.
    s = kda.make_shape(2, 2, 2, 2, 32, 32)
    rc = _call(kda, s, _fake_args(kda))
    import torch
    if not torch.cuda.is_available():
        assert rc > 0


# ---- kda_commit argument checks (fake pointers, nothing launched) -----------

def _commit(kda, shape, acc=0x7f0000000000, inter=0x7f0100000000, snaps=0x7f0200000000,
            S=0x7f0300000000, cs=0x7f0400000000, status=None):
    L = kda.lib()
    v = lambda x: ctypes.c_void_p(x) if x is not None else None
    return L.kda_commit(ctypes.byref(shape), v(acc), v(inter), v(snaps), v(S), v(cs), v(status), None)


def test_commit_rejects_bad_arguments(kda):
    s = kda.make_shape(4, 3, 2, 2, 32, 32)
    assert _commit(kda, s, acc=None) == -1
    assert _commit(kda, s, S=None) == -1
    assert _commit(kda, s, inter=0x7f0100000008) == -4
    assert _commit(kda, s, acc=0x7f0000000002) == -4
    assert _commit(kda, s, S=0x7f0100000000 + 4096) == -5   # state out inside inter_ssm
    assert _commit(kda, s, cs=0x7f0300000000 + 16) == -5     # two outputs overlap
    assert _commit(kda, kda.make_shape(4, 0, 2, 2, 32, 32)) == -2
    assert _commit(kda, kda.make_shape(0, 3, 2, 2, 32, 32), acc=None, S=None) == 0


# ---- state-pool indirection argument checks --------------------------------

def _call_indexed(kda, shape, ptrs, idx, ws_bytes=1 << 20):
    L = kda.lib()
    v = lambda n: ctypes.c_void_p(ptrs[n]) if ptrs[n] is not None else None
    return L.kda_conv_verify_indexed(
        ctypes.byref(shape), ctypes.byref(idx), v("mixed_qkv"), v("conv_w"), v("conv_state"),
        v("A_log"), v("dt_bias"), v("a"), v("b"), v("S0"), 0, v("o"), v("inter_ssm"),
        v("conv_snapshots"), v("workspace"), ws_bytes, None, None)


def test_indexed_rejects_bad_pools(kda):
    s = kda.make_shape(4, 2, 2, 2, 32, 32)
    ptrs = _fake_args(kda)
    good_idx = 0x7e0000000000
    # an index array with an empty pool
    assert _call_indexed(kda, s, ptrs, kda.KdaStateIndices(good_idx, None, None, 0, 0, 0)) == -2
    # misaligned index array
    assert _call_indexed(kda, s, ptrs, kda.KdaStateIndices(good_idx + 2, None, None, 8, 0, 0)) == -4
    # an index array inside an output buffer
    inside = ptrs["inter_ssm"] + 64
    assert _call_indexed(kda, s, ptrs, kda.KdaStateIndices(None, None, inside, 0, 0, 8)) == -5
    # a pool larger than N makes the state buffers larger: S0 now overlaps the next buffer
    big = kda.KdaStateIndices(good_idx, None, None, 1 << 20, 0, 0)
    assert _call_indexed(kda, s, ptrs, big) == -5


def test_decode_rejects_bad_arguments(kda):
    L = kda.lib()
    s = kda.make_shape(4, 2, 2, 2, 32, 32)
    p = _fake_args(kda)
    v = lambda x: ctypes.c_void_p(x) if x is not None else None

    def call(S=p["S0"], o=p["o"], plan=None):
        return L.kda_conv_decode(ctypes.byref(s), None, v(p["mixed_qkv"]), v(p["conv_w"]),
                                 v(p["conv_state"]), v(p["A_log"]), v(p["dt_bias"]), v(p["a"]),
                                 v(p["b"]), v(S), 0, v(o), v(p["workspace"]), 1 << 20,
                                 ctypes.byref(plan) if plan is not None else None, None)
    assert call(S=None) == -1
    assert call(o=p["S0"] + 64) == -5                 # output inside the in/out state
    assert call(plan=kda.parse_plan("pipe:64")) == -8
    assert call(plan=kda.parse_plan("item:64")) == -8  # wider than V = 32


def test_plan_head_dim_256_layout(kda):
    # K = 256: 16 row groups x 2 column quads per warp, 8 columns per warp, so an
    # 8-warp tile is 64 columns wide
    p = kda.make_plan(kda.make_shape(64, 4, 8, 16, K=256, V=256), 152)
    assert p.variant == kda.VARIANT_ONE_ITEM and p.bv == 64 and p.warps == 8
    assert p.items == 64 * 16 * 4
    p1 = kda.make_plan(kda.make_shape(512, 1, 8, 16, K=256, V=256), 152)
    assert p1.variant == kda.VARIANT_ONE_ITEM and p1.bv == 64 and p1.warps == 8
    q = kda.make_plan(kda.make_shape(64, 4, 8, 16, K=128, V=256), 152)
    assert q.variant == kda.VARIANT_ONE_ITEM and q.bv == 128 and q.items == 64 * 16 * 2
    with pytest.raises(kda.KdaError) as e:
        kda.make_plan(kda.make_shape(4, 2, 1, 1, K=256, V=128), 152, "pipelined")
    assert e.value.code == -8
    s = kda.make_shape(2, 2, 1, 1, K=256, V=128)
    assert kda.resolve_plan(s, 152, "item:32").warps == 4
    assert kda.resolve_plan(s, 152, "smem:32").warps == 4
    for bad in ("item:128", "smem:128", "item:8", "pipe:64"):  # 16 warps / 1 warp / pipelined: not built
        assert _call_plan(kda, s, _fake_args(kda), kda.parse_plan(bad)) == -8, bad


def test_selftest_rejects_bad_arguments_on_the_host(kda):
    # checked before any CUDA call (no GPU here)
    L = kda.lib()
    st = ctypes.c_void_p(0x7f0000000000)
    assert L.kda_selftest_bounded_wait(0, 1000, None, None) == -1
    assert L.kda_selftest_bounded_wait(4, 1000, st, None) == -2
    assert L.kda_selftest_bounded_wait(-1, 1000, st, None) == -2
    assert L.kda_selftest_bounded_wait(0, -1, st, None) == -2
    assert L.kda_selftest_bounded_wait(0, 3_000_000_000, st, None) == -2


def test_dispatcher_invariants_over_random_shapes(kda):
    # whatever the shape, the dispatcher's plans are well formed: the tile
    # width divides V and matches the warps, one item per (sequence, v-head,
    # tile), a grid that covers them, one or two launches, and the plan
    # resolves to itself; the decode dispatcher never picks a variant without
    # a decode form.  A cluster q/k roll groups the items of one q/k head:
    # at most 8 of them (a portable cluster), the register-state kernel at 4
    # or 8 warps, a grid of whole clusters, and clusters that never span two
    # sequences (a sequence's items are a whole number of groups), so a
    # padding sequence skips whole clusters and every cluster barrier ends
    import numpy as np
    rng = np.random.default_rng(77)
    wc = {32: 16, 64: 16, 128: 16, 256: 8}
    for _ in range(3000):
        K = int(rng.choice([32, 64, 128, 256]))
        V = int(rng.choice([32, 64, 128, 256]))
        H = int(rng.integers(1, 65))
        HV = H * int(rng.choice([1, 2, 3, 4, 8]))
        N = int(rng.integers(1, 2049))
        T = int(rng.integers(1, 17))
        act = str(rng.choice(["bf16", "f32"]))
        s = kda.make_shape(N, T, H, HV, K, V, act)
        for decode in (False, True):
            p = kda.make_plan(s, 152, decode=decode)
            assert V % p.bv == 0 and p.bv == p.warps * wc[K], (N, T, H, HV, K, V, decode)
            assert p.items == N * HV * (V // p.bv)
            assert 1 <= p.grid and (p.grid == p.items or p.variant == kda.VARIANT_PIPELINED)
            assert p.launches in (1, 2) and p.ctas_per_sm >= 1
            if decode:
                assert p.variant in (kda.VARIANT_ONE_ITEM, kda.VARIANT_ONE_ITEM_SMEM)
            label = kda.plan_label(p)
            q = kda.resolve_plan(s, 152, label, decode=decode)
            assert (q.variant, q.bv, q.warps, q.items, q.grid) == (p.variant, p.bv, p.warps, p.items, p.grid)
            group = (HV // H) * (V // p.bv)
            if p.qk_roll == kda.QK_ROLL_CLUSTER:
                assert 2 <= group <= 8 and p.variant == kda.VARIANT_ONE_ITEM and p.warps in (4, 8)
                assert p.grid % group == 0 and (HV * (V // p.bv)) % group == 0
                assert p.launches == 1
                # below 2 waves of resident CTAs only; the roll kernel from there
                assert p.items < 2 * 152 * p.ctas_per_sm
            elif group > 1 and p.variant != kda.VARIANT_SPLIT:
                assert p.qk_roll in (kda.QK_ROLL_COUNTER, kda.QK_ROLL_KERNEL)
