"""Thin ctypes binding of the C ABI in include/kda_verify.h.

Argument marshalling only: every step of the verify decode runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  If the
library is missing the import of this module fails loudly; there is no CPU
fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import torch

from . import _build

GATE_SOFTPLUS = 0
GATE_SAFE = 1
VARIANT_AUTO = 0
VARIANT_ONE_ITEM = 1
VARIANT_PIPELINED = 2
VARIANT_ONE_ITEM_SMEM = 3
VARIANT_SPLIT = 4
VARIANTS = {"auto": VARIANT_AUTO, "one_item": VARIANT_ONE_ITEM, "pipelined": VARIANT_PIPELINED,
            "one_item_smem": VARIANT_ONE_ITEM_SMEM, "split": VARIANT_SPLIT}
# plan-string prefix of each variant ("item:128", "pipe:128", "smem:128", "split:128")
PLAN_PREFIX = {VARIANT_ONE_ITEM: "item", VARIANT_PIPELINED: "pipe", VARIANT_ONE_ITEM_SMEM: "smem",
               VARIANT_SPLIT: "split"}
F32 = 0
BF16 = 1
MAX_T = 16

# The names declared in include/kda_verify.h.
EXPORTED = ("kda_conv_verify", "kda_conv_verify_variant", "kda_conv_verify_plan",
            "kda_conv_verify_indexed", "kda_conv_decode", "kda_commit", "kda_commit_indexed",
            "kda_conv_verify_noalloc", "kda_noalloc_read_status", "kda_workspace_bytes",
            "kda_make_plan", "kda_make_decode_plan", "kda_resolve_plan", "kda_read_status",
            "kda_selftest_bounded_wait", "kda_strerror", "kda_version")
NOALLOC_MAX_SCRATCH_BYTES = 256 * 1024


class KdaShape(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("HV", ctypes.c_int), ("K", ctypes.c_int), ("V", ctypes.c_int),
                ("W", ctypes.c_int), ("act", ctypes.c_int)]


class KdaPlan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("bv", ctypes.c_int), ("warps", ctypes.c_int),
                ("grid", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("items", ctypes.c_longlong), ("prefetch", ctypes.c_int), ("qk_roll", ctypes.c_int),
                ("launches", ctypes.c_int)]


class KdaStateIndices(ctypes.Structure):
    _fields_ = [("cache_indices", ctypes.c_void_p), ("conv_state_indices", ctypes.c_void_p),
                ("intermediate_state_indices", ctypes.c_void_p), ("state_pool", ctypes.c_int),
                ("conv_pool", ctypes.c_int), ("inter_pool", ctypes.c_int)]


def state_indices(cache=None, conv=None, inter=None, state_pool=0, conv_pool=0,
                  inter_pool=0) -> KdaStateIndices:
    """Pool slots (int32 device tensors [N] or None for the identity)."""
    ptr = lambda t: None if t is None else t.data_ptr()
    return KdaStateIndices(ptr(cache), ptr(conv), ptr(inter), state_pool, conv_pool, inter_pool)


class KdaError(RuntimeError):
    def __init__(self, code: int, what: str = "kda_conv_verify"):
        self.code = code
        super().__init__(f"{what} failed with code {code}: {strerror(code)}")


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not built ({path}); run __graft_entry__.build() "
                          "or python -m linear_attention_speculative_gb300._build")
    L = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    sp = ctypes.POINTER(KdaShape)
    args_common = [sp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp, vp, sz]
    L.kda_conv_verify.restype = ctypes.c_int
    L.kda_conv_verify.argtypes = args_common + [vp]
    L.kda_conv_verify_variant.restype = ctypes.c_int
    L.kda_conv_verify_variant.argtypes = args_common + [ctypes.c_int, vp]
    L.kda_conv_verify_plan.restype = ctypes.c_int
    L.kda_conv_verify_plan.argtypes = args_common + [ctypes.POINTER(KdaPlan), vp]
    L.kda_commit.restype = ctypes.c_int
    L.kda_commit.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp]
    ip = ctypes.POINTER(KdaStateIndices)
    L.kda_conv_verify_indexed.restype = ctypes.c_int
    L.kda_conv_verify_indexed.argtypes = ([sp, ip] + args_common[1:]
                                          + [ctypes.POINTER(KdaPlan), vp])
    L.kda_conv_decode.restype = ctypes.c_int
    L.kda_conv_decode.argtypes = [sp, ip, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, sz,
                                  ctypes.POINTER(KdaPlan), vp]
    L.kda_commit_indexed.restype = ctypes.c_int
    L.kda_commit_indexed.argtypes = [sp, ip, vp, vp, vp, vp, vp, vp, vp]
    L.kda_conv_verify_noalloc.restype = ctypes.c_int
    L.kda_conv_verify_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                          vp, vp, vp, vp]
    L.kda_noalloc_read_status.restype = ctypes.c_int
    L.kda_noalloc_read_status.argtypes = [sp, ctypes.POINTER(ctypes.c_int), vp]
    L.kda_workspace_bytes.restype = sz
    L.kda_workspace_bytes.argtypes = [sp]
    L.kda_make_plan.restype = ctypes.c_int
    L.kda_make_plan.argtypes = [sp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(KdaPlan)]
    L.kda_make_decode_plan.restype = ctypes.c_int
    L.kda_make_decode_plan.argtypes = [sp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(KdaPlan)]
    L.kda_resolve_plan.restype = ctypes.c_int
    L.kda_resolve_plan.argtypes = [sp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(KdaPlan)]
    L.kda_read_status.restype = ctypes.c_int
    L.kda_read_status.argtypes = [sp, vp, ctypes.POINTER(ctypes.c_int), vp]
    L.kda_selftest_bounded_wait.restype = ctypes.c_int
    L.kda_selftest_bounded_wait.argtypes = [ctypes.c_int, ctypes.c_longlong, vp, vp]
    L.kda_strerror.restype = ctypes.c_char_p
    L.kda_strerror.argtypes = [ctypes.c_int]
    L.kda_version.restype = ctypes.c_int
    L.kda_version.argtypes = []
    _lib = L
    return L


def lib():
    return _load()


def strerror(code: int) -> str:
    return lib().kda_strerror(code).decode()


def make_shape(N, T, H, HV, K=128, V=128, act="bf16", W=4) -> KdaShape:
    a = {"bf16": BF16, "f32": F32, torch.bfloat16: BF16, torch.float32: F32}[act]
    return KdaShape(N, T, H, HV, K, V, W, a)


def shape_of(mixed_qkv: torch.Tensor, a: torch.Tensor, S0: torch.Tensor) -> KdaShape:
    """Infer the problem shape from the tensors (dim = 2HK + HV V)."""
    N, T, dim = mixed_qkv.shape
    HV, K = a.shape[2], a.shape[3]
    V = S0.shape[3]
    H = (dim - HV * V) // (2 * K)
    return make_shape(N, T, H, HV, K, V, mixed_qkv.dtype)


def workspace_bytes(shape: KdaShape) -> int:
    return int(lib().kda_workspace_bytes(ctypes.byref(shape)))


def alloc_workspace(shape: KdaShape, device) -> torch.Tensor:
    """A zeroed workspace (the kernel leaves it zeroed after every launch)."""
    n = max(256, workspace_bytes(shape))
    return torch.zeros(n, dtype=torch.uint8, device=device)


def make_plan(shape: KdaShape, num_sms: int, variant: str = "auto", decode: bool = False) -> KdaPlan:
    """The dispatcher's plan for kda_conv_verify (or, with decode, kda_conv_decode)."""
    plan = KdaPlan()
    fn = lib().kda_make_decode_plan if decode else lib().kda_make_plan
    rc = fn(ctypes.byref(shape), num_sms, VARIANTS[variant], ctypes.byref(plan))
    if rc != 0:
        raise KdaError(rc, "kda_make_decode_plan" if decode else "kda_make_plan")
    return plan


def resolve_plan(shape: KdaShape, num_sms: int, plan, decode: bool = False) -> KdaPlan:
    """A hand-written plan (KdaPlan or plan string) with its derived fields
    filled in as the verify call would (launches, q/k roll, grid, ...)."""
    p = parse_plan(plan) if isinstance(plan, str) else plan
    rc = lib().kda_resolve_plan(ctypes.byref(shape), num_sms, int(decode), ctypes.byref(p))
    if rc != 0:
        raise KdaError(rc, "kda_resolve_plan")
    return p


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# ---- argument checks of the Python entry points ------------------------------
# The C ABI takes raw pointers and cannot know the size of a buffer; here each
# tensor is checked against the shape the call implies (its layout in
# include/kda_verify.h), so a wrong-sized, wrongly typed, strided or host
# tensor raises ValueError instead of being read or written out of bounds.
# validate=False skips the checks (to exercise the library's own rejections).

def _act(shape: KdaShape):
    return torch.bfloat16 if shape.act == BF16 else torch.float32


def _expect(name, t, dims, dtype, rows=None, optional=False):
    """t: a contiguous tensor of `dtype` and shape `dims`; rows, when given,
    replaces the first dimension by a lower bound (state pools).  That every
    tensor lives on the GPU is checked last (_on_cuda), once the shapes are."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    got = tuple(t.shape)
    want = tuple(int(d) for d in dims)
    if rows is None:
        ok = got == want
    else:
        ok = len(got) == len(want) and got[1:] == want[1:] and got[0] >= rows
        want = (f">={rows}",) + want[1:]
    if not ok:
        raise ValueError(f"{name} must have shape {want}, got {got}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on_cuda(**tensors):
    for name, t in tensors.items():
        if t is not None and t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor, got {t.device}")


def _check_inputs(shape: KdaShape, gate, mixed_qkv, conv_w, A_log, dt_bias, a, b):
    N, T, H, HV, K, V = shape.N, shape.T, shape.H, shape.HV, shape.K, shape.V
    dim, act = 2 * H * K + HV * V, _act(shape)
    softplus = gate in ("softplus", GATE_SOFTPLUS)
    _expect("mixed_qkv", mixed_qkv, (N, T, dim), act)
    _expect("conv_w", conv_w, (dim, 4), act)
    _expect("A_log", A_log, (HV,), torch.float32, optional=not softplus)
    _expect("dt_bias", dt_bias, (HV, K), torch.float32, optional=not softplus)
    _expect("a", a, (N, T, HV, K), act)
    _expect("b", b, (N, T, HV), act)
    return dim, act


def _pool_rows(shape: KdaShape, idx: Optional["KdaStateIndices"]):
    """Rows each state pool must hold: its pool size where the call gives
    slots for it, else N."""
    N = shape.N
    if idx is None:
        return N, N, N
    return (idx.state_pool if idx.cache_indices else N,
            idx.conv_pool if idx.conv_state_indices else N,
            idx.inter_pool if idx.intermediate_state_indices else N)


def _check_verify(shape, gate, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, o,
                  inter_ssm, conv_snapshots, idx=None):
    N, T, HV, K, V = shape.N, shape.T, shape.HV, shape.K, shape.V
    dim, act = _check_inputs(shape, gate, mixed_qkv, conv_w, A_log, dt_bias, a, b)
    rs, rc, ri = _pool_rows(shape, idx)
    _expect("conv_state", conv_state, (rc, dim, 3), act, rows=rc)
    _expect("S0", S0, (rs, HV, K, V), torch.float32, rows=rs)
    _expect("o", o, (N, T, HV, V), act)
    _expect("inter_ssm", inter_ssm, (ri, T, HV, K, V), torch.float32, rows=ri)
    _expect("conv_snapshots", conv_snapshots, (ri, T, dim, 3), act, rows=ri)
    _on_cuda(mixed_qkv=mixed_qkv, conv_w=conv_w, conv_state=conv_state, A_log=A_log, dt_bias=dt_bias,
             a=a, b=b, S0=S0, o=o, inter_ssm=inter_ssm, conv_snapshots=conv_snapshots)


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


QK_ROLL_AUTO, QK_ROLL_COUNTER, QK_ROLL_KERNEL, QK_ROLL_CLUSTER = 0, 1, 2, 3
QK_ROLL_NAMES = {"auto": QK_ROLL_AUTO, "counter": QK_ROLL_COUNTER, "kernel": QK_ROLL_KERNEL,
                 "cluster": QK_ROLL_CLUSTER}


def parse_plan(spec: str) -> KdaPlan:
    """'item:32' / 'pipe:128' / 'smem:128' / 'pipe:128:300' / 'item:128:0:-1' /
    'smem:128:0:0:kernel' (variant, v-tile width, grid, L2 prefetch distance: -1 off,
    0 default, q/k conv_state roll: 'counter', 'kernel' or 'cluster', default the
    dispatcher's)."""
    parts = spec.split(":")
    plan = KdaPlan()
    plan.variant = {"item": VARIANT_ONE_ITEM, "pipe": VARIANT_PIPELINED,
                    "smem": VARIANT_ONE_ITEM_SMEM, "split": VARIANT_SPLIT}[parts[0]]
    plan.bv = int(parts[1])
    plan.grid = int(parts[2]) if len(parts) > 2 else 0
    plan.prefetch = int(parts[3]) if len(parts) > 3 else 0
    plan.qk_roll = QK_ROLL_NAMES[parts[4]] if len(parts) > 4 else QK_ROLL_AUTO
    return plan


def conv_verify(mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate: str,
                o, inter_ssm, conv_snapshots, workspace, stream=None, variant: str = "auto",
                shape: Optional[KdaShape] = None, plan=None, validate: bool = True) -> None:
    """Launch the fused verify decode on `stream` (default: current stream).

    Tensors must be contiguous CUDA tensors in the layouts of the header
    (checked unless validate=False; ValueError otherwise); conv_state is
    updated in place; o / inter_ssm / conv_snapshots are written.  `plan` (a
    KdaPlan or a 'item:32'-style string) overrides the dispatcher.  Raises
    KdaError on any non-zero return code."""
    if shape is None:
        shape = shape_of(mixed_qkv, a, S0)
    if validate:
        _check_verify(shape, gate, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, o,
                      inter_ssm, conv_snapshots)
    gm = GATE_SOFTPLUS if gate in ("softplus", GATE_SOFTPLUS) else GATE_SAFE
    args = (ctypes.byref(shape), _ptr(mixed_qkv), _ptr(conv_w), _ptr(conv_state), _ptr(A_log),
            _ptr(dt_bias), _ptr(a), _ptr(b), _ptr(S0), gm, _ptr(o), _ptr(inter_ssm),
            _ptr(conv_snapshots), _ptr(workspace), workspace.numel() * workspace.element_size())
    if plan is not None:
        if isinstance(plan, str):
            plan = parse_plan(plan)
        rc = lib().kda_conv_verify_plan(*args, ctypes.byref(plan), _stream_handle(stream))
    else:
        rc = lib().kda_conv_verify_variant(*args, VARIANTS[variant], _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc)


def conv_verify_noalloc(mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, gate: str,
                        o, inter_ssm, conv_snapshots, stream=None,
                        shape: Optional[KdaShape] = None, validate: bool = True) -> None:
    """The allocation-free entry point: no workspace argument, the scratch is
    the library's built-in device array (calls must not overlap on the GPU)."""
    if shape is None:
        shape = shape_of(mixed_qkv, a, S0)
    if validate:
        _check_verify(shape, gate, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, o,
                      inter_ssm, conv_snapshots)
    gm = GATE_SOFTPLUS if gate in ("softplus", GATE_SOFTPLUS) else GATE_SAFE
    rc = lib().kda_conv_verify_noalloc(
        ctypes.byref(shape), _ptr(mixed_qkv), _ptr(conv_w), _ptr(conv_state), _ptr(A_log),
        _ptr(dt_bias), _ptr(a), _ptr(b), _ptr(S0), gm, _ptr(o), _ptr(inter_ssm),
        _ptr(conv_snapshots), _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_conv_verify_noalloc")


def noalloc_read_status(shape: KdaShape, stream=None) -> int:
    """Read and clear the status word of the allocation-free entry point's
    built-in scratch (for the call of shape `shape`; synchronises `stream`)."""
    st = ctypes.c_int(0)
    rc = lib().kda_noalloc_read_status(ctypes.byref(shape), ctypes.byref(st),
                                       _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_noalloc_read_status")
    return st.value


STATUS_TMA_TIMEOUT = 1
STATUS_BAD_ACCEPT = 2
STATUS_BAD_INDEX = 4


def conv_verify_indexed(shape: KdaShape, idx: KdaStateIndices, mixed_qkv, conv_w, conv_state,
                        A_log, dt_bias, a, b, S0, gate: str, o, inter_ssm, conv_snapshots,
                        workspace, stream=None, plan=None, validate: bool = True) -> None:
    """The verify over state pools (conv_state, S0, inter_ssm, conv_snapshots
    are pools addressed through `idx`; see kda_state_indices)."""
    if validate:
        _check_verify(shape, gate, mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0, o,
                      inter_ssm, conv_snapshots, idx)
    gm = GATE_SOFTPLUS if gate in ("softplus", GATE_SOFTPLUS) else GATE_SAFE
    if isinstance(plan, str):
        plan = parse_plan(plan)
    rc = lib().kda_conv_verify_indexed(
        ctypes.byref(shape), ctypes.byref(idx), _ptr(mixed_qkv), _ptr(conv_w), _ptr(conv_state),
        _ptr(A_log), _ptr(dt_bias), _ptr(a), _ptr(b), _ptr(S0), gm, _ptr(o), _ptr(inter_ssm),
        _ptr(conv_snapshots), _ptr(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(plan) if plan is not None else None, _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_conv_verify_indexed")


def conv_decode(mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S, gate: str, o, workspace,
                stream=None, plan=None, idx: Optional[KdaStateIndices] = None,
                shape: Optional[KdaShape] = None, validate: bool = True) -> None:
    """Plain decode: S (f32, the state pool or [N,HV,K,V]) is updated in place,
    conv_state rolled, o written; no snapshots."""
    if shape is None:
        shape = shape_of(mixed_qkv, a, S if idx is None else S[: mixed_qkv.shape[0]])
    if validate:
        dim, act = _check_inputs(shape, gate, mixed_qkv, conv_w, A_log, dt_bias, a, b)
        rs, rc, _ = _pool_rows(shape, idx)
        _expect("conv_state", conv_state, (rc, dim, 3), act, rows=rc)
        _expect("S", S, (rs, shape.HV, shape.K, shape.V), torch.float32, rows=rs)
        _expect("o", o, (shape.N, shape.T, shape.HV, shape.V), act)
        _on_cuda(mixed_qkv=mixed_qkv, conv_w=conv_w, conv_state=conv_state, A_log=A_log,
                 dt_bias=dt_bias, a=a, b=b, S=S, o=o)
    gm = GATE_SOFTPLUS if gate in ("softplus", GATE_SOFTPLUS) else GATE_SAFE
    if isinstance(plan, str):
        plan = parse_plan(plan)
    rc = lib().kda_conv_decode(
        ctypes.byref(shape), ctypes.byref(idx) if idx is not None else None, _ptr(mixed_qkv),
        _ptr(conv_w), _ptr(conv_state), _ptr(A_log), _ptr(dt_bias), _ptr(a), _ptr(b), _ptr(S), gm,
        _ptr(o), _ptr(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(plan) if plan is not None else None, _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_conv_decode")


def _check_commit(shape, accepted, inter_ssm, conv_snapshots, S, conv_state, status, idx=None):
    N, T, HV, K, V = shape.N, shape.T, shape.HV, shape.K, shape.V
    dim, act = 2 * shape.H * K + HV * V, _act(shape)
    rs, rc, ri = _pool_rows(shape, idx)
    _expect("accepted", accepted, (N,), torch.int32)
    _expect("inter_ssm", inter_ssm, (ri, T, HV, K, V), torch.float32, rows=ri)
    _expect("conv_snapshots", conv_snapshots, (ri, T, dim, 3), act, rows=ri)
    _expect("S", S, (rs, HV, K, V), torch.float32, rows=rs)
    _expect("conv_state", conv_state, (rc, dim, 3), act, rows=rc)
    if status is not None:
        _expect("status", status, (1,), torch.int32, rows=1)
    _on_cuda(accepted=accepted, inter_ssm=inter_ssm, conv_snapshots=conv_snapshots, S=S,
             conv_state=conv_state, status=status)


def commit_indexed(shape: KdaShape, idx: KdaStateIndices, accepted, inter_ssm, conv_snapshots,
                   S, conv_state, status=None, stream=None, validate: bool = True) -> None:
    if validate:
        _check_commit(shape, accepted, inter_ssm, conv_snapshots, S, conv_state, status, idx)
    rc = lib().kda_commit_indexed(ctypes.byref(shape), ctypes.byref(idx), _ptr(accepted),
                                  _ptr(inter_ssm), _ptr(conv_snapshots), _ptr(S),
                                  _ptr(conv_state), _ptr(status), _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_commit_indexed")


def commit(accepted, inter_ssm, conv_snapshots, S, conv_state, status=None, stream=None,
           shape: Optional[KdaShape] = None, validate: bool = True) -> None:
    """Accept accepted[n] (int32, device) verified tokens of every sequence:
    S[n] <- inter_ssm[n, acc-1], conv_state[n] <- conv_snapshots[n, acc-1]."""
    if shape is None:
        N, T, HV, K, V = inter_ssm.shape
        dim = conv_snapshots.shape[2]
        H = (dim - HV * V) // (2 * K)
        shape = make_shape(N, T, H, HV, K, V, conv_snapshots.dtype)
    if validate:
        _check_commit(shape, accepted, inter_ssm, conv_snapshots, S, conv_state, status)
    rc = lib().kda_commit(ctypes.byref(shape), _ptr(accepted), _ptr(inter_ssm),
                          _ptr(conv_snapshots), _ptr(S), _ptr(conv_state), _ptr(status),
                          _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_commit")


def read_status(shape: KdaShape, workspace: torch.Tensor, stream=None) -> int:
    st = ctypes.c_int(0)
    rc = lib().kda_read_status(ctypes.byref(shape), _ptr(workspace), ctypes.byref(st),
                               _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_read_status")
    return st.value


def run(inputs: Dict[str, torch.Tensor], gate: str, variant: str = "auto",
        workspace: Optional[torch.Tensor] = None, stream=None, plan=None) -> Dict[str, torch.Tensor]:
    """Convenience: allocate outputs on the inputs' device and launch.
    `inputs["conv_state"]` is rolled in place."""
    x = inputs["mixed_qkv"]
    shape = shape_of(x, inputs["a"], inputs["S0"])
    dev = x.device
    N, T, dim = x.shape
    HV, K, V = shape.HV, shape.K, shape.V
    out = {
        "o": torch.empty((N, T, HV, V), dtype=x.dtype, device=dev),
        "inter_ssm": torch.empty((N, T, HV, K, V), dtype=torch.float32, device=dev),
        "conv_snapshots": torch.empty((N, T, dim, 3), dtype=x.dtype, device=dev),
    }
    ws = workspace if workspace is not None else alloc_workspace(shape, dev)
    conv_verify(x, inputs["conv_w"], inputs["conv_state"], inputs.get("A_log"),
                inputs.get("dt_bias"), inputs["a"], inputs["b"], inputs["S0"], gate,
                out["o"], out["inter_ssm"], out["conv_snapshots"], ws, stream=stream,
                variant=variant, shape=shape, plan=plan)
    return out


def selftest_bounded_wait(mode: int, limit_ns: int = 0, stream=None):
    """Run the kernels' bounded waits until they give up (no fault); returns
    (status word, mask of the waits that gave up: 1 one-item, 2 pipelined,
    4 the one-item wait inside a cluster, mode 3)."""
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    rc = lib().kda_selftest_bounded_wait(int(mode), int(limit_ns), _ptr(out), _stream_handle(stream))
    if rc != 0:
        raise KdaError(rc, "kda_selftest_bounded_wait")
    torch.cuda.synchronize()
    return int(out[0]), int(out[1])


def plan_label(plan: KdaPlan) -> str:
    """'item:128' etc.: the plan-string prefix of the variant and the v-tile width."""
    return f"{PLAN_PREFIX[plan.variant]}:{plan.bv}"
