"""CPU oracle for the fused causal-conv1d + KDA verify decode.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline may import this package; the product path never does.  It shares no
code with the CUDA library (see ``kda_oracle.c`` for the definition and the
page it follows).  Parity pins live in ``tests/test_oracle_*.py``.

``verify`` runs the plain fp64 C oracle sequence by sequence; ``seqs`` picks a
subset of sequences so that full-size workloads can be checked on samples.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Iterable, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")

GATE_SOFTPLUS = 0
GATE_SAFE = 1
L2NORM_EPS = 1e-6

_lib = None
_lock = threading.Lock()
_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into oracle/_build (idempotent)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(L):
    for name in ("orc_silu", "orc_sigmoid", "orc_softplus", "orc_gate_safe"):
        f = getattr(L, name)
        f.restype = ctypes.c_double
        f.argtypes = [ctypes.c_double]
    L.orc_gate_softplus.restype = ctypes.c_double
    L.orc_gate_softplus.argtypes = [ctypes.c_double] * 3
    L.orc_causal_conv1d_silu.restype = None
    L.orc_causal_conv1d_silu.argtypes = [ctypes.c_int, ctypes.c_int, _dp, _dp, _dp]
    L.orc_l2norm.restype = None
    L.orc_l2norm.argtypes = [ctypes.c_int, _dp, ctypes.c_double]
    L.orc_delta_rule_step.restype = None
    L.orc_delta_rule_step.argtypes = [ctypes.c_int, ctypes.c_int, _dp, _dp, _dp, _dp,
                                      ctypes.c_double, _dp, ctypes.c_double, _dp]
    L.orc_commit_seq.restype = ctypes.c_int
    L.orc_commit_seq.argtypes = [ctypes.c_int] * 7 + [_dp] * 4
    L.orc_kda_conv_verify_seq.restype = ctypes.c_int
    L.orc_kda_conv_verify_seq.argtypes = ([ctypes.c_int] * 7 + [ctypes.c_double]
                                          + [_dp] * 12)
    return L


def lib():
    """The compiled oracle (built from kda_oracle.c on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def use_library(path: str) -> None:
    """Load another build of kda_oracle.c in place of the default one, for the
    rest of this process.  Only the mutation test's child process calls this:
    it plants a mistake in a copy of the source and checks that the pins
    catch it."""
    global _lib
    with _lock:
        _lib = _bind(ctypes.CDLL(path))


def _f64(x) -> np.ndarray:
    """Any array-like (numpy or torch, any float dtype) -> contiguous float64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor; bf16/f32 -> f64 is exact
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(_dp)


# ---- scalar and step functions (for the pins) ------------------------------

def silu(y: float) -> float:
    return lib().orc_silu(y)


def sigmoid(x: float) -> float:
    return lib().orc_sigmoid(x)


def softplus(x: float) -> float:
    return lib().orc_softplus(x)


def gate_softplus(A_log: float, a: float, dt_bias: float) -> float:
    return lib().orc_gate_softplus(A_log, a, dt_bias)


def gate_safe(a: float) -> float:
    return lib().orc_gate_safe(a)


def causal_conv1d_silu(xext, w, T: int) -> np.ndarray:
    xext, w = _f64(xext), _f64(w)
    W = w.shape[0]
    assert xext.shape[0] == T + W - 1
    y = np.empty(T, np.float64)
    lib().orc_causal_conv1d_silu(T, W, _ptr(xext), _ptr(w), _ptr(y))
    return y


def l2norm(x, eps: float = L2NORM_EPS) -> np.ndarray:
    x = _f64(x).copy()
    lib().orc_l2norm(x.shape[0], _ptr(x), eps)
    return x


def delta_rule_step(S, g, k, v, beta: float, q, scale: float):
    """One recurrence token; returns (S_new, o)."""
    S = _f64(S).copy()
    K, V = S.shape
    g, k, v, q = _f64(g), _f64(k), _f64(v), _f64(q)
    o = np.empty(V, np.float64)
    lib().orc_delta_rule_step(K, V, _ptr(S), _ptr(g), _ptr(k), _ptr(v), beta, _ptr(q),
                              scale, _ptr(o))
    return S, o


# ---- the whole call ---------------------------------------------------------

def verify(inputs: Dict, gate: str, seqs: Optional[Iterable[int]] = None,
           threads: int = 1, eps: float = L2NORM_EPS) -> Dict[str, np.ndarray]:
    """Run the oracle on the sequences `seqs` (default: all).

    `inputs` holds mixed_qkv, conv_w, conv_state, A_log, dt_bias, a, b, S0 in
    the layouts of the workload module (torch or numpy, any float dtype).
    Returns float64 arrays indexed by position in `seqs`:
    o [n,T,HV,V], inter_ssm [n,T,HV,K,V], conv_snapshots [n,T,dim,W-1],
    conv_state [n,dim,W-1] (the rolled state).
    """
    L = lib()
    if seqs is not None:
        # keep only the requested sequences before converting to float64
        seqs = list(seqs)
        inputs = dict(inputs)
        for key in ("mixed_qkv", "conv_state", "a", "b", "S0"):
            v = inputs[key]
            inputs[key] = v[seqs] if hasattr(v, "detach") else np.asarray(v)[seqs]
    x = _f64(inputs["mixed_qkv"])
    N, T, dim = x.shape
    w = _f64(inputs["conv_w"])
    W = w.shape[1]
    cs = _f64(inputs["conv_state"])
    a = _f64(inputs["a"])
    HV, K = a.shape[2], a.shape[3]
    b = _f64(inputs["b"])
    S0 = _f64(inputs["S0"])
    V = S0.shape[3]
    H = (dim - HV * V) // (2 * K)
    gm = GATE_SOFTPLUS if gate == "softplus" else GATE_SAFE
    A_log = _f64(inputs.get("A_log")) if gm == GATE_SOFTPLUS else None
    dt_bias = _f64(inputs.get("dt_bias")) if gm == GATE_SOFTPLUS else None
    seqs = list(range(N))  # positions within the (possibly sliced) inputs
    n = len(seqs)
    out = {
        "o": np.empty((n, T, HV, V)),
        "inter_ssm": np.empty((n, T, HV, K, V)),
        "conv_snapshots": np.empty((n, T, dim, W - 1)),
        "conv_state": np.empty((n, dim, W - 1)),
    }

    def one(i: int) -> int:
        s = seqs[i]
        return L.orc_kda_conv_verify_seq(
            T, H, HV, K, V, W, gm, eps, _ptr(x[s]), _ptr(w), _ptr(cs[s]), _ptr(A_log),
            _ptr(dt_bias), _ptr(a[s]), _ptr(b[s]), _ptr(S0[s]), _ptr(out["o"][i]),
            _ptr(out["inter_ssm"][i]), _ptr(out["conv_snapshots"][i]),
            _ptr(out["conv_state"][i]))

    if threads <= 1:
        codes = [one(i) for i in range(n)]
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            codes = list(ex.map(one, range(n)))
    bad = [c for c in codes if c != 0]
    if bad:
        raise ValueError(f"oracle rejected the call (code {bad[0]})")
    return out


def commit(acc, inter_ssm, conv_snapshots) -> Dict[str, np.ndarray]:
    """Accept acc[n] tokens of every sequence: returns the committed state
    S [N,HV,K,V] and conv_state [N,dim,W-1] (float64)."""
    L = lib()
    inter = _f64(inter_ssm)
    snap = _f64(conv_snapshots)
    N, T, HV, K, V = inter.shape
    dim, W1 = snap.shape[2], snap.shape[3]
    acc = [int(a) for a in (acc.tolist() if hasattr(acc, "tolist") else acc)]
    S = np.empty((N, HV, K, V))
    cs = np.empty((N, dim, W1))
    for n in range(N):
        rc = L.orc_commit_seq(T, HV, K, V, dim, W1 + 1, acc[n], _ptr(inter[n]), _ptr(snap[n]),
                              _ptr(S[n]), _ptr(cs[n]))
        if rc != 0:
            raise ValueError(f"oracle commit rejected acc[{n}] = {acc[n]}")
    return {"S": S, "conv_state": cs}
