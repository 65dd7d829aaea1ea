"""Shared helpers of the GPU parity tests: error metrics and launch wrappers.

Tolerance (written here once, used by every parity test and the smoke check).
The bound is 2e-3 relative on o and on the state snapshots, measured element
by element as |x - y| / max(|y|, rms(y)) against the float64 oracle y, where
the rms floor keeps elements that cancel to ~0 from dominating.

o is stored in the activation type.  A bf16 value carries an 8-bit
significand, so rounding the exact result to bf16 alone moves it by up to
2^-8 = 3.9e-3 of its magnitude: no bf16 output can sit within 2e-3 of the
exact value everywhere.  The bound is therefore applied to the computation,
and the final round-to-nearest into the output type is allowed on top of it:
an element passes when |x - y| <= 2e-3 * max(|y|, rms(y)) + ulp(x) / 2.
For fp32 outputs the extra term is ~6e-8 relative.  The relative RMS error
of o must also stay below 2e-3, measured against the oracle rounded into the
output type (||x - round(y)|| / ||y||), as the verify-decode page measures its
own o (its Tests & Accuracy section reports o's relative RMS error against a
reference in the same dtype, <= 1.7e-4, apart from the 1.5e-3 - 1.7e-3 that
bf16 rounding alone leaves against fp32).  Against the unrounded y that floor
fluctuates with the sample: on a few hundred elements rounding alone can give
2.1e-3.

Conv snapshots and the rolled conv_state are copies and must match bit for
bit.
"""

import numpy as np
import torch

TOL = 2e-3


def max_rel_err(x, y) -> float:
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    if y.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(y * y)))
    den = np.maximum(np.abs(y), rms)
    den[den == 0] = 1.0
    return float(np.max(np.abs(x - y) / den))


def half_ulp(x, dtype) -> np.ndarray:
    """Half the spacing of `dtype` (torch.bfloat16 / torch.float32) at x."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    bits = 8 if dtype == torch.bfloat16 else 24  # significand bits
    e = np.floor(np.log2(np.where(x > 0, x, 1.0)))
    h = np.ldexp(1.0, (e - bits).astype(np.int64))
    return np.where(x > 0, h, 0.0)


def max_rel_err_rounded(x, y, dtype) -> float:
    """Largest error left after allowing the final rounding into `dtype`,
    relative to max(|y|, rms(y))."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    if y.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(y * y)))
    den = np.maximum(np.abs(y), rms)
    den[den == 0] = 1.0
    excess = np.maximum(np.abs(x - y) - half_ulp(x, dtype), 0.0)
    return float(np.max(excess / den))


def round_to(y, dtype) -> np.ndarray:
    """y (float64) rounded once, to nearest even, to the significand of
    `dtype` (torch.bfloat16: 8 bits, torch.float32: 24 bits)."""
    y = np.asarray(y, dtype=np.float64)
    bits = 8 if dtype == torch.bfloat16 else 24
    m, e = np.frexp(y)  # y = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, bits)), e - bits)


def rel_rmse(x, y) -> float:
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    d = float(np.sqrt(np.mean((x - y) ** 2)))
    r = float(np.sqrt(np.mean(y * y)))
    return d / r if r > 0 else d


def rel_rmse_rounded(x, y, dtype) -> float:
    """||x - round(y)|| / ||y||: the relative RMS error left once the exact
    result is rounded into the output type."""
    y = np.asarray(y, dtype=np.float64)
    r = float(np.sqrt(np.mean(y * y))) if y.size else 0.0
    d = float(np.sqrt(np.mean((np.asarray(x, dtype=np.float64) - round_to(y, dtype)) ** 2))) if y.size else 0.0
    return d / r if r > 0 else d


def to_device(inputs, device="cuda"):
    return {k: (v.to(device) if v is not None else None) for k, v in inputs.items()}


def run_kernel(inputs_cpu, gate, variant="auto"):
    """Copy inputs to the GPU, run one call, return (device outputs, rolled
    conv_state on the device).  `variant` is auto / one_item / pipelined
    or an explicit plan such as 'item:64' or 'pipe:64'."""
    from linear_attention_speculative_gb300 import kda
    dev = to_device(inputs_cpu)
    if ":" in variant:
        out = kda.run(dev, gate, plan=variant)
    else:
        out = kda.run(dev, gate, variant=variant)
    torch.cuda.synchronize()
    return out, dev["conv_state"]


def assert_parity(out, conv_state_dev, ref, seqs=None, tol=TOL):
    """Compare device outputs (optionally only sequences `seqs`) to the oracle."""
    def pick(t):
        t = t if seqs is None else t[list(seqs)]
        return t.detach().to("cpu", torch.float64).numpy()

    o = pick(out["o"])
    e_o = max_rel_err_rounded(o, ref["o"], out["o"].dtype)
    r_o = rel_rmse_rounded(o, ref["o"], out["o"].dtype)
    e_s = max_rel_err(pick(out["inter_ssm"]), ref["inter_ssm"])
    assert np.array_equal(pick(out["conv_snapshots"]), ref["conv_snapshots"]), "conv snapshots differ"
    assert np.array_equal(pick(conv_state_dev), ref["conv_state"]), "rolled conv_state differs"
    assert e_o <= tol, f"o max rel err beyond output rounding {e_o:.3e} > {tol}"
    assert r_o <= tol, f"o rel rmse {r_o:.3e} > {tol}"
    assert e_s <= tol, f"inter_ssm max rel err {e_s:.3e} > {tol}"
    return e_o, e_s


def assert_decode_parity(o, S_final, conv_state_dev, ref, seqs=None, t=-1, tol=TOL):
    """Compare a plain decode (or one token of a chain) with the oracle's
    verify of the same inputs: the state it leaves against the oracle's state
    snapshot after token `t`, its o against the oracle's o (rounded check,
    relative RMS), and the rolled conv_state bit for bit (None: not checked).
    `o` holds the tokens the decode ran; `ref` the oracle's whole call."""
    def pick(x):
        x = x if seqs is None else x[list(seqs)]
        return x.detach().to("cpu", torch.float64).numpy()

    T = ref["o"].shape[1]
    toks = list(range(T)) if o.shape[1] == T else [t % T]
    y_o = ref["o"][:, toks]
    x_o = pick(o)
    e_o = max_rel_err_rounded(x_o, y_o, o.dtype)
    r_o = rel_rmse_rounded(x_o, y_o, o.dtype)
    e_s = max_rel_err(pick(S_final), ref["inter_ssm"][:, t])
    assert e_o <= tol, f"o max rel err beyond output rounding {e_o:.3e} > {tol}"
    assert r_o <= tol, f"o rel rmse {r_o:.3e} > {tol}"
    assert e_s <= tol, f"state max rel err {e_s:.3e} > {tol}"
    if conv_state_dev is not None:
        assert np.array_equal(pick(conv_state_dev), ref["conv_state"]), "rolled conv_state differs"
    return e_o, e_s


def conv_window_properties(inputs_cpu, out, conv_state_dev):
    """Full-size check that holds at any size: every snapshot and the rolled
    state are the right raw window of [old conv_state || tokens] (pure
    indexing on the device, compared bit for bit)."""
    x = inputs_cpu["mixed_qkv"].cuda()
    cs = inputs_cpu["conv_state"].cuda()
    T = x.shape[1]
    xext = torch.cat([cs, x.transpose(1, 2)], dim=2)  # [N, dim, T+3]
    snaps = out["conv_snapshots"]                       # [N, T, dim, 3]
    for t in range(T):
        assert torch.equal(snaps[:, t], xext[:, :, t + 1:t + 4]), f"snapshot {t}"
    assert torch.equal(conv_state_dev, xext[:, :, T:T + 3]), "rolled conv_state"


def _stage_floats(T, K, BV):
    rows = K // 8 if K <= 128 else K // 16
    rs = rows + (0 if (rows // 4) & 1 else 4)
    ks = (8 if K <= 128 else 16) * rs
    return 3 * T * ks + T * BV + (T + 3) // 4 * 4


def split_fits(K, V, T, bv, G, act="bf16") -> bool:
    """The split variant's limits: each item's stage within its K x bv slice
    of the last token's snapshot, the prep kernel's staging within one CTA."""
    ks = _stage_floats(1, K, 0) - 4  # 3 * KS
    prep = 4 * ((2 + G) * T * ks // 3 + G * T * V + G * ((T + 3) // 4 * 4)) \
        + (2 * K + G * V) * 3 * (4 if act == "f32" else 2)
    return _stage_floats(T, K, bv) <= K * bv and prep <= 232448


def variant_built(variant, K, V, decode=False, T=1, G=1, act="bf16") -> bool:
    """Whether a named variant runs for head dims K x V (the pipelined kernel
    needs K <= 128, V >= 64 and no decode; the split variant K <= 128, no
    decode and a stage that fits)."""
    if variant == "pipelined":
        return K <= 128 and V >= 64 and not decode
    if variant == "split":
        return K <= 128 and not decode and split_fits(K, V, T, min(V, 128), G, act)
    return True


def plan_built(plan, K, V, decode=False, T=1, act="bf16", G=1) -> bool:
    """Whether an explicit plan string names a kernel the library builds for
    head dims K x V: one-item tiles are 1/2/4/8 warps of 16 columns (K <= 128;
    1 warp not for K = 256, whose warps hold 8 columns), the shared-memory
    state 4 or 8 warps, the pipelined kernel 4 or 8 consumer warps at
    K <= 128 and no decode (T and act matter only for its shared memory)."""
    if plan in (None, "auto"):
        return True
    kind, bv = plan.split(":")[0], int(plan.split(":")[1])
    wc = 8 if K == 256 else 16
    if bv > V or V % bv:
        return False
    if plan.split(":")[4:5] == ["cluster"]:
        # the cluster roll: the one-item kernel with the state in registers at
        # 4 or 8 warps, a group of at most 8 items
        if kind != "item" or bv not in (4 * wc, 8 * wc) or G * (V // bv) > 8:
            return False
    if kind == "split":
        return (K <= 128 and not decode and bv in (32, 64, 128)
                and split_fits(K, V, T, bv, G, act))
    if kind == "pipe":
        # its shared memory fits one CTA except 128-wide K = 128 tiles at
        # T = 16 with fp32 activations
        too_big = bv == 128 and K == 128 and T >= 16 and act == "f32"
        return K <= 128 and not decode and bv in (64, 128) and not too_big
    if kind == "smem":
        return bv in (4 * wc, 8 * wc)
    return bv in (2 * wc, 4 * wc, 8 * wc) or (K <= 128 and bv == wc)
