"""Static checks of the launch protocol in the CUDA sources (no GPU).

Every kernel of the library is launched as a programmatic dependent of the
kernel before it on the stream, so its CTAs may start while that kernel is
still running.  Two rules keep stream order intact, and a mistake in either
would only show as a rare race on the GPU:
  * a kernel touches no global memory before `griddepcontrol.wait`;
  * a kernel triggers its own dependents (`griddepcontrol.launch_dependents`)
    only after that wait, because two of its dependents -- the q/k roll
    kernel and the split variant's recurrence kernel -- load before their
    own waits and rely on everything before their primary being complete.
These tests read the kernel bodies and the launch sites as text."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "linear_attention_speculative_gb300", "csrc")

# kernels that wait for the previous kernel first, then trigger
WAIT_THEN_TRIGGER = {
    "kda_kernel.cuh": ("kda_tile_kernel", "kda_prep_kernel", "kda_pipe_kernel"),
    "kda_commit.cu": ("kda_commit_kernel",),
}


def _read(name):
    with open(os.path.join(CSRC, name), encoding="utf-8") as f:
        return f.read()


def _strip_comments(code):
    code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
    return re.sub(r"//[^\n]*", " ", code)


def _body(code, kernel):
    """Text of the body of __global__ function `kernel` (brace-matched)."""
    m = re.search(r"__global__[^{;]*?\b" + kernel + r"\s*\(", code, flags=re.S)
    assert m, kernel
    i = code.index("{", m.end())
    depth = 0
    for j in range(i, len(code)):
        depth += {"{": 1, "}": -1}.get(code[j], 0)
        if depth == 0:
            return code[i:j + 1]
    raise AssertionError(f"unbalanced body of {kernel}")


def test_every_kernel_waits_before_it_triggers_its_dependents():
    for name, kernels in WAIT_THEN_TRIGGER.items():
        code = _strip_comments(_read(name))
        for k in kernels:
            body = _body(code, k)
            w = body.find("griddepcontrol.wait")
            t = body.find("griddepcontrol.launch_dependents")
            assert w >= 0 and t >= 0, k
            assert w < t, f"{k} triggers its dependents before waiting for the kernel before it"


def test_nothing_global_before_the_first_wait():
    # before its first wait a kernel only computes from its parameters and
    # indices: no pointer dereference, no load/store helper, no atomic
    suspicious = re.compile(r"__ldg|ld_|st_|atomic|\bp\.(idx|mixed|conv_state|S0|a\b|b\b|o\b|inter|S_out|acc)|->|\*\s*\(")
    for name, kernels in WAIT_THEN_TRIGGER.items():
        code = _strip_comments(_read(name))
        for k in kernels:
            body = _body(code, k)
            pre = body[:body.find("griddepcontrol.wait")]
            pre = re.sub(r"&\s*\w+\s*->\s*\w+", " ", pre)  # taking a (shared-memory) address reads nothing
            assert not suspicious.search(pre), (k, suspicious.search(pre).group(0))


def test_the_roll_kernel_stores_only_after_its_wait_and_triggers_after_it():
    body = _body(_strip_comments(_read("kda_roll.cu")), "kda_qk_roll_kernel")
    w = body.find("griddepcontrol.wait")
    t = body.find("griddepcontrol.launch_dependents")
    assert 0 <= w < t
    assert "st_16" not in body[:w] and "st_16" in body[w:]


def test_product_kernels_are_launched_as_programmatic_dependents():
    # the only triple-chevron launch left is the bounded-wait self-test
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh")) or name == "kda_selftest.cu":
            continue
        code = _strip_comments(_read(name))
        assert "<<<" not in code, name
        code = re.sub(r"inline void set_programmatic\(.*?\n}", " ", code, flags=re.S)  # the helper itself
        # one launch configuration per kernel launched (the roll kernel's two
        # instantiations share one), each carrying the programmatic attribute
        n_cfg = len(re.findall(r"cudaLaunchConfig_t\s+\w+\s*=", code))
        n_pdl = code.count("set_programmatic(") + code.count("programmaticStreamSerializationAllowed = 1")
        assert n_pdl == n_cfg, (name, n_cfg, n_pdl)
        assert code.count("cudaLaunchKernelEx(") >= n_cfg, name
