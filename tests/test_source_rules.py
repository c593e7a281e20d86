"""Rules on the library's source text that claims elsewhere rest on, checked
without a GPU:

- every kernel launch goes through the launch counter that the benchmark
  reports as gpu_launches;
- every kernel that is launched as a programmatic dependent (it may start
  while the kernel before it still runs) waits for that kernel with
  griddepcontrol.wait, so its reads see the finished results."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "..",
                    "dense_fp32_gemm_05_gb300", "csrc")


def _sources():
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, f)) as fh:
                yield f, fh.read()


def _code(line):
    return line.split("//")[0]


def test_every_kernel_launch_is_counted():
    launches = 0
    for f, text in _sources():
        lines = text.splitlines()
        for i, line in enumerate(lines):
            code = _code(line)
            if "<<<" in code or "cudaLaunchKernelEx(" in code:
                launches += 1
                window = "\n".join(_code(x) for x in lines[max(0, i - 3):i])
                assert "count_launch();" in window, f"{f}:{i + 1}: launch not counted"
    # FFMA main, scale, GEMV dot/axpy/staged, split pre-pass (2), tensor-core
    # main (cluster, plain), and the dependent-launch helper
    assert launches >= 10


def _kernel_body(text, name):
    m = re.search(r"__global__[^{;]*?\b" + name + r"\s*\(", text, re.S)
    if not m:
        return None
    start = text.index("{", m.end())
    depth = 0
    for j in range(start, len(text)):
        if text[j] == "{":
            depth += 1
        elif text[j] == "}":
            depth -= 1
            if depth == 0:
                return text[start:j]
    return None


def test_dependent_kernels_wait_for_their_predecessor():
    texts = dict(_sources())
    # kernels passed to launch_dependent() or launched with the programmatic
    # attribute: the K-split sum, both stream-K fixups, the tensor-core main
    # kernel (after the split pre-pass), the FFMA kernel (after the transpose
    # pre-pass)
    dependents = [("gemv.cu", "gemv_ksum_kernel"), ("ffma_kernel.cuh", "sk_fixup_kernel"),
                  ("tc_gemm.cu", "sk_fixup_kernel"), ("tc_gemm.cu", "tc_gemm_kernel"),
                  ("ffma_kernel.cuh", "ffma_gemm_kernel")]
    for f, name in dependents:
        body = _kernel_body(texts[f], name)
        assert body is not None, (f, name)
        assert "pdl_wait();" in body, (f, name)
    # and nothing else is launched that way
    named = set()
    for f, text in texts.items():
        for m in re.finditer(r"launch_dependent\(\s*([\w:<>, ]+?)\s*,", text):
            named.add(m.group(1).split("::")[-1])
    assert named <= {"gemv_ksum_kernel", "sk_fixup_kernel", "fix", "kern",
                     "void (*kern)(KArgs...)"}, named
    assert "cudaLaunchAttributeProgrammaticStreamSerialization" not in texts["gemv.cu"]
    assert "cudaLaunchAttributeProgrammaticStreamSerialization" not in texts["sgemm_api.cu"]
