"""Source-level rules of the CUDA kernels, checked on the CPU.

Every kernel is launched with programmatic stream serialization, so its
blocks may start while the previous kernel in the stream is still running;
each must wait for that kernel (pdl_enter: griddepcontrol.wait) before it
touches memory.  A kernel without the wait would race with its predecessor.
"""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "collective_reduction_virtual_gb300", "csrc")
# launched with a plain cudaLaunchKernel, never after a kernel of ours
EXEMPT = {"vc_selftest_wait_timeout"}


def _kernels():
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh")):
            continue
        src = open(os.path.join(CSRC, name)).read()
        for m in re.finditer(r"__global__\s+void\s+(?:__launch_bounds__\([^)]*\)\s*)?(\w+)\s*\(", src):
            body_start = src.index("{", m.end())
            yield name, m.group(1), src[body_start + 1:body_start + 400]


def test_every_kernel_waits_for_its_predecessor_first():
    found = list(_kernels())
    assert len(found) >= 20
    for name, kernel, body in found:
        if kernel in EXEMPT:
            continue
        first = body.strip().split(";")[0].strip()
        assert first == "pdl_enter()", f"{name}: {kernel} does not start with pdl_enter()"


def test_launches_go_through_the_dependent_launch_helper():
    src = open(os.path.join(CSRC, "api.cpp")).read()
    plain = [ln.strip() for ln in src.splitlines() if "cudaLaunchKernel(" in ln]
    assert len(plain) == 1 and "selftest_timeout_kernel" in plain[0], plain
