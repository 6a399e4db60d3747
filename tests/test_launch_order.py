"""Launch-order rule of the CUDA sources, checked on the text (no GPU).

The library launches its kernels with programmatic stream serialisation
(``launch_dep``): a kernel's CTAs may be scheduled while the previous kernel
in the stream still runs.  That is only correct if every kernel launched that
way waits for its predecessor (``grid_dep_wait()``) before anything else: before
it reads an input the previous kernel wrote, before it touches the workspace
counter the previous kernel resets, and before it allocates TMEM.  A kernel
without the wait could also complete before its predecessor, and the kernel
after it would then no longer be ordered behind the earlier ones.  This test
finds every kernel passed to ``launch_dep`` and checks that the first
statements of its body are the wait and then the trigger, and that the plain
``<<<>>>`` form (fully ordered, no overlap) is left to the two kernels that are
not on any step's path (the plan export and the failure-path self-test) and to
the backward preprocessing, launched plainly by measurement; a plain launch
is always ordered behind everything before it."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "io_aware_exact_09_gb300", "csrc")


def sources():
    out = {}
    for n in sorted(os.listdir(CSRC)):
        if n.endswith((".cu", ".cuh", ".h")):
            out[n] = re.sub(r"//[^\n]*", "", open(os.path.join(CSRC, n)).read())
    return out


def kernel_bodies(src):
    """name -> body text of every __global__ function defined in src."""
    out = {}
    for m in re.finditer(r"__global__\s+void\s+(?:__launch_bounds__\([^)]*\)\s*)?(\w+)\s*\(", src):
        i = src.index("{", m.end())
        depth, j = 0, i
        while True:
            if src[j] == "{":
                depth += 1
            elif src[j] == "}":
                depth -= 1
                if depth == 0:
                    break
            j += 1
        out[m.group(1)] = src[i + 1:j]
    return out


def dep_launched(src):
    """Kernel names passed to launch_dep (template arguments stripped; a
    local function-pointer variable resolved to the kernel it holds)."""
    names = set()
    for m in re.finditer(r"launch_dep\(\s*([\w:]+)", src):
        name = m.group(1)
        alias = re.search(r"auto\s+%s\s*=\s*(\w+)" % name, src)
        names.add(alias.group(1) if alias else name)
    return names


def test_every_dependent_launch_waits_first():
    srcs = sources()
    bodies = {}
    for s in srcs.values():
        bodies.update(kernel_bodies(s))
    launched = set()
    for n, s in srcs.items():
        if n == "fa_internal.h":
            continue
        launched |= dep_launched(s)
    assert {"fa_fwd_kernel", "fa_bwd64_kernel", "fa_bwd128_kernel",
            "fa_bwd_convert_kernel", "fa_decode_kernel", "fa_decode_merge_kernel", "fa_fwd_fp8_kernel",
            "fa_quant_fp8_kernel"} <= launched
    for k in sorted(launched):
        assert k in bodies, k
        stmts = [x.strip() for x in bodies[k].split(";") if x.strip()]
        assert stmts[0] == "grid_dep_wait()", (k, stmts[:2])
        assert stmts[1] == "grid_dep_launch()", (k, stmts[:2])


def test_plain_launches_are_the_listed_ones():
    plain = set()
    for s in sources().values():
        plain |= set(re.findall(r"(\w+)(?:<[^<>;]*>)?<<<", s))
    # the plan export and the self-test are off every step's path; the
    # backward preprocessing is launched plainly by measurement (launched to
    # overlap the forward's tail it slowed the main kernel after it down) and
    # still waits first and triggers its successor early
    assert plain == {"fa_plan_kernel", "fa_selftest_wait_kernel", "fa_bwd_pre_kernel"}, plain


def test_plainly_launched_step_kernels_keep_the_wait_and_trigger():
    bodies = {}
    for s in sources().values():
        bodies.update(kernel_bodies(s))
    stmts = [x.strip() for x in bodies["fa_bwd_pre_kernel"].split(";") if x.strip()]
    assert stmts[:2] == ["grid_dep_wait()", "grid_dep_launch()"], stmts[:2]


def test_the_wait_is_the_griddepcontrol_pair():
    ptx = open(os.path.join(CSRC, "fa_ptx.cuh")).read()
    assert re.search(r"grid_dep_wait\(\)\s*\{\s*asm volatile\(\"griddepcontrol\.wait;\"", ptx)
    assert re.search(r"grid_dep_launch\(\)\s*\{\s*asm volatile\(\"griddepcontrol\.launch_dependents;\"", ptx)
    h = open(os.path.join(CSRC, "fa_internal.h")).read()
    assert "cudaLaunchAttributeProgrammaticStreamSerialization" in h
