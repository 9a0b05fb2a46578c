"""The library builds for sm_103a with no register spills in any kernel
instance: every gemm_kernel instantiation fits its 168-register budget (11 or
fewer warps a CTA), which the epilogue's 32-value chunks and the pipelines'
bookkeeping are sized for.  Reads ptxas's -v report of the in-tree build."""

import os
import re

from grouped_gemm_epilogues_gb300 import build as gge_build


def test_no_spills_in_any_kernel_instance():
    gge_build.build()
    log = open(os.path.join(gge_build.BUILD, "ptxas.log")).read()
    current, seen, spills = None, 0, []
    for line in log.splitlines():
        m = re.search(r"Compiling entry function '(\S*gemm_kernel\S*)'", line)
        if m:
            current = m.group(1)
            continue
        if current is None:
            continue
        s = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if s:
            seen += 1
            if int(s.group(1)) or int(s.group(2)):
                spills.append((current, line.strip()))
        r = re.search(r"Used (\d+) registers", line)
        if r:
            assert int(r.group(1)) <= 168, (current, line)
            current = None
    assert seen >= 10, "no kernel instances found in the ptxas report"
    assert not spills, spills
