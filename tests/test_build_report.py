"""The compiler's resource report for the kernels (no GPU needed): every
kernel entry compiles without register spills (the routing kernel's 32 logits
per lane stay in registers), and the two step kernels stay within 168
registers per thread, the budget their 384-thread blocks have
(384 x 168 <= 65536)."""
import os
import re

from quantized_moe_routed_gb300 import build as libbuild


def _entries(unit):
    log = os.path.join(libbuild.BUILD, unit + ".log")
    if not os.path.exists(log):
        libbuild.build(force=True)
    text = open(log).read()
    out = {}
    for block in re.split(r"ptxas info\s*: Compiling entry function ", text)[1:]:
        name = re.match(r"'([^']+)'", block).group(1)
        regs = int(re.search(r"Used (\d+) registers", block).group(1))
        spills = [int(a) + int(b) for a, b in re.findall(r"(\d+) bytes spill stores, (\d+) bytes spill loads", block)]
        out[name] = (regs, spills)
    return out


def test_kernels_do_not_spill_and_fit_the_register_budget():
    libbuild.build()
    for unit, kernel in (("moe_kernels.cu", "moe_step_kernel"), ("moe_tc.cu", "moe_tc_kernel"),
                         ("moe_route.cu", "moe_route_kernel")):
        entries = _entries(unit)
        steps = {n: v for n, v in entries.items() if kernel in n}
        assert steps, f"no {kernel} entries in the {unit} report"
        for name, (regs, spills) in entries.items():
            assert all(s == 0 for s in spills), f"{name} spills"
        for name, (regs, _) in steps.items():
            assert regs <= 168, f"{name} uses {regs} registers"
