"""Register-spill budget of every kernel, read from the ``-Xptxas -v`` report
the build writes beside each object (``_build/<unit>.ptxas.txt``).  A spill
puts loads and stores to local memory on a kernel's critical path, so a
change that makes a kernel spill (or spill more) fails here, on the CPU,
before any GPU time is spent.  The pipeline's own kernels must not spill at
all; the two kernels listed in SPILL_BYTES spill a few bytes outside their
inner loops and are held at what they spill now."""
import glob
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BUILD = os.path.join(ROOT, "combine_moe_dispatch_layout_gb300", "_build")
CSRC = os.path.join(ROOT, "combine_moe_dispatch_layout_gb300", "csrc")

# largest spill-store bytes allowed per kernel (every instantiation)
SPILL_BYTES = {
    "grouped_gemm_kernel": 68,       # epilogue address set-up
    "swiglu_quant_kernel": 8,
    "swiglu_quant_warp_kernel": 4,
}


@pytest.fixture(scope="module")
def reports():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    import __graft_entry__
    __graft_entry__._load_builder().build()
    out = {}
    for src in glob.glob(os.path.join(CSRC, "*.cu")):
        unit = os.path.splitext(os.path.basename(src))[0]
        path = os.path.join(BUILD, unit + ".ptxas.txt")
        assert os.path.exists(path), "no ptxas report for " + unit
        out[unit] = open(path).read()
    return out


def _kernel_name(mangled):
    """The ``*_kernel`` identifier inside an Itanium-mangled name, whose
    identifiers are written as <decimal length><characters>.  The length can
    follow digits of a hashed namespace name, so every suffix of a run of
    digits is tried as the length."""
    for m in re.finditer(r"\d+", mangled):
        run, start = m.group(0), m.end()
        for i in range(len(run)):
            n = int(run[i:])
            ident = mangled[start:start + n]
            if (len(ident) == n and ident.endswith("_kernel")
                    and re.fullmatch(r"[A-Za-z_]\w*", ident)):
                return ident
    return mangled


def _kernels(text):
    """(kernel name, registers, spill store bytes, spill load bytes) for every
    entry function of one report."""
    rows = []
    name = None
    spill = None
    for line in text.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            name = _kernel_name(m.group(1))
            spill = None
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and name:
            spill = (int(m.group(1)), int(m.group(2)))
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and name:
            rows.append((name, int(m.group(1))) + (spill or (0, 0)))
            name = None
    return rows


def test_every_unit_reports_its_kernels(reports):
    names = {k[0] for text in reports.values() for k in _kernels(text)}
    for must in ("layout_kernel", "notify_small_kernel", "dispatch_quant_kernel",
                 "dispatch_copy_kernel", "combine_kernel", "combine_quant_kernel",
                 "fused_dispatch_kernel", "grouped_gemm_kernel", "deq_combine_kernel"):
        assert must in names, must


def test_spill_budget(reports):
    over = []
    for unit, text in sorted(reports.items()):
        for name, regs, st, ld in _kernels(text):
            limit = SPILL_BYTES.get(name, 0)
            if st > limit:
                over.append("%s: %s spills %d bytes (%d registers), budget %d"
                            % (unit, name, st, regs, limit))
    assert not over, "\n".join(over)
