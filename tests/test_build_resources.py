"""Resource use of the kernels on the measured path, from ptxas's own report of
this build (CPU: nvcc cross-compiles for sm_103a): the sources compile without
warnings (device code, and host code under -Wall -Wextra), and the GEMM, dGLU
and NVFP4 cast instantiations that the forward and backward time keep every
value in registers (no spill stores or loads)."""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from mxfp8_nvfp4_block_gb300 import build as B  # noqa: E402

# demangled instantiations: gemm_kernel<format, epilogue, CTAs per tile, X4 scales, extra outputs>
SPILL_FREE = [
    "gemm_kernel<0, 0, 1, false, false>",   # MXFP8 fc1 + SwiGLU + requant
    "gemm_kernel<0, 1, 1, false, false>",   # MXFP8 fc1 + SReLU + requant
    "gemm_kernel<0, 2, 1, false, false>",   # MXFP8 fc2 and the fc1 dgrad
    "gemm_kernel<0, 4, 1, false, false>",   # MXFP8 fc2 dGLU (SwiGLU)
    "gemm_kernel<0, 5, 1, false, false>",   # MXFP8 fc2 dGLU (SReLU)
    "gemm_kernel<1, 1, 1, true, false>",    # NVFP4 fc1 + SReLU + amaxes
    "gemm_kernel<1, 2, 1, true, false>",    # NVFP4 fc2
    "row_quant_kernel<1, true>",            # NVFP4 casts (x, fc2_x)
    "row_quant_kernel<0, true>",            # MXFP8 casts (x, dy)
    "rowcol_quant_kernel<true, true, true, true>",    # NVFP4 row + column (RHT) cast, GEMM_TILED row scales
    "rowcol_quant_kernel<true, true, false, true>",   # the same, compact row scales
    "rowcol_quant_kernel<false, true, false, true>",  # column (RHT) only
    "rowcol_quant_kernel<true, true, true, false>",   # forward fc2_x: rowwise + post-RHT amax
    "colq_kernel<0>", "colq_kernel<1>", "colq_kernel<2>",
]


@pytest.fixture(scope="module")
def ptxas_report(tmp_path_factory):
    out_dir = tmp_path_factory.mktemp("ptxas")
    procs = []
    for src in B.SOURCES:
        cmd = [B.nvcc()] + B.ARCH + B.FLAGS + ["-Xptxas", "-v", "-c", os.path.join(B.CSRC, src), "-o",
                                               str(out_dir / src.replace(".cu", ".o"))]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    reports = {}
    for src, p in procs:
        text, _ = p.communicate(timeout=600)
        assert p.returncode == 0, text.decode(errors="replace")[-3000:]
        reports[src] = text.decode(errors="replace")
    return reports


def per_kernel(reports):
    """{demangled kernel name: (registers, spill store bytes, spill load bytes)}"""
    info = {}
    for text in reports.values():
        name = None
        spill = None
        for line in text.splitlines():
            m = re.search(r"Compiling entry function '([^']+)'", line)
            if m:
                name = subprocess.run(["c++filt", m.group(1)], capture_output=True, text=True).stdout.strip()
                name = name.replace("gmlp::(anonymous namespace)::", "").replace("gmlp::", "")
                name = re.sub(r"^void ", "", name.split("(")[0])
                continue
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m and name:
                spill = (int(m.group(1)), int(m.group(2)))
            m = re.search(r"Used (\d+) registers", line)
            if m and name:
                info[name] = (int(m.group(1)),) + (spill or (0, 0))
                name, spill = None, None
    return info


def test_sources_compile_without_warnings(ptxas_report):
    for src, text in ptxas_report.items():
        assert "warning" not in text, (src, [ln for ln in text.splitlines() if "warning" in ln])


def test_measured_kernels_do_not_spill(ptxas_report):
    info = per_kernel(ptxas_report)
    for k in SPILL_FREE:
        assert k in info, (k, sorted(info))
        regs, st, ld = info[k]
        assert st == 0 and ld == 0, (k, info[k])
    # the GEMM's 576 threads at one CTA per SM cap it at 96 registers a thread
    assert max(v[0] for k, v in info.items() if k.startswith("gemm_kernel")) <= 96
