"""Every bf16 activation against every bf16 group maximum: the library's
group quantiser (compiled from its own device header) gives the code of the
definition, clamp(rint(x / sx), -7, 7) with sx = amax / 7 by IEEE division,
for all 1.05e9 pairs with |x| <= amax."""
import os
import shutil
import subprocess
import tempfile

import pytest

from gpuhelp import need_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_group_quantiser_exhaustive():
    need_gpu()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    src = os.path.join(ROOT, "tests", "cuda", "quant_exhaustive.cu")
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "quant_exhaustive")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(ROOT, "quantized_speculative_decoding_shared_gb300", "csrc"),
                        src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    fields = out.stdout.split()
    vals = dict(zip(fields[0::2], fields[1::2]))
    assert out.returncode == 0, out.stdout + out.stderr
    assert int(vals["pairs"]) > 1_000_000_000
    assert int(vals["code_mismatches"]) == 0 and int(vals["scale_mismatches"]) == 0, out.stdout
