"""Which tcgen05.mma kinds assemble for sm_103a (compile only, CPU).

The expert-grouped GEMM runs its exact integer block dots as kind::f16 MMAs
(every operand a small integer, exact in fp16).  This records why: ptxas
rejects kind::i8 for sm_103a (and accepts it for sm_100a), while kind::f16
and kind::f8f6f4 assemble for sm_103a."""

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
PROBE = os.path.join(HERE, "probes", "tcgen05_mma_kinds.cu")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    pytest.skip("nvcc not found")


def _assemble(arch, kind, tmp_path):
    out = tmp_path / f"{arch}_{kind}.o"
    r = subprocess.run([_nvcc(), "-gencode", f"arch=compute_{arch},code=sm_{arch}", f"-DPROBE_{kind}", "-c", PROBE,
                        "-o", str(out)], capture_output=True, text=True)
    return r.returncode, r.stderr


def test_kind_i8_is_rejected_on_sm_103a(tmp_path):
    rc, err = _assemble("103a", "I8", tmp_path)
    assert rc != 0
    assert "kind::i8" in err and "sm_103a" in err


def test_kind_i8_assembles_on_sm_100a(tmp_path):
    rc, err = _assemble("100a", "I8", tmp_path)
    assert rc == 0, err


@pytest.mark.parametrize("kind", ["F16", "F8F6F4"])
def test_kinds_that_assemble_on_sm_103a(tmp_path, kind):
    rc, err = _assemble("103a", kind, tmp_path)
    assert rc == 0, err
