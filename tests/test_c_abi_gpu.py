"""The C ABI used from C alone: tests/c/decode_step.c plans and runs one decode
step through libpka.so (no Python in that process) and writes its inputs and
outputs; here they are compared with the fp64 oracle."""

import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    assert cc is not None, "a C compiler is needed to build the C-ABI test program"
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    lib = os.path.join(ROOT, "paged_kv_attention_32_gb300", "_lib")
    assert os.path.exists(os.path.join(lib, "libpka.so")), "build the library first"
    exe = str(tmp_path / "decode_step")
    subprocess.run([cc, "-std=c11", "-O1", os.path.join(ROOT, "tests", "c", "decode_step.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-L", lib, "-lpka", "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{lib}:{os.path.join(cuda, 'lib64')}", "-lm", "-o", exe],
                   check=True, capture_output=True, text=True)
    return exe


@pytest.mark.parametrize("hq,mma_min_rows,kernel", [(8, 16, 0), (8, 0, 1), (16, 0, 1)])
def test_decode_step_from_c(tmp_path, hq, mma_min_rows, kernel):
    """Groups of 4 and 8 rows on the tensor-core kernel (the default) and 4 rows on the
    CUDA-core one (mma_min_rows 16); 3 requests on a GB300 are split into chunks, so the
    in-kernel merge runs too."""
    exe = _build(tmp_path)
    r = subprocess.run([exe, str(tmp_path), str(hq), str(mma_min_rows)], capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    meta = dict(kv.split("=") for kv in r.stdout.split())
    B, Hkv, D, ps, C, P = (int(meta[x]) for x in ("B", "Hkv", "D", "ps", "C", "P"))
    assert int(meta["Hq"]) == hq and int(meta["kernel"]) == kernel
    assert int(meta["num_split"]) > 0

    def load(name, dtype, shape):
        return np.fromfile(str(tmp_path / name), dtype=dtype).reshape(shape)

    q = load("q.bin", np.uint16, (B, hq, D))
    k = load("k.bin", np.uint16, (P, Hkv, ps, D))
    v = load("v.bin", np.uint16, (P, Hkv, ps, D))
    tables = load("tables.bin", np.int32, (B, C))
    lens = load("lens.bin", np.int32, (B,))
    out_bits = load("out.bin", np.uint16, (B, hq, D))
    lse = load("lse.bin", np.float32, (B, hq))
    ref_o, ref_l = oracle.paged_decode(q, k, v, tables, lens, Hkv, ps, q_len=1)
    out = torch.from_numpy(out_bits.astype(np.int32) << 16).view(torch.float32)
    assert_close(out, torch.from_numpy(lse), ref_o, ref_l)
