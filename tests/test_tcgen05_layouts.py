"""GPU check of the tcgen05 building blocks (descriptors, TMEM operand packing) that the
tensor-core chunk kernels rely on: every operand layout they use, against torch.matmul."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    from gated_delta_rule_07_gb300 import build
    out = tmp_path_factory.mktemp("probe") / "libprobe.so"
    subprocess.run([build.nvcc(), "-O2", "-std=c++17", *build.ARCH, "-Xcompiler", "-fPIC",
                    "-shared", f"-I{build.CSRC}", f"-I{build.INCLUDE}",
                    os.path.join(HERE, "probes", "tcgen05_layouts.cu"), "-o", str(out)],
                   check=True)
    lib = ctypes.CDLL(str(out))
    lib.probe_run.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p] * 4
    return lib


# (name, N, K, a_src, b_mn, a_cap, b_cap, b_roff) -- the layouts of the chunk kernels
CASES = [
    ("SQ: K-major A and B, K=128, B in a 128-row tile", 64, 128, 0, 0, 128, 128, 0),
    ("WU: MN-major A (128-row blocks), K-major B", 64, 64, 1, 0, 128, 64, 0),
    ("delta: TMEM A, MN-major B, K=128", 64, 128, 2, 1, 128, 128, 0),
    ("O1: TMEM A, K-major B at row 64 of a 128-row tile", 64, 128, 2, 0, 128, 128, 64),
    ("O2: TMEM A, K-major B", 64, 64, 2, 0, 128, 64, 0),
    ("Dh: TMEM A, MN-major B, N=128 over two blocks", 128, 64, 2, 1, 128, 128, 0),
    ("plain K-major, K=64", 64, 64, 0, 0, 128, 64, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mma_layout(probe, case):
    name, N, K, a_src, b_mn, a_cap, b_cap, b_roff = case
    g = torch.Generator(device="cuda").manual_seed(1)
    A = torch.randn(128, K, device="cuda", generator=g).half()
    B = torch.randn(K, N, device="cuda", generator=g).half()
    D = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.probe_run(N, K, a_src, b_mn, a_cap, b_cap, b_roff, A.data_ptr(), B.data_ptr(),
                         D.data_ptr(), st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    ref = A.float() @ B.float()
    err = (D - ref).abs().max().item()
    assert err < 1e-2, f"{name}: max error {err}"
