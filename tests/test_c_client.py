"""The C ABI from plain C: a client compiled with gcc against include/fa.h and
linked to libfa.so (no Python, no torch in the client). On the CPU it checks
the host-side contract; on the GPU it also runs a forward pass whose values
are compared with the oracle."""
import os
import subprocess

import numpy as np
import pytest

from exact_io_aware_attention_gb300 import build as fa_build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def client(tmp_path):
    lib = fa_build.build()
    exe = str(tmp_path / "abi_client")
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(fa_build.nvcc())), "lib64")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O2",
           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "c", "abi_client.c"),
           "-o", exe, "-L", os.path.dirname(lib), "-lfa", f"-Wl,-rpath,{os.path.dirname(lib)}",
           "-L", cuda_lib, "-lcudart", f"-Wl,-rpath,{cuda_lib}", "-lm"]
    subprocess.check_call(cmd)
    return exe


def test_c_client_host_checks(tmp_path):
    out = subprocess.run([client(tmp_path)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert "host checks passed" in out.stdout


@pytest.mark.gpu
def test_c_client_forward_matches_the_oracle(tmp_path):
    import torch
    import oracle
    out = subprocess.run([client(tmp_path), "gpu"], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    o_129_5, lse_129, lse_0 = (float(x) for x in out.stdout.split())
    n, d = 130, 64
    idx = np.arange(n * d)
    mk = lambda scale, mul, mod, off: torch.tensor(
        scale * ((idx * mul) % mod - off), dtype=torch.float32).to(torch.bfloat16).double()
    q, k, v = (t.numpy().reshape(1, 1, n, d) for t in
               (mk(0.01, 7, 23, 11), mk(0.02, 5, 19, 9), mk(0.05, 3, 17, 8)))
    o_ref, lse_ref = oracle.forward(q, k, v, causal=True, scale=0.125)
    assert abs(o_129_5 - o_ref[0, 0, 129, 5]) <= 1e-2 * max(1.0, abs(o_ref[0, 0, 129, 5])) + 4e-3
    assert abs(lse_129 - lse_ref[0, 0, 129]) <= 1e-3
    assert abs(lse_0 - lse_ref[0, 0, 0]) <= 1e-3
