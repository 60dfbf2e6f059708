"""Runs one named attention case through the library, for profilers.

``python -m exact_io_aware_attention_gb300.profile_case CASE [--steps K] [--warmup W]``
runs W + K forward and backward calls of CASE on cuda:0 with seeded inputs
(the generator of ``inputs.py``) and exits 0, so that a profiler can capture
kernels that the benchmark's workload does not launch:

  decode_n65536     B1 H16, one query against 65536 keys, d=128, causal: the
                    split forward and its merge kernel (fa_fwd_combine)
  d256_causal       B4 H8 N4096 d=256 causal: the head-dimension-256 kernels
  block_sparse      B4 H16 N8192 d=64, the 128x128 block mask kept with
                    p=0.25 (diagonal kept)
  gpt2_small        B8 H12 N1024 d=64 causal
"""
from __future__ import annotations

import argparse

CASES = {
    #              B   H   Nq     Nk     d    causal sparse
    "decode_n65536": (1, 16, 1, 65536, 128, True, None),
    "d256_causal": (4, 8, 4096, 4096, 256, True, None),
    "block_sparse": (4, 16, 8192, 8192, 64, False, 0.25),
    "gpt2_small": (8, 12, 1024, 1024, 64, True, None),
}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--steps", type=int, default=1)
    ap.add_argument("--warmup", type=int, default=3)
    a = ap.parse_args(argv)

    import torch

    import exact_io_aware_attention_gb300 as fa
    from exact_io_aware_attention_gb300 import inputs as gen

    B, H, Nq, Nk, d, causal, density = CASES[a.case]
    x = gen.make_inputs(B, H, Nq, d, case=900, Nk=Nk)
    q, k, v, do = (x[t].cuda() for t in ("q", "k", "v", "do"))
    mask = None
    if density is not None:
        mask = gen.block_mask(Nq // gen.TILE, density, seed=904).cuda()
    for _ in range(a.warmup + a.steps):
        o, lse = fa.forward(q, k, v, causal=causal, block_mask=mask)
        fa.backward(q, k, v, o, do, lse, causal=causal, block_mask=mask)
    torch.cuda.synchronize()
    if fa.device_status() != 0:
        raise SystemExit("a kernel-side wait gave up")


if __name__ == "__main__":
    main()
