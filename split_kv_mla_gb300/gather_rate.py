"""Gather-rate probe: the split kernel's row fetch run alone, by four copy mechanisms.

Compiles ``probes/gather_rate.cu`` for sm_103a into ``_build_probe/`` and runs
it.  One CTA per SM streams 128-row blocks of random 576-byte pool rows (two
blocks in flight, no compute) by TMA ``tile::gather4`` (the split kernel's
copies), by TMA for the latent boxes plus ``cp.async`` for the RoPE bytes, by
16-byte ``cp.async`` alone, and by one ``cp.async.bulk`` per row (a row-major
layout the tensor cores cannot read, shown as the copy engine's ceiling).  The
table it prints (CSV) bounds what the split kernel's fetch can deliver: at 128
CTAs and four blocks each (B=8, H=16, S=8192 with 16 splits) the gathers alone
take about as long as the whole split kernel.

    python -m split_kv_mla_gb300.gather_rate
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "probes", "gather_rate.cu")
OUT = os.path.join(HERE, "_build_probe")


def build() -> str:
    from split_kv_mla_gb300 import build as b
    os.makedirs(OUT, exist_ok=True)
    exe = os.path.join(OUT, "gather_rate")
    cmd = [b._nvcc(), *b.ARCH, "-O3", "-std=c++17", SRC, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed:\n{r.stdout}\n{r.stderr}")
    return exe


def main() -> int:
    exe = build()
    return subprocess.run([exe]).returncode


if __name__ == "__main__":
    sys.exit(main())
