"""The bounds-checked debug build (TQ2_BOUNDS_CHECK): in a child process
that loads it, a sweep over tiny shapes (K in {256, 512, 768}, every N in
1..70, every M in 1..16, each kernel that takes the shape), the decoder
layer shapes at M = 1..16, grouped calls (one launch up to M = 16, and
consecutive calls), the affine-int4 kernel and the tcgen05 GEMM (narrow
tiles over split-K clusters, with and without the prologue pass) must report no out-of-buffer
index (TQ2_FLAG_BOUNDS clear) and match the oracle (tests/bounds_sweep.py).
The checks skip a bad access and set a flag; nothing traps."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.gpu
def test_bounds_checked_sweep():
    env = dict(os.environ, TQ2_BOUNDS_CHECK="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_sweep.py")], env=env, capture_output=True,
                       text=True, timeout=1200)
    print(r.stdout)
    assert r.returncode == 0, f"bounds sweep failed:\n{r.stdout[-3000:]}\n{r.stderr[-3000:]}"
    assert r.stdout.strip().endswith("OK")


def test_checked_library_exports_the_abi():
    """The debug library is built from the same sources and exports every
    symbol the header declares (no GPU needed)."""
    code = ("import quantized_gemv_tq2_gb300 as tq2; import quantized_gemv_tq2_gb300.build as b; "
            "L = tq2.load(); assert tq2.bounds_checked(); assert L._name == b.CHECK_LIB_PATH, L._name; "
            "missing = [n for n in tq2.declared_symbols() if not hasattr(L, n)]; assert not missing, missing; "
            "print('ok')")
    env = dict(os.environ, TQ2_BOUNDS_CHECK="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900,
                       cwd=os.path.dirname(HERE))
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
