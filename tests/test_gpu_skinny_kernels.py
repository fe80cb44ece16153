"""Every decode-shaped kernel against the oracle at every M it can serve.

The library picks the decode kernel of gemv.cuh for M <= 16 and the tcgen05
skinny kernel for 17 <= M <= 32.  TERNARY_SKINNY_IMPL forces the tcgen05 kernel
(tc) or the older warp-MMA kernel (mma) for every M <= 32; it is read once per
process, so each choice runs in a child process of its own.
"""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys, torch
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import oracle
    import ternary_weight_linear_02_gb300 as tl
    from ternary_weight_linear_02_gb300 import synth
    from parity import check, oracle_ref
    tl.build(); oracle.build(); tl.load()
    cases = [
        (1, 200, 320, torch.bfloat16, 0, torch.float32),
        (1, 131, 2048, torch.float16, 128, torch.float32),
        (2, 257, 4096, torch.bfloat16, 0, torch.bfloat16),
        (2, 96, 1024, torch.bfloat16, 128, torch.float32),
        (5, 300, 1152, torch.float16, 0, torch.float16),
        (16, 129, 11008, torch.bfloat16, 0, torch.float32),
        (20, 75, 1536, torch.bfloat16, 128, torch.float32),
        (32, 4100, 512, torch.float16, 128, torch.float32),
    ]
    for M, N, K, xdt, gs, odt in cases:
        x, p, s = synth.layer(M, N, K, xdt, gs, 0.005, 0.05, ("impl", M, N, K, gs), "cpu", 0.01)
        x, p, s = x.cuda(), p.cuda(), s.cuda()
        y = tl.linear(x, p, s, gs, out_dtype=odt, path="skinny")
        torch.cuda.synchronize()
        check(y, oracle_ref(x, p, s, gs), x, s, what=f"{{M}}x{{N}}x{{K}} gs={{gs}}")
        assert tl.device_status() == 0
    print("ok")
""")


@pytest.mark.parametrize("impl", ["auto", "tc", "mma"])
def test_skinny_kernel_forced(impl):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, TERNARY_SKINNY_IMPL=impl)
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
