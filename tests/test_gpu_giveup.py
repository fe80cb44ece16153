"""The decode kernel's bounded waits give up cleanly.

ternary_test_set_wait_limit makes the next launches first wait on a barrier
that nothing arrives on, with a short give-up time.  The wait runs out (no
fault, no hang): the call returns, the device status word reads
TL_ERR_TIMEOUT, no output is written, every copy in flight has landed and
every cluster barrier has been joined -- so the next normal call on the same
device is correct and leaves the status word clear.
"""
import pytest
import torch

import oracle
import ternary_weight_linear_02_gb300 as tl
from ternary_weight_linear_02_gb300 import synth

from parity import check, check_silu, oracle_ref, silu_refs

pytestmark = pytest.mark.gpu

DEV = "cuda"
TL_ERR_TIMEOUT = 7


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tl.build()
    oracle.build()
    tl.load()
    yield
    tl.load().ternary_test_set_wait_limit(0, 0)


# shapes the decode kernel serves (64-wide groups and the 11008-row layer at
# M = 1 stay on it; the dispatch sends other M > 8 calls to the tcgen05 kernel)
@pytest.mark.parametrize("M,N,K,gs", [(4, 4096, 4096, 64),   # split K: cluster barriers
                                      (1, 11008, 4096, 128),  # no split K, group scales
                                      (16, 300, 18944, 64)])  # two token tiles, split K
def test_wait_gives_up_then_recovers(M, N, K, gs):
    lib = tl.load()
    x, p, s = synth.layer(M, N, K, torch.bfloat16, gs, 0.005, 0.05, ("giveup", M, N, K), DEV)
    out = torch.full((M, N), 123.0, dtype=torch.float32, device=DEV)
    tl.linear(x, p, s, gs, out=out, out_dtype=torch.float32)  # creates the status word
    torch.cuda.synchronize()
    assert tl.device_status(clear=True) == 0
    out.fill_(123.0)
    lib.ternary_test_set_wait_limit(1 << 16, 1)  # ~30 us, and a wait nothing satisfies
    try:
        tl.linear(x, p, s, gs, out=out, out_dtype=torch.float32, static_weights=True)
        torch.cuda.synchronize()
    finally:
        lib.ternary_test_set_wait_limit(0, 0)
    assert tl.device_status(clear=True) == TL_ERR_TIMEOUT
    assert torch.all(out == 123.0)  # a call whose wait gave up writes nothing
    y = tl.linear(x, p, s, gs, out_dtype=torch.float32, static_weights=True)
    torch.cuda.synchronize()
    assert tl.device_status(clear=True) == 0
    rows = torch.arange(0, N, max(1, N // 64)).numpy()
    check(y[:, rows], oracle_ref(x, p, s, gs, rows=rows), x, s, rows=rows, what="after give-up")


def test_gated_wait_gives_up_then_recovers():
    lib = tl.load()
    M, N, K = 4, 1000, 8192
    x, p, s = synth.layer(M, 2 * N, K, torch.bfloat16, 0, 0.005, 0.05, ("giveup", "silu"), DEV)
    h = torch.full((M, N), 5.0, dtype=torch.float32, device=DEV)
    lib.ternary_test_set_wait_limit(1 << 16, 1)
    try:
        tl.linear_silu_mul(x, p, s, 0, out=h, out_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        lib.ternary_test_set_wait_limit(0, 0)
    assert tl.device_status(clear=True) == TL_ERR_TIMEOUT
    assert torch.all(h == 5.0)
    h = tl.linear_silu_mul(x, p, s, 0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tl.device_status(clear=True) == 0
    h_ref, g_ref, u_ref = silu_refs(x, p, s, 0)
    check_silu(h, h_ref, g_ref, u_ref, x, s, what="gated, after give-up")


def test_async_status_reports_the_give_up():
    lib = tl.load()
    x, p, s = synth.layer(2, 512, 2048, torch.bfloat16, 0, 0.005, 0.05, ("giveup", "async"), DEV)
    dst = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.ternary_test_set_wait_limit(1 << 16, 1)
    try:
        tl.linear(x, p, s, 0)
        tl.device_status_async(dst, clear=True)
        torch.cuda.synchronize()
    finally:
        lib.ternary_test_set_wait_limit(0, 0)
    assert int(dst.item()) == TL_ERR_TIMEOUT
    assert tl.device_status(clear=False) == 0  # cleared by the async read
