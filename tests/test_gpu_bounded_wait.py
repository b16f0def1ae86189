"""The bounded-wait path on the GPU: a wait on a barrier that nothing arrives
at (a flag nothing sets) runs out after its limit, the kernel reports
KDA_DEVERR_TIMEOUT and returns, and the context stays usable -- a decode step
launched right after is bit-exact against one run on a fresh copy."""
import pytest
import torch

import kda_inputs as gen

pytestmark = pytest.mark.gpu
DEV = "cuda"
KD = VD = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_state_gb300 import _build
    _build.build()


def kda():
    import kda_state_gb300
    return kda_state_gb300


def test_wait_runs_out_and_context_stays_usable():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda().kda_selftest_bounded_wait(err, wait_us=2000)
    torch.cuda.synchronize()
    assert int(err.item()) == kda().KDA_DEVERR_TIMEOUT

    g = gen.make_gen(91)
    B, H, S = 4, 2, 6
    pool = gen.checkpoint((S, H, KD, VD), g).to(DEV)
    ref = pool.clone()
    x = {n: t.to(DEV) for n, t in gen.token_inputs(1, H, torch.bfloat16, g, lead=(B,)).items()}
    ids = torch.tensor([3, 0, 5, 1], dtype=torch.int32, device=DEV)
    args = [x[n][:, 0].contiguous() for n in ("q", "k", "v", "gk", "beta")]
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    o1 = kda().kda_decode_step(*args, ids, pool, dev_err=err2)
    o2 = kda().kda_decode_step(*args, ids, ref)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    assert torch.equal(o1, o2) and torch.equal(pool, ref)
