"""The Python binding's argument checks on the device: a tensor of the wrong
dtype, shape or layout, a ring of the wrong shape, or a missing dev_err
element raises before anything is launched, and the state pool is left as it
was.  (The C entry points take bare pointers and cannot see any of this.)"""
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, K = 2, 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from kda_state_gb300 import _build
    _build.build()


def kda():
    import kda_state_gb300
    return kda_state_gb300


def _inputs(lead, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(5)
    x = {n: torch.randn(*lead, H, K, generator=g).to(dtype).to(DEV) for n in ("q", "k", "v", "gk")}
    x["beta"] = torch.rand(*lead, H, generator=g).to(dtype).to(DEV)
    return x


def test_prefill_argument_checks():
    T = 70
    x = _inputs((T,))
    cu_h = torch.tensor([0, 30, T], dtype=torch.int32)
    cu = cu_h.to(DEV)
    ids = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    pool = torch.randn(3, H, K, K, device=DEV)
    before = pool.clone()
    call = lambda **kw: kda().kda_chunk_prefill(**{**dict(q=x["q"], k=x["k"], v=x["v"], gk=x["gk"],
                                                         beta=x["beta"], cu_seqlens=cu,
                                                         cu_seqlens_host=cu_h, state_pool=pool,
                                                         init_slot=ids, out_slot=ids), **kw})
    with pytest.raises(TypeError, match="k has dtype"):
        call(k=x["k"].float())
    with pytest.raises(ValueError, match="must be contiguous"):
        call(q=x["q"].transpose(0, 1).contiguous().transpose(0, 1))
    with pytest.raises(ValueError, match="beta has shape"):
        call(beta=x["beta"][:, :1].contiguous())
    with pytest.raises(TypeError, match="state_pool has dtype"):
        call(state_pool=pool.to(torch.bfloat16))
    with pytest.raises(TypeError, match="init_slot has dtype"):
        call(init_slot=ids.long())
    with pytest.raises(ValueError, match="cu_seqlens has shape"):
        call(cu_seqlens=cu[:2].contiguous())
    with pytest.raises(ValueError, match="o has shape"):
        call(o=torch.empty(T, H, K + 1, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError, match="dev_err needs at least one element"):
        call(dev_err=torch.empty(0, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(pool, before)
    call()                              # the same call, well formed, runs
    torch.cuda.synchronize()


def test_decode_verify_fold_argument_checks():
    B, G = 3, 4
    pool = torch.randn(4, H, K, K, device=DEV)
    before = pool.clone()
    ids = torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV)
    x = _inputs((B,))
    with pytest.raises(ValueError, match="slot_ids has shape"):
        kda().kda_decode_step(x["q"], x["k"], x["v"], x["gk"], x["beta"], ids[:2], pool)
    xv = _inputs((B, G))
    ring = kda().make_ring(4, 8, H)
    bad = kda().make_ring(4, 8, H + 1)
    with pytest.raises(ValueError, match="ring.k has shape"):
        kda().kda_verify_store_inputs(xv["q"], xv["k"], xv["v"], xv["gk"], xv["beta"], ids, pool, bad)
    with pytest.raises(TypeError, match="ring.k has dtype"):
        kda().kda_verify_store_inputs(xv["q"], xv["k"], xv["v"], xv["gk"], xv["beta"], ids, pool,
                                      kda().make_ring(4, 8, H, dtype=torch.float32))
    acc = torch.tensor([1, 2, 3], dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError, match="accept_len has shape"):
        kda().kda_replay_fold([pool], [ring], ids, acc[:1], max_accept=G)
    with pytest.raises(ValueError, match="state_pools\\[1\\] has shape"):
        kda().kda_replay_fold([pool, pool[:2]], [ring, ring], ids, acc, max_accept=G)
    torch.cuda.synchronize()
    assert torch.equal(pool, before)
