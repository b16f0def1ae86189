"""The seeded input recipe shared by the tests, smoke and the benchmark: a
seed fixes every tensor, and the draws have the structure the recipe states
(unit q and k per token-head, gk <= 0, beta in (0, 1), lengths and counts in
their ranges, the acceptance-length mean of its closed form)."""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import kda_inputs as gen  # noqa: E402


def test_a_seed_fixes_every_tensor():
    a = gen.token_inputs(37, 3, torch.bfloat16, gen.make_gen(5))
    b = gen.token_inputs(37, 3, torch.bfloat16, gen.make_gen(5))
    c = gen.token_inputs(37, 3, torch.bfloat16, gen.make_gen(6))
    for n in a:
        assert torch.equal(a[n], b[n]) and not torch.equal(a[n], c[n])
    w1, w2 = gen.varlen_batch(H=2), gen.varlen_batch(H=2)
    assert w1["lengths"] == w2["lengths"] and torch.equal(w1["x"]["q"], w2["x"]["q"])


def test_token_input_structure():
    x = gen.token_inputs(500, 4, torch.float32, gen.make_gen(7))
    for n in ("q", "k"):
        nrm = x[n].double().norm(dim=-1)
        assert torch.allclose(nrm, torch.ones_like(nrm), atol=1e-6)
    assert x["q"].shape == (500, 4, 128) and x["v"].shape == (500, 4, 128)
    assert x["beta"].shape == (500, 4)
    assert (x["gk"] <= 0).all() and (x["gk"] > -30).all()
    assert ((x["beta"] > 0) & (x["beta"] < 1)).all()
    # -softplus(N(0, 1)) has mean about -0.806; sigmoid(N(0, 1)) mean 1/2
    assert abs(x["gk"].double().mean().item() + 0.806) < 0.02
    assert abs(x["beta"].double().mean().item() - 0.5) < 0.02
    xb = gen.token_inputs(50, 2, torch.bfloat16, gen.make_gen(7))
    assert all(t.dtype == torch.bfloat16 and t.is_contiguous() for t in xb.values())


def test_lengths_counts_and_slots():
    g = gen.make_gen(8)
    L = gen.varlen_lengths(400, 64, 2048, g)
    assert min(L) >= 64 and max(L) <= 2048
    cu = gen.cu_seqlens([3, 0, 5])
    assert cu.dtype == torch.int32 and cu.tolist() == [0, 3, 3, 8]
    d = gen.draft_lengths(1000, 8, g)
    assert d.min() >= 1 and d.max() <= 8
    p = gen.slot_permutation(128, g)
    assert sorted(p.tolist()) == list(range(128))
    a = gen.accept_lengths(200000, 8, 0.64, g)
    assert a.min() >= 1 and a.max() <= 8
    want = 1 + sum(0.64 ** i for i in range(1, 8))          # 2.70: 1 + run of accepts, capped
    assert abs(a.double().mean().item() - want) < 0.01


def test_checkpoint_scale():
    ck = gen.checkpoint((64, 128, 128), gen.make_gen(9))
    assert ck.dtype == torch.float32 and abs(ck.std().item() - 0.02) < 2e-4
