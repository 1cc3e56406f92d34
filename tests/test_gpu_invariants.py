"""Invariants of the packed forward on the GPU, through the C ABI.

Splitting a sequence across a context-parallel group must not change what the
model computes ("Scaling video training with parallelism", opening section),
and packed samples stay independent of one another (Dynamic-CP article,
dynamic rescheduling and packing, Fig. 1).  So on one seeded ragged batch:

* cpattn_fwd gives the oracle's result for every virtual CP size and split
  (cp = 1, 2, 4, 8; zigzag and contiguous), element by element, and the
  results agree with one another;
* changing the keys and values of the other sequences leaves a sequence's
  O and LSE bit-identical;
* changing the keys and values after position p leaves every query at
  position <= p bit-identical (causality).
"""

import itertools

import numpy as np
import pytest
import torch

import inputs
from oracle import attention as A
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

# ragged lengths (57 ... 1390), every one >= 2*8 so cp = 8 zigzag is defined
CU = (0, 57, 357, 614, 1214, 1300, 2690)
H, HKV, D = 8, 2, 128


@pytest.fixture(scope="module")
def cp():
    import context_attention_cpattn_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    m.build()
    m.lib()
    return m


@pytest.fixture(scope="module")
def batch():
    w = inputs.custom(CU, H, HKV, D, dtype="bf16", causal=True, mode="zigzag", cp=1)
    (q, k, v), dev = U.device_inputs(w)
    O, L = A.packed_attention(q, k, v, CU, True, w.scale)
    return w, (q, k, v), dev, (O, L)


def _fwd(cp, w, dev, cps, mode):
    plan = cp.cpattn_plan(CU, cps, mode)
    return U.run_fwd(cp, plan, w, *dev)


def test_every_cp_size_and_split_gives_the_oracle_result(cp, batch):
    w, _, dev, (O, L) = batch
    results = {}
    for mode in ("zigzag", "contiguous"):
        for cps in (1, 2, 4, 8):
            o, lse = _fwd(cp, w, dev, cps, mode)
            U.check(o, lse, O, L, "bf16", f"{mode} cp={cps}")
            results[(mode, cps)] = (o, lse)
    # and with one another: each pair within the same bounds, with each
    # other's output in place of the oracle's
    for (ka, (oa, la)), (kb, (ob, lb)) in itertools.combinations(results.items(), 2):
        U.check(oa, la, ob.to("cpu", torch.float64).numpy(), lb.to("cpu", torch.float64).numpy(), "bf16",
                f"{ka} vs {kb}")


@pytest.mark.parametrize("mode,cps", [("zigzag", 4), ("contiguous", 3), ("zigzag", 8)])
def test_other_sequences_do_not_leak(cp, batch, mode, cps):
    """New values in every other sequence's K and V leave the sequence's rows
    bit-identical."""
    w, _, (qd, kd, vd), _ = batch
    plan = cp.cpattn_plan(CU, cps, mode)
    o_ref, l_ref = U.run_fwd(cp, plan, w, qd, kd, vd)
    g = torch.Generator(device="cuda").manual_seed(7)
    for s in range(len(CU) - 1):
        a, b = CU[s], CU[s + 1]
        k2, v2 = kd.clone(), vd.clone()
        other = torch.ones(w.T, dtype=torch.bool, device="cuda")
        other[a:b] = False
        k2[other] = (3 * torch.randn(int(other.sum()), HKV, D, device="cuda", generator=g)).to(kd.dtype)
        v2[other] = (3 * torch.randn(int(other.sum()), HKV, D, device="cuda", generator=g)).to(vd.dtype)
        o, l = U.run_fwd(cp, plan, w, qd, k2, v2)
        assert torch.equal(o[a:b], o_ref[a:b]), f"sequence {s}: O changed"
        assert torch.equal(l[:, a:b], l_ref[:, a:b]), f"sequence {s}: LSE changed"
        assert not torch.equal(o[other], o_ref[other])   # the perturbation did reach the others


@pytest.mark.parametrize("mode,cps", [("zigzag", 4), ("contiguous", 3), ("zigzag", 8)])
def test_future_keys_do_not_leak(cp, batch, mode, cps):
    """New values in K and V after position p of a sequence leave every
    query at position <= p bit-identical."""
    w, _, (qd, kd, vd), _ = batch
    plan = cp.cpattn_plan(CU, cps, mode)
    o_ref, l_ref = U.run_fwd(cp, plan, w, qd, kd, vd)
    g = torch.Generator(device="cuda").manual_seed(11)
    rng = np.random.default_rng(3)
    for s in (1, 3, 5):
        a, b = CU[s], CU[s + 1]
        for p in sorted(rng.choice(b - a - 1, size=3, replace=False)):
            cut = a + int(p) + 1                       # tokens [cut, b) are after position p
            k2, v2 = kd.clone(), vd.clone()
            k2[cut:b] = (3 * torch.randn(b - cut, HKV, D, device="cuda", generator=g)).to(kd.dtype)
            v2[cut:b] = (3 * torch.randn(b - cut, HKV, D, device="cuda", generator=g)).to(vd.dtype)
            o, l = U.run_fwd(cp, plan, w, qd, k2, v2)
            assert torch.equal(o[:cut], o_ref[:cut]), f"sequence {s}, p={p}: O before the cut changed"
            assert torch.equal(l[:, :cut], l_ref[:, :cut]), f"sequence {s}, p={p}: LSE before the cut changed"
            assert torch.equal(o[b:], o_ref[b:]) and torch.equal(l[:, b:], l_ref[:, b:])
