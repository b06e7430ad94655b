"""Linear-layer state composition through the C ABI (pic_compose_states) against the
float64 oracle's compose_states, on small chains of every shape the two-level fold
produces and on the full long-context and batched chains."""

import numpy as np
import pytest
import torch

import oracle.pic_oracle as O
import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build
from position_independent_kv_pic_gb300 import inputs
from position_independent_kv_pic_gb300.states import ComposeBatch

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pic_build.build()
    pic.load()


def _pool(n, H, seed):
    wl = inputs.custom([[1] * n], [1], [0], seed=seed)
    T, S, _ = inputs.linear_states(wl, H=H, d=D)
    return T, S


def tolerance(n):
    """Error bound of a chain of n elements, relative to max |S_ref| over the chain's
    output.  Each fold step splits both factors into bf16 hi + lo (each part within
    2^-16 of its value, relative) and drops lo.lo: every product term T_mk X_kn
    carries a rounding error below about 3 * 2^-16 |T_mk||X_kn|.  Summed with one
    sign over the 128 terms of an entry that is at most 5 * 2^-16 of max |X| for
    these inputs (|T| rows sum to about 1.5), 10 * 2^-16 with the fp32 accumulation.
    The terms' rounding errors are independent with random signs, so their sum
    grows as sqrt(128) ~ 11 times one term rather than 128 times: one step's error
    stays below 2^-16 max |X| (the worst case divided by 10).  The error of step j
    reaches the output through the later transitions, whose norm is below 0.95,
    so the chain's error stays below sum_j 0.95^(n-1-j) <= min(n - 1, 20) steps'
    worth.  (HYPIC, section 2.1, reports the composed state within 6e-5 of a full
    recompute on a real model, inside FP16 noise; 2^-16 per step is 1.5e-5.)"""
    return max(min(n - 1, 20), 1) * 2.0 ** -16


def check(batch, T, S, chains):
    out = batch.out.double().cpu().numpy()
    Td, Sd = T.double().numpy(), S.double().numpy()
    worst = 0.0
    for r, ids in enumerate(chains):
        for h in range(batch.H):
            if len(ids) == 0:
                assert np.all(out[r, h] == 0.0)
                continue
            ref = O.compose_states(Td[ids, h], Sd[ids, h])
            err = np.abs(out[r, h] - ref).max() / np.abs(ref).max()
            worst = max(worst, err / tolerance(len(ids)))
            assert err <= tolerance(len(ids)), (r, h, len(ids), err, tolerance(len(ids)))
    return worst


CHAINS = [[], [4], [1, 2], [0, 1, 2, 3, 4], [5, 5, 3, 9, 0, 1, 7, 2, 6, 8, 4, 3, 3],
          list(np.random.default_rng(7).integers(0, 10, 40))]


@pytest.mark.parametrize("seg", [0, 2, 3, 5, 16, 40])
def test_small_chains(seg):
    T, S = _pool(10, 3, seed=11)
    b = ComposeBatch(T, S, CHAINS, seg=seg)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0, pic.pic_strerror(b.error())
    check(b, T, S, CHAINS)


def test_one_element_chain_is_a_copy():
    T, S = _pool(4, 2, seed=12)
    chains = [[3], [0], [2]]
    b = ComposeBatch(T, S, chains, seg=0)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    for r, ids in enumerate(chains):
        assert torch.equal(b.out[r].cpu(), S[ids[0]])


def test_segment_choice_and_two_levels():
    """The automatic choice folds the long chain in two launches and matches."""
    T, S = _pool(8, 4, seed=13)
    chains = [list(np.random.default_rng(3).integers(0, 8, 100))]
    b = ComposeBatch(T, S, chains)
    assert 1 < b.seg < 100 and b.launches == 2  # level 0 and level 1; the CTAs plan themselves
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    check(b, T, S, chains)


@pytest.mark.parametrize("n_req", [352, 360])
def test_many_requests(n_req):
    """Up to 352 requests the CTAs find their (request, head, segment) themselves;
    above, a planner launch writes the counts: both compose every chain."""
    T, S = _pool(6, 1, seed=16)
    rng = np.random.default_rng(n_req)
    chains = [list(rng.integers(0, 6, int(rng.integers(0, 5)))) for _ in range(n_req)]
    b = ComposeBatch(T, S, chains, seg=2)
    assert b.launches == (2 if n_req <= 352 else 3)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0, pic.pic_strerror(b.error())
    check(b, T, S, chains)


@pytest.mark.parametrize("preset", ["long_context_100x1000", "batched_shared_16req"])
def test_full_workloads(preset):
    wl = inputs.PRESETS[preset]()
    T, S, chains = inputs.linear_states(wl, H=32, d=D)
    b = ComposeBatch(T, S, chains)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0, pic.pic_strerror(b.error())
    worst = check(b, T, S, chains)
    print(f"{preset}: seg {b.seg}, worst error / bound {worst:.3f}")


def test_bad_id_is_flagged():
    T, S = _pool(4, 2, seed=14)
    b = ComposeBatch(T, S, [[0, 1], [2, 3]], seg=0)
    b.ids[3] = 7  # outside the pool of 4
    b.run()
    torch.cuda.synchronize()
    assert b.error() == pic.PIC_ERR_RANGE
    # the good chain is still composed
    ref = O.compose_states(T[[0, 1], 0].double().numpy(), S[[0, 1], 0].double().numpy())
    assert np.abs(b.out[0, 0].double().cpu().numpy() - ref).max() <= tolerance(2) * np.abs(ref).max()


def test_unsupported_head_dim():
    assert pic.pic_compose_workspace(1, 4, 2, 64, 0) == 0
    T = torch.zeros(2, 1, 64, 64, device="cuda")
    with pytest.raises(pic.PicError):
        pic.pic_compose_states(T, T, torch.zeros(2, dtype=torch.int32, device="cuda"),
                               torch.tensor([0, 2], dtype=torch.int32, device="cuda"), 1, 2, 2, 1, 64, 0,
                               torch.empty(1, 1, 64, 64, device="cuda"), torch.empty(256, dtype=torch.uint8,
                                                                                     device="cuda"),
                               torch.zeros(1, dtype=torch.int32, device="cuda"))


def test_split_t_is_the_bf16_hi_lo_pair():
    T, _ = _pool(3, 2, seed=15)
    Td = T.cuda()
    out = torch.empty((3, 2, 2, D, D), dtype=torch.bfloat16, device="cuda")
    pic.pic_compose_split_t(Td, out)
    torch.cuda.synchronize()
    hi = Td.to(torch.bfloat16)
    lo = (Td - hi.float()).to(torch.bfloat16)
    assert torch.equal(out[:, :, 0], hi) and torch.equal(out[:, :, 1], lo)
    rel = ((out[:, :, 0].double() + out[:, :, 1].double()) - Td.double()).abs() / Td.double().abs().clamp_min(1e-30)
    assert rel.max().item() <= 2.0 ** -16
