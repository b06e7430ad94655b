"""Decode after link: the CUDA decode step (through the C ABI) against the float64
oracle's decode_after_link over the oracle's own linked context, after a link by
the rotary correction and after a rotate-on-read link (whose pages keep every
chunk's keys in the chunk's frame)."""

import numpy as np
import pytest
import torch

import oracle.pic_oracle as O
import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build
from position_independent_kv_pic_gb300 import inputs
from position_independent_kv_pic_gb300.link import LinkBatch

from parity_util import TOL_MAX, TOL_MEAN, oracle_request

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pic_build.build()
    pic.load()


def _decode(wl, scheme="rotary"):
    b = LinkBatch(wl, scheme=scheme)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0, pic.pic_strerror(b.error())
    b.setup_decode()
    b.run_decode()
    torch.cuda.synchronize()
    assert b.error() == 0, pic.pic_strerror(b.error())
    return b


def _check(b, reqs):
    wl = b.wl
    got = b.dec_out.double().cpu().numpy()
    dq, dk, dv = (t.double().numpy() for t in inputs.decode_inputs(wl))
    errs = []
    for r in reqs:
        link = oracle_request(b, r, which=[])
        assert link["K_ctx"].shape[0] == b.dec_pos_h[r]
        expect = O.decode_after_link(link["K_ctx"], link["V_ctx"], dq[r], dk[r], dv[r], wl.theta, wl.dtype)
        errs.append(np.abs(got[r] - expect))
    e = np.concatenate([x.ravel() for x in errs])
    return float(e.max()), float(e.mean())


@pytest.mark.parametrize("scheme", ["rotary", "ror"])
@pytest.mark.parametrize("preset", ["rag_prompt_6chunks", "many_chunk_sink_20", "long_context_100x1000"])
def test_decode_single_request(preset, scheme):
    b = _decode(inputs.PRESETS[preset](), scheme)
    emax, emean = _check(b, [0])
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)


@pytest.mark.parametrize("scheme", ["rotary", "ror"])
def test_decode_batched(scheme):
    """Every request of the 16-request batch (shared chunks: rotated into private
    pages by the rotary correction, read in place by rotate-on-read)."""
    b = _decode(inputs.batched_shared(), scheme)
    emax, emean = _check(b, range(b.n_req))
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)


@pytest.mark.parametrize("n_req", [160, 170])
def test_decode_many_requests(n_req):
    """Up to 160 requests the decode CTAs split the work themselves; above, a planner
    launch writes their descriptors: both give every request its own decode."""
    rng = np.random.default_rng(n_req)
    lens = [[int(x) for x in rng.integers(1, 60, size=int(rng.integers(1, 4)))] for _ in range(n_req)]
    wl = inputs.custom(lens, [1] * n_req, [2] * n_req, Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=n_req)
    b = _decode(wl)
    emax, emean = _check(b, [0, n_req // 2, n_req - 1])
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)


@pytest.mark.parametrize("scheme", ["rotary", "ror"])
@pytest.mark.parametrize("Hq", [8, 16, 32, 64])
def test_decode_gqa_groups(Hq, scheme):
    wl = inputs.custom([[130, 70, 45], [55, 8, 200]], [20, 1], [2, 16], Hq=Hq, Hkv=8, d=128, theta=5e5,
                       dtype="bf16", seed=60 + Hq)
    b = _decode(wl, scheme)
    emax, emean = _check(b, [0, 1])
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)


def test_decode_unsupported_shape_is_refused():
    assert pic.pic_decode_workspace(1, 4, 2, 16, pic.PIC_FP32) == 0
    assert pic.pic_decode_workspace(1, 32, 8, 128, pic.PIC_BF16) > 0


def test_link_attention_on_decode_rows_repeated():
    """One row per request through the link attention kernel, many calls back to
    back (the shape that exposed the V-zeroing warps' parity wait on a slot's K
    phase): no error, the decode kernel's result, the same bits every call."""
    wl = inputs.batched_shared()
    b = LinkBatch(wl)
    b.run()
    b.setup_decode()
    b.run_decode()
    torch.cuda.synchronize()
    assert b.error() == 0
    row_off = torch.arange(b.n_req + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(pic.pic_link_attention_workspace(b.n_req, b.n_req, wl.Hq, wl.Hkv, wl.d, b.pic_dtype), 256),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(12):
        out = torch.empty_like(b.dec_out)
        pic.pic_link_attention(b.dec_q, b.dec_table, b.dec_pos, row_off, b.k_pool, b.v_pool, b.pic_dtype,
                               b.dec_pages, b.dec_page_off, b.n_req, b.n_req, wl.Hq, wl.Hkv, wl.d, b.scale, out, ws,
                               b.err)
        outs.append(out)
    torch.cuda.synchronize()
    assert b.error() == 0, pic.pic_strerror(b.error())
    assert all(torch.equal(o, outs[0]) for o in outs)
    assert (outs[0].float() - b.dec_out.float()).abs().max().item() <= 2e-3


def test_decode_bad_block_is_flagged_and_skipped():
    """A page whose V block id is past the pool is reported (PIC_ERR_RANGE) and not
    read; the call still ends (no wait runs out) and the other heads' pages are
    untouched by it."""
    wl = inputs.custom([[40, 50, 60]], [3], [4], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=97)
    b = _decode(wl)
    bad = b.dec_pages.clone()
    bad[1, 1] = b.num_blocks + 7
    good = b.dec_pages
    b.dec_pages = bad
    b.run_decode()
    torch.cuda.synchronize()
    assert b.error() == pic.PIC_ERR_RANGE
    assert torch.isfinite(b.dec_out.float()).all()
    b.dec_pages = good
    b.err.zero_()
    b.run_decode()
    torch.cuda.synchronize()
    assert b.error() == 0
