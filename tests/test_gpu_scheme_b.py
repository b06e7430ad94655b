"""Scheme B through the C ABI: chunks cached without position encoding, encoded at
their global positions by pic_rope_cached_k, against the float64 oracle (link_request with scheme "nope"):
in place, and out of place into private pages when chunks are shared."""

import numpy as np
import pytest
import torch

import oracle.pic_oracle as O
import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build
from position_independent_kv_pic_gb300 import inputs
from position_independent_kv_pic_gb300.link import LinkBatch

from parity_util import TOL_MAX, TOL_MEAN, check_attention, check_fresh_kv, check_rows, storage_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pic_build.build()
    pic.load()


def _run(wl):
    b = LinkBatch(wl, scheme="nope")
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0, pic.pic_strerror(b.error())
    return b


def _check_k(b):
    """Every kept cached K slot (chunk 0 included) within one ulp of the oracle's
    encoding at the global position."""
    wl = b.wl
    starts = b.chunk_start.cpu().numpy()
    for r, req in enumerate(wl.requests):
        c0, c1 = int(b.chunk_off[r]), int(b.chunk_off[r + 1])
        for ci, c in enumerate(range(c0, c1)):
            sid = int(b.flat_store_ids[c])
            stored = b.store_k[b.store_off[sid]:b.store_off[sid + 1]].double().numpy()
            got = b.rotated_chunk_k(c).double().numpy()
            m = 0 if ci == 0 else min(req.k, stored.shape[0])
            expect = O.rope_cached_k(stored, int(starts[c]), wl.theta, wl.dtype)
            ratio = (np.abs(got[m:] - expect[m:]) / storage_ulp(expect[m:], wl.dtype)).max() if m < len(stored) else 0
            assert ratio <= (1.0 if wl.dtype == "bf16" else 4.0), (r, ci, ratio)


def _check_attention(b):
    return check_attention(b, scheme="nope")


@pytest.mark.parametrize("preset", ["rag_prompt_6chunks", "many_chunk_sink_20", "long_context_100x1000"])
def test_scheme_b_workloads(preset):
    """Every kept cached slot, every fresh slot and every row of the workload."""
    b = _run(inputs.PRESETS[preset]())
    check_rows(b)
    _check_k(b)
    check_fresh_kv(b)
    emax, emean = _check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)


@pytest.mark.parametrize("case", [
    ([[300, 17, 1, 64, 129]], [37], [8]),
    ([[40, 50, 60]], [3], [40]),
    ([[130, 70], [55, 8, 200, 31]], [20, 1], [2, 16]),
])
def test_scheme_b_edge_cases(case):
    lens, qs, ks = case
    b = _run(inputs.custom(lens, qs, ks, Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=70 + len(lens)))
    check_rows(b)
    _check_k(b)
    check_fresh_kv(b)
    emax, emean = _check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)


def test_scheme_b_fp32_small():
    b = _run(inputs.custom([[21, 13, 40]], [6], [5], Hq=4, Hkv=2, d=32, theta=1e4, dtype="fp32", seed=77))
    _check_k(b)
    emax, emean = _check_attention(b)
    assert emax < 1e-4 and emean < 1e-5, (emax, emean)


def test_scheme_b_shared_chunks():
    """16 requests over a shared store: every chunk (the first too) is encoded at its
    global position into the request's private pages, against the oracle on every
    kept slot and every row; the shared sources stay as cached (un-encoded)."""
    b = _run(inputs.batched_shared())
    check_rows(b)
    _check_k(b)
    check_fresh_kv(b)
    emax, emean = _check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)
    for c, blocks in enumerate(b.store_blocks):
        L = int(b.wl.chunk_lens[c])
        j = np.arange(L)
        got = b.k_pool[torch.from_numpy(blocks[j // 16]).cuda(), :, torch.from_numpy(j % 16).cuda(), :].cpu()
        assert torch.equal(got, b.store_k[b.store_off[c]:b.store_off[c + 1]])
