"""The allocation-free attention entry point, called through the C ABI.

pic_link_attention_noalloc serves callers that cannot allocate device memory
when they run the link step (an engine whose KV pool already holds nearly all of
HBM, or a plugin handed only device pointers by a framework that owns
allocation).  It must give what pic_link_attention gives, within the attention
tolerance, on repeated calls that reuse its fixed scratch.  This file is
collected last so a stop-at-first-failure run has already run everything else.
"""

import numpy as np
import pytest
import torch

import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build
from position_independent_kv_pic_gb300 import inputs
from position_independent_kv_pic_gb300.link import LinkBatch

from parity_util import TOL_MAX, TOL_MEAN

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pic_build.build()
    pic.load()


def _noalloc(b, out):
    wl, dv = b.wl, b.dev
    pic.pic_link_attention_noalloc(dv["q_raw"], b.row_table, b.rows, dv["row_off"], b.k_pool, b.v_pool,
                                   b.pic_dtype, b.pages, dv["page_off"], b.n_req, b.n_rows, wl.Hq, wl.Hkv,
                                   wl.d, b.scale, out, b.err)


WORKLOADS = [
    lambda: inputs.rag_prompt(),
    lambda: inputs.custom([[130, 70], [55, 8, 200, 31], [500]], [20, 1, 33], [2, 16, 8], Hq=32, Hkv=8, d=128,
                          theta=5e5, dtype="bf16", seed=77),
    lambda: inputs.custom([[2000, 3000, 1500]], [40], [8], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=78),
    lambda: inputs.worked_example(),
]


@pytest.mark.parametrize("case", range(len(WORKLOADS)))
def test_noalloc_matches_workspace_entry_point(case):
    b = LinkBatch(WORKLOADS[case]())
    b.run()                         # the existing entry point, with a caller workspace
    torch.cuda.synchronize()
    assert b.error() == 0
    ref = b.out.double().clone()
    for call in range(2):           # two calls in a row share the fixed scratch
        out = torch.full_like(b.out, float("nan"))
        b.err.zero_()
        _noalloc(b, out)
        torch.cuda.synchronize()
        assert b.error() == 0, pic.pic_strerror(b.error())
        diff = (out.double() - ref).abs()
        assert torch.isfinite(diff).all(), f"call {call}"
        tol = (1e-5, 1e-6) if b.wl.dtype == "fp32" else (TOL_MAX, TOL_MEAN)
        assert diff.max().item() <= tol[0] and diff.mean().item() <= tol[1], (call, diff.max().item())


def _refused(lib, n_rows, n_req=1):
    """Host-side answer for a call of n_rows rows with NULL pointers: the size check
    comes first, so PIC_ERR_WORKSPACE means over the limit, PIC_ERR_INVALID under."""
    return lib.pic_link_attention_noalloc(None, None, None, None, None, None, 10, pic.PIC_BF16, None, None,
                                          n_req, n_rows, 32, 8, 128, 0.1, None, None, None)


def _row_limit(lib):
    """Largest row count of one request that the fixed scratch takes (bisection)."""
    lo, hi = 1, 1 << 20
    assert _refused(lib, lo) == pic.PIC_ERR_INVALID and _refused(lib, hi) == pic.PIC_ERR_WORKSPACE
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _refused(lib, mid) == pic.PIC_ERR_WORKSPACE:
            hi = mid
        else:
            lo = mid
    return lo


def _compare(b, calls=2):
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    ref = b.out.double().clone()
    for call in range(calls):
        out = torch.full_like(b.out, float("nan"))
        b.err.zero_()
        _noalloc(b, out)
        torch.cuda.synchronize()
        assert b.error() == 0, pic.pic_strerror(b.error())
        diff = (out.double() - ref).abs()
        assert torch.isfinite(diff).all(), f"call {call}"
        assert diff.max().item() <= TOL_MAX and diff.mean().item() <= TOL_MEAN, (call, diff.max().item())


def test_noalloc_just_under_the_row_limit():
    """One request with as many rows as the scratch takes (its Q operands reach the
    array's deepest region) and a 30k-token context."""
    lib = pic.load()
    n = _row_limit(lib)
    assert n == 959, n  # the limit the header states for one request at Hq = 32, Hkv = 8
    # 30 chunks of 1000 tokens, k = 16: 29 * 16 seam rows + the query = n rows
    q = n - 29 * 16
    _compare(LinkBatch(inputs.custom([[1000] * 30], [q], [16], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16",
                                     seed=79)))


def test_noalloc_with_nearly_all_split_units():
    """One tile pair over a 60k-token context: split into about 60 extra units."""
    _compare(LinkBatch(inputs.custom([[50000, 10000]], [48], [16], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16",
                                     seed=80)))


def test_noalloc_refused_just_over_the_row_limit():
    lib = pic.load()
    n = _row_limit(lib)
    assert _refused(lib, n + 1) == pic.PIC_ERR_WORKSPACE
    assert _refused(lib, n) == pic.PIC_ERR_INVALID


def test_noalloc_warm_up_call_without_rows():
    """A call with no rows launches nothing and returns PIC_OK once the device code is
    loaded and the scratch address looked up."""
    lib = pic.load()
    for n_req, n_rows in ((0, 0), (1, 0)):
        assert lib.pic_link_attention_noalloc(None, None, None, None, None, None, 10, pic.PIC_BF16, None, None,
                                              n_req, n_rows, 32, 8, 128, 0.1, None, None, None) == pic.PIC_OK


def test_noalloc_refuses_calls_beyond_its_scratch():
    """A call needing more than PIC_NOALLOC_SCRATCH_BYTES is refused on the host,
    before its pointers are looked at and before any launch."""
    lib = pic.load()
    status = lib.pic_link_attention_noalloc(None, None, None, None, None, None, 10, pic.PIC_BF16, None, None,
                                            1, 10 ** 6, 32, 8, 128, 0.1, None, None, None)
    assert status == pic.PIC_ERR_WORKSPACE
    assert lib.pic_link_attention_noalloc(None, None, None, None, None, None, 10, pic.PIC_BF16, None, None,
                                          1, 100, 32, 8, 128, 0.1, None, None, None) == pic.PIC_ERR_INVALID
