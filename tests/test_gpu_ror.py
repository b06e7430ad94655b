"""Rotate-on-read through the C ABI: the cached K pages stay at local positions and
pic_link_attention_ror rotates them inside the attention kernel.  Its K is, by
construction, the re-rotation pass's K, so its output must equal the rotary
correction path's output bit for bit; it is also checked against the float64
oracle directly, and the cached pages must come out of the step untouched."""

import numpy as np
import pytest
import torch

import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build
from position_independent_kv_pic_gb300 import inputs
from position_independent_kv_pic_gb300.link import LinkBatch

from parity_util import TOL_MAX, TOL_MEAN, check_attention, oracle_request

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pic_build.build()
    pic.load()


def _pair(wl):
    """The same link step by the rotary correction and by rotate-on-read."""
    rot = LinkBatch(wl, scheme="rotary")
    ror = LinkBatch(wl, scheme="ror", rows_inputs=(rot.q_raw_h, rot.k_new_h, rot.v_new_h))
    rot.run()
    ror.run()
    torch.cuda.synchronize()
    assert rot.error() == 0, pic.pic_strerror(rot.error())
    assert ror.error() == 0, pic.pic_strerror(ror.error())
    return rot, ror


def _cached_pages_untouched(b):
    """Every cached chunk's K is still as compiled after a rotate-on-read step."""
    for sid, blocks in enumerate(b.store_blocks):
        L = int(b.wl.chunk_lens[sid])
        j = np.arange(L)
        blk = torch.from_numpy(blocks[j // 16].astype(np.int64)).to(b.device)
        got = b.k_pool[blk, :, torch.from_numpy(j % 16).to(b.device), :].cpu()
        assert torch.equal(got, b.store_k[b.store_off[sid]:b.store_off[sid + 1]]), f"cached chunk {sid} written"


@pytest.mark.parametrize("preset", ["rag_prompt_6chunks", "many_chunk_sink_20", "long_context_100x1000",
                                    "batched_shared_16req"])
def test_bit_identical_to_rerotation(preset):
    rot, ror = _pair(inputs.PRESETS[preset]())
    assert torch.equal(ror.out, rot.out)
    _cached_pages_untouched(ror)


def test_page_tab_marks_cached_pages_after_the_first_chunk():
    b = LinkBatch(inputs.batched_shared(), scheme="ror")
    b.run()
    torch.cuda.synchronize()
    tab = b.page_tab.cpu().numpy()
    pages = b.pages.cpu().numpy()
    starts = b.chunk_start.cpu().numpy()
    src = set(b.k_src.tolist())
    po = b.offs["page_off"]
    for r in range(b.n_req):
        c0 = int(b.chunk_off[r])
        for p in range(int(po[r]), int(po[r + 1])):
            t = int(tab[p])
            if t < 0:
                continue
            # a cached page of a later chunk of this request, at that chunk's offset
            assert c0 < t < int(b.chunk_off[r + 1])
            assert int(pages[p, 0]) in src
            assert (int(pages[p, 2]) - int(starts[t])) % 16 == 0
    n_rotating = int((tab >= 0).sum())
    assert n_rotating == b.n_rot  # one page per entry the re-rotation pass would have run


@pytest.mark.parametrize("case", [
    ([[300, 17, 1, 64, 129]], [37], [8]),
    ([[40, 50, 60]], [3], [40]),
    ([[130, 70], [55, 8, 200, 31]], [20, 1], [2, 16]),
])
def test_edge_cases_against_oracle(case):
    lens, qs, ks = case
    wl = inputs.custom(lens, qs, ks, Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=90 + len(lens))
    rot, ror = _pair(wl)
    assert torch.equal(ror.out, rot.out)
    out = ror.out.double().cpu().numpy()
    errs = []
    for r in range(ror.n_req):
        a, e = int(ror.offs["row_off"][r]), int(ror.offs["row_off"][r + 1])
        res = oracle_request(ror, r)
        errs.append(np.abs(out[a:e] - res["out"]).ravel())
    x = np.concatenate(errs)
    assert x.max() <= TOL_MAX and x.mean() <= TOL_MEAN, (x.max(), x.mean())


def test_rag_prompt_against_oracle():
    wl = inputs.rag_prompt()
    b = LinkBatch(wl, scheme="ror")
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    emax, emean = check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)


def test_bad_table_row_is_flagged():
    wl = inputs.custom([[40, 50, 60]], [3], [4], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=95)
    b = LinkBatch(wl, scheme="ror")
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    t = b.page_tab.clone()
    rotating = torch.nonzero(t >= 0).flatten()
    assert len(rotating) > 0
    # run the attention alone with one page pointing past the table
    b.page_tab[rotating[0]] = b.n_chunks + 3
    pic.pic_link_attention_ror(b.dev["q_raw"], b.row_table, b.rows, b.dev["row_off"], b.k_pool, b.v_pool,
                               b.pic_dtype, b.pages, b.page_tab, b.delta_table, b.dev["page_off"], b.n_req,
                               b.n_rows, wl.Hq, wl.Hkv, wl.d, b.scale, b.out, b.ws, b.err)
    torch.cuda.synchronize()
    assert b.error() == pic.PIC_ERR_RANGE


def test_unsupported_shapes():
    wl = inputs.custom([[21, 13, 40]], [6], [5], Hq=4, Hkv=2, d=32, theta=1e4, dtype="fp32", seed=77)
    b = LinkBatch(wl, scheme="ror")
    with pytest.raises(pic.PicError):
        b.run()
    with pytest.raises(NotImplementedError):
        LinkBatch(inputs.rag_prompt(), scheme="ror").setup_decode()


def test_plan_and_run_equal_the_single_call():
    """The step plans the attention beside the re-rotation pass (side stream) and runs
    it after both: the same bits as one pic_link_attention call."""
    wl = inputs.rag_prompt()
    b = LinkBatch(wl)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    out = torch.empty_like(b.out)
    pic.pic_link_attention(b.dev["q_raw"], b.row_table, b.rows, b.dev["row_off"], b.k_pool, b.v_pool, b.pic_dtype,
                           b.pages, b.dev["page_off"], b.n_req, b.n_rows, wl.Hq, wl.Hkv, wl.d, b.scale, out, b.ws,
                           b.err)
    torch.cuda.synchronize()
    assert b.error() == 0
    assert torch.equal(out, b.out)


def test_pipelined_steps_match_single_steps():
    """LinkPipeline (uploads and read-backs on copy streams, double-buffered inputs and
    outputs) gives every step the single step's result: shared chunks rotated out of
    place, so repeated steps are identical."""
    from position_independent_kv_pic_gb300.link import LinkPipeline

    b = LinkBatch(inputs.batched_shared())
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    ref = b.out.cpu()
    b.pin_host_inputs()
    pipe = LinkPipeline(b)
    pipe.begin()
    outs = []
    for _ in range(5):
        host, ev = pipe.submit(b.host_pinned)
        ev.synchronize()
        outs.append(host.clone())
    torch.cuda.synchronize()
    assert b.error() == 0
    assert all(torch.equal(o, ref) for o in outs)
    # overlapped: four steps queued back to back, the last two results (the two
    # host buffers) checked once everything has arrived
    results = [pipe.submit(b.host_pinned) for _ in range(4)]
    torch.cuda.synchronize()
    assert b.error() == 0
    assert torch.equal(results[-1][0], ref) and torch.equal(results[-2][0], ref)
