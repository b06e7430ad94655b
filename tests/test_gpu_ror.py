"""Rotate-on-read through the C ABI (RoPE article 3.3: the correction applied where
the kernel reads the cache).  The step splices the framed layout: every chunk's
keys stay in the chunk's own frame (cached pages never written, the recomputed
head rows' fresh K encoded at their position in the chunk) and every key tile
lies in one chunk; pic_link_attention_ror rotates Q back by the chunk's offset
for the key tiles of that chunk instead of rotating K.  Checked against the float64
oracle on every row of every workload, with the pool read back: cached pages
untouched, fresh K in its frame."""

import numpy as np
import pytest
import torch

import oracle.pic_oracle as O
import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build
from position_independent_kv_pic_gb300 import inputs
from position_independent_kv_pic_gb300.link import LinkBatch

from parity_util import TOL_MAX, TOL_MEAN, check_attention, check_fresh_kv, check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pic_build.build()
    pic.load()


def _run(wl):
    b = LinkBatch(wl, scheme="ror")
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0, pic.pic_strerror(b.error())
    return b


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
def test_against_oracle(preset):
    b = _run(inputs.PRESETS[preset]())
    check_rows(b)
    check_fresh_kv(b)
    emax, emean = check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)
    _cached_pages_untouched(b)


def test_framed_layout():
    """Every chunk's run of pages starts on a key-tile boundary of its request's list
    and is padded with empty entries; page_tab names the chunk for every page of a
    chunk after the first (fresh, cached and padding) and -1 for chunk 0 and the
    query; the fresh rows' frame positions are their positions in the chunk."""
    b = _run(inputs.batched_shared())
    pages = b.pages_host()
    tab = b.page_tab.cpu().numpy()
    starts = b.chunk_start.cpu().numpy()
    frame_pos = b.row_frame_pos.cpu().numpy()
    rows = b.rows.cpu().numpy()
    po, ro = b.offs["page_off"], b.offs["row_off"]
    for r, req in enumerate(b.wl.requests):
        c0, c1 = int(b.chunk_off[r]), int(b.chunk_off[r + 1])
        p = int(po[r])
        for c in range(c0, c1):
            L = int(b.chunk_lens[c])
            end = int(starts[c]) + L
            run = [p]
            while p < int(po[r + 1]) and pages["lo"][p] < pages["hi"][p] and pages["gpos0"][p] < end:
                p += 1
            n_real = p - run[0]
            while p < int(po[r + 1]) and pages["lo"][p] == pages["hi"][p] and pages["gpos0"][p] == end:
                assert pages["k_block"][p] == -1 and pages["v_block"][p] == -1
                p += 1
            assert (run[0] - int(po[r])) % pic.PIC_TILE_PAGES == 0 and (p - run[0]) % pic.PIC_TILE_PAGES == 0
            assert p - run[0] - n_real < pic.PIC_TILE_PAGES
            want = c if c > c0 else -1
            assert np.all(tab[run[0]:p] == want), (r, c)
        assert np.all(tab[p:int(po[r + 1])] == -1)  # the query pages
        lens = b.wl.chunk_lens[req.chunk_ids]
        o_rows, o_starts, T = O.select_rows(lens, req.q, req.k)
        a, e = int(ro[r]), int(ro[r + 1])
        assert np.array_equal(rows[a:e], o_rows)
        c = np.searchsorted(o_starts, o_rows, side="right") - 1
        assert np.array_equal(frame_pos[a:e], np.where(o_rows >= T, o_rows, o_rows - o_starts[c]))


@pytest.mark.parametrize("case", [
    ([[300, 17, 1, 64, 129]], [37], [8]),
    ([[40, 50, 60]], [3], [40]),
    ([[130, 70], [55, 8, 200, 31]], [20, 1], [2, 16]),
    ([[1, 1, 1, 1, 1, 1]], [1], [1]),
    ([[77, 91, 33]], [5], [0]),
    ([[100, 250]], [0], [16]),
])
def test_edge_cases_against_oracle(case):
    lens, qs, ks = case
    wl = inputs.custom(lens, qs, ks, Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=90 + len(lens))
    b = _run(wl)
    check_rows(b)
    check_fresh_kv(b)
    emax, emean = check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)
    _cached_pages_untouched(b)


@pytest.mark.parametrize("Hq", [8, 16, 64])
def test_gqa_groups_against_oracle(Hq):
    wl = inputs.custom([[90, 140, 20]], [29], [8], Hq=Hq, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=97)
    b = _run(wl)
    emax, emean = check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)


def test_bad_table_row_is_flagged():
    wl = inputs.custom([[40, 50, 60]], [3], [4], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=95)
    b = _run(wl)
    framed = torch.nonzero(b.page_tab >= 0).flatten()
    assert len(framed) > 0
    # run the attention alone with the frames of one chunk pointing past the table
    b.page_tab[framed] = b.n_chunks + 3
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


def test_plan_parts_in_either_order_equal_the_single_call():
    """The plan in its two parts (the Q operands, which need no page list, and the
    unit plan), the units first here, then the run: the same bits as one
    pic_link_attention call."""
    wl = inputs.many_chunk()
    b = LinkBatch(wl)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    ref = torch.empty_like(b.out)
    pic.pic_link_attention(b.dev["q_raw"], b.row_table, b.rows, b.dev["row_off"], b.k_pool, b.v_pool, b.pic_dtype,
                           b.pages, b.dev["page_off"], b.n_req, b.n_rows, wl.Hq, wl.Hkv, wl.d, b.scale, ref, b.ws,
                           b.err)
    b.ws.fill_(0xFF)  # nothing may survive from the previous plan
    pic.pic_link_attention_plan_units(b.rows, b.dev["row_off"], b.pages, b.dev["page_off"], b.n_req, b.n_rows,
                                      wl.Hq, wl.Hkv, wl.d, b.pic_dtype, b.ws, b.err)
    pic.pic_link_attention_plan_q(b.dev["q_raw"], b.row_table, b.dev["row_off"], b.n_req, b.n_rows, wl.Hq, wl.Hkv,
                                  wl.d, b.pic_dtype, b.ws, b.err)
    out = torch.empty_like(b.out)
    pic.pic_link_attention_run(b.dev["q_raw"], b.row_table, b.rows, b.dev["row_off"], b.k_pool, b.v_pool,
                               b.pic_dtype, b.pages, b.dev["page_off"], b.n_req, b.n_rows, wl.Hq, wl.Hkv, wl.d,
                               b.scale, out, b.ws, b.err)
    torch.cuda.synchronize()
    assert b.error() == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("graphs", [False, True])
def test_pipelined_steps_match_single_steps(graphs):
    """LinkPipeline (uploads and read-backs on copy streams, double-buffered inputs and
    outputs; eagerly or as one CUDA graph per buffer set) gives every step the single
    step's result: shared chunks rotated out of place, so repeated steps are identical."""
    from position_independent_kv_pic_gb300.link import LinkPipeline

    b = LinkBatch(inputs.batched_shared())
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    ref = b.out.cpu()
    b.pin_host_inputs()
    pipe = LinkPipeline(b, graphs=graphs)
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


@pytest.mark.parametrize("scheme", ["rotary", "ror", "nope"])
def test_graph_replay_equals_the_eager_step(scheme):
    """The step captured as a CUDA graph (LinkGraph) gives the eager step's output bit
    for bit, replay after replay (the pool reset to the cached chunks each time)."""
    from position_independent_kv_pic_gb300.link import LinkGraph

    b = LinkBatch(inputs.rag_prompt(), scheme=scheme)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    ref = b.out.clone()
    g = LinkGraph(b)
    for _ in range(3):
        b.reset_pool()
        b.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert b.error() == 0
        assert torch.equal(b.out, ref)
