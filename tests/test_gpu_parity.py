"""Parity of the CUDA path (through the C ABI) against the float64 oracle.

Rows and chunk starts: bit-exact.  Re-rotated K and the recomputed rows' fresh K:
within 1 ulp of the storage dtype; fresh V bit-identical.  Attention: max-abs <=
2e-2 and mean-abs <= 2e-3 (fp32 accumulate, bf16 out).  Every workload, the
~100k-token and batched ones included (the sizes and launch configuration the
benchmark times), is compared on every row and every re-rotated chunk.  Two
mistakes planted in the step's host sequence (no re-rotation; a row table on
local positions) must each miss the attention tolerance by more than 10x.
"""

import numpy as np
import pytest
import torch

import oracle.pic_oracle as O
import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build
from position_independent_kv_pic_gb300 import inputs
from position_independent_kv_pic_gb300.link import LinkBatch

from parity_util import TOL_MAX, TOL_MEAN, check_attention, check_fresh_kv, check_rerotated_k, check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pic_build.build()
    pic.load()


def _run(wl, **kw):
    b = LinkBatch(wl, **kw)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0, pic.pic_strerror(b.error())
    return b


# ---------------------------------------------------------------- tensor-core layouts

def test_selftest_umma():
    g = torch.Generator().manual_seed(0)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    bm = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    dk = torch.zeros(128, 128, device="cuda")
    dmn = torch.zeros(128, 128, device="cuda")
    dts = torch.zeros(128, 128, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pic.pic_selftest_umma(a.cuda(), bm.cuda(), dk, dmn, dts, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    A, B = a.double(), bm.double()
    assert (dk.double().cpu() - A @ B.T).abs().max() < 1e-3
    assert (dmn.double().cpu() - A @ B).abs().max() < 1e-3
    assert (dts.double().cpu() - A @ B).abs().max() < 1e-3


def test_selftest_umma_pair():
    """The CTA-pair products: S = A.B^T with M = N = 256 (each CTA 128 rows of A and
    128 keys of B), P.V with P from TMEM and V split by columns between the CTAs."""
    g = torch.Generator().manual_seed(1)
    a = torch.randn(256, 128, generator=g).to(torch.bfloat16)
    b = torch.randn(256, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    ds = torch.full((256, 256), float("nan"), device="cuda")
    dpv = torch.full((256, 128), float("nan"), device="cuda")
    info = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pic.pic_selftest_umma_pair(a.cuda(), b.cuda(), v.cuda(), ds, dpv, info, err)
    torch.cuda.synchronize()
    A, B, V = a.double(), b.double(), v.double()
    es = (ds.double().cpu() - A @ B.T).abs().nan_to_num(1e9)
    epv = (dpv.double().cpu() - A @ V).abs().nan_to_num(1e9)
    print("tmem bases", info.tolist(), "err", err.item(), "S err by quadrant",
          [[float(es[128 * i:128 * i + 128, 128 * j:128 * j + 128].max()) for j in range(2)] for i in range(2)],
          "PV err by quadrant",
          [[float(epv[128 * i:128 * i + 128, 64 * j:64 * j + 64].max()) for j in range(2)] for i in range(2)])
    assert err.item() == 0
    assert es.max() < 1e-3 and epv.max() < 1e-3


# ---------------------------------------------------------------- the workloads

def test_worked_example_fp32():
    b = _run(inputs.worked_example())
    check_rows(b)
    assert b.rows.cpu().tolist() == [4, 5, 9, 10, 14, 15, 16]
    check_rerotated_k(b)
    check_fresh_kv(b)
    emax, emean = check_attention(b)
    assert emax < 1e-5 and emean < 1e-6, (emax, emean)


@pytest.mark.parametrize("preset", ["rag_prompt_6chunks", "many_chunk_sink_20", "long_context_100x1000",
                                    "batched_shared_16req"])
def test_bf16_workload(preset):
    """Every row, every re-rotated chunk and every fresh slot of the workload."""
    b = _run(inputs.PRESETS[preset]())
    check_rows(b)
    check_rerotated_k(b)
    check_fresh_kv(b)
    emax, emean = check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)
    if b.wl.out_of_place:  # the shared sources are untouched
        for c, blocks in enumerate(b.store_blocks):
            L = int(b.wl.chunk_lens[c])
            j = np.arange(L)
            got = b.k_pool[torch.from_numpy(blocks[j // 16]).cuda(), :, torch.from_numpy(j % 16).cuda(), :].cpu()
            assert torch.equal(got, b.store_k[b.store_off[c]:b.store_off[c + 1]])


# ---------------------------------------------------------------- planted mistakes (host sequence)

def _assert_caught(b):
    emax, emean = check_attention(b)
    assert emax > 10 * TOL_MAX or emean > 10 * TOL_MEAN, (emax, emean)


def test_mutation_skipped_rerotation_is_caught(monkeypatch):
    """The step without pic_rerotate_k (cached K left at local positions) fails parity."""
    import position_independent_kv_pic_gb300.link as link
    monkeypatch.setattr(link, "pic_rerotate_k", lambda *a, **kw: None)
    _assert_caught(_run(inputs.rag_prompt()))


def test_mutation_local_position_row_table_is_caught(monkeypatch):
    """The step with the per-row RoPE table built on chunk-local positions (the row's
    offset in its chunk, or in the query) fails parity."""
    import position_independent_kv_pic_gb300.link as link
    wl = inputs.rag_prompt()
    b = LinkBatch(wl)
    local = []
    for req in wl.requests:
        rows, starts, T = O.select_rows(wl.chunk_lens[req.chunk_ids], req.q, req.k)
        c = np.searchsorted(starts, rows, side="right") - 1
        local.append(np.where(rows >= T, rows - T, rows - starts[c]))
    local_dev = torch.from_numpy(np.concatenate(local).astype(np.int32)).cuda()
    real = link.pic_rope_table

    def table_on_local_rows(pos, d, theta, table, stream=None):
        return real(local_dev if pos.data_ptr() == b.rows.data_ptr() else pos, d, theta, table, stream)

    monkeypatch.setattr(link, "pic_rope_table", table_on_local_rows)
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    _assert_caught(b)


# ---------------------------------------------------------------- edge cases

EDGE = [
    # (chunk lengths per request, q per request, k per request, Hq, Hkv, dtype)
    ([[300, 17, 1, 64, 129]], [37], [8], 32, 8, "bf16"),      # L_c < k, single-token chunk, ragged tails
    ([[100, 250]], [0], [16], 32, 8, "bf16"),                 # q = 0
    ([[77, 91, 33]], [5], [0], 32, 8, "bf16"),                # k = 0: only query rows
    ([[200]], [45], [4], 32, 8, "bf16"),                      # one chunk: no seam rows
    ([[40, 50, 60]], [3], [40], 32, 8, "bf16"),               # k >= L_c: whole chunks recomputed, k > 16
    ([[1, 1, 1, 1, 1, 1]], [1], [1], 32, 8, "bf16"),          # one-token chunks
    ([[130, 70], [55, 8, 200, 31], [500]], [20, 1, 33], [2, 16, 8], 32, 8, "bf16"),  # several requests
    ([[90, 140, 20]], [29], [8], 64, 8, "bf16"),              # GQA group 8 (16 rows per MMA tile)
    ([[90, 140, 20]], [29], [8], 8, 8, "bf16"),               # no GQA (128 rows per MMA tile)
    ([[90, 140, 20]], [29], [8], 16, 8, "bf16"),              # group 2
    ([[33, 47, 12]], [9], [3], 8, 2, "fp32"),                 # fp32 SIMT, d = 128
]


@pytest.mark.parametrize("case", range(len(EDGE)))
def test_edge_cases(case):
    lens, qs, ks, Hq, Hkv, dtype = EDGE[case]
    d = 128
    wl = inputs.custom(lens, qs, ks, Hq=Hq, Hkv=Hkv, d=d, theta=5e5, dtype=dtype, seed=50 + case)
    b = _run(wl)
    check_rows(b)
    check_rerotated_k(b)
    check_fresh_kv(b)
    emax, emean = check_attention(b)
    tol = (1e-4, 1e-5) if dtype == "fp32" else (TOL_MAX, TOL_MEAN)
    assert emax <= tol[0] and emean <= tol[1], (emax, emean)


def test_more_q_tile_pairs_than_the_planner_holds_in_shared_memory():
    """Over 1,024 Q-tile pairs in one call (520 requests of 66-79 recomputed rows, two
    pairs of 64 rows each at Hq = 32, Hkv = 8): the unit planner takes its path for
    tile tables larger than its shared-memory arrays (a search per tile instead of
    the staged counts).  Every row against the oracle."""
    rng = np.random.default_rng(123)
    n = 520
    lens = [[int(rng.integers(20, 60)), int(rng.integers(10, 40))] for _ in range(n)]
    qs = [int(rng.integers(58, 72)) for _ in range(n)]
    wl = inputs.custom(lens, qs, [8] * n, Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=123)
    b = _run(wl)
    ro = b.offs["row_off"]
    pairs = sum(-(-int(ro[r + 1] - ro[r]) // 64) for r in range(b.n_req))
    assert pairs > 1024, pairs
    check_rows(b)
    emax, emean = check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)


def test_request_limit_of_one_call():
    """The tensor-core path plans at most 1,024 requests per call: 1,024 requests link
    and match the oracle on every row, 1,025 are refused with PIC_ERR_UNSUPPORTED."""
    def wl_of(n):
        return inputs.custom([[6, 5]] * n, [2] * n, [2] * n, Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16",
                             seed=7)

    b = _run(wl_of(1024))
    assert b.n_req == 1024
    check_rows(b)
    emax, emean = check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)
    over = LinkBatch(wl_of(1025))
    with pytest.raises(pic.PicError) as e:
        over.run()
    torch.cuda.synchronize()
    assert e.value.status == pic.PIC_ERR_UNSUPPORTED


def test_no_rows_is_a_no_op():
    wl = inputs.custom([[50]], [0], [4], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=3)
    b = _run(wl)
    assert b.n_rows == 0


def test_fp32_small_head_dims():
    for d in (16, 32, 64):
        wl = inputs.custom([[21, 13, 40]], [6], [5], Hq=4, Hkv=2, d=d, theta=1e4, dtype="fp32", seed=d)
        b = _run(wl)
        check_rows(b)
        check_rerotated_k(b)
        check_fresh_kv(b)
        emax, emean = check_attention(b)
        assert emax < 1e-4 and emean < 1e-5, (d, emax, emean)


def test_in_place_leaves_other_slots_alone():
    """In-place re-rotation touches only the cached, non-recomputed slots of chunks >= 1;
    V pages of cached chunks are never written."""
    wl = inputs.custom([[40, 37, 50]], [7], [5], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=7)
    b = LinkBatch(wl)
    k0, v0 = b.k_pool.clone(), b.v_pool.clone()
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    fresh = torch.from_numpy(b.fresh_blocks.astype(np.int64)).cuda()
    keep = torch.ones(b.num_blocks, dtype=torch.bool, device="cuda")
    keep[fresh] = False
    assert torch.equal(b.v_pool[keep], v0[keep])
    # seam slots of chunks >= 1 and chunk 0 are untouched in the K pool
    for ci, sid in enumerate(b.flat_store_ids):
        blocks = b.store_blocks[sid]
        L = int(wl.chunk_lens[sid])
        m = L if ci == 0 else min(5, L)
        j = np.arange(m)
        bi = torch.from_numpy(blocks[j // 16]).cuda()
        si = torch.from_numpy(j % 16).cuda()
        assert torch.equal(b.k_pool[bi, :, si, :], k0[bi, :, si, :])


def test_out_of_range_block_sets_error_flag():
    """A corrupted block table is reported through err_flag; nothing faults."""
    wl = inputs.custom([[40, 37, 50]], [7], [5], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=8)
    b = LinkBatch(wl)
    b.dev["k_src"][3] = b.num_blocks + 5
    b.run()
    torch.cuda.synchronize()
    assert b.error() == pic.PIC_ERR_RANGE
    assert torch.isfinite(b.out.float()).all()
