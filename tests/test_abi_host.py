"""The C-ABI library without a GPU: it loads, exports every symbol pic.h declares,
and its host-side sizing agrees with the oracle's row selection and with a direct
enumeration of the page layout the header documents."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle.pic_oracle as O
import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build

from conftest import ROOT


@pytest.fixture(scope="module", autouse=True)
def built():
    pic_build.build()
    pic.load()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "pic.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pic_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    declared = _declared_symbols()
    assert len(declared) >= 12
    lib = ctypes.CDLL(pic.library_path())
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(pic.EXPORTED) == declared


def test_strerror():
    for s in range(7):
        assert pic.pic_strerror(s)
    assert pic.pic_strerror(99) == "unknown status"


@pytest.mark.parametrize("seed", range(30))
def test_count_rows_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 300, size=rng.integers(0, 40))
    q, k = int(rng.integers(0, 300)), int(rng.integers(0, 70))
    expect = O.count_rows(lens, q, k)
    assert pic.pic_count_rows(lens, q, k) == expect


def test_count_rows_worked_example():
    assert pic.pic_count_rows([4, 5, 5], 3, 2) == 7


def test_count_rows_invalid():
    assert pic.pic_count_rows([3, 0, 2], 1, 1) == -1
    assert pic.pic_count_rows([3], -1, 1) == -1
    assert pic.pic_count_rows([3], 1, -2) == -1


def _enumerate_layout(lens, q, k):
    """The layout pic.h documents, enumerated slot by slot."""
    link, rot, fresh, chunk_pages = [], 0, 0, 0
    s = 0
    for c, L in enumerate(lens):
        m = 0 if c == 0 else min(k, L)
        for f in range(-(-m // 16)):
            link.append((s + 16 * f, 0, min(16, m - 16 * f)))
            fresh += 1
        for j in range(-(-L // 16)):
            chunk_pages += 1
            lo, hi = max(0, m - 16 * j), min(16, L - 16 * j)
            if lo < hi:
                link.append((s + 16 * j, lo, hi))
                rot += c > 0
        s += L
    for f in range(-(-q // 16)):
        link.append((s + 16 * f, 0, min(16, q - 16 * f)))
        fresh += 1
    return link, rot, fresh, chunk_pages, s


@pytest.mark.parametrize("seed", range(30))
def test_request_sizes_match_layout(seed):
    rng = np.random.default_rng(100 + seed)
    lens = rng.integers(1, 80, size=rng.integers(1, 12)).tolist()
    q, k = int(rng.integers(0, 70)), int(rng.integers(0, 40))
    link, rot, fresh, cpages, T = _enumerate_layout(lens, q, k)
    sz = pic.pic_request_sizes_of(lens, q, k)
    assert sz == dict(tokens=T + q, rows=O.count_rows(lens, q, k), link_pages=len(link), rot_pages=rot,
                      fresh_pages=fresh, chunk_pages=cpages)
    # the layout covers every position 0 .. T+q-1 exactly once, and first positions increase
    covered = sorted(p for g0, lo, hi in link for p in range(g0 + lo, g0 + hi))
    assert covered == list(range(T + q))
    firsts = [g0 + lo for g0, lo, hi in link]
    assert all(a < b for a, b in zip(firsts, firsts[1:]))
    # recomputed positions (oracle) are exactly the fresh pages' slots
    rows = O.select_rows(lens, q, k)[0].tolist()
    fresh_slots = []
    s = 0
    for c, L in enumerate(lens):
        m = 0 if c == 0 else min(k, L)
        fresh_slots += list(range(s, s + m))
        s += L
    fresh_slots += list(range(T, T + q))
    assert fresh_slots == rows


@pytest.mark.parametrize("seed", range(20))
def test_framed_layout_sizes(seed):
    """The framed layout (rotate-on-read) pads every chunk's run of link pages to whole
    key tiles: the count follows from the spliced layout's pages grouped by chunk."""
    rng = np.random.default_rng(300 + seed)
    lens = rng.integers(1, 200, size=rng.integers(1, 12)).tolist()
    q, k = int(rng.integers(0, 70)), int(rng.integers(0, 40))
    link, rot, fresh, cpages, T = _enumerate_layout(lens, q, k)
    starts = np.concatenate([[0], np.cumsum(lens)])
    per_chunk = [sum(1 for g0, lo, hi in link if starts[c] <= g0 + lo < starts[c + 1]) for c in range(len(lens))]
    assert sum(per_chunk) + -(-q // 16) == len(link)
    tile = pic.PIC_TILE_PAGES
    framed = pic.pic_request_sizes_of(lens, q, k, pic.PIC_LAYOUT_FRAMED)
    spliced = pic.pic_request_sizes_of(lens, q, k, pic.PIC_LAYOUT_SPLICED)
    assert framed["link_pages"] == sum(-(-n // tile) * tile for n in per_chunk) + -(-q // 16)
    assert {f: v for f, v in framed.items() if f != "link_pages"} == \
        {f: v for f, v in spliced.items() if f != "link_pages"}
    offs = pic.pic_plan_offsets(lens, [0, len(lens)], [q], [k], pic.PIC_LAYOUT_FRAMED)
    assert offs["page_off"].tolist() == [0, framed["link_pages"]]
    with pytest.raises(pic.PicError):
        pic.pic_request_sizes_of(lens, q, k, 7)


def test_plan_offsets():
    lens = [4, 5, 5, 7, 33, 1]
    chunk_off = [0, 3, 3, 6]
    q, k = [3, 5, 0], [2, 1, 40]
    offs = pic.pic_plan_offsets(lens, chunk_off, q, k)
    rows = [O.count_rows(lens[a:b], qq, kk) for a, b, qq, kk in zip(chunk_off, chunk_off[1:], q, k)]
    assert offs["row_off"].tolist() == [0] + np.cumsum(rows).tolist()
    sizes = [pic.pic_request_sizes_of(lens[a:b], qq, kk) for a, b, qq, kk in zip(chunk_off, chunk_off[1:], q, k)]
    assert offs["page_off"].tolist() == [0] + np.cumsum([s["link_pages"] for s in sizes]).tolist()
    assert offs["rot_off"].tolist() == [0] + np.cumsum([s["rot_pages"] for s in sizes]).tolist()
    assert offs["fresh_off"].tolist() == [0] + np.cumsum([s["fresh_pages"] for s in sizes]).tolist()
    assert offs["chunk_page_off"].tolist() == [0] + np.cumsum([-(-L // 16) for L in lens]).tolist()
    with pytest.raises(pic.PicError):
        pic.pic_plan_offsets([4, 0], [0, 2], [1], [1])


def test_workspace_size():
    small = pic.pic_link_attention_workspace(100, 1, 32, 8, 128, pic.PIC_BF16)
    big = pic.pic_link_attention_workspace(5000, 16, 32, 8, 128, pic.PIC_BF16)
    assert 0 < small < big
    assert small % 256 == 0
    assert pic.pic_link_attention_workspace(100, 1, 4, 2, 16, pic.PIC_FP32) == 0   # SIMT path needs none
    assert pic.pic_link_attention_workspace(100, 1, 30, 8, 128, pic.PIC_BF16) == 0  # Hq % Hkv != 0


def test_device_entry_points_reject_bad_arguments_without_launch():
    """Argument checks happen on the host, before any CUDA call."""
    lib = pic.load()
    assert lib.pic_rope_table(None, -1, 16, 1e4, None, None) == pic.PIC_ERR_INVALID
    assert lib.pic_rope_table(None, 4, 15, 1e4, None, None) == pic.PIC_ERR_INVALID
    assert lib.pic_rope_table(None, 0, 16, 1e4, None, None) == pic.PIC_OK       # empty is a no-op
    assert lib.pic_rerotate_k(None, 10, 0, 8, 128, None, -1, None, 1, None, None) == pic.PIC_ERR_INVALID
    assert lib.pic_rerotate_k(None, 10, 7, 8, 128, None, 1, None, 1, None, None) == pic.PIC_ERR_INVALID
    assert lib.pic_rerotate_k(None, 10, 0, 8, 128, None, 0, None, 1, None, None) == pic.PIC_OK
    assert lib.pic_select_rows(None, None, None, None, None, -1, None, None, None, None) == pic.PIC_ERR_INVALID
    assert lib.pic_select_rows(None, None, None, None, None, 0, None, None, None, None) == pic.PIC_OK
    bad = lib.pic_link_attention(None, None, None, None, None, None, 10, 0, None, None, 1, 5, 30, 8, 128,
                                 0.1, None, None, 0, None, None)
    assert bad == pic.PIC_ERR_INVALID                                               # Hq % Hkv != 0
    assert lib.pic_link_attention(None, None, None, None, None, None, 10, 0, None, None, 0, 0, 32, 8, 128,
                                  0.1, None, None, 0, None, None) == pic.PIC_OK


def test_compose_segment_and_workspace():
    """Host sizing of the state composition: one level when the chains fill the SMs,
    else the shortest segment whose level-0 CTAs fit one wave; the workspace holds
    two levels' (T, S) intermediates only when there are two levels."""
    assert pic.pic_compose_segment(16, 264, 30, 32, 152) == 0          # 512 chains: one level
    seg = pic.pic_compose_segment(1, 100, 100, 32, 152)
    assert seg == 25 and 32 * -(-100 // seg) <= 152 and 32 * -(-100 // (seg - 1)) > 152
    assert pic.pic_compose_segment(1, 3, 3, 1, 152) == 2
    assert pic.pic_compose_segment(0, 0, 0, 32, 152) == 0
    one = pic.pic_compose_workspace(1, 100, 32, 128, 0)
    two = pic.pic_compose_workspace(1, 100, 32, 128, 25)
    assert 0 < one < 4096 and two >= one + 2 * 32 * 4 * 128 * 128 * 4
    assert pic.pic_compose_workspace(1, 100, 32, 64, 25) == 0          # d = 128 only
    lib = pic.load()
    assert lib.pic_compose_states(None, None, 0, None, None, 0, 0, 0, 32, 128, 0, None, None, 0, None,
                                  None) == pic.PIC_OK                  # no requests: a no-op
    assert lib.pic_compose_states(None, None, 4, None, None, 1, 5, 6, 32, 128, 0, None, None, 0, None,
                                  None) == pic.PIC_ERR_INVALID         # max_chain > n_elems
    assert lib.pic_compose_states(None, None, 4, None, None, 1, 5, 5, 32, 64, 0, None, None, 0, None,
                                  None) == pic.PIC_ERR_UNSUPPORTED


def test_rotate_on_read_entry_checks_without_launch():
    lib = pic.load()
    args = lambda n_tab, dtype, Hq, Hkv, d, n_req, n_rows: (None, None, None, None, None, None, 10, dtype, None,
                                                             None, None, n_tab, None, n_req, n_rows, Hq, Hkv, d,
                                                             0.1, None, None, 0, None, None)
    assert lib.pic_link_attention_ror(*args(0, pic.PIC_BF16, 32, 8, 128, 0, 0)) == pic.PIC_OK
    assert lib.pic_link_attention_ror(*args(-1, pic.PIC_BF16, 32, 8, 128, 0, 0)) == pic.PIC_ERR_INVALID
    assert lib.pic_link_attention_ror(*args(0, pic.PIC_FP32, 4, 2, 16, 0, 0)) == pic.PIC_ERR_UNSUPPORTED
    assert lib.pic_link_attention_ror(*args(0, pic.PIC_BF16, 30, 8, 128, 1, 5)) == pic.PIC_ERR_INVALID


def test_compose_split_checks_without_launch():
    lib = pic.load()
    assert lib.pic_compose_split_t(None, -1, 128, None, None) == pic.PIC_ERR_INVALID
    assert lib.pic_compose_split_t(None, 4, 64, None, None) == pic.PIC_ERR_UNSUPPORTED
    assert lib.pic_compose_split_t(None, 0, 128, None, None) == pic.PIC_OK
