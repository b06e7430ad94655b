"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: values the
pages print (tests/golden), closed forms, an independent formulation (complex
numbers, explicit rotation matrices), a library routine (torch SDPA in float64,
torch's bfloat16 conversion), or an invariant.  The mutation tests at the end
plant the mistakes the KV-cache blog plants (reset positions, dropped mask
offset) plus a skipped re-rotation, in the oracle, and check that each one moves
the output far outside the parity tolerance.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.pic_oracle as O
from position_independent_kv_pic_gb300 import inputs

from conftest import GOLDEN

TOL_MAX, TOL_MEAN = 2e-2, 2e-3  # attention parity tolerance (fp32 accumulate, bf16 out)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# (a) row selection: the worked example and the k sweep
# ---------------------------------------------------------------------------

def test_worked_example_rows():
    g = _golden("legolink_worked_example.json")
    rows, starts, T = O.select_rows(g["chunk_lens"], g["q"], g["k"])
    assert rows.tolist() == g["rows"]
    assert starts.tolist() == g["chunk_starts"]
    assert T == g["T"]
    assert T + g["q"] == g["total_tokens"]
    assert len(rows) == g["n_recomputed"]
    assert rows[-g["q"]:].tolist() == g["query_rows"]
    key_pos = np.arange(g["total_tokens"])
    counts = [int(O.visible(key_pos, p).sum()) for p in O.query_positions(rows, starts, T)]
    assert counts == g["visible_key_counts"]


def test_k_sweep_counts():
    g = _golden("legolink_k_sweep.json")
    for row in g["sweep"]:
        n = O.count_rows(g["chunk_lens"], g["q"], row["k"])
        assert n == row["recompute_tokens"]
        assert round(100.0 * n / g["total_tokens"], 1) == row["pct_of_total"]


@pytest.mark.parametrize("seed", range(20))
def test_select_rows_brute_force(seed):
    """Brute force on tiny inputs: a token is recomputed iff it is one of the first k
    tokens of a chunk other than the first, or a query token."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 9, size=rng.integers(1, 6)).tolist()
    q, k = int(rng.integers(0, 5)), int(rng.integers(0, 10))
    owner, local = [], []
    for c, L in enumerate(lens):
        owner += [c] * L
        local += list(range(L))
    T = len(owner)
    expect = [p for p in range(T) if owner[p] > 0 and local[p] < k] + list(range(T, T + q))
    rows, starts, T2 = O.select_rows(lens, q, k)
    assert T2 == T and rows.tolist() == expect
    assert len(rows) == sum(min(k, L) for L in lens[1:]) + q
    assert starts.tolist() == [owner.index(c) for c in range(len(lens))]


def test_select_rows_degenerate():
    assert O.select_rows([7], 0, 5)[0].tolist() == []          # one chunk, no query
    assert O.select_rows([3, 2], 0, 0)[0].tolist() == []       # k = 0, q = 0
    assert O.select_rows([3, 2], 2, 0)[0].tolist() == [5, 6]   # k = 0: only query rows
    assert O.select_rows([3, 2], 0, 9)[0].tolist() == [3, 4]   # L_c < k
    with pytest.raises(ValueError):
        O.select_rows([3, 0], 1, 1)
    with pytest.raises(ValueError):
        O.select_rows([3], 1, -1)


# ---------------------------------------------------------------------------
# (e) the offset causal mask: the KV-cache blog's exercise
# ---------------------------------------------------------------------------

def test_offset_mask_exercise():
    g = _golden("offset_mask_exercise.json")
    for case in g["cases"]:
        P, C = case["cached"], case["new"]
        rows, starts, T = O.select_rows([P], C, 0)
        qpos = O.query_positions(rows, starts, T)
        assert qpos.tolist() == case["query_positions"]
        key_pos = np.arange(T + C)
        mask = np.stack([O.visible(key_pos, p) for p in qpos])
        assert list(mask.shape) == case["scores_shape"]
        assert mask.sum(axis=1).tolist() == case["visible_key_counts"]
        top_left = np.stack([O.visible(key_pos, i) for i in range(C)])
        assert top_left.sum(axis=1).tolist() == case["top_left_visible_key_counts"]


# ---------------------------------------------------------------------------
# RoPE: independent formulations and the identities the RoPE article states
# ---------------------------------------------------------------------------

def test_inv_freq_shape_of_spectrum():
    """Footnote 3 of the RoPE article: inv_freq runs from 1 (index 0, fastest) down
    towards 1/base, as a geometric sequence."""
    for d, base in [(16, 1e4), (128, 5e5), (64, 1e4)]:
        f = O.inv_freq(d, base)
        assert f.shape == (d // 2,)
        assert f[0] == 1.0
        ratio = f[1:] / f[:-1]
        assert np.allclose(ratio, ratio[0], rtol=1e-13, atol=0)
        # one more step of the sequence would land exactly on 1/base
        assert math.isclose(f[-1] * ratio[0], 1.0 / base, rel_tol=1e-12)
        assert np.all(np.diff(f) < 0)


def test_rope_single_pair_closed_form():
    """x = e_0 rotated by position 1 at frequency 1 lands on (cos 1) e_0 + (sin 1) e_{d/2}:
    half-split pairing, counter-clockwise rotation."""
    for d in (2, 16, 128):
        x = np.zeros((1, d))
        x[0, 0] = 1.0
        y = O.rope(x, [1], 10000.0)
        expect = np.zeros(d)
        expect[0], expect[d // 2] = math.cos(1.0), math.sin(1.0)
        assert np.allclose(y[0], expect, atol=1e-15)


def test_rope_matches_complex_multiplication():
    """RoPE as complex multiplication: pair (x_i, x_{i+d/2}) is z_i = x_i + 1j x_{i+d/2},
    rotated to z_i * exp(1j * p * base**(-2i/d))."""
    rng = np.random.default_rng(0)
    d, base = 128, 5e5
    x = rng.standard_normal((50, 3, d))
    pos = rng.integers(0, 200000, size=50)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    w = np.exp(1j * np.outer(pos, base ** (-np.arange(0, d, 2) / d)))[:, None, :]
    zr = z * w
    expect = np.concatenate([zr.real, zr.imag], axis=-1)
    assert np.allclose(O.rope(x, pos, base), expect, rtol=0, atol=1e-12)


def test_rope_matches_rotation_matrix():
    """RoPE as an explicit block rotation matrix R(p) acting on dimension pairs."""
    rng = np.random.default_rng(1)
    d, base, p = 16, 1e4, 37
    R = np.zeros((d, d))
    for i in range(d // 2):
        a = p * base ** (-2.0 * i / d)
        c, s = math.cos(a), math.sin(a)
        R[i, i], R[i, i + d // 2] = c, -s
        R[i + d // 2, i], R[i + d // 2, i + d // 2] = s, c
    x = rng.standard_normal((4, d))
    assert np.allclose(O.rope(x, [p] * 4, base), x @ R.T, atol=1e-13)
    assert np.allclose(R @ R.T, np.eye(d), atol=1e-14)  # orthogonal


@pytest.mark.parametrize("seed", range(4))
def test_rotation_additivity(seed):
    """(b) Rotating by Delta after encoding at p equals encoding at p + Delta
    (rotary correction, RoPE article 3.3), up to float64 rounding, for positions and
    offsets up to 2e5."""
    rng = np.random.default_rng(seed)
    d, base = 128, 5e5
    x = rng.standard_normal((64, 8, d))
    p = rng.integers(0, 200000, size=64)
    delta = int(rng.integers(0, 200000))
    lhs = O.rope(O.rope(x, p, base), np.full(64, delta), base)
    rhs = O.rope(x, p + delta, base)
    err = np.abs(lhs - rhs).max() / np.abs(rhs).max()
    # angles reach 4e5 rad; cos/sin of such arguments carry ~4e5 * 2^-53 absolute error
    assert err < 1e-10


def test_rerotate_equals_rope_at_global_position():
    """(b) A chunk compiled at local positions and re-rotated by its start equals RoPE
    applied directly at the global positions (exact mode: no storage rounding)."""
    rng = np.random.default_rng(2)
    k_raw = rng.standard_normal((40, 2, 16))
    s = 12345
    moved = O.rerotate_k(O.compile_chunk_k(k_raw, 1e4, "fp64"), s, 1e4, "fp64")
    direct = O.rope(k_raw, np.arange(40) + s, 1e4)
    assert np.allclose(moved, direct, rtol=0, atol=1e-11)


@pytest.mark.parametrize("seed", range(4))
def test_relative_position(seed):
    """(c) <RoPE_m(q), RoPE_n(k)> depends only on m - n (RoPE article 2.2)."""
    rng = np.random.default_rng(seed)
    d, base = 128, 5e5
    q, k = rng.standard_normal((1, d)), rng.standard_normal((1, d))
    m, n, t = (int(v) for v in rng.integers(0, 100000, size=3))
    a = float((O.rope(q, [m], base) @ O.rope(k, [n], base).T)[0, 0])
    b = float((O.rope(q, [m + t], base) @ O.rope(k, [n + t], base).T)[0, 0])
    assert abs(a - b) < 1e-9 * max(1.0, abs(a))


def test_rerotate_by_zero_is_identity():
    """(f) Delta = 0 (chunk 0) leaves stored bits unchanged."""
    k, _, _ = inputs.chunk_store(inputs.rag_prompt())
    x = k[:300].double().numpy()
    assert np.array_equal(O.rerotate_k(x, 0, 5e5, "bf16"), x)


# ---------------------------------------------------------------------------
# bf16 rounding against torch's conversion
# ---------------------------------------------------------------------------

def test_round_bf16_matches_torch():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ours = O.round_to(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(ours, ref)


def test_round_bf16_ties_to_even():
    # float32 values exactly halfway between two bf16 neighbours
    bits = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x40490000 | 0x8000], np.uint32)
    x = bits.view(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.round_to(x.astype(np.float64), "bf16"), ref)
    assert O.round_to(np.array([1.0 + 2.0 ** -8]), "bf16")[0] == 1.0            # tie -> even
    assert O.round_to(np.array([1.0 + 3 * 2.0 ** -8]), "bf16")[0] == 1.0 + 2.0 ** -6


# ---------------------------------------------------------------------------
# (d) brute force: with k >= every chunk length, link == full recompute
# ---------------------------------------------------------------------------

def _full_recompute_sdpa(q_raw_all, k_raw_all, v_all, base, dtype, Hq, Hkv):
    """Full causal attention over the whole sequence with torch SDPA (float64, CPU,
    explicit boolean mask): the full-recompute (FR) baseline of the EPIC comparison."""
    N, _, d = q_raw_all.shape
    qr = O.round_to(O.rope(q_raw_all, np.arange(N), base), dtype)
    kr = O.round_to(O.rope(k_raw_all, np.arange(N), base), dtype)
    Q = torch.from_numpy(qr).permute(1, 0, 2)[None]
    K = torch.from_numpy(kr).permute(1, 0, 2)[None]
    V = torch.from_numpy(np.asarray(v_all, np.float64)).permute(1, 0, 2)[None]
    mask = torch.ones(N, N, dtype=torch.bool).tril()
    out = torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, attn_mask=mask, scale=1.0 / math.sqrt(d), enable_gqa=(Hq != Hkv))
    return out[0].permute(1, 0, 2).numpy()


def _naive_full_attention(q_raw_all, k_raw_all, v_all, base, dtype, Hq, Hkv):
    """Triple loop, for the tiniest case."""
    N, _, d = q_raw_all.shape
    qr = O.round_to(O.rope(q_raw_all, np.arange(N), base), dtype)
    kr = O.round_to(O.rope(k_raw_all, np.arange(N), base), dtype)
    out = np.zeros((N, Hq, d))
    for i in range(N):
        for h in range(Hq):
            kv = h // (Hq // Hkv)
            s = [sum(qr[i, h, t] * kr[j, kv, t] for t in range(d)) / math.sqrt(d) for j in range(i + 1)]
            m = max(s)
            w = [math.exp(v - m) for v in s]
            z = sum(w)
            for t in range(d):
                out[i, h, t] = sum(w[j] * v_all[j, kv, t] for j in range(i + 1)) / z
    return out


@pytest.mark.parametrize("dtype,lens,q,Hq,Hkv,d", [
    ("fp32", [4, 5, 5], 3, 4, 2, 16),
    ("bf16", [6, 3, 7, 2], 5, 8, 2, 32),
    ("fp64", [5, 9], 4, 4, 4, 8),
])
def test_full_recompute_equivalence(dtype, lens, q, Hq, Hkv, d):
    rng = np.random.default_rng(7)
    base = 1e4
    N = sum(lens) + q
    k = max(lens)
    q_raw = O.round_to(rng.standard_normal((N, Hq, d)), dtype)
    k_raw = O.round_to(rng.standard_normal((N, Hkv, d)), dtype)
    v = O.round_to(rng.standard_normal((N, Hkv, d)), dtype)
    # chunk 0 is compiled at local = global positions; every other chunk is recomputed
    chunks_k, chunks_v, s = [], [], 0
    for L in lens:
        chunks_k.append(O.compile_chunk_k(k_raw[s:s + L], base, dtype))
        chunks_v.append(v[s:s + L])
        s += L
    rows = O.select_rows(lens, q, k)[0]
    assert len(rows) == N - lens[0]
    res = O.link_request(chunks_k, chunks_v, q, k, q_raw[rows], k_raw[rows], v[rows], base, dtype)
    fr = _full_recompute_sdpa(q_raw, k_raw, v, base, dtype, Hq, Hkv)
    assert np.abs(res["out"] - fr[rows]).max() < 1e-12
    if dtype == "fp32":
        naive = _naive_full_attention(q_raw, k_raw, v, base, dtype, Hq, Hkv)
        assert np.abs(naive - fr).max() < 1e-12


def test_chunked_prefill_equivalence():
    """(f) k = 0 with one cached chunk of P tokens and q new tokens is plain chunked
    prefill: new token i at position P + i sees keys 0 .. P + i (offset mask)."""
    rng = np.random.default_rng(8)
    P, q, Hq, Hkv, d, base = 10, 3, 4, 2, 16, 1e4
    q_raw = rng.standard_normal((q, Hq, d))
    k_raw = rng.standard_normal((P + q, Hkv, d))
    v = rng.standard_normal((P + q, Hkv, d))
    cached = O.compile_chunk_k(k_raw[:P], base, "fp64")
    res = O.link_request([cached], [v[:P]], q, 0, q_raw, k_raw[P:], v[P:], base, "fp64")
    assert res["rows"].tolist() == [10, 11, 12]
    Q = torch.from_numpy(O.rope(q_raw, np.arange(P, P + q), base)).permute(1, 0, 2)[None]
    K = torch.from_numpy(O.rope(k_raw, np.arange(P + q), base)).permute(1, 0, 2)[None]
    V = torch.from_numpy(v).permute(1, 0, 2)[None]
    allowed = torch.arange(P + q)[None, :] <= (P + torch.arange(q))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, attn_mask=allowed, enable_gqa=True)[0].permute(1, 0, 2).numpy()
    assert np.abs(res["out"] - ref).max() < 1e-12


# ---------------------------------------------------------------------------
# (g) layer-0 invariance: fresh K/V equal to the chunk's own K_raw / V
# ---------------------------------------------------------------------------

def _layer0_case(dtype, k, seed=9):
    rng = np.random.default_rng(seed)
    lens, q, Hq, Hkv, d, base = [9, 12, 7, 10], 6, 8, 2, 32, 5e5
    N = sum(lens) + q
    k_raw = O.round_to(rng.standard_normal((N, Hkv, d)), dtype)
    v = O.round_to(rng.standard_normal((N, Hkv, d)), dtype)
    q_raw = O.round_to(rng.standard_normal((q, Hq, d)), dtype)
    chunks_k, chunks_v, s = [], [], 0
    for L in lens:
        chunks_k.append(O.compile_chunk_k(k_raw[s:s + L], base, dtype))
        chunks_v.append(v[s:s + L])
        s += L
    rows = O.select_rows(lens, q, k)[0]
    n_seam = len(rows) - q
    q_all = np.concatenate([np.zeros((n_seam, Hq, d)), q_raw])
    res = O.link_request(chunks_k, chunks_v, q, k, q_all, k_raw[rows], v[rows], base, dtype)
    return res["out"][n_seam:]


def test_layer0_invariance_exact():
    """With layer-0-like fresh K/V (context independent), re-rotation is exact in float64,
    so the query rows' output does not depend on k."""
    ref = _layer0_case("fp64", 0)
    for k in (1, 3, 12):
        assert np.abs(_layer0_case("fp64", k) - ref).max() < 1e-12


def test_layer0_invariance_bf16():
    """The same invariant holds up to bf16 storage rounding of K."""
    ref = _layer0_case("bf16", 0)
    for k in (2, 12):
        diff = np.abs(_layer0_case("bf16", k) - ref)
        assert diff.max() < TOL_MAX and diff.mean() < TOL_MEAN


# ---------------------------------------------------------------------------
# (h) mutations planted in the oracle must be caught by the parity tolerance
# ---------------------------------------------------------------------------

def _mutation_workload():
    wl = inputs.custom([[24, 40, 33, 51, 29]], [19], [4], Hq=8, Hkv=2, d=64, theta=1e4,
                       dtype="bf16", seed=11)
    kst, vst, off = inputs.chunk_store(wl)
    req = wl.requests[0]
    lens = wl.chunk_lens[req.chunk_ids]
    n = O.count_rows(lens, req.q, req.k)
    qr, kn, vn = inputs.row_inputs(wl, n)
    chunks_k = [kst[off[c]:off[c + 1]].double().numpy() for c in req.chunk_ids]
    chunks_v = [vst[off[c]:off[c + 1]].double().numpy() for c in req.chunk_ids]
    return (chunks_k, chunks_v, req.q, req.k, qr.double().numpy(), kn.double().numpy(),
            vn.double().numpy(), wl.theta, wl.dtype)


def _run():
    return O.link_request(*_mutation_workload())


def _assert_caught(good, bad):
    diff = np.abs(bad["out"] - good["out"])
    assert diff.max() > 10 * TOL_MAX or diff.mean() > 10 * TOL_MEAN, (diff.max(), diff.mean())


def test_mutation_no_rerotation(monkeypatch):
    good = _run()
    monkeypatch.setattr(O, "rerotate_k", lambda k, delta, theta, dtype: O.round_to(k, dtype))
    _assert_caught(good, _run())


def test_mutation_top_left_mask(monkeypatch):
    good = _run()
    rank = {int(p): i for i, p in enumerate(good["rows"])}
    real = O.visible
    monkeypatch.setattr(O, "visible", lambda key_pos, qp: real(key_pos, rank[int(qp)]))
    _assert_caught(good, _run())


def test_mutation_local_query_positions(monkeypatch):
    good = _run()

    def local(rows, starts, T):
        c = np.searchsorted(starts, rows, side="right") - 1
        return np.where(rows >= T, rows - T, rows - starts[c])

    monkeypatch.setattr(O, "query_positions", local)
    _assert_caught(good, _run())


# ---------------------------------------------------------------------------
# Decode after link ([EPIC] decode tokens after the query; [KVC] single-token decode)
# ---------------------------------------------------------------------------

def _decode_case(dtype, lens, q, k, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    base = 1e4
    chunks_k = [O.compile_chunk_k(O.round_to(rng.standard_normal((L, Hkv, d)), dtype), base, dtype) for L in lens]
    chunks_v = [O.round_to(rng.standard_normal((L, Hkv, d)), dtype) for L in lens]
    n = O.count_rows(np.array(lens), q, k)
    q_raw = O.round_to(rng.standard_normal((n + 1, Hq, d)), dtype)
    k_raw = O.round_to(rng.standard_normal((n + 1, Hkv, d)), dtype)
    v = O.round_to(rng.standard_normal((n + 1, Hkv, d)), dtype)
    return base, chunks_k, chunks_v, q_raw, k_raw, v, n


@pytest.mark.parametrize("dtype", ["fp64", "bf16"])
def test_decode_after_link_equals_longer_link(dtype):
    """Decoding one token after a link with q query rows gives the output the same
    token gets as the last query row of a link with q + 1 query rows."""
    lens, q, k, Hq, Hkv, d = [6, 9, 4, 7], 3, 2, 4, 2, 16
    base, ck, cv, q_raw, k_raw, v, n = _decode_case(dtype, lens, q, k, Hq, Hkv, d, seed=21)
    longer = O.link_request(ck, cv, q + 1, k, q_raw, k_raw, v, base, dtype)
    link = O.link_request(ck, cv, q, k, q_raw[:n], k_raw[:n], v[:n], base, dtype)
    assert link["K_ctx"].shape[0] == sum(lens) + q
    dec = O.decode_after_link(link["K_ctx"], link["V_ctx"], q_raw[n], k_raw[n], v[n], base, dtype)
    assert np.abs(dec - longer["out"][-1]).max() < 1e-12


def test_decode_matches_full_recompute():
    """With k >= every chunk length the linked context is the fully recomputed one, so
    the decode row equals the last row of full causal attention over N + 1 tokens
    (torch SDPA, float64)."""
    rng = np.random.default_rng(23)
    lens, q, Hq, Hkv, d, base, dtype = [5, 4, 6], 2, 4, 2, 16, 1e4, "fp64"
    N = sum(lens) + q
    q_raw = rng.standard_normal((N + 1, Hq, d))
    k_raw = rng.standard_normal((N + 1, Hkv, d))
    v = rng.standard_normal((N + 1, Hkv, d))
    ck, cv, s = [], [], 0
    for L in lens:
        ck.append(O.compile_chunk_k(k_raw[s:s + L], base, dtype))
        cv.append(v[s:s + L])
        s += L
    rows = O.select_rows(lens, q, max(lens))[0]
    link = O.link_request(ck, cv, q, max(lens), q_raw[rows], k_raw[rows], v[rows], base, dtype)
    dec = O.decode_after_link(link["K_ctx"], link["V_ctx"], q_raw[N], k_raw[N], v[N], base, dtype)
    fr = _full_recompute_sdpa(q_raw, k_raw, v, base, dtype, Hq, Hkv)
    assert np.abs(dec - fr[N]).max() < 1e-12


def test_decode_mutations_caught():
    """A decode that forgets its own K/V, or encodes its query at the last context
    position instead of its own, moves the output far past the GPU tolerance."""
    lens, q, k, Hq, Hkv, d = [6, 9, 4, 7], 3, 2, 4, 2, 16
    base, ck, cv, q_raw, k_raw, v, n = _decode_case("fp64", lens, q, k, Hq, Hkv, d, seed=22)
    link = O.link_request(ck, cv, q, k, q_raw[:n], k_raw[:n], v[:n], base, "fp64")
    K, V = link["K_ctx"], link["V_ctx"]
    good = O.decode_after_link(K, V, q_raw[n], k_raw[n], v[n], base, "fp64")
    N = K.shape[0]
    q_rot = O.rope(q_raw[n][None], np.array([N]), base)
    no_self = O.attention_rows(q_rot, np.array([N - 1]), K, V, 1.0 / math.sqrt(d))[0]
    q_wrong = O.rope(q_raw[n][None], np.array([N - 1]), base)
    k_new = O.rope(k_raw[n][None], np.array([N]), base)
    wrong_pos = O.attention_rows(q_wrong, np.array([N]), np.concatenate([K, k_new]), np.concatenate([V, v[n][None]]),
                                 1.0 / math.sqrt(d))[0]
    for bad in (no_self, wrong_pos):
        assert np.abs(bad - good).max() > 10 * 2e-2 or np.abs(bad - good).mean() > 10 * 2e-3


# ---------------------------------------------------------------------------
# Scheme B ([ROPE] 3.2): K cached without position encoding, encoded on use
# ---------------------------------------------------------------------------

def _scheme_case(dtype, lens, q, k, Hq, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    nope = [O.round_to(rng.standard_normal((L, Hkv, d)), dtype) for L in lens]
    cv = [O.round_to(rng.standard_normal((L, Hkv, d)), dtype) for L in lens]
    n = O.count_rows(np.array(lens), q, k)
    q_raw = O.round_to(rng.standard_normal((n, Hq, d)), dtype)
    k_raw = O.round_to(rng.standard_normal((n, Hkv, d)), dtype)
    v = O.round_to(rng.standard_normal((n, Hkv, d)), dtype)
    return nope, cv, q_raw, k_raw, v


def test_scheme_b_equals_rotary_correction_exactly():
    """In exact arithmetic, caching K un-encoded and encoding it at s_c + j gives the
    same context and outputs as caching it encoded at j and rotating by s_c."""
    lens, q, k, Hq, Hkv, d, base = [7, 12, 5, 9], 4, 3, 4, 2, 16, 1e4
    nope, cv, q_raw, k_raw, v = _scheme_case("fp64", lens, q, k, Hq, Hkv, d, seed=31)
    compiled = [O.compile_chunk_k(x, base, "fp64") for x in nope]
    a = O.link_request(nope, cv, q, k, q_raw, k_raw, v, base, "fp64", scheme="nope")
    b = O.link_request(compiled, cv, q, k, q_raw, k_raw, v, base, "fp64", scheme="rotary")
    assert np.abs(a["K_ctx"] - b["K_ctx"]).max() < 1e-12
    assert np.abs(a["out"] - b["out"]).max() < 1e-12


def test_scheme_b_full_recompute():
    """With k >= every chunk length, scheme B's link equals full causal attention
    over the whole sequence (torch SDPA, float64)."""
    rng = np.random.default_rng(32)
    lens, q, Hq, Hkv, d, base = [5, 4, 6], 3, 4, 2, 16, 1e4
    N = sum(lens) + q
    q_raw = rng.standard_normal((N, Hq, d))
    k_raw = rng.standard_normal((N, Hkv, d))
    v = rng.standard_normal((N, Hkv, d))
    nope, cv, s = [], [], 0
    for L in lens:
        nope.append(k_raw[s:s + L])
        cv.append(v[s:s + L])
        s += L
    rows = O.select_rows(lens, q, max(lens))[0]
    res = O.link_request(nope, cv, q, max(lens), q_raw[rows], k_raw[rows], v[rows], base, "fp64", scheme="nope")
    fr = _full_recompute_sdpa(q_raw, k_raw, v, base, "fp64", Hq, Hkv)
    assert np.abs(res["out"] - fr[rows]).max() < 1e-12


def test_scheme_b_bf16_close_to_rotary():
    """In bf16, scheme B rounds once (RoPE at the global position) where rotary
    correction rounds twice (at the local position, then after the rotation).  A
    rotation keeps the norm of each dimension pair, so the two contexts differ by
    at most a few roundings of that norm: |a - b| <= 2^-7 |pair| per element."""
    lens, q, k, Hq, Hkv, d, base = [40, 33, 21], 2, 4, 4, 2, 32, 1e4
    nope, cv, q_raw, k_raw, v = _scheme_case("bf16", lens, q, k, Hq, Hkv, d, seed=33)
    compiled = [O.compile_chunk_k(x, base, "bf16") for x in nope]
    Ka = O.splice_context(nope, cv, q, k, k_raw, v, base, "bf16", "nope")[0]
    Kb = O.splice_context(compiled, cv, q, k, k_raw, v, base, "bf16", "rotary")[0]
    h = d // 2
    norm = np.sqrt(Ka[..., :h] ** 2 + Ka[..., h:] ** 2)
    norm = np.concatenate([norm, norm], axis=-1)
    assert (np.abs(Ka - Kb) <= 2.0 ** -7 * norm + 1e-30).all()
    assert np.abs(Ka - Kb).max() > 0  # the roundings do differ somewhere


def test_scheme_b_mutation_unencoded_chunk0_caught(monkeypatch):
    """Scheme B must encode chunk 0 as well (it is cached un-encoded): leaving it as
    cached moves the output far past the GPU tolerance."""
    lens, q, k, Hq, Hkv, d, base = [9, 7, 8], 3, 2, 4, 2, 16, 1e4
    nope, cv, q_raw, k_raw, v = _scheme_case("fp64", lens, q, k, Hq, Hkv, d, seed=34)
    good = O.link_request(nope, cv, q, k, q_raw, k_raw, v, base, "fp64", scheme="nope")["out"]
    real = O.rope_cached_k

    def skip_chunk0(k_nope, start, theta, dtype):
        return np.asarray(k_nope, np.float64) if start == 0 else real(k_nope, start, theta, dtype)

    monkeypatch.setattr(O, "rope_cached_k", skip_chunk0)
    bad = O.link_request(nope, cv, q, k, q_raw, k_raw, v, base, "fp64", scheme="nope")["out"]
    assert np.abs(bad - good).max() > 10 * 2e-2 or np.abs(bad - good).mean() > 10 * 2e-3


# ---------------------------------------------------------------------------
# Linear-layer state composition ([HYPIC] 2.1)
# ---------------------------------------------------------------------------

def _delta_rule_tokens(rng, L, dk, dv):
    """Gated delta rule: A_t = alpha_t (I - beta_t k_t k_t^T), B_t = beta_t k_t v_t^T."""
    k = rng.standard_normal((L, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, dv))
    alpha = rng.uniform(0.9, 1.0, L)
    beta = rng.uniform(0.1, 0.9, L)
    A = np.stack([alpha[t] * (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) for t in range(L)])
    B = np.stack([beta[t] * np.outer(k[t], v[t]) for t in range(L)])
    return A, B


@pytest.mark.parametrize("family", ["delta", "retnet"])
def test_composition_equals_token_recurrence(family):
    """Composing cached per-segment (T_C, S(C|0)) reproduces the state of the token
    recurrence over the concatenated segments."""
    rng = np.random.default_rng(41)
    dk, dv, lens = 8, 6, [5, 9, 3, 7]
    segs = []
    for L in lens:
        if family == "delta":
            A, B = _delta_rule_tokens(rng, L, dk, dv)
        else:
            A = np.stack([0.97 * np.eye(dk)] * L)
            B = np.einsum("ti,tj->tij", rng.standard_normal((L, dk)), rng.standard_normal((L, dv)))
        segs.append((A, B))
    T, S = zip(*[O.segment_operator(A, B) for A, B in segs])
    direct = O.recurrence(np.concatenate([a for a, _ in segs]), np.concatenate([b for _, b in segs]))
    assert np.abs(O.compose_states(np.array(T), np.array(S)) - direct).max() < 1e-12


def test_composition_is_associative():
    """Composing sub-chains first (a scan in any tree order) gives the same state."""
    rng = np.random.default_rng(42)
    d, n = 6, 9
    T = 0.9 * np.eye(d) + 0.05 * rng.standard_normal((n, d, d))
    S = rng.standard_normal((n, d, d))
    seq = O.compose_states(T, S)
    # (0..3) then (4..8) as sub-chains: T of a sub-chain is the product of its T
    def sub(a, b):
        Tp = np.eye(d)
        for i in range(a, b):
            Tp = T[i] @ Tp
        return Tp, O.compose_states(T[a:b], S[a:b])
    (T1, S1), (T2, S2) = sub(0, 4), sub(4, 9)
    assert np.abs(T2 @ S1 + S2 - seq).max() < 1e-12


def test_naive_sum_exact_only_without_transition():
    """Plain linear attention (A_t = I): composition is the plain sum of the segment
    states.  With decay the sum drops T(C2) and is structurally wrong."""
    rng = np.random.default_rng(43)
    d, n = 6, 5
    S = rng.standard_normal((n, d, d))
    assert np.abs(O.compose_states(np.stack([np.eye(d)] * n), S) - S.sum(0)).max() < 1e-12
    T = np.stack([0.8 * np.eye(d)] * n)
    good = O.compose_states(T, S)
    assert np.linalg.norm(good - S.sum(0)) > 0.2 * np.linalg.norm(good)
