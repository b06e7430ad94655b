"""Oracle for the PIC link step.  TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 CPU restatement of what the link step computes (NumPy,
and PyTorch CPU operations for the attention's products).  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import it; the product path (the CUDA library and its binding)
never does.  It shares no code, tables or constants with the CUDA path and works
on dense per-chunk arrays (no pages, no tables, no tiling).

Sources (page title, then section):
  [EPIC]  blog review "EPIC: Efficient Position-Independent Caching for Serving
          Large Language Models" (juhe.plus): the compile/link walk-through
          (chunks of 4, 5, 5 tokens + a 3-token query), ``link_legolink``
          Steps 1-3, the method comparison table and the k-sweep table (Step 5).
  [ROPE]  article on RoPE and prefix caching (10100.com): section 2.2 (RoPE
          rotates dimension pairs by an angle proportional to the position;
          q.k depends only on the position difference), section 3.3 (rotary
          correction: a cached K at position a is moved to position b by one
          rotation by b - a), footnote 3 (inv_freq = 1 / base^(2i/d), HF Llama).
  [HYPIC] HYPIC article (joto.ai), section 2.2: the first w tokens of every
          internal segment (seam window) are recomputed under the full prefix.
  [KVC]   blog "KV cache from scratch: two-layer decoder, position offset and
          correctness checks" (chenhuiyu.github.io), section on the offset
          causal mask: allowed[i, j] = [j <= P + i].

Readings where the pages are silent or garbled:
  * RoPE pairs dimension i with i + d/2 (HF Llama "rotate half", [ROPE] fn. 3);
    no frequency scaling.
  * A chunk compiled at local positions 0..L-1 and placed at start s_c is moved
    to its global positions by one rotation by Delta_c = s_c ([ROPE] 3.3).
  * Chunk 0 (in link order) is never recomputed; every query row is
    ([EPIC] Step 1).  Recomputed rows of chunk c are its first min(k, L_c) tokens.
  * Masked keys are left out of the softmax (not added as a large negative);
    the scale is 1/sqrt(d) ([EPIC] Step 3, [KVC] mask section).
  * GQA: query head h reads KV head floor(h / (Hq/Hkv)) (contiguous groups).
  * Rounding mirrors storage: every value the link step stores (re-rotated K,
    fresh K, the position-encoded Q that feeds the matrix unit) is rounded to the
    storage dtype (bf16 round-to-nearest-even, or fp32) once; everything else is
    float64.  The softmax weights are not rounded.

Parity pins for every function here live in tests/test_oracle_pins.py.
"""

from __future__ import annotations

import math

import numpy as np
import torch

__all__ = [
    "select_rows", "count_rows", "inv_freq", "rope", "round_to", "compile_chunk_k",
    "rerotate_k", "visible", "query_positions", "splice_context", "attention_rows",
    "link_request",
]


# ---------------------------------------------------------------------------
# Row selection  ([EPIC] link_legolink Step 1 and the worked example)
# ---------------------------------------------------------------------------

def select_rows(chunk_lens, q: int, k: int):
    """LegoLink-k row selection.

    Walk the chunks in link order keeping a running offset (the chunk's start
    s_c).  Every chunk except the first contributes its first min(k, L_c) tokens;
    then all q query tokens (global positions T .. T+q-1) are appended.

    Returns (rows, starts, T): rows int64 [n_sel] ascending global positions,
    starts int64 [C] the chunk starts s_c, T the total cached length.
    """
    if k < 0 or q < 0:
        raise ValueError("k and q must be >= 0")
    rows, starts, offset = [], [], 0
    for c, L in enumerate(chunk_lens):
        L = int(L)
        if L < 1:
            raise ValueError("every chunk needs at least one token")
        starts.append(offset)
        if c > 0:
            for j in range(min(k, L)):
                rows.append(offset + j)
        offset += L
    T = offset
    rows.extend(range(T, T + q))
    return np.array(rows, np.int64), np.array(starts, np.int64), T


def count_rows(chunk_lens, q: int, k: int) -> int:
    """Number of recomputed rows of one request (length of select_rows)."""
    return len(select_rows(chunk_lens, q, k)[0])


# ---------------------------------------------------------------------------
# RoPE  ([ROPE] 2.2, footnote 3)
# ---------------------------------------------------------------------------

def inv_freq(d: int, theta: float) -> np.ndarray:
    """theta_i = base^(-2i/d) for i = 0 .. d/2-1 (float64 pow)."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / d)


def rope(x, pos, theta: float) -> np.ndarray:
    """Rotate every pair (x_i, x_{i+d/2}) of the last axis by the angle pos * theta_i.

    ``x`` has shape [n, ..., d]; ``pos`` has one position per leading index
    (shape [n]).  y_i = x_i cos - x_{i+d/2} sin,  y_{i+d/2} = x_{i+d/2} cos + x_i sin.
    """
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    h = d // 2
    p = np.asarray(pos, np.float64).reshape((x.shape[0],) + (1,) * (x.ndim - 1))
    ang = p * inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def round_to(x, dtype: str) -> np.ndarray:
    """Round float64 values to the storage dtype and return them as float64.

    bf16: round to 8 significant bits, ties to even (np.rint rounds half to even);
    valid for values that are zero or in bf16's normal range, which covers every
    value the workloads produce.  fp32: IEEE float32 conversion (ties to even).
    fp64: no rounding (exact-arithmetic mode, used by the oracle's own pins).
    """
    x = np.asarray(x, np.float64)
    if dtype == "fp64":
        return x
    if dtype == "bf16":
        m, e = np.frexp(x)
        return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    if dtype == "fp32":
        return x.astype(np.float32).astype(np.float64)
    raise ValueError(dtype)


def compile_chunk_k(k_raw, theta: float, dtype: str) -> np.ndarray:
    """What a chunk compiled on its own stores: K roped at local positions 0..L-1
    ([EPIC] compile_chunk, positions from 0)."""
    k_raw = np.asarray(k_raw, np.float64)
    return round_to(rope(k_raw, np.arange(k_raw.shape[0]), theta), dtype)


def rerotate_k(k_stored, delta: int, theta: float, dtype: str) -> np.ndarray:
    """Rotary correction ([ROPE] 3.3): move a cached K from local to global positions
    with ONE rotation by Delta, then store it (round to dtype)."""
    k_stored = np.asarray(k_stored, np.float64)
    return round_to(rope(k_stored, np.full(k_stored.shape[0], delta), theta), dtype)


# ---------------------------------------------------------------------------
# Mask and positions  ([KVC] offset causal mask; [EPIC] Step 2, global positions)
# ---------------------------------------------------------------------------

def visible(key_pos, query_pos) -> np.ndarray:
    """Causal visibility of keys at ``key_pos`` for a query at ``query_pos``."""
    return np.asarray(key_pos) <= query_pos


def query_positions(rows, starts, T):
    """Positions at which recomputed rows are encoded: their global positions."""
    return np.asarray(rows, np.int64)


# ---------------------------------------------------------------------------
# Splice and attention  ([EPIC] Step 3; [HYPIC] 2.2)
# ---------------------------------------------------------------------------

def rope_cached_k(k_nope, start: int, theta: float, dtype: str) -> np.ndarray:
    """Scheme B ([ROPE] 3.2): a chunk's K cached without its position encoding is
    encoded on use at its global positions start + j, then stored (rounded once)."""
    k_nope = np.asarray(k_nope, np.float64)
    return round_to(rope(k_nope, start + np.arange(k_nope.shape[0]), theta), dtype)


def splice_context(chunks_k, chunks_v, q, k, k_new_raw, v_new, theta, dtype, scheme="rotary"):
    """Build the spliced K/V of one request at global positions.

    Cached chunks are concatenated in link order.  scheme "rotary" (rotary
    correction, [ROPE] 3.3): chunk c's K was cached encoded at local positions and
    is re-rotated by Delta_c = s_c.  scheme "nope" (scheme B, [ROPE] 3.2): chunk
    c's K was cached without position encoding and is encoded at s_c + j.  Then
    the recomputed rows' fresh K (roped at their global position) and fresh V
    overwrite / append at their positions.

    Returns (K_ctx, V_ctx, rows, starts, T) with K_ctx, V_ctx float64 [T+q][Hkv][d].
    """
    lens = [int(c.shape[0]) for c in chunks_k]
    rows, starts, T = select_rows(lens, q, k)
    Hkv, d = chunks_k[0].shape[1], chunks_k[0].shape[2]
    N = T + q
    K = np.zeros((N, Hkv, d), np.float64)
    V = np.zeros((N, Hkv, d), np.float64)
    for c, (kc, vc) in enumerate(zip(chunks_k, chunks_v)):
        s = int(starts[c])
        if scheme == "rotary":
            K[s:s + lens[c]] = rerotate_k(kc, s, theta, dtype)
        elif scheme == "nope":
            K[s:s + lens[c]] = rope_cached_k(kc, s, theta, dtype)
        else:
            raise ValueError(scheme)
        V[s:s + lens[c]] = np.asarray(vc, np.float64)
    if len(rows):
        K[rows] = round_to(rope(k_new_raw, rows, theta), dtype)
        V[rows] = np.asarray(v_new, np.float64)
    return K, V, rows, starts, T


def attention_rows(q_rot, q_pos, K_ctx, V_ctx, scale, which=None, group=16) -> np.ndarray:
    """Masked softmax attention of position-encoded queries over the spliced context.

    q_rot [n][Hq][d], q_pos [n]; key j sits at global position j.  For every
    selected row and head: O = sum_j softmax_j(q.K_j * scale) V_j over visible j,
    KV head floor(h/g).  ``which`` restricts the rows computed (others are NaN).

    Rows are independent.  They are taken ``group`` at a time so that one matrix
    product per KV head serves the group's g * group query vectors; each row keeps
    its own visibility mask (built by ``visible`` for that row alone), masked
    scores are -inf and so get weight exactly 0.  Everything is float64; the
    products and elementwise passes are PyTorch CPU operations, which use every
    host core.
    """
    n, Hq, d = q_rot.shape
    N, Hkv, _ = K_ctx.shape
    g = Hq // Hkv
    Q = torch.from_numpy(np.ascontiguousarray(q_rot, np.float64))
    Kt = torch.from_numpy(np.ascontiguousarray(np.asarray(K_ctx, np.float64).transpose(1, 0, 2)))  # [Hkv][N][d]
    Vt = torch.from_numpy(np.ascontiguousarray(np.asarray(V_ctx, np.float64).transpose(1, 0, 2)))
    key_pos = np.arange(N)
    out = torch.full((n, Hq, d), float("nan"), dtype=torch.float64)
    todo = list(range(n)) if which is None else [int(i) for i in which]
    for b0 in range(0, len(todo), group):
        sel = todo[b0:b0 + group]
        vis = np.stack([visible(key_pos, int(q_pos[i])) for i in sel])   # [nb][N]
        if not vis.any(axis=1).all():
            raise ValueError("a query row sees no key")
        last = int(np.flatnonzero(vis.any(axis=0))[-1]) + 1
        mask = torch.from_numpy(vis[:, None, :last])                        # [nb][1][last]
        nb = len(sel)
        idx = torch.tensor(sel, dtype=torch.int64)
        for h in range(Hkv):
            qh = Q[idx, h * g:(h + 1) * g, :].reshape(nb * g, d)
            s = (qh @ Kt[h, :last].T).reshape(nb, g, last)
            s.mul_(scale)
            s.masked_fill_(~mask, float("-inf"))
            s.sub_(s.amax(dim=2, keepdim=True))
            s.exp_()
            s.div_(s.sum(dim=2, keepdim=True))
            out[idx, h * g:(h + 1) * g, :] = (s.reshape(nb * g, last) @ Vt[h, :last]).reshape(nb, g, d)
    return out.numpy()


def link_request(chunks_k, chunks_v, q, k, q_raw, k_new_raw, v_new, theta, dtype,
                 scale=None, which=None, scheme="rotary"):
    """The whole link step of one request.

    chunks_k / chunks_v: lists of stored per-chunk K / V, each [L_c][Hkv][d]
    (float64 values of the stored dtype), in link order.  q_raw [n_sel][Hq][d],
    k_new_raw / v_new [n_sel][Hkv][d]: the recomputed rows' un-roped Q, K and V.
    Returns dict(rows, starts, T, K_ctx, V_ctx, out) with out float64 [n_sel][Hq][d].
    """
    K, V, rows, starts, T = splice_context(chunks_k, chunks_v, q, k, k_new_raw, v_new,
                                           theta, dtype, scheme)
    d = K.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qpos = query_positions(rows, starts, T)
    q_rot = round_to(rope(q_raw, qpos, theta), dtype) if len(rows) else np.zeros((0,) + np.shape(q_raw)[1:])
    out = attention_rows(q_rot, qpos, K, V, scale, which)
    return dict(rows=rows, starts=starts, T=T, K_ctx=K, V_ctx=V, out=out)


# ---------------------------------------------------------------------------
# Decode after link  ([EPIC] the query and decode tokens gather the information;
# [KVC] single-token cache decode: the new position is encoded, its K/V appended,
# and its query reads every cached position)
# ---------------------------------------------------------------------------

def decode_after_link(K_ctx, V_ctx, q_raw, k_raw, v_raw, theta, dtype, scale=None):
    """One decode row after a link step.

    K_ctx / V_ctx [N][Hkv][d]: the linked context (cached chunks, recomputed rows and
    query rows at positions 0..N-1, as ``link_request`` returns it).  The new token
    sits at position P = N: its K is roped at P and stored (rounded to dtype), its V
    stored, and its Q (roped at P, rounded as every tensor-core operand) attends
    over keys 0..P.  q_raw [Hq][d], k_raw / v_raw [Hkv][d] (un-roped).
    Returns out [Hq][d] float64.
    """
    N, Hkv, d = K_ctx.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pos = np.array([N])
    k_new = round_to(rope(np.asarray(k_raw, np.float64)[None], pos, theta), dtype)
    K = np.concatenate([K_ctx, k_new], axis=0)
    V = np.concatenate([V_ctx, round_to(np.asarray(v_raw, np.float64)[None], dtype)], axis=0)
    q_rot = round_to(rope(np.asarray(q_raw, np.float64)[None], pos, theta), dtype)
    return attention_rows(q_rot, pos, K, V, scale)[0]


# ---------------------------------------------------------------------------
# Linear-attention layers  ([HYPIC] 2.1: cache each segment's transition operator)
# ---------------------------------------------------------------------------
# A linear-attention layer keeps a state S (d_k x d_v) per head, updated per token
# as S_t = A_t S_{t-1} + B_t (A_t: d_k x d_k transition -- identity for plain
# linear attention, gamma I for RetNet, alpha_t (I - beta_t k_t k_t^T) for the
# gated delta rule; B_t: the token's rank-one write).  A segment C of tokens is
# summarised by its cumulative transition T_C = A_L ... A_1 and its end state from
# zero S(C|0); both depend only on the segment's own tokens.

def recurrence(A, B, S0=None) -> np.ndarray:
    """End state of S_t = A_t S_{t-1} + B_t over the tokens (A [L][dk][dk], B [L][dk][dv])."""
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    S = np.zeros(B.shape[1:]) if S0 is None else np.asarray(S0, np.float64).copy()
    for t in range(A.shape[0]):
        S = A[t] @ S + B[t]
    return S


def segment_operator(A, B):
    """(T_C, S(C|0)) of one segment from its tokens."""
    A = np.asarray(A, np.float64)
    T = np.eye(A.shape[1])
    for t in range(A.shape[0]):
        T = A[t] @ T
    return T, recurrence(A, B)


def compose_states(T, S) -> np.ndarray:
    """End state of a chain of segments from their cached (T_c, S_c), in chain order:
    S(C1 C2) = T(C2) S(C1) + S(C2), applied left to right.  T, S [n][d][d]."""
    T = np.asarray(T, np.float64)
    S = np.asarray(S, np.float64)
    acc = S[0].copy()
    for i in range(1, S.shape[0]):
        acc = T[i] @ acc + S[i]
    return acc
