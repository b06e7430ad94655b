"""Helpers that run the oracle on a LinkBatch's inputs and compare the CUDA results."""

import numpy as np
import torch

import oracle.pic_oracle as O
from position_independent_kv_pic_gb300 import inputs

TOL_MAX, TOL_MEAN = 2e-2, 2e-3   # attention: fp32 accumulate, bf16 out


def request_inputs(batch, r):
    """float64 views of request r's stored chunks and recomputed-row inputs."""
    wl = batch.wl
    req = wl.requests[r]
    a, b = int(batch.offs["row_off"][r]), int(batch.offs["row_off"][r + 1])
    chunks_k = [batch.store_k[batch.store_off[c]:batch.store_off[c + 1]].double().numpy() for c in req.chunk_ids]
    chunks_v = [batch.store_v[batch.store_off[c]:batch.store_off[c + 1]].double().numpy() for c in req.chunk_ids]
    return (chunks_k, chunks_v, req.q, req.k, batch.q_raw_h[a:b].double().numpy(),
            batch.k_new_h[a:b].double().numpy(), batch.v_new_h[a:b].double().numpy())


def oracle_request(batch, r, which=None, scheme="rotary"):
    wl = batch.wl
    ck, cv, q, k, qr, kn, vn = request_inputs(batch, r)
    return O.link_request(ck, cv, q, k, qr, kn, vn, wl.theta, wl.dtype, which=which, scheme=scheme)


# Oracle outputs of whole requests of the preset workloads, kept for the session:
# the rotary-correction and rotate-on-read steps of one preset share their inputs,
# so they share the oracle's answer (the oracle's cost dominates these tests).
_ORACLE_CACHE = {}


def oracle_out(batch, r, scheme="rotary"):
    """float64 oracle output [n_rows(r)][Hq][d] of request r (every row)."""
    wl = batch.wl
    key = (wl.name, wl.seed, r, scheme) if wl.name in inputs.PRESETS else None
    if key is not None and key in _ORACLE_CACHE:
        return _ORACLE_CACHE[key]
    out = oracle_request(batch, r, scheme=scheme)["out"]
    if key is not None:
        _ORACLE_CACHE[key] = out
    return out


def bf16_ulp(x):
    x = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(np.maximum(x, 2.0 ** -126))
    return np.ldexp(1.0, e - 8)


def storage_ulp(x, dtype):
    if dtype == "bf16":
        return bf16_ulp(x)
    x = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(np.maximum(x, 2.0 ** -126))
    return np.ldexp(1.0, e - 24)


def check_rows(batch):
    rows = batch.rows.cpu().numpy()
    starts = batch.chunk_start.cpu().numpy()
    for r, req in enumerate(batch.wl.requests):
        lens = batch.wl.chunk_lens[req.chunk_ids]
        o_rows, o_starts, _ = O.select_rows(lens, req.q, req.k)
        a, b = batch.offs["row_off"][r], batch.offs["row_off"][r + 1]
        assert np.array_equal(rows[a:b], o_rows), f"rows of request {r}"
        c0, c1 = batch.chunk_off[r], batch.chunk_off[r + 1]
        assert np.array_equal(starts[c0:c1], o_starts), f"chunk starts of request {r}"


def check_rerotated_k(batch, max_chunks=None):
    """Every cached, non-recomputed K of every linked chunk within 1 ulp of the oracle;
    chunk 0 of each request bit-identical to the stored chunk."""
    wl = batch.wl
    starts = batch.chunk_start.cpu().numpy()
    worst = 0.0
    for r, req in enumerate(wl.requests):
        c0, c1 = int(batch.chunk_off[r]), int(batch.chunk_off[r + 1])
        for ci, c in enumerate(range(c0, c1)):
            if max_chunks is not None and ci >= max_chunks and c < c1 - 1:
                continue
            sid = int(batch.flat_store_ids[c])
            stored = batch.store_k[batch.store_off[sid]:batch.store_off[sid + 1]].double().numpy()
            got = batch.rotated_chunk_k(c).double().numpy()
            if ci == 0:
                assert np.array_equal(got, stored), f"chunk 0 of request {r} changed"
                continue
            m = min(req.k, stored.shape[0])
            if m == stored.shape[0]:
                continue
            expect = O.rerotate_k(stored[m:], int(starts[c]), wl.theta, wl.dtype)
            diff = np.abs(got[m:] - expect)
            ratio = (diff / storage_ulp(expect, wl.dtype)).max()
            worst = max(worst, float(ratio))
            # bf16: within one ulp of the exactly rounded rotation.  fp32: the
            # compensated rotation is good to ~2^-23 relative, i.e. a few fp32 ulps.
            bound = 1.0 if wl.dtype == "bf16" else 4.0
            assert ratio <= bound, f"request {r} chunk {ci}: {ratio} ulp"
    return worst


def sample_rows(n, k_first=8, k_last=8, k_rand=16, seed=0):
    rng = np.random.default_rng(seed)
    idx = set(range(min(n, k_first))) | set(range(max(0, n - k_last), n))
    if n > 0:
        idx |= set(rng.choice(n, size=min(n, k_rand), replace=False).tolist())
    return sorted(idx)


def check_attention(batch, which_per_request=None, scheme="rotary"):
    """Max-abs and mean-abs error of the attention output against the oracle
    (every row of every request unless ``which_per_request`` picks rows)."""
    out = batch.out.double().cpu().numpy()
    errs = []
    for r in range(batch.n_req):
        a, b = int(batch.offs["row_off"][r]), int(batch.offs["row_off"][r + 1])
        if b == a:
            continue
        if which_per_request is None:
            errs.append(np.abs(out[a:b] - oracle_out(batch, r, scheme)).reshape(-1))
        else:
            which = which_per_request(b - a)
            res = oracle_request(batch, r, which, scheme)
            errs.append(np.abs(out[a:b][which] - res["out"][which]).reshape(-1))
    if not errs:
        return 0.0, 0.0
    e = np.concatenate(errs)
    assert np.isfinite(e).all()
    return float(e.max()), float(e.mean())


def frame_positions(rows, starts, T):
    """Positions at which the framed layout encodes recomputed rows' fresh K: a seam
    row's position within its chunk, a query row's global position."""
    c = np.searchsorted(starts, rows, side="right") - 1
    return np.where(rows >= T, rows, rows - starts[c])


def check_fresh_kv(batch):
    """a4, read back from the pools: the slot of every recomputed row (row_block,
    row_slot from the splice) holds K = RoPE(K_new, p_r) rounded to the pool dtype,
    within one ulp of the oracle's rounding of the float64 rotation, and V = V_new
    bit for bit.  p_r comes from the oracle's row selection: the global position, or
    in the framed layout (rotate-on-read) the position in the row's frame.  Returns
    the worst K error in ulps."""
    wl = batch.wl
    if batch.n_rows == 0:
        return 0.0
    blk, slot = batch.row_block.long(), batch.row_slot.long()
    k_got = batch.k_pool[blk, :, slot, :].double().cpu().numpy()
    v_got = batch.v_pool[blk, :, slot, :].cpu()
    assert torch.equal(v_got, batch.v_new_h), "fresh V differs from V_new"
    worst = 0.0
    bound = 1.0 if wl.dtype == "bf16" else 4.0
    for r, req in enumerate(wl.requests):
        a, b = int(batch.offs["row_off"][r]), int(batch.offs["row_off"][r + 1])
        if b == a:
            continue
        rows, starts, T = O.select_rows(wl.chunk_lens[req.chunk_ids], req.q, req.k)
        pos = frame_positions(rows, starts, T) if batch.scheme == "ror" else rows
        expect = O.round_to(O.rope(batch.k_new_h[a:b].double().numpy(), pos, wl.theta), wl.dtype)
        ratio = float((np.abs(k_got[a:b] - expect) / storage_ulp(expect, wl.dtype)).max())
        worst = max(worst, ratio)
        assert ratio <= bound, f"fresh K of request {r}: {ratio} ulp"
    return worst
