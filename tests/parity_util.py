"""Helpers that run the oracle on a LinkBatch's inputs and compare the CUDA results."""

import numpy as np
import torch

import oracle.pic_oracle as O

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


def oracle_request(batch, r, which=None):
    wl = batch.wl
    ck, cv, q, k, qr, kn, vn = request_inputs(batch, r)
    return O.link_request(ck, cv, q, k, qr, kn, vn, wl.theta, wl.dtype, which=which)


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


def check_attention(batch, which_per_request=None):
    """Max-abs and mean-abs error of the attention output against the oracle."""
    out = batch.out.double().cpu().numpy()
    errs = []
    for r in range(batch.n_req):
        a, b = int(batch.offs["row_off"][r]), int(batch.offs["row_off"][r + 1])
        if b == a:
            continue
        which = None if which_per_request is None else which_per_request(b - a)
        res = oracle_request(batch, r, which)
        sel = list(range(b - a)) if which is None else which
        errs.append(np.abs(out[a:b][sel] - res["out"][sel]).reshape(-1))
    if not errs:
        return 0.0, 0.0
    e = np.concatenate(errs)
    assert np.isfinite(e).all()
    return float(e.max()), float(e.mean())
