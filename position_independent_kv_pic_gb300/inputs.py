"""Seeded synthetic workloads for the PIC link step.

This module only draws random inputs and describes their structure (chunk
lengths, link order, query length, k, physical block placement). It holds
none of the method's arithmetic: no row selection, no RoPE, no attention.
Both the oracle-side tests and the CUDA path are fed from here.

Value recipe: every tensor is drawn as float32 N(0, 1) from NumPy's PCG64
(``default_rng``), one spawned sub-stream per role, then cast to the storage
dtype with round-to-nearest-even (torch's float32 -> bfloat16 conversion).

Cached K is drawn directly as the *stored* (already position-encoded) key of
each chunk.  A chunk compiled at local positions 0..L-1 stores
RoPE(K_raw, j); for K_raw with i.i.d. N(0,1) entries each rotated pair is
again i.i.d. N(0,1), so drawing the stored key directly has the same
distribution as compiling a Gaussian K_raw.  The attention-sink workload
scales the stored key at local position 0 of every chunk by 4 (RoPE at
position 0 is the identity, so this equals scaling K_raw there).

Workload shapes follow the RAG prompts the EPIC / HYPIC pages describe
(a few to ~100 retrieved chunks, up to ~100k tokens, 16-token KV pages).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 16  # tokens per KV page

_STREAMS = ("lens", "order", "q", "kstore", "vstore", "knew", "vnew", "blocks", "qlen", "decode", "states")


@dataclass
class Request:
    chunk_ids: np.ndarray  # int32 [C] ids into the chunk store, in link order
    q: int                 # query length
    k: int                 # LegoLink k (seam window)


@dataclass
class Workload:
    name: str
    Hq: int
    Hkv: int
    d: int
    theta: float
    dtype: str                      # "bf16" or "fp32"
    chunk_lens: np.ndarray          # int32 [n_store] lengths of the distinct cached chunks
    requests: list = field(default_factory=list)
    sink_scale: float = 1.0         # factor on the stored K at local position 0
    out_of_place: bool = False      # rotate K into per-request pages (shared chunks)
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def total_tokens(self) -> int:
        """Sum over requests of (sum of linked chunk lengths + query length)."""
        return int(sum(int(self.chunk_lens[r.chunk_ids].sum()) + r.q for r in self.requests))


def _rngs(seed: int) -> dict:
    ss = np.random.SeedSequence(seed)
    return {name: np.random.default_rng(s) for name, s in zip(_STREAMS, ss.spawn(len(_STREAMS)))}


# --------------------------------------------------------------------------
# Workload presets (structure only; tensors are drawn by the functions below)
# --------------------------------------------------------------------------

def worked_example(seed: int = 1) -> Workload:
    """EPIC blog's LegoLink walk-through: chunks of 4, 5, 5 tokens + 3-token query, k=2.
    Tiny fp32 layer: Hq=4, Hkv=2, d=16, RoPE base 1e4."""
    wl = Workload("worked_example_fp32", 4, 2, 16, 1.0e4, "fp32",
                  np.array([4, 5, 5], np.int32), seed=seed)
    wl.requests = [Request(np.arange(3, dtype=np.int32), 3, 2)]
    return wl


def rag_prompt(seed: int = 2) -> Workload:
    """RAG prompt on a Llama-3-8B-shaped attention layer (Hq=32, Hkv=8, d=128, base 5e5):
    a 128-token system chunk + 5 retrieved chunks of 512 tokens + 64-token query, k=16."""
    lens = np.array([128] + [512] * 5, np.int32)
    wl = Workload("rag_prompt_6chunks", 32, 8, 128, 5.0e5, "bf16", lens, seed=seed)
    wl.requests = [Request(np.arange(6, dtype=np.int32), 64, 16)]
    return wl


def many_chunk(seed: int = 3) -> Workload:
    """20 chunks with lengths uniform in [512, 2048] + 128-token query, k=8; the stored K of
    every chunk's first token is scaled by 4 to mimic attention sinks."""
    r = _rngs(seed)
    lens = r["lens"].integers(512, 2049, size=20).astype(np.int32)
    wl = Workload("many_chunk_sink_20", 32, 8, 128, 5.0e5, "bf16", lens, sink_scale=4.0, seed=seed)
    wl.requests = [Request(np.arange(20, dtype=np.int32), 128, 8)]
    return wl


def long_context(seed: int = 4, n_chunks: int = 100, chunk_len: int = 1000, q: int = 256,
                 k: int = 8) -> Workload:
    """100 chunks x 1000 tokens + 256-token query (~100k tokens), k=8 (seam window w=8).
    The chunks are linked in a random order relative to how they sit in the cache."""
    r = _rngs(seed)
    lens = np.full(n_chunks, chunk_len, np.int32)
    order = r["order"].permutation(n_chunks).astype(np.int32)
    wl = Workload(f"long_context_{n_chunks}x{chunk_len}", 32, 8, 128, 5.0e5, "bf16", lens, seed=seed)
    wl.requests = [Request(order, q, k)]
    return wl


def batched_shared(seed: int = 5, n_req: int = 16, n_store: int = 64) -> Workload:
    """16 requests, each linking 3-30 distinct chunks drawn from a shared store of 64 chunks
    (lengths uniform in [256, 4096]) + a 32-256-token query; k=2 for even and k=16 for odd
    requests.  The same chunk lands at different offsets in different requests, so K is
    rotated out of place into per-request pages while V pages stay shared."""
    r = _rngs(seed)
    lens = r["lens"].integers(256, 4097, size=n_store).astype(np.int32)
    wl = Workload(f"batched_shared_{n_req}req", 32, 8, 128, 5.0e5, "bf16", lens,
                  out_of_place=True, seed=seed)
    for i in range(n_req):
        n_c = int(r["order"].integers(3, 31))
        ids = r["order"].choice(n_store, size=n_c, replace=False).astype(np.int32)
        q = int(r["qlen"].integers(32, 257))
        wl.requests.append(Request(ids, q, 2 if i % 2 == 0 else 16))
    return wl


PRESETS = {
    "worked_example_fp32": worked_example,
    "rag_prompt_6chunks": rag_prompt,
    "many_chunk_sink_20": many_chunk,
    "long_context_100x1000": long_context,
    "batched_shared_16req": batched_shared,
}


def custom(chunk_lens_per_request, qs, ks, Hq=4, Hkv=2, d=16, theta=1.0e4, dtype="fp32",
           seed=0, sink_scale=1.0, out_of_place=False, name="custom") -> Workload:
    """A workload where request i links its own private chunks ``chunk_lens_per_request[i]``."""
    lens, reqs, base = [], [], 0
    for cl, q, k in zip(chunk_lens_per_request, qs, ks):
        cl = [int(x) for x in cl]
        lens.extend(cl)
        reqs.append(Request(np.arange(base, base + len(cl), dtype=np.int32), int(q), int(k)))
        base += len(cl)
    wl = Workload(name, Hq, Hkv, d, float(theta), dtype, np.array(lens, np.int32),
                  sink_scale=sink_scale, out_of_place=out_of_place, seed=seed)
    wl.requests = reqs
    return wl


# --------------------------------------------------------------------------
# Tensor draws
# --------------------------------------------------------------------------

def _cast(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def chunk_store(wl: Workload):
    """Stored (compiled) K and V of every distinct chunk, concatenated along tokens.

    Returns (K, V, off): K, V are CPU tensors [sum(L)][Hkv][d] in the workload dtype and
    ``off`` int64 [n_store+1] gives each chunk's token range."""
    r = _rngs(wl.seed)
    n = int(wl.chunk_lens.sum())
    off = np.zeros(len(wl.chunk_lens) + 1, np.int64)
    off[1:] = np.cumsum(wl.chunk_lens)
    k = r["kstore"].standard_normal((n, wl.Hkv, wl.d), dtype=np.float32)
    if wl.sink_scale != 1.0:
        k[off[:-1]] *= np.float32(wl.sink_scale)
    v = r["vstore"].standard_normal((n, wl.Hkv, wl.d), dtype=np.float32)
    return _cast(k, wl.dtype), _cast(v, wl.dtype), off


def row_inputs(wl: Workload, n_rows: int):
    """Per-row inputs of the recomputed rows, for ``n_rows`` rows in total over all requests:
    Q_raw [n_rows][Hq][d] (not yet position-encoded), K_new_raw [n_rows][Hkv][d]
    (not yet position-encoded) and V_new [n_rows][Hkv][d]."""
    r = _rngs(wl.seed)
    q = r["q"].standard_normal((n_rows, wl.Hq, wl.d), dtype=np.float32)
    kn = r["knew"].standard_normal((n_rows, wl.Hkv, wl.d), dtype=np.float32)
    vn = r["vnew"].standard_normal((n_rows, wl.Hkv, wl.d), dtype=np.float32)
    return _cast(q, wl.dtype), _cast(kn, wl.dtype), _cast(vn, wl.dtype)


def decode_inputs(wl: Workload):
    """Inputs of one decode row per request: Q_raw [n_req][Hq][d], K_raw [n_req][Hkv][d]
    (not yet position-encoded) and V [n_req][Hkv][d]."""
    r = _rngs(wl.seed)["decode"]
    n = len(wl.requests)
    q = r.standard_normal((n, wl.Hq, wl.d), dtype=np.float32)
    k = r.standard_normal((n, wl.Hkv, wl.d), dtype=np.float32)
    v = r.standard_normal((n, wl.Hkv, wl.d), dtype=np.float32)
    return _cast(q, wl.dtype), _cast(k, wl.dtype), _cast(v, wl.dtype)


def linear_states(wl: Workload, H: int = 32, d: int = 128):
    """Cached per-chunk pairs (T_c, S_c) of a linear-attention layer with H heads and
    d x d states (HYPIC blog, section 2.1), for every distinct chunk of the workload,
    and each request's chain of chunk ids in link order.

    Recipe: T_c = g I + E with g ~ U[0.5, 0.75] per (chunk, head) and E i.i.d.
    N(0, 0.01 / d) (so the spectral norm of T_c stays below about 0.95, like a
    decayed delta-rule transition), S_c i.i.d. N(0, 1).  Returns (T, S, chains):
    T, S float32 CPU tensors [n_store][H][d][d], chains a list of int32 arrays."""
    r = _rngs(wl.seed)["states"]
    n = len(wl.chunk_lens)
    g = r.uniform(0.5, 0.75, size=(n, H, 1, 1)).astype(np.float32)
    T = r.standard_normal((n, H, d, d), dtype=np.float32)
    T *= np.float32(0.1 / np.sqrt(d))
    T += g * np.eye(d, dtype=np.float32)
    S = r.standard_normal((n, H, d, d), dtype=np.float32)
    return torch.from_numpy(T), torch.from_numpy(S), [np.asarray(q.chunk_ids, np.int32) for q in wl.requests]


def block_shuffle(wl: Workload, n_blocks: int) -> np.ndarray:
    """A seeded permutation of physical block ids, so that logically adjacent pages land
    at scattered places in the pool."""
    return _rngs(wl.seed)["blocks"].permutation(n_blocks).astype(np.int32)
