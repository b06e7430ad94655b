"""One link step over a batch of requests, through the C ABI.

Host side of the step, as a serving engine would drive it:
  * the paged KV pool (K and V, [num_blocks][Hkv][16][d]) holds every cached chunk as
    it was compiled, one chunk per run of pages (a block manager's job: this module
    assigns the physical block ids, scattered by a seeded permutation);
  * per-request metadata (chunk lengths in link order, q, k, block tables, fresh
    blocks) and the recomputed rows' un-roped Q, K and V are the step's inputs;
  * ``run()`` issues the device calls: row selection, splice, RoPE tables,
    re-rotation of cached K, fresh K/V, link attention.  Every one is a kernel of
    libpic.so; nothing here computes on the data.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from . import (PIC_BF16, PIC_FP32, PIC_LAYOUT_FRAMED, PIC_LAYOUT_SPLICED, PIC_PAGE, pic_decode_attention,
               pic_decode_workspace, pic_link_attention, pic_link_attention_plan_q, pic_link_attention_plan_units,
               pic_link_attention_ror, pic_link_attention_run, pic_link_attention_workspace,
               pic_plan_offsets, pic_rerotate_k, pic_rope_cached_k, pic_rope_table, pic_select_rows,
               pic_splice_pages, pic_write_fresh_kv)
from .inputs import Workload, block_shuffle, chunk_store, decode_inputs, row_inputs


def _cdiv(a, b):
    return (a + b - 1) // b


class LinkBatch:
    """Device state and inputs of one link step for the requests of a workload."""

    def __init__(self, wl: Workload, device="cuda", rows_inputs=None, scheme="rotary"):
        """scheme "rotary": the pool's cached K is encoded at local positions and the step
        re-rotates it by the chunk offset (rotary correction).  scheme "ror": the same
        correction applied on read inside link attention (rotate-on-read, on the framed
        page layout): every chunk's keys stay in the chunk's frame (the cached pages are
        never written, the recomputed head rows' fresh K is encoded at its position in
        the chunk) and Q is rotated back by the chunk's offset instead, so shared chunks
        need no per-request copies.  scheme
        "nope": the pool's cached K carries no position encoding and the step encodes
        every kept cached slot at its global position (scheme B; with shared chunks into
        per-request pages, the first chunk's too)."""
        if scheme not in ("rotary", "ror", "nope"):
            raise ValueError(scheme)
        self.scheme = scheme
        self.wl = wl
        self.device = torch.device(device)
        self.dtype = wl.torch_dtype
        self.pic_dtype = PIC_BF16 if wl.dtype == "bf16" else PIC_FP32
        Hkv, d = wl.Hkv, wl.d

        # ---- request metadata (host)
        flat_ids = np.concatenate([r.chunk_ids for r in wl.requests]).astype(np.int64) \
            if wl.requests else np.zeros(0, np.int64)
        self.flat_store_ids = flat_ids
        self.chunk_lens = wl.chunk_lens[flat_ids].astype(np.int32)
        self.chunk_off = np.zeros(len(wl.requests) + 1, np.int32)
        self.chunk_off[1:] = np.cumsum([len(r.chunk_ids) for r in wl.requests])
        self.q_len = np.array([r.q for r in wl.requests], np.int32)
        self.k = np.array([r.k for r in wl.requests], np.int32)
        self.layout = PIC_LAYOUT_FRAMED if scheme == "ror" else PIC_LAYOUT_SPLICED
        offs = pic_plan_offsets(self.chunk_lens, self.chunk_off, self.q_len, self.k, self.layout)
        self.offs = offs
        self.n_req = len(wl.requests)
        self.n_rows = int(offs["row_off"][-1])
        self.n_pages = int(offs["page_off"][-1])
        self.n_rot = int(offs["rot_off"][-1])
        self.n_fresh = int(offs["fresh_off"][-1])
        self.n_chunks = len(self.chunk_lens)
        self.tokens = int(self.chunk_lens.sum()) + int(self.q_len.sum())

        # ---- block allocation
        store_np = np.array([_cdiv(int(L), PIC_PAGE) for L in wl.chunk_lens], np.int64)
        store_base = np.zeros(len(store_np) + 1, np.int64)
        store_base[1:] = np.cumsum(store_np)
        n_store_pages = int(store_base[-1])
        n_chunk_pages = int(offs["chunk_page_off"][-1])
        # shared chunks: rotated (or, scheme B, encoded) into per-request pages; rotate-on-read
        # reads them in place
        copies = wl.out_of_place and scheme in ("rotary", "nope")
        n_dst = n_chunk_pages if copies else 0
        n_link_blocks = n_store_pages + n_dst + self.n_fresh
        # one more block per request takes the row a decode step appends after the link
        self.decode_blocks = np.arange(n_link_blocks, n_link_blocks + self.n_req, dtype=np.int32)
        self.num_blocks = n_link_blocks + self.n_req
        perm = block_shuffle(wl, n_link_blocks).astype(np.int64)
        self.store_blocks = [perm[store_base[c]:store_base[c + 1]] for c in range(len(store_np))]
        k_src = np.concatenate([self.store_blocks[c] for c in flat_ids]) if len(flat_ids) else np.zeros(0, np.int64)
        self.k_src = k_src.astype(np.int32)
        self.v_blocks = self.k_src.copy()
        self.k_dst = perm[n_store_pages:n_store_pages + n_dst].astype(np.int32) if copies else None
        self.fresh_blocks = perm[n_store_pages + n_dst:].astype(np.int32)

        # ---- pool: the cached chunks as compiled
        kst, vst, soff = chunk_store(wl)
        self.store_k, self.store_v, self.store_off = kst, vst, soff
        shape = (self.num_blocks, Hkv, PIC_PAGE, d)
        self.k_pool = torch.zeros(shape, dtype=self.dtype, device=self.device)
        self.v_pool = torch.zeros(shape, dtype=self.dtype, device=self.device)
        self.reset_pool()

        # ---- recomputed rows' inputs
        if rows_inputs is None:
            rows_inputs = row_inputs(wl, self.n_rows)
        self.q_raw_h, self.k_new_h, self.v_new_h = rows_inputs

        # ---- device buffers
        dev, i32 = self.device, torch.int32
        self.host = {
            "chunk_lens": torch.from_numpy(self.chunk_lens), "chunk_off": torch.from_numpy(self.chunk_off),
            "q_len": torch.from_numpy(self.q_len), "k": torch.from_numpy(self.k),
            "row_off": torch.from_numpy(offs["row_off"]), "page_off": torch.from_numpy(offs["page_off"]),
            "rot_off": torch.from_numpy(offs["rot_off"]), "fresh_off": torch.from_numpy(offs["fresh_off"]),
            "chunk_page_off": torch.from_numpy(offs["chunk_page_off"]),
            "k_src": torch.from_numpy(self.k_src), "v_blocks": torch.from_numpy(self.v_blocks),
            "fresh_blocks": torch.from_numpy(self.fresh_blocks),
            "q_raw": self.q_raw_h, "k_new": self.k_new_h, "v_new": self.v_new_h,
        }
        if self.k_dst is not None:
            self.host["k_dst"] = torch.from_numpy(self.k_dst)
        self.dev = {n: t.to(dev) for n, t in self.host.items()}
        self.rows = torch.empty(self.n_rows, dtype=i32, device=dev)
        self.chunk_start = torch.empty(self.n_chunks, dtype=i32, device=dev)
        self.pages = torch.empty((self.n_pages, 4), dtype=i32, device=dev)   # pic_link_page, 16 B
        self.rot = torch.empty((self.n_rot, 4), dtype=i32, device=dev)       # pic_rot_page, 16 B
        self.page_tab = torch.empty(self.n_pages, dtype=i32, device=dev) if scheme == "ror" else None
        # rotate-on-read: each recomputed row's position in its frame, and the table the
        # fresh K is encoded with
        self.row_frame_pos = torch.empty(self.n_rows, dtype=i32, device=dev) if scheme == "ror" else None
        self.fresh_table = torch.empty((self.n_rows, d // 2, 4), dtype=torch.float32, device=dev) \
            if scheme == "ror" else None
        self.row_block = torch.empty(self.n_rows, dtype=i32, device=dev)
        self.row_slot = torch.empty(self.n_rows, dtype=i32, device=dev)
        self.delta_table = torch.empty((self.n_chunks, d // 2, 4), dtype=torch.float32, device=dev)
        self.row_table = torch.empty((self.n_rows, d // 2, 4), dtype=torch.float32, device=dev)
        self.out = torch.empty((self.n_rows, wl.Hq, d), dtype=self.dtype, device=dev)
        ws = pic_link_attention_workspace(self.n_rows, self.n_req, wl.Hq, wl.Hkv, d, self.pic_dtype)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev) if ws > 0 else None
        self.err = torch.zeros(1, dtype=i32, device=dev)
        self.scale = 1.0 / math.sqrt(d)
        self._side = None  # stream of the cached-K pass (created on first use)
        self._plan_s = None  # stream of the row table and the attention plan (created on first use)
        if scheme == "nope":
            # the model's position table (every position a cached slot can take), built once
            self.n_pos = max([int(wl.chunk_lens[r.chunk_ids].sum()) for r in wl.requests] + [1])
            pos_all = torch.arange(self.n_pos, dtype=i32, device=dev)
            self.pos_table = torch.empty((self.n_pos, d // 2, 4), dtype=torch.float32, device=dev)
            pic_rope_table(pos_all, d, wl.theta, self.pos_table)

    # ------------------------------------------------------------------ state
    def reset_pool(self):
        """Write every cached chunk, as compiled, into its pages (zeroing the rest)."""
        wl = self.wl
        self.k_pool.zero_()
        self.v_pool.zero_()
        blk, slot, src = [], [], []
        for c, blocks in enumerate(self.store_blocks):
            L = int(wl.chunk_lens[c])
            j = np.arange(L)
            blk.append(blocks[j // PIC_PAGE])
            slot.append(j % PIC_PAGE)
            src.append(self.store_off[c] + j)
        if blk:
            b = torch.from_numpy(np.concatenate(blk)).to(self.device)
            s = torch.from_numpy(np.concatenate(slot)).to(self.device)
            idx = torch.from_numpy(np.concatenate(src)).to(self.device)
            self.k_pool[b, :, s, :] = self.store_k.to(self.device)[idx]
            self.v_pool[b, :, s, :] = self.store_v.to(self.device)[idx]

    def pin_host_inputs(self):
        """Page-locked copies of the step's per-request inputs (for end-to-end timing)."""
        self.host_pinned = {n: t.pin_memory() for n, t in self.host.items()}
        self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()

    def upload(self):
        """Host -> device copies of the step's inputs (async on the current stream)."""
        for n, t in self.host_pinned.items():
            self.dev[n].copy_(t, non_blocking=True)

    def download(self):
        """Device -> host copy of the step's result (async on the current stream)."""
        self.out_host.copy_(self.out, non_blocking=True)
        return self.out_host

    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def d2h_bytes(self) -> int:
        return self.out.numel() * self.out.element_size()

    # ------------------------------------------------------------------ step
    # kernels one run() launches: select, splice, 2 tables, re-rotate, fresh K/V, and the
    # attention (its tile rows, Q operands and unit plan, the attention, the LSE merge)
    LAUNCHES_PER_STEP = 11  # rotary correction and rotate-on-read (a third table, no re-rotation); scheme B: 10

    @property
    def launches_per_step(self) -> int:
        return self.LAUNCHES_PER_STEP - (1 if self.scheme == "nope" else 0)

    def run(self, stream=None, marks=None, inputs=None, out=None):
        """The link step: a1 select, splice, a2 tables, a3 re-rotate, a4 fresh K/V, a5+a6 attention.

        The cached-K pass (re-rotation, or scheme B's encoding) runs on a side stream
        beside the work that reads no cached K — the row table, the fresh K/V, the
        attention plan — and the attention run waits for both.  ``marks`` (optional)
        maps "rerotate" / "attention" to (start, end) CUDA events recorded around the
        cached-K pass (on the side stream) and the attention run.  ``inputs`` / ``out``
        (optional) replace the step's device inputs (a dict like ``self.dev``) and its
        output tensor, for a caller that double-buffers them (LinkPipeline)."""
        wl = self.wl
        dv = self.dev if inputs is None else inputs
        out_t = self.out if out is None else out
        mk = marks or {}
        if stream is None:
            main = torch.cuda.current_stream(self.device)
        elif isinstance(stream, int):
            main = torch.cuda.ExternalStream(stream)
        else:
            main = stream
        pic_select_rows(dv["chunk_lens"], dv["chunk_off"], dv["q_len"], dv["k"], dv["row_off"], self.rows,
                        self.chunk_start, self.err, main)
        # the side stream forks once the chunk starts exist: the offset table (which
        # needs only them) runs beside the splice, the pass itself waits for the splice
        pass_stream = main
        if self.scheme in ("rotary", "nope"):
            if self._side is None:
                self._side = torch.cuda.Stream(self.device)
                self._ev_fork, self._ev_join = torch.cuda.Event(), torch.cuda.Event()
                self._ev_spliced = torch.cuda.Event()
            pass_stream = self._side
            self._ev_fork.record(main)
            pass_stream.wait_event(self._ev_fork)
        if self.scheme == "rotary":
            pic_rope_table(self.chunk_start, wl.d, wl.theta, self.delta_table, pass_stream)
        # a third stream, also forked after row selection, takes the row table and the
        # attention plan's Q operands (which need no page list), beside the splice
        plan_stream = main
        if self.scheme in ("rotary", "nope"):
            if self._plan_s is None:
                self._plan_s = torch.cuda.Stream(self.device)
                self._ev_rowtab, self._ev_planned = torch.cuda.Event(), torch.cuda.Event()
            plan_stream = self._plan_s
            plan_stream.wait_event(self._ev_fork)
            pic_rope_table(self.rows, wl.d, wl.theta, self.row_table, plan_stream)
            self._ev_rowtab.record(plan_stream)
            # the Q operands need only the rows: written beside the splice
            pic_link_attention_plan_q(dv["q_raw"], self.row_table, dv["row_off"], self.n_req, self.n_rows, wl.Hq,
                                      wl.Hkv, wl.d, self.pic_dtype, self.ws, self.err, plan_stream)
        # scheme B with shared chunks: the page list reads every chunk from its private pages
        list_src = dv["k_dst"] if (self.scheme == "nope" and "k_dst" in dv) else dv["k_src"]
        pic_splice_pages(dv["chunk_lens"], dv["chunk_off"], dv["q_len"], dv["k"], self.chunk_start,
                         dv["chunk_page_off"], list_src, dv.get("k_dst"), dv["v_blocks"], dv["fresh_off"],
                         dv["fresh_blocks"], dv["row_off"], dv["page_off"], dv["rot_off"], self.pages, self.rot,
                         self.row_block, self.row_slot, self.err, main, page_tab=self.page_tab, layout=self.layout,
                         row_frame_pos=self.row_frame_pos)
        if pass_stream is not main:
            self._ev_spliced.record(main)
            pass_stream.wait_event(self._ev_spliced)
        if plan_stream is not main:
            # the unit plan (one block) runs on the pass stream just before the pass: beside
            # the pass it would find no SM with room until the pass ended
            pic_link_attention_plan_units(self.rows, dv["row_off"], self.pages, dv["page_off"], self.n_req,
                                          self.n_rows, wl.Hq, wl.Hkv, wl.d, self.pic_dtype, self.ws, self.err,
                                          pass_stream)
            self._ev_planned.record(plan_stream)
        if self.scheme == "ror":
            pic_rope_table(self.chunk_start, wl.d, wl.theta, self.delta_table, pass_stream)
        if "rerotate" in mk:
            mk["rerotate"][0].record(pass_stream)
        if self.scheme == "rotary":
            pic_rerotate_k(self.k_pool, self.pic_dtype, wl.Hkv, wl.d, self.rot, self.n_rot, self.delta_table,
                           self.n_chunks, self.err, pass_stream)
        elif self.scheme == "nope":
            pic_rope_cached_k(self.k_pool, self.pic_dtype, wl.Hkv, wl.d, dv["chunk_lens"], dv["chunk_off"], dv["k"],
                              self.n_req, self.chunk_start, dv["chunk_page_off"], self.n_chunks,
                              int(self.offs["chunk_page_off"][-1]), dv["k_src"], dv.get("k_dst"), self.pos_table,
                              self.err, pass_stream)
        if "rerotate" in mk:
            mk["rerotate"][1].record(pass_stream)
        if pass_stream is not main:
            self._ev_join.record(pass_stream)
        if plan_stream is main:
            pic_rope_table(self.rows, wl.d, wl.theta, self.row_table, main)
        else:
            main.wait_event(self._ev_rowtab)
        fresh_table = self.row_table
        if self.scheme == "ror":  # fresh K in its chunk's frame
            pic_rope_table(self.row_frame_pos, wl.d, wl.theta, self.fresh_table, main)
            fresh_table = self.fresh_table
        pic_write_fresh_kv(self.k_pool, self.v_pool, self.pic_dtype, wl.Hkv, wl.d, dv["k_new"], dv["v_new"],
                           fresh_table, self.row_block, self.row_slot, self.n_rows, self.err, main)
        if self.scheme == "ror":
            if "attention" in mk:
                mk["attention"][0].record(main)
            pic_link_attention_ror(dv["q_raw"], self.row_table, self.rows, dv["row_off"], self.k_pool, self.v_pool,
                                   self.pic_dtype, self.pages, self.page_tab, self.delta_table, dv["page_off"],
                                   self.n_req, self.n_rows, wl.Hq, wl.Hkv, wl.d, self.scale, out_t, self.ws,
                                   self.err, main)
        else:
            main.wait_event(self._ev_planned)
            main.wait_event(self._ev_join)
            if "attention" in mk:
                mk["attention"][0].record(main)
            pic_link_attention_run(dv["q_raw"], self.row_table, self.rows, dv["row_off"], self.k_pool, self.v_pool,
                                   self.pic_dtype, self.pages, dv["page_off"], self.n_req, self.n_rows, wl.Hq,
                                   wl.Hkv, wl.d, self.scale, out_t, self.ws, self.err, main)
        if "attention" in mk:
            mk["attention"][1].record(main)

    # ------------------------------------------------------------------ decode after the link
    def setup_decode(self):
        """Inputs and page lists of one decode row per request, at position T_r + q_r right
        after the request's query rows.  Call after run() has built the link page list: a
        request's decode page list is its link pages followed by one page holding the new
        row (a serving engine keeps this list; building it is not part of the step)."""
        wl, dev, i32 = self.wl, self.device, torch.int32
        q, k, v = decode_inputs(wl)
        self.dec_q, self.dec_k, self.dec_v = q.to(dev), k.to(dev), v.to(dev)
        pos = np.array([int(wl.chunk_lens[r.chunk_ids].sum()) + r.q for r in wl.requests], np.int32)
        self.dec_pos_h = pos
        self.dec_pos = torch.from_numpy(pos).to(dev)
        self.dec_block = torch.from_numpy(self.decode_blocks).to(dev)
        self.dec_slot = torch.zeros(self.n_req, dtype=i32, device=dev)
        po = self.offs["page_off"].astype(np.int64)
        src, new_off = [], np.zeros(self.n_req + 1, np.int32)
        for r in range(self.n_req):
            src += list(range(po[r], po[r + 1])) + [-1]
            new_off[r + 1] = len(src)
        src = np.array(src, np.int64)
        pages = self.pages[torch.from_numpy(np.maximum(src, 0)).to(dev)].clone()
        extra = np.flatnonzero(src < 0)
        ent = np.stack([self.decode_blocks, self.decode_blocks, pos, np.full(self.n_req, 1 << 16, np.int32)], 1)
        pages[torch.from_numpy(extra).to(dev)] = torch.from_numpy(ent.astype(np.int32)).to(dev)
        self.dec_pages = pages
        self.dec_page_off = torch.from_numpy(new_off).to(dev)
        # after a rotate-on-read link the linked pages keep their frames; the new row's
        # page is in the global frame
        self.dec_page_tab = None
        if self.scheme == "ror":
            tab = self.page_tab[torch.from_numpy(np.maximum(src, 0)).to(dev)].clone()
            tab[torch.from_numpy(extra).to(dev)] = -1
            self.dec_page_tab = tab
        self.dec_table = torch.empty((self.n_req, wl.d // 2, 4), dtype=torch.float32, device=dev)
        self.dec_out = torch.empty((self.n_req, wl.Hq, wl.d), dtype=self.dtype, device=dev)
        ws = pic_decode_workspace(self.n_req, wl.Hq, wl.Hkv, wl.d, self.pic_dtype)
        self.dec_ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev) if ws > 0 else None
        # HBM bytes a decode step must read: every listed valid K and V row, plus Q and out
        lohi = self.dec_pages[:, 3].cpu().numpy()
        slots = int(((lohi >> 16) - (lohi & 0xffff)).clip(min=0).sum())
        elt = 2 if self.dtype == torch.bfloat16 else 4
        self.dec_bytes = 2 * slots * wl.Hkv * wl.d * elt + 2 * self.n_req * wl.Hq * wl.d * elt

    def run_decode(self, stream=None, marks=None):
        """One decode step: the new rows' RoPE table, their K/V written into the decode
        blocks, and the decode attention (split-KV + merge).  ``marks`` may map "decode" to
        (start, end) events recorded around the attention call."""
        wl, mk = self.wl, marks or {}
        pic_rope_table(self.dec_pos, wl.d, wl.theta, self.dec_table, stream)
        pic_write_fresh_kv(self.k_pool, self.v_pool, self.pic_dtype, wl.Hkv, wl.d, self.dec_k, self.dec_v,
                           self.dec_table, self.dec_block, self.dec_slot, self.n_req, self.err, stream)
        if "decode" in mk:
            mk["decode"][0].record()
        pic_decode_attention(self.dec_q, self.dec_table, self.k_pool, self.v_pool, self.pic_dtype, self.dec_pages,
                             self.dec_page_off, self.n_req, wl.Hq, wl.Hkv, wl.d, self.scale, self.dec_out, self.dec_ws,
                             self.err, stream, page_tab=self.dec_page_tab,
                             rot_table=self.delta_table if self.dec_page_tab is not None else None)
        if "decode" in mk:
            mk["decode"][1].record()

    # ------------------------------------------------------------------ read-back helpers (tests)
    def error(self) -> int:
        return int(self.err.item())

    def pages_host(self) -> np.ndarray:
        return self.pages.cpu().numpy().view(np.uint8).view(
            np.dtype([("k_block", "<i4"), ("v_block", "<i4"), ("gpos0", "<i4"), ("lo", "<i2"), ("hi", "<i2")]))[:, 0]

    def rotated_chunk_k(self, flat_chunk: int) -> torch.Tensor:
        """K of one linked chunk as it sits in the pool after the step ([L][Hkv][d], CPU)."""
        L = int(self.chunk_lens[flat_chunk])
        cp0 = int(self.offs["chunk_page_off"][flat_chunk])
        r = int(np.searchsorted(self.chunk_off, flat_chunk, side="right") - 1)
        first = flat_chunk == int(self.chunk_off[r])
        # private pages when chunks were copied; the first chunk is copied only by scheme B
        table = self.k_src if (self.k_dst is None or (first and self.scheme != "nope")) else self.k_dst
        j = np.arange(L)
        b = torch.from_numpy(table[cp0 + j // PIC_PAGE].astype(np.int64)).to(self.device)
        s = torch.from_numpy(j % PIC_PAGE).to(self.device)
        return self.k_pool[b, :, s, :].cpu()


def _main():
    """Run the link step of a seeded preset workload a few times and print one JSON
    line (mean time of the timed steps, context tokens/s)."""
    import argparse
    import json

    from . import build
    from .inputs import PRESETS

    ap = argparse.ArgumentParser(description=_main.__doc__.splitlines()[0])
    ap.add_argument("--workload", default="long_context_100x1000", choices=sorted(PRESETS))
    ap.add_argument("--scheme", default="rotary", choices=["rotary", "ror", "nope"])
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--runs", type=int, default=2)
    ap.add_argument("--decode", action="store_true", help="time one decode step after the link instead")
    a = ap.parse_args()
    build.build()
    b = LinkBatch(PRESETS[a.workload](), scheme=a.scheme)
    if a.decode:
        b.run()
        b.setup_decode()
        step = b.run_decode
    else:
        step = b.run
    for _ in range(a.warmup):
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.runs)]
    for e0, e1 in ev:
        e0.record()
        step()
        e1.record()
    torch.cuda.synchronize()
    if b.error():
        raise SystemExit(f"device error {b.error()}")
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / max(len(ev), 1)
    print(json.dumps({"workload": a.workload, "scheme": a.scheme, "decode": a.decode, "ms_per_step": ms,
                      "tokens_per_s": b.tokens / (ms / 1e3), "launches_per_step": b.launches_per_step}))


if __name__ == "__main__":
    _main()


class LinkGraph:
    """One link step (every kernel of LinkBatch.run on its three streams) captured as a
    CUDA graph, so that a step costs one graph launch instead of ten kernel launches
    from the host.  The graph reads and writes the batch's own device buffers: update
    their contents (same shapes) between replays, not the tensors."""

    def __init__(self, batch: LinkBatch):
        self.b = batch
        batch.run()  # loads the device code and sets kernel attributes outside the capture
        torch.cuda.synchronize(batch.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            batch.run()
        torch.cuda.synchronize(batch.device)

    def replay(self):
        """Launch the captured step on the current stream."""
        self.graph.replay()


class LinkPipeline:
    """Link steps back to back with every step's input upload (host -> device, from
    pinned memory) and output read-back (device -> host) on their own copy streams,
    overlapped with the neighbouring steps' kernels: the device inputs and outputs
    are double-buffered, so step i + 1's upload and step i - 1's read-back run while
    step i computes.  The step itself is LinkBatch.run on the current stream, or with
    ``graphs`` one CUDA graph per buffer set (captured once, replayed per step)."""

    def __init__(self, batch: LinkBatch, graphs: bool = False):
        self.b = batch
        dev = batch.device
        self.sets = [batch.dev, {n: t.clone() for n, t in batch.dev.items()}]
        self.outs = [batch.out, torch.empty_like(batch.out)]
        self.graphs = None
        if graphs:
            self.graphs = []
            for k in range(2):
                batch.run(inputs=self.sets[k], out=self.outs[k])  # outside the capture first
                torch.cuda.synchronize(dev)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    batch.run(inputs=self.sets[k], out=self.outs[k])
                self.graphs.append(g)
            torch.cuda.synchronize(dev)
        self.host_out = [torch.empty(batch.out.shape, dtype=batch.out.dtype).pin_memory() for _ in range(2)]
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.uploaded = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.read = [torch.cuda.Event() for _ in range(2)]
        self.i = 0

    def begin(self, stream=None):
        """Order the copy streams after everything issued so far on ``stream``."""
        main = torch.cuda.current_stream(self.b.device) if stream is None else stream
        ev = torch.cuda.Event()
        ev.record(main)
        self.h2d.wait_event(ev)
        self.d2h.wait_event(ev)

    def submit(self, host_inputs, stream=None):
        """Queue one step on ``host_inputs`` (pinned tensors named as LinkBatch.host).
        Returns (pinned host output, event recorded once it has arrived)."""
        main = torch.cuda.current_stream(self.b.device) if stream is None else stream
        k = self.i % 2
        if self.i >= 2:
            self.h2d.wait_event(self.computed[k])  # the step two back has finished reading set k
        for n, t in host_inputs.items():
            with torch.cuda.stream(self.h2d):
                self.sets[k][n].copy_(t, non_blocking=True)
        self.uploaded[k].record(self.h2d)
        main.wait_event(self.uploaded[k])
        if self.i >= 2:
            main.wait_event(self.read[k])  # out k's previous result has been read back
        if self.graphs is not None:
            with torch.cuda.stream(main):
                self.graphs[k].replay()
        else:
            self.b.run(stream=main, inputs=self.sets[k], out=self.outs[k])
        self.computed[k].record(main)
        self.d2h.wait_event(self.computed[k])
        with torch.cuda.stream(self.d2h):
            self.host_out[k].copy_(self.outs[k], non_blocking=True)
        self.read[k].record(self.d2h)
        self.i += 1
        return self.host_out[k], self.read[k]
