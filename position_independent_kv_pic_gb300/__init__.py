"""Python binding of the PIC link-step library (libpic.so, C ABI in include/pic.h).

Argument marshalling only: every function here has the name of its C entry point,
takes torch tensors (device tensors for device pointers, numpy/host arrays for
``*_host`` arguments), passes raw pointers and the current CUDA stream, and turns a
non-OK status into an exception.  All computation happens in the library's CUDA
kernels.  If libpic.so is missing the import of any entry point raises: there is
no fallback.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "load", "library_path", "PicError", "PIC_OK", "PIC_ERR_INVALID", "PIC_ERR_CUDA",
    "PIC_ERR_UNSUPPORTED", "PIC_ERR_TIMEOUT", "PIC_ERR_RANGE", "PIC_ERR_WORKSPACE",
    "PIC_BF16", "PIC_FP32", "PIC_PAGE", "PIC_TILE_PAGES", "PIC_LAYOUT_SPLICED", "PIC_LAYOUT_FRAMED",
    "LINK_PAGE_DTYPE", "ROT_PAGE_DTYPE",
    "pic_count_rows", "pic_request_sizes_of", "pic_plan_offsets", "pic_strerror",
    "pic_select_rows", "pic_splice_pages", "pic_rope_table", "pic_rerotate_k",
    "pic_write_fresh_kv", "pic_link_attention_workspace", "pic_link_attention",
    "pic_selftest_umma", "pic_selftest_umma_pair", "pic_link_attention_noalloc", "PIC_NOALLOC_SCRATCH_BYTES",
    "EXPORTED",
    "pic_decode_workspace", "pic_decode_attention", "pic_rope_cached_k",
    "pic_compose_segment", "pic_compose_workspace", "pic_compose_states", "pic_link_attention_ror",
    "pic_link_attention_plan", "pic_link_attention_plan_q", "pic_link_attention_plan_units",
    "pic_link_attention_run", "pic_compose_split_t",
]

PIC_OK, PIC_ERR_INVALID, PIC_ERR_CUDA, PIC_ERR_UNSUPPORTED = 0, 1, 2, 3
PIC_ERR_TIMEOUT, PIC_ERR_RANGE, PIC_ERR_WORKSPACE = 4, 5, 6
PIC_BF16, PIC_FP32 = 0, 1
PIC_PAGE = 16
PIC_TILE_PAGES = 8
PIC_LAYOUT_SPLICED, PIC_LAYOUT_FRAMED = 0, 1
PIC_NOALLOC_SCRATCH_BYTES = 32 << 20

# numpy views of the 16-byte structs of pic.h
LINK_PAGE_DTYPE = np.dtype([("k_block", "<i4"), ("v_block", "<i4"), ("gpos0", "<i4"),
                            ("lo", "<i2"), ("hi", "<i2")])
ROT_PAGE_DTYPE = np.dtype([("src_block", "<i4"), ("dst_block", "<i4"), ("tab", "<i4"),
                           ("lo", "<i2"), ("hi", "<i2")])

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

# every symbol include/pic.h declares
EXPORTED = (
    "pic_count_rows", "pic_request_sizes_of", "pic_plan_offsets", "pic_strerror",
    "pic_select_rows", "pic_splice_pages", "pic_rope_table", "pic_rerotate_k",
    "pic_write_fresh_kv", "pic_link_attention_workspace", "pic_link_attention",
    "pic_selftest_umma", "pic_selftest_umma_pair", "pic_link_attention_noalloc", "pic_decode_workspace",
    "pic_decode_attention",
    "pic_rope_cached_k", "pic_compose_segment", "pic_compose_workspace", "pic_compose_states",
    "pic_link_attention_ror", "pic_link_attention_plan", "pic_link_attention_plan_q",
    "pic_link_attention_plan_units", "pic_link_attention_run", "pic_compose_split_t",
)


class PicError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {pic_strerror(status)} (status {status})")


class _Sizes(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("rows", ctypes.c_int64), ("link_pages", ctypes.c_int64),
                ("rot_pages", ctypes.c_int64), ("fresh_pages", ctypes.c_int64),
                ("chunk_pages", ctypes.c_int64)]


def library_path() -> str:
    """The in-tree libpic.so, or the build of the library that the environment
    variable PIC_LIBRARY names (a file name in this package's directory, e.g. the
    failure-injection test build)."""
    return os.path.join(_HERE, os.environ.get("PIC_LIBRARY", "libpic.so"))


_P = ctypes.c_void_p
_I32, _I64, _F32, _F64, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_size_t

_SIGS = {
    "pic_count_rows": (_I64, [_P, _I32, _I32, _I32]),
    "pic_request_sizes_of": (ctypes.c_int, [_P, _I32, _I32, _I32, ctypes.c_int, ctypes.POINTER(_Sizes)]),
    "pic_plan_offsets": (ctypes.c_int, [_P, _P, _P, _P, _I32, ctypes.c_int, _P, _P, _P, _P, _P]),
    "pic_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "pic_select_rows": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P, _P, _P, _P]),
    "pic_splice_pages": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P]),
    "pic_rope_table": (ctypes.c_int, [_P, _I64, _I32, _F64, _P, _P]),
    "pic_rerotate_k": (ctypes.c_int, [_P, _I64, ctypes.c_int, _I32, _I32, _P, _I64, _P, _I64, _P, _P]),
    "pic_write_fresh_kv": (ctypes.c_int, [_P, _P, _I64, ctypes.c_int, _I32, _I32, _P, _P, _P, _P, _P,
                                          _I64, _P, _P]),
    "pic_link_attention_workspace": (_SZ, [_I64, _I32, _I32, _I32, _I32, ctypes.c_int]),
    "pic_link_attention": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, ctypes.c_int, _P, _P, _I32,
                                          _I64, _I32, _I32, _I32, _F32, _P, _P, _SZ, _P, _P]),
    "pic_selftest_umma": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P]),
    "pic_selftest_umma_pair": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P]),
    "pic_link_attention_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, ctypes.c_int, _P, _P, _I32,
                                                  _I64, _I32, _I32, _I32, _F32, _P, _P, _P]),
    "pic_decode_workspace": (_SZ, [_I32, _I32, _I32, _I32, ctypes.c_int]),
    "pic_rope_cached_k": (ctypes.c_int, [_P, _I64, ctypes.c_int, _I32, _I32, _P, _P, _P, _I32, _P, _P, _I32, _I64,
                                         _P, _P, _P, _I64, _P, _P]),
    "pic_link_attention_ror": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, ctypes.c_int, _P, _P, _P, _I64, _P,
                                              _I32, _I64, _I32, _I32, _I32, _F32, _P, _P, _SZ, _P, _P]),
    "pic_link_attention_plan": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I32, _I64, _I32, _I32, _I32, ctypes.c_int,
                                               _P, _SZ, _P, _P]),
    "pic_link_attention_plan_q": (ctypes.c_int, [_P, _P, _P, _I32, _I64, _I32, _I32, _I32, ctypes.c_int, _P, _SZ,
                                                 _P, _P]),
    "pic_link_attention_plan_units": (ctypes.c_int, [_P, _P, _P, _P, _I32, _I64, _I32, _I32, _I32, ctypes.c_int, _P,
                                                     _SZ, _P, _P]),
    "pic_link_attention_run": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, ctypes.c_int, _P, _P, _I32, _I64, _I32,
                                              _I32, _I32, _F32, _P, _P, _SZ, _P, _P]),
    "pic_compose_split_t": (ctypes.c_int, [_P, _I64, _I32, _P, _P]),
    "pic_compose_segment": (_I32, [_I32, _I64, _I32, _I32, _I32]),
    "pic_compose_workspace": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "pic_compose_states": (ctypes.c_int, [_P, _P, _I64, _P, _P, _I32, _I64, _I32, _I32, _I32, _I32, _P, _P, _SZ,
                                          _P, _P]),
    "pic_decode_attention": (ctypes.c_int, [_P, _P, _P, _P, _I64, ctypes.c_int, _P, _P, _P, _P, _I64, _I32, _I32,
                                            _I32, _I32, _F32, _P, _P, _SZ, _P, _P]),
}


def load():
    """Load libpic.so (built by ``python -m position_independent_kv_pic_gb300.build``)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{os.path.basename(path)} not built ({path}); run position_independent_kv_pic_gb300.build")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _ptr(t):
    """Device (or host) address of a tensor / ndarray, or None."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, where: str):
    if status != PIC_OK:
        raise PicError(status, where)


def _host_i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


# ----------------------------------------------------------------- host helpers

def pic_strerror(status: int) -> str:
    return load().pic_strerror(int(status)).decode()


def pic_count_rows(chunk_lens_host, q: int, k: int) -> int:
    a = _host_i32(chunk_lens_host)
    return int(load().pic_count_rows(_ptr(a), len(a), int(q), int(k)))


def pic_request_sizes_of(chunk_lens_host, q: int, k: int, layout: int = 0) -> dict:
    a = _host_i32(chunk_lens_host)
    s = _Sizes()
    _check(load().pic_request_sizes_of(_ptr(a), len(a), int(q), int(k), int(layout), ctypes.byref(s)),
           "pic_request_sizes_of")
    return {f: int(getattr(s, f)) for f, _ in _Sizes._fields_}


def pic_plan_offsets(chunk_lens_host, chunk_off_host, q_len_host, k_host, layout: int = 0) -> dict:
    """Host offsets (row_off, page_off, rot_off, fresh_off, chunk_page_off) as int32 arrays."""
    lens, coff = _host_i32(chunk_lens_host), _host_i32(chunk_off_host)
    ql, kk = _host_i32(q_len_host), _host_i32(k_host)
    n_req = len(ql)
    outs = {n: np.zeros(n_req + 1, np.int32) for n in ("row_off", "page_off", "rot_off", "fresh_off")}
    outs["chunk_page_off"] = np.zeros(len(lens) + 1, np.int32)
    _check(load().pic_plan_offsets(_ptr(lens), _ptr(coff), _ptr(ql), _ptr(kk), n_req, int(layout),
                                   _ptr(outs["row_off"]),
                                   _ptr(outs["page_off"]), _ptr(outs["rot_off"]), _ptr(outs["fresh_off"]),
                                   _ptr(outs["chunk_page_off"])), "pic_plan_offsets")
    return outs


def pic_link_attention_workspace(n_rows: int, n_req: int, Hq: int, Hkv: int, d: int, dtype: int) -> int:
    return int(load().pic_link_attention_workspace(int(n_rows), int(n_req), int(Hq), int(Hkv), int(d), int(dtype)))


# ----------------------------------------------------------------- device entry points

def pic_select_rows(chunk_lens, chunk_off, q_len, k, row_off, rows, chunk_start, err_flag, stream=None):
    n_req = q_len.numel()
    _check(load().pic_select_rows(_ptr(chunk_lens), _ptr(chunk_off), _ptr(q_len), _ptr(k), _ptr(row_off), n_req,
                                  _ptr(rows), _ptr(chunk_start), _ptr(err_flag), _stream(stream)), "pic_select_rows")


def pic_splice_pages(chunk_lens, chunk_off, q_len, k, chunk_start, chunk_page_off, k_src_blocks, k_dst_blocks,
                     v_blocks, fresh_off, fresh_blocks, row_off, page_off, rot_off, pages, rot, row_block,
                     row_slot, err_flag, stream=None, page_tab=None, layout: int = 0, row_frame_pos=None):
    n_req = q_len.numel()
    _check(load().pic_splice_pages(
        _ptr(chunk_lens), _ptr(chunk_off), _ptr(q_len), _ptr(k), n_req, _ptr(chunk_start), _ptr(chunk_page_off),
        _ptr(k_src_blocks), _ptr(k_dst_blocks), _ptr(v_blocks), _ptr(fresh_off), _ptr(fresh_blocks), _ptr(row_off),
        _ptr(page_off), _ptr(rot_off), int(layout), _ptr(pages), _ptr(rot), _ptr(row_block), _ptr(row_slot),
        _ptr(row_frame_pos), _ptr(page_tab), _ptr(err_flag), _stream(stream)), "pic_splice_pages")


def pic_rope_table(pos, d: int, theta: float, table, stream=None):
    _check(load().pic_rope_table(_ptr(pos), pos.numel(), int(d), float(theta), _ptr(table), _stream(stream)),
           "pic_rope_table")


def pic_rerotate_k(k_pool, dtype: int, Hkv: int, d: int, rot, n_rot: int, table, n_tab: int, err_flag,
                   stream=None):
    _check(load().pic_rerotate_k(_ptr(k_pool), k_pool.shape[0], int(dtype), int(Hkv), int(d), _ptr(rot), int(n_rot),
                                 _ptr(table), int(n_tab), _ptr(err_flag), _stream(stream)), "pic_rerotate_k")


def pic_write_fresh_kv(k_pool, v_pool, dtype: int, Hkv: int, d: int, k_raw, v_raw, row_table, row_block, row_slot,
                       n_rows: int, err_flag, stream=None):
    _check(load().pic_write_fresh_kv(_ptr(k_pool), _ptr(v_pool), k_pool.shape[0], int(dtype), int(Hkv), int(d),
                                     _ptr(k_raw), _ptr(v_raw), _ptr(row_table), _ptr(row_block), _ptr(row_slot),
                                     int(n_rows), _ptr(err_flag), _stream(stream)), "pic_write_fresh_kv")


def pic_link_attention(q, row_table, rows, row_off, k_pool, v_pool, dtype: int, pages, page_off, n_req: int,
                       n_rows: int, Hq: int, Hkv: int, d: int, scale: float, out, ws, err_flag, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pic_link_attention(
        _ptr(q), _ptr(row_table), _ptr(rows), _ptr(row_off), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], int(dtype),
        _ptr(pages), _ptr(page_off), int(n_req), int(n_rows), int(Hq), int(Hkv), int(d), float(scale), _ptr(out),
        _ptr(ws), ws_bytes, _ptr(err_flag), _stream(stream)), "pic_link_attention")


def pic_rope_cached_k(k_pool, dtype: int, Hkv: int, d: int, chunk_lens, chunk_off, k, n_req: int, chunk_start,
                      chunk_page_off, n_chunks: int, n_chunk_pages: int, k_src, k_dst, pos_table, err_flag,
                      stream=None):
    _check(load().pic_rope_cached_k(
        _ptr(k_pool), k_pool.shape[0], int(dtype), int(Hkv), int(d), _ptr(chunk_lens), _ptr(chunk_off), _ptr(k),
        int(n_req), _ptr(chunk_start), _ptr(chunk_page_off), int(n_chunks), int(n_chunk_pages), _ptr(k_src),
        _ptr(k_dst), _ptr(pos_table), pos_table.shape[0], _ptr(err_flag), _stream(stream)), "pic_rope_cached_k")


def pic_decode_workspace(n_req: int, Hq: int, Hkv: int, d: int, dtype: int) -> int:
    return int(load().pic_decode_workspace(int(n_req), int(Hq), int(Hkv), int(d), int(dtype)))


def pic_decode_attention(q, q_table, k_pool, v_pool, dtype: int, pages, page_off, n_req: int, Hq: int, Hkv: int,
                         d: int, scale: float, out, ws, err_flag, stream=None, page_tab=None, rot_table=None):
    """page_tab / rot_table: the page frames and offset table of a rotate-on-read link (None: every key is
    at its global position)."""
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    n_tab = 0 if rot_table is None else rot_table.shape[0]
    _check(load().pic_decode_attention(
        _ptr(q), _ptr(q_table), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], int(dtype), _ptr(pages), _ptr(page_off),
        _ptr(page_tab), _ptr(rot_table), int(n_tab), int(n_req), int(Hq), int(Hkv), int(d), float(scale), _ptr(out),
        _ptr(ws), ws_bytes, _ptr(err_flag), _stream(stream)), "pic_decode_attention")


def pic_link_attention_plan(q, row_table, rows, row_off, pages, page_off, n_req: int, n_rows: int, Hq: int,
                            Hkv: int, d: int, dtype: int, ws, err_flag, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pic_link_attention_plan(
        _ptr(q), _ptr(row_table), _ptr(rows), _ptr(row_off), _ptr(pages), _ptr(page_off), int(n_req), int(n_rows),
        int(Hq), int(Hkv), int(d), int(dtype), _ptr(ws), ws_bytes, _ptr(err_flag), _stream(stream)),
        "pic_link_attention_plan")


def pic_link_attention_plan_q(q, row_table, row_off, n_req: int, n_rows: int, Hq: int, Hkv: int, d: int, dtype: int,
                              ws, err_flag, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pic_link_attention_plan_q(
        _ptr(q), _ptr(row_table), _ptr(row_off), int(n_req), int(n_rows), int(Hq), int(Hkv), int(d), int(dtype),
        _ptr(ws), ws_bytes, _ptr(err_flag), _stream(stream)), "pic_link_attention_plan_q")


def pic_link_attention_plan_units(rows, row_off, pages, page_off, n_req: int, n_rows: int, Hq: int, Hkv: int, d: int,
                                  dtype: int, ws, err_flag, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pic_link_attention_plan_units(
        _ptr(rows), _ptr(row_off), _ptr(pages), _ptr(page_off), int(n_req), int(n_rows), int(Hq), int(Hkv), int(d),
        int(dtype), _ptr(ws), ws_bytes, _ptr(err_flag), _stream(stream)), "pic_link_attention_plan_units")


def pic_link_attention_run(q, row_table, rows, row_off, k_pool, v_pool, dtype: int, pages, page_off, n_req: int,
                           n_rows: int, Hq: int, Hkv: int, d: int, scale: float, out, ws, err_flag, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pic_link_attention_run(
        _ptr(q), _ptr(row_table), _ptr(rows), _ptr(row_off), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], int(dtype),
        _ptr(pages), _ptr(page_off), int(n_req), int(n_rows), int(Hq), int(Hkv), int(d), float(scale), _ptr(out),
        _ptr(ws), ws_bytes, _ptr(err_flag), _stream(stream)), "pic_link_attention_run")


def pic_link_attention_ror(q, row_table, rows, row_off, k_pool, v_pool, dtype: int, pages, page_tab, rot_table,
                           page_off, n_req: int, n_rows: int, Hq: int, Hkv: int, d: int, scale: float, out, ws,
                           err_flag, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pic_link_attention_ror(
        _ptr(q), _ptr(row_table), _ptr(rows), _ptr(row_off), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], int(dtype),
        _ptr(pages), _ptr(page_tab), _ptr(rot_table), rot_table.shape[0], _ptr(page_off), int(n_req), int(n_rows),
        int(Hq), int(Hkv), int(d), float(scale), _ptr(out), _ptr(ws), ws_bytes, _ptr(err_flag), _stream(stream)),
        "pic_link_attention_ror")


def pic_compose_segment(n_req: int, n_elems: int, max_chain: int, H: int, sms: int) -> int:
    return int(load().pic_compose_segment(int(n_req), int(n_elems), int(max_chain), int(H), int(sms)))


def pic_compose_workspace(n_req: int, max_chain: int, H: int, d: int, seg: int) -> int:
    return int(load().pic_compose_workspace(int(n_req), int(max_chain), int(H), int(d), int(seg)))


def pic_compose_split_t(T, T_split, stream=None):
    """T [..][d][d] fp32 -> T_split [..][2][d][d] bf16 (hi, lo planes)."""
    n = T.numel() // (T.shape[-1] * T.shape[-2])
    _check(load().pic_compose_split_t(_ptr(T), n, int(T.shape[-1]), _ptr(T_split), _stream(stream)),
           "pic_compose_split_t")


def pic_compose_states(T_split, S_pool, ids, chain_off, n_req: int, n_elems: int, max_chain: int, H: int, d: int,
                       seg: int, out, ws, err_flag, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(load().pic_compose_states(
        _ptr(T_split), _ptr(S_pool), S_pool.shape[0], _ptr(ids), _ptr(chain_off), int(n_req), int(n_elems),
        int(max_chain), int(H), int(d), int(seg), _ptr(out), _ptr(ws), ws_bytes, _ptr(err_flag), _stream(stream)),
        "pic_compose_states")


def pic_selftest_umma(a, b, d_kmajor, d_mnmajor, d_tmem_a, err_flag, stream=None):
    _check(load().pic_selftest_umma(_ptr(a), _ptr(b), _ptr(d_kmajor), _ptr(d_mnmajor), _ptr(d_tmem_a),
                                    _ptr(err_flag), _stream(stream)), "pic_selftest_umma")


def pic_selftest_umma_pair(a, b, v, d_s, d_pv, info, err_flag, stream=None):
    _check(load().pic_selftest_umma_pair(_ptr(a), _ptr(b), _ptr(v), _ptr(d_s), _ptr(d_pv), _ptr(info),
                                         _ptr(err_flag), _stream(stream)), "pic_selftest_umma_pair")


def pic_link_attention_noalloc(q, row_table, rows, row_off, k_pool, v_pool, dtype: int, pages, page_off,
                               n_req: int, n_rows: int, Hq: int, Hkv: int, d: int, scale: float, out, err_flag,
                               stream=None):
    """pic_link_attention for callers that cannot allocate: the library's fixed device
    scratch replaces the workspace (see pic.h for its size limit and sharing rules)."""
    _check(load().pic_link_attention_noalloc(
        _ptr(q), _ptr(row_table), _ptr(rows), _ptr(row_off), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], int(dtype),
        _ptr(pages), _ptr(page_off), int(n_req), int(n_rows), int(Hq), int(Hkv), int(d), float(scale), _ptr(out),
        _ptr(err_flag), _stream(stream)), "pic_link_attention_noalloc")
