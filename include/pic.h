/*
 * pic.h -- C ABI of the position-independent-caching (PIC) "link" step for
 * NVIDIA GB300 (sm_103a).
 *
 * The link step takes KV caches that were computed per chunk at local positions
 * 0..L_c-1 and
 *   1. selects the rows to recompute: the first min(k, L_c) tokens of every chunk
 *      except the first, plus every query token (EPIC's LegoLink-k);
 *   2. splices the chunks into one context at global positions (a page list);
 *   3. re-rotates every cached K of chunk c by its offset Delta_c = s_c, one
 *      rotation R(theta * Delta_c) ("rotary correction");
 *   4. writes the recomputed rows' fresh K (RoPE at the global position) and V;
 *   5. runs causal attention (key_pos <= query_pos, scale 1/sqrt(d)) for the
 *      recomputed rows only, against the whole spliced K/V, Q roped at global
 *      positions.
 *
 * Sources: blog review "EPIC: Efficient Position-Independent Caching for Serving
 * Large Language Models" (compile/link walk-through; link_legolink Steps 1-3);
 * article on RoPE and prefix caching, sections 2.2 (RoPE) and 3.3 (rotary
 * correction); HYPIC article, section 2.2 (seam window = recomputed chunk heads);
 * blog "KV cache from scratch", mask section (offset causal mask).
 *
 * Conventions shared by every entry point
 *   - Pointers are DEVICE pointers unless their name ends in _host.  The caller
 *     owns all memory and streams; the library allocates nothing and keeps no
 *     state between calls (one exception, pic_link_attention_noalloc, is
 *     described where it is declared).
 *   - Every device entry point is asynchronous on `stream`.  Its return value
 *     reports only what the host can check synchronously: PIC_ERR_INVALID for a
 *     bad argument, PIC_ERR_UNSUPPORTED for a valid but unimplemented shape,
 *     PIC_ERR_WORKSPACE for a short workspace, PIC_ERR_CUDA when a launch fails.
 *   - Problems only the device can see (an out-of-range block id, metadata that
 *     disagrees with the host-computed sizes, a bounded wait that ran out) are
 *     written to *err_flag (int32, device), first error wins.  The caller zeroes
 *     it before the calls and reads it after synchronising.  Kernels never trap.
 *   - KV pools: K and V each [num_blocks][Hkv][PIC_PAGE][d] in the pool dtype
 *     (bf16 or fp32), row-major, 16-byte aligned.  A block is one 16-token page
 *     of one layer for all KV heads.
 *   - Request metadata is CSR: request r links chunks chunk_off[r] ..
 *     chunk_off[r+1]-1 (indices into the flat chunk arrays), in link order.
 *   - GQA: query head h reads KV head h / (Hq / Hkv).
 *   - Positions are int32 (sequence length < 2^31).
 *   - RoPE pairs dimension i with i + d/2, angle p * theta^(-2i/d).
 */
#ifndef PIC_H_
#define PIC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (binary compatible); NULL means the legacy default stream. */
typedef struct CUstream_st* pic_stream_t;

typedef enum {
  PIC_OK = 0,
  PIC_ERR_INVALID = 1,     /* bad argument (host check) or bad metadata (device flag) */
  PIC_ERR_CUDA = 2,        /* a CUDA runtime / driver call failed */
  PIC_ERR_UNSUPPORTED = 3, /* dtype / head-dim / GQA-group combination not implemented */
  PIC_ERR_TIMEOUT = 4,     /* device: a bounded pipeline wait ran out (err_flag only) */
  PIC_ERR_RANGE = 5,       /* device: block id, slot or count outside its buffer (err_flag only) */
  PIC_ERR_WORKSPACE = 6    /* workspace smaller than pic_link_attention_workspace() */
} pic_status;

typedef enum { PIC_BF16 = 0, PIC_FP32 = 1 } pic_dtype;

#define PIC_PAGE 16 /* tokens per KV page (block) */
#define PIC_TILE_PAGES 8 /* pages per key tile of the tensor-core attention (128 keys) */

/* How a request's link page list is laid out (pic_request_sizes_of,
 * pic_plan_offsets, pic_splice_pages):
 *   PIC_LAYOUT_SPLICED  the chunks' pages back to back at their global positions;
 *                       every key the attention reads is encoded at its global
 *                       position (rotary correction by pic_rerotate_k, or scheme B
 *                       by pic_rope_cached_k).
 *   PIC_LAYOUT_FRAMED   for rotate-on-read: every chunk's run of pages (its fresh
 *                       head pages, then its cached pages) is padded with empty
 *                       entries to a whole number of key tiles (PIC_TILE_PAGES), so
 *                       that every key tile lies in one chunk; each chunk's keys stay
 *                       in the chunk's own frame (encoded at positions local to the
 *                       chunk: the cached pages as cached, the recomputed head rows
 *                       at their position within the chunk); chunk 0 and the query
 *                       are in the global frame (their local and global positions
 *                       coincide, or the query's fresh K is at its global position). */
typedef enum { PIC_LAYOUT_SPLICED = 0, PIC_LAYOUT_FRAMED = 1 } pic_layout;

/* One entry of a request's spliced context: 16 key slots at global positions
 * gpos0 .. gpos0+15, of which slots [lo, hi) are valid.  K comes from block
 * k_block of the K pool and V from block v_block of the V pool (they differ
 * when K was rotated out of place while V stays shared).  A request's entries
 * are sorted by gpos0 + lo: strictly increasing over entries with valid slots;
 * an empty entry (lo == hi, blocks -1: the padding of the framed layout) carries
 * the gpos0 of the next chunk's start.  16 bytes. */
typedef struct {
  int32_t k_block;
  int32_t v_block;
  int32_t gpos0;
  int16_t lo, hi;
} pic_link_page;

/* One unit of re-rotation work: rotate slots [lo, hi) of every KV head of K
 * block src_block by the offset in row `tab` of the offset table and store
 * them into dst_block (dst_block == src_block: in place).  16 bytes. */
typedef struct {
  int32_t src_block;
  int32_t dst_block;
  int32_t tab;
  int16_t lo, hi;
} pic_rot_page;

/* Sizes of one request, all closed-form in the chunk lengths, q and k. */
typedef struct {
  int64_t tokens;      /* T + q: spliced context length                         */
  int64_t rows;        /* n_sel = sum_{c>=1} min(k, L_c) + q: recomputed rows   */
  int64_t link_pages;  /* entries of the request's pic_link_page list           */
  int64_t rot_pages;   /* entries of the request's pic_rot_page list            */
  int64_t fresh_pages; /* fresh blocks the recomputed rows are written into     */
  int64_t chunk_pages; /* pages of the request's cached chunks: sum ceil(L_c/16) */
} pic_request_sizes;

/* ------------------------------------------------------------------------
 * Host helpers (no device work).
 * ------------------------------------------------------------------------ */

/* Number of recomputed rows of one request: sum over chunks c >= 1 of
 * min(k, L_c), plus q (EPIC link_legolink Step 1; the worked example gives 7 of
 * 17 for lengths {4,5,5}, q = 3, k = 2).  chunk_lens_host: n_chunks lengths in
 * link order, each >= 1.  Returns -1 on invalid input (n_chunks < 0, q < 0,
 * k < 0, a length < 1, or a NULL pointer with n_chunks > 0). */
int64_t pic_count_rows(const int32_t* chunk_lens_host, int32_t n_chunks, int32_t q, int32_t k);

/* All sizes of one request (see pic_request_sizes).  The layout they describe:
 *   link pages, in order, for each chunk c: ceil(m_c/16) fresh pages holding the
 *   recomputed head rows (m_c = min(k, L_c) for c >= 1, 0 for c = 0), then the
 *   chunk's cached pages j that keep at least one slot (valid slots
 *   [max(0, m_c - 16j), min(16, L_c - 16j))); finally ceil(q/16) fresh query pages.
 *   In PIC_LAYOUT_FRAMED every chunk's fresh + cached pages are followed by empty
 *   entries up to a multiple of PIC_TILE_PAGES (link_pages counts them).
 *   rot pages: the kept cached pages of chunks c >= 1 (chunk 0 has Delta = 0).
 *   fresh pages: the fresh link pages above, in the same order.
 * Returns PIC_ERR_INVALID on the same conditions as pic_count_rows, or for an
 * unknown layout. */
pic_status pic_request_sizes_of(const int32_t* chunk_lens_host, int32_t n_chunks, int32_t q,
                                int32_t k, pic_layout layout, pic_request_sizes* out);

/* Exclusive prefix offsets over n_req requests, from host copies of the
 * metadata: row_off, page_off, rot_off, fresh_off and chunk_page_off receive
 * n_req+1 (chunk_page_off: n_chunks_total+1) entries; any output may be NULL.
 * chunk_page_off[c] is the first page of chunk c in a per-chunk page table that
 * gives every chunk ceil(L_c/16) pages.  page_off follows `layout` (the framed
 * layout's padding included).  Returns PIC_ERR_INVALID on bad input. */
pic_status pic_plan_offsets(const int32_t* chunk_lens_host, const int32_t* chunk_off_host,
                            const int32_t* q_len_host, const int32_t* k_host, int32_t n_req,
                            pic_layout layout, int32_t* row_off_host, int32_t* page_off_host,
                            int32_t* rot_off_host, int32_t* fresh_off_host,
                            int32_t* chunk_page_off_host);

/* Message for a status code (static string, never NULL). */
const char* pic_strerror(pic_status status);

/* ------------------------------------------------------------------------
 * a1  Row selection (EPIC link_legolink Step 1; worked example).
 * ------------------------------------------------------------------------
 * For every request r (one thread block each): walks its chunks in link order,
 * writes each chunk's start s_c (exclusive prefix sum of the lengths) to
 * chunk_start[c], and writes the recomputed rows' global positions, ascending,
 * to rows[row_off[r] ...]: the first min(k[r], L_c) positions of every chunk
 * c >= 1, then T .. T + q[r] - 1.
 *   chunk_lens  [n_chunks_total] int32, >= 1       (device)
 *   chunk_off   [n_req+1] int32 CSR                 (device)
 *   q_len, k    [n_req] int32, >= 0                 (device)
 *   row_off     [n_req+1] int32 from pic_plan_offsets (device)
 *   rows        [row_off[n_req]] int32  out         (device)
 *   chunk_start [n_chunks_total] int32  out         (device)
 * Device errors: PIC_ERR_INVALID (length < 1, q or k < 0), PIC_ERR_RANGE (the
 * request's row count disagrees with row_off). */
pic_status pic_select_rows(const int32_t* chunk_lens, const int32_t* chunk_off,
                           const int32_t* q_len, const int32_t* k, const int32_t* row_off,
                           int32_t n_req, int32_t* rows, int32_t* chunk_start,
                           int32_t* err_flag, pic_stream_t stream);

/* ------------------------------------------------------------------------
 * Splice: build each request's link page list, its re-rotation work list and
 * the pool slot of every recomputed row (EPIC Step 3: cached K/V are copied to
 * their global positions and the recomputed rows overwrite theirs; HYPIC 2.2:
 * seam rows are not taken from the cache).  Layout as in pic_request_sizes_of.
 *   chunk_lens, chunk_off, q_len, k, n_req: as for pic_select_rows
 *   chunk_start     [n_chunks_total] from pic_select_rows
 *   chunk_page_off  [n_chunks_total+1] CSR into the three per-chunk page tables
 *   k_src_blocks    [chunk_page_off[n]] K-pool block of each chunk page as cached
 *   k_dst_blocks    same shape: where the rotated K goes; NULL = in place
 *   v_blocks        same shape: V-pool block of each chunk page (never written)
 *   fresh_off       [n_req+1] CSR into fresh_blocks
 *   fresh_blocks    block ids (same id in the K and V pools) for recomputed rows
 *   page_off, rot_off [n_req+1] from pic_plan_offsets (with the same layout)
 *   layout  PIC_LAYOUT_SPLICED, or PIC_LAYOUT_FRAMED for rotate-on-read (each
 *                 chunk's run padded to whole key tiles with entries {-1, -1,
 *                 next chunk's start, 0, 0}; k_dst_blocks must be NULL)
 *   pages   out [page_off[n_req]]   link page lists (gpos0 global)
 *   rot     out [rot_off[n_req]]    re-rotation work (tab = flat chunk index)
 *   row_block, row_slot out [n_rows]: pool block and slot of each recomputed row
 *                 (row order as written by pic_select_rows; row_off gives n_rows)
 *   row_frame_pos out [n_rows] or NULL: the position at which each recomputed
 *                 row's fresh K is to be encoded: its global position in the
 *                 spliced layout; in the framed layout its position within its
 *                 chunk (seam rows of chunks c >= 1) or its global position
 *                 (query rows).  pic_rope_table over it gives the table for
 *                 pic_write_fresh_kv.
 *   page_tab out [page_off[n_req]] or NULL: per link page, the offset-table row
 *                 of the page's frame: the flat chunk index for the pages of a
 *                 chunk after the first (in the framed layout its fresh pages and
 *                 padding too), -1 for pages in the global frame (chunk 0, query
 *                 pages; fresh pages in the spliced layout); the input of
 *                 pic_link_attention_ror
 *   row_off [n_req+1]
 * With k_dst_blocks NULL the cached pages of the list are the cached blocks
 * themselves: rotated in place by pic_rerotate_k, or left as cached for
 * rotate-on-read.
 * Device errors: PIC_ERR_RANGE when a count disagrees with the offsets. */
pic_status pic_splice_pages(const int32_t* chunk_lens, const int32_t* chunk_off,
                            const int32_t* q_len, const int32_t* k, int32_t n_req,
                            const int32_t* chunk_start, const int32_t* chunk_page_off,
                            const int32_t* k_src_blocks, const int32_t* k_dst_blocks,
                            const int32_t* v_blocks, const int32_t* fresh_off,
                            const int32_t* fresh_blocks, const int32_t* row_off,
                            const int32_t* page_off, const int32_t* rot_off, pic_layout layout,
                            pic_link_page* pages, pic_rot_page* rot, int32_t* row_block,
                            int32_t* row_slot, int32_t* row_frame_pos, int32_t* page_tab,
                            int32_t* err_flag, pic_stream_t stream);

/* ------------------------------------------------------------------------
 * a2  RoPE tables (RoPE article 2.2 and footnote 3).
 * ------------------------------------------------------------------------
 * table[i][j] = { cos_hi, sin_hi, cos_lo, sin_lo } of the angle pos[i] * theta^(-2j/d),
 * j < d/2: theta^(-2j/d) by the host's fp64 pow (once per call, passed to the
 * kernel), cos and sin computed in fp64 on the device and stored as two fp32
 * parts each (hi = v rounded to 16 significant bits, lo = fp32(v - hi)).  With
 * them the rotation kernels reach ~2^-23 relative error (bf16 inputs times a
 * 16-bit hi are exact in fp32) and store K within one bf16 ulp of the exact
 * rotation.  Used with pos = chunk_start (offset table for the rotary correction
 * by Delta_c) and with pos = rows (per-row table for fresh K and for Q).
 *   pos [n] int32 (device); table out [n][d/2][4] fp32 (device, 16-byte aligned);
 *   d even, 2..256.
 * Errors: PIC_ERR_INVALID (n < 0, bad d, theta <= 0). */
pic_status pic_rope_table(const int32_t* pos, int64_t n, int32_t d, double theta, float* table,
                          pic_stream_t stream);

/* ------------------------------------------------------------------------
 * a3  Re-rotation of cached K by the chunk offset (rotary correction, RoPE
 *     article 3.3): K <- R(theta * Delta) K, one rotation, fp32 math, one
 *     rounding to the pool dtype (bf16 round-to-nearest-even).  V untouched.
 * ------------------------------------------------------------------------
 *   k_pool     [num_blocks][Hkv][16][d] (read and written)
 *   rot        [n_rot] work entries (pic_splice_pages); tab < n_tab
 *   table      [n_tab][d/2][4] offset table (pic_rope_table over chunk_start)
 * In place entries read and write the same slots; out-of-place entries must not
 * overlap another entry's source.  Device errors: PIC_ERR_RANGE (block id outside
 * [0, num_blocks), tab outside [0, n_tab), lo/hi outside [0, 16]).
 * Supported: bf16 or fp32 pools, d even, 2 <= d <= 256, d % 16 == 0 for bf16. */
pic_status pic_rerotate_k(void* k_pool, int64_t num_blocks, pic_dtype dtype, int32_t Hkv,
                          int32_t d, const pic_rot_page* rot, int64_t n_rot, const float* table,
                          int64_t n_tab, int32_t* err_flag, pic_stream_t stream);

/* ------------------------------------------------------------------------
 * a3' Scheme B (RoPE article 3.2): the cached chunks hold K WITHOUT position
 *     encoding; on link every kept cached slot is encoded at its global
 *     position: slot s of page j of chunk c <- RoPE(K, s_c + 16 j + s), fp32 math,
 *     one rounding to the pool dtype.  Chunk 0 is encoded too (at 0..L_0 - 1).
 *     Replaces the offset table and pic_rerotate_k of the rotary correction.
 * ------------------------------------------------------------------------
 *   k_pool            [num_blocks][Hkv][16][d] (read and written)
 *   chunk_lens, chunk_off, k, n_req, chunk_start: as pic_select_rows (chunk_start
 *                     is its output)
 *   chunk_page_off    [n_chunks+1], n_chunk_pages = chunk_page_off[n_chunks] (host)
 *   k_src_blocks      [n_chunk_pages] block of each cached page
 *   k_dst_blocks      [n_chunk_pages] destination, or NULL for in place.  With
 *                     chunks shared by requests every chunk (the first too) is
 *                     encoded out of place into the request's private pages, and
 *                     pic_splice_pages is given those pages as its k_src_blocks
 *                     so that the page list reads them
 *   pos_table         [n_pos][d/2][4]: pic_rope_table over positions 0..n_pos-1
 *                     (a per-model table; every encoded position must be < n_pos)
 * Slots [0, min(k, L_c)) of chunks after the first (recomputed rows) are left
 * alone.  Device errors: PIC_ERR_RANGE (block id, or a position >= n_pos).
 * Supported: as pic_rerotate_k. */
pic_status pic_rope_cached_k(void* k_pool, int64_t num_blocks, pic_dtype dtype, int32_t Hkv, int32_t d,
                             const int32_t* chunk_lens, const int32_t* chunk_off, const int32_t* k,
                             int32_t n_req, const int32_t* chunk_start, const int32_t* chunk_page_off,
                             int32_t n_chunks, int64_t n_chunk_pages, const int32_t* k_src_blocks,
                             const int32_t* k_dst_blocks, const float* pos_table, int64_t n_pos,
                             int32_t* err_flag, pic_stream_t stream);

/* ------------------------------------------------------------------------
 * a4  Fresh K/V of the recomputed rows (EPIC Step 3: the new K/V replace the
 *     cached slots / append the query): K <- RoPE(k_raw[i], p_i) rounded to the
 *     pool dtype, V <- v_raw[i], written to slot row_slot[i] of block
 *     row_block[i] in both pools.
 * ------------------------------------------------------------------------
 *   k_raw, v_raw [n_rows][Hkv][d] pool dtype (un-roped K, V)
 *   row_table    [n_rows][d/2][4] (pic_rope_table over rows)
 *   row_block, row_slot [n_rows] (pic_splice_pages)
 * Device errors: PIC_ERR_RANGE (block or slot out of range). */
pic_status pic_write_fresh_kv(void* k_pool, void* v_pool, int64_t num_blocks, pic_dtype dtype,
                              int32_t Hkv, int32_t d, const void* k_raw, const void* v_raw,
                              const float* row_table, const int32_t* row_block,
                              const int32_t* row_slot, int64_t n_rows, int32_t* err_flag,
                              pic_stream_t stream);

/* ------------------------------------------------------------------------
 * a5+a6  Recompute-row link attention (EPIC Step 3; offset causal mask of the
 *        KV-cache blog).  For every recomputed row i of request r and query
 *        head h:  out[i][h] = sum_j softmax_j(scale * RoPE(q[i][h], p_i) . K_j) V_j
 *        over the request's pages, keys at global positions <= p_i, KV head
 *        h / (Hq/Hkv).  Q is roped on load and rounded to the pool dtype; scores,
 *        softmax and accumulation are fp32; out is written in the pool dtype.
 * ------------------------------------------------------------------------
 *   q           [n_rows][Hq][d] un-roped Q (pool dtype)
 *   row_table   [n_rows][d/2][4] (pic_rope_table over rows)
 *   rows        [n_rows] global positions (pic_select_rows); row_off [n_req+1]
 *   k_pool, v_pool [num_blocks][Hkv][16][d]
 *   pages       link page lists (pic_splice_pages); page_off [n_req+1]
 *   out         [n_rows][Hq][d] pool dtype
 *   ws          workspace of at least pic_link_attention_workspace() bytes,
 *               256-byte aligned; contents need not be initialised.
 * bf16 pools with d = 128 and Hq/Hkv in {1, 2, 4, 8, 16} run on the tensor cores
 * (tcgen05, TMEM accumulators, TMA page loads; at most 1024 requests per call,
 * else PIC_ERR_UNSUPPORTED); fp32 pools and other bf16 shapes run on the SIMT
 * kernel.  Every bounded wait that runs out sets
 * PIC_ERR_TIMEOUT in *err_flag and the kernel returns.
 * Errors: PIC_ERR_INVALID (Hq % Hkv != 0, bad d, n_req < 0, ...),
 * PIC_ERR_WORKSPACE, PIC_ERR_UNSUPPORTED, PIC_ERR_CUDA. */
size_t pic_link_attention_workspace(int64_t n_rows, int32_t n_req, int32_t Hq, int32_t Hkv,
                                    int32_t d, pic_dtype dtype);

pic_status pic_link_attention(const void* q, const float* row_table, const int32_t* rows,
                              const int32_t* row_off, const void* k_pool, const void* v_pool,
                              int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                              const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                              int32_t Hkv, int32_t d, float scale, void* out, void* ws,
                              size_t ws_bytes, int32_t* err_flag, pic_stream_t stream);

/* ------------------------------------------------------------------------
 * Link attention without a caller workspace.  (No counterpart in the
 * papers: this is a packaging variant of pic_link_attention.)
 * ------------------------------------------------------------------------
 * Some callers cannot allocate device memory at the point where they run the
 * link step: a serving engine that has already reserved nearly all of HBM for
 * its KV pool (a cudaMalloc then fails, and it also synchronises the device,
 * stalling every other stream), or a plugin that is handed device pointers by a
 * host framework that owns all allocation.  For them this entry point computes
 * exactly what pic_link_attention computes, same arguments minus ws/ws_bytes,
 * with its planning and split-KV scratch in one fixed device array of
 * PIC_NOALLOC_SCRATCH_BYTES inside the library.  It calls no cudaMalloc,
 * cudaFree or allocating routine.
 *   - The array is reserved on a GPU when the library's device code is loaded
 *     there.  CUDA loads device code lazily by default: at the first launch of
 *     one of this library's attention kernels on that GPU, or at this entry
 *     point's first call, whichever comes first; it then stays reserved until
 *     the process exits.  Loading may also synchronise the device.
 *   - Warm-up: call this entry point once on each device, with that device
 *     current, BEFORE reserving most of HBM and before any stream capture.  A
 *     call with n_req = 0 or n_rows = 0 does exactly this (it launches nothing,
 *     loads the device code, looks up and keeps the array's device address) and
 *     returns PIC_OK, or PIC_ERR_CUDA if the device code cannot be loaded (for
 *     example when HBM is already full).
 *   - The looked-up address is kept for the life of the process: do not use
 *     the library across a cudaDeviceReset.
 *   - Every call on a device uses the same array, which keeps the previous
 *     call's contents (nothing in it needs to start at zero).  Calls whose work
 *     overlaps on the GPU (different streams, or host threads without ordering)
 *     race on the array: order them.
 *   - The tensor-core path (bf16, d = 128) splits long key ranges into at most
 *     60 extra work units; a call whose scratch would exceed the array (more
 *     than 959 recomputed rows of one request at Hq = 32, Hkv = 8, more than
 *     767 over 4 requests) is refused with PIC_ERR_WORKSPACE before any other check or
 *     launch.  The SIMT path (fp32 pools, other shapes) needs no scratch.
 * Results match pic_link_attention within the attention tolerance (the split
 * of key ranges, and so the summation order, can differ). */
#define PIC_NOALLOC_SCRATCH_BYTES (32u << 20)

pic_status pic_link_attention_noalloc(const void* q, const float* row_table, const int32_t* rows,
                                      const int32_t* row_off, const void* k_pool, const void* v_pool,
                                      int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                                      const int32_t* page_off, int32_t n_req, int64_t n_rows,
                                      int32_t Hq, int32_t Hkv, int32_t d, float scale, void* out,
                                      int32_t* err_flag, pic_stream_t stream);

/* The same call in two halves, so that the part that reads no K or V can overlap
 * the re-rotation pass on another stream:
 *   pic_link_attention_plan  plans the work units and writes the roped Q operands
 *       into ws (reads q, row_table, rows, row_off, pages, page_off only; a no-op
 *       for shapes off the tensor cores);
 *   pic_link_attention_run   the attention and the merge, from that plan.
 * run must follow plan (stream order or an event) with the same arguments and the
 * same ws, untouched in between; plan + run = pic_link_attention, bit for bit. */
pic_status pic_link_attention_plan(const void* q, const float* row_table, const int32_t* rows,
                                   const int32_t* row_off, const pic_link_page* pages, const int32_t* page_off,
                                   int32_t n_req, int64_t n_rows, int32_t Hq, int32_t Hkv, int32_t d,
                                   pic_dtype dtype, void* ws, size_t ws_bytes, int32_t* err_flag,
                                   pic_stream_t stream);

pic_status pic_link_attention_run(const void* q, const float* row_table, const int32_t* rows,
                                  const int32_t* row_off, const void* k_pool, const void* v_pool,
                                  int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                                  const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                                  int32_t Hkv, int32_t d, float scale, void* out, void* ws, size_t ws_bytes,
                                  int32_t* err_flag, pic_stream_t stream);

/* pic_link_attention_plan in two parts, so that the part that needs no page list
 * can run before the splice has written it:
 *   pic_link_attention_plan_q      the tile pairs' rows and the roped Q operands
 *                                  (reads q, row_table, row_off);
 *   pic_link_attention_plan_units  the work units (reads rows, row_off, pages,
 *                                  page_off).
 * Arguments as pic_link_attention_plan.  They write different fields of the
 * plan in ws (the tiles' rows and the Q operands; the units and the tiles' key
 * ranges), so they run in either order or at the same time on two streams; both
 * together are pic_link_attention_plan, bit for bit, and both precede the run. */
pic_status pic_link_attention_plan_q(const void* q, const float* row_table, const int32_t* row_off,
                                     int32_t n_req, int64_t n_rows, int32_t Hq, int32_t Hkv, int32_t d,
                                     pic_dtype dtype, void* ws, size_t ws_bytes, int32_t* err_flag,
                                     pic_stream_t stream);
pic_status pic_link_attention_plan_units(const int32_t* rows, const int32_t* row_off, const pic_link_page* pages,
                                         const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                                         int32_t Hkv, int32_t d, pic_dtype dtype, void* ws, size_t ws_bytes,
                                         int32_t* err_flag, pic_stream_t stream);

/* ------------------------------------------------------------------------
 * a3+a5  Rotate-on-read link attention (RoPE article 3.3: the rotary correction
 *     applied where the kernel reads the cache, a mixed reuse + correction
 *     path).  Over a page list of the framed layout (PIC_LAYOUT_FRAMED): every
 *     chunk's keys stay in the chunk's own frame — the cached pages as cached,
 *     the recomputed head rows encoded at their position in the chunk — and
 *     every key tile (PIC_TILE_PAGES pages) lies in one chunk.  Since
 *     RoPE(q, p) . R(Delta) k = R(-Delta) RoPE(q, p) . k, the kernel rotates Q
 *     back by the chunk's offset (fp32, cos / sin = hi + lo of the table row, one
 *     more bf16 rounding) for the key tiles of that chunk instead of rotating K:
 *     no re-rotation pass, cached pages never written, no per-request copies of
 *     shared chunks.  Not bit-identical to pic_rerotate_k + pic_link_attention
 *     (Q is rounded in another frame); checked against the same float64
 *     reference at the same tolerance.
 * ------------------------------------------------------------------------
 *   arguments as pic_link_attention, plus
 *   page_tab   [page_off[n_req]] int32: each link page's frame — the row of its
 *              chunk's offset in rot_table, < 0 for the global frame (chunk 0,
 *              the query) — pic_splice_pages' page_tab output for the framed
 *              layout, with k_dst_blocks NULL so that the list points at the
 *              cached blocks
 *   rot_table  [n_tab][d/2][4] fp32 offset table (pic_rope_table over chunk_start)
 * Tensor-core shapes only (bf16 pools, d = 128, Hq / Hkv in {1, 2, 4, 8, 16});
 * otherwise PIC_ERR_UNSUPPORTED.  A frame >= n_tab sets PIC_ERR_RANGE in
 * *err_flag and that key tile is read in the global frame. */
pic_status pic_link_attention_ror(const void* q, const float* row_table, const int32_t* rows,
                                  const int32_t* row_off, const void* k_pool, const void* v_pool,
                                  int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                                  const int32_t* page_tab, const float* rot_table, int64_t n_tab,
                                  const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                                  int32_t Hkv, int32_t d, float scale, void* out, void* ws, size_t ws_bytes,
                                  int32_t* err_flag, pic_stream_t stream);

/* ------------------------------------------------------------------------
 * Decode after link (EPIC review: the query and the tokens decoded after it
 * gather the information of all chunks; "KV cache from scratch", single-token
 * cache decode: a new position reads the whole cache once).
 * ------------------------------------------------------------------------
 * One new query row per request, at position P_r, attends over the keys listed
 * in the request's page list (every listed key is visible: the list holds the
 * linked context, the recomputed rows and the new row's own K/V, which the caller
 * wrote first with pic_write_fresh_kv):
 *   out[r][h] = softmax_j(RoPE(q[r][h], P_r) . K_j[h / g] * scale) . V_j[h / g]
 * with RoPE(q) rounded to bf16 as on the link path.
 *   q         [n_req][Hq][d] bf16, un-roped
 *   q_table   [n_req][d/2][4] fp32: pic_rope_table over the positions P_r
 *   k_pool, v_pool, num_blocks, pages, page_off: as pic_link_attention (the
 *             lo/hi slot range of every page entry is honoured; gpos0 is unused)
 *   page_tab, rot_table, n_tab: NULL / NULL / 0 when every listed key is encoded
 *             at its global position (the spliced layout).  After a rotate-on-read
 *             link (the framed layout) the page list's page_tab from
 *             pic_splice_pages (-1 for the new row's own page) and the offset table
 *             of pic_link_attention_ror: the keys of a page with row f >= 0 are in
 *             that chunk's frame, and the consumer rotates Q back by its offset,
 *             R(-theta * Delta_f) RoPE(q, P), rounded to bf16, for them.  A row
 *             >= n_tab sets PIC_ERR_RANGE and the page is read in the global frame
 *   out       [n_req][Hq][d] bf16
 *   ws        at least pic_decode_workspace() bytes, 256-byte aligned, any contents
 * bf16 pools with d = 128 and g = Hq / Hkv in {1, 2, 4, 8}; otherwise
 * PIC_ERR_UNSUPPORTED (0 from pic_decode_workspace).  Every request gets splits in
 * proportion to its pages so that all CTAs fit in one wave — found by the decode
 * CTAs themselves up to 160 requests, by a one-block planner launch above —,
 * the split-KV decode (pages moved into shared memory by TMA, each page's two
 * small contractions on warp-level bf16 MMAs with fp32 accumulate, P rounded to
 * bf16 as on the link path), and the merge of the splits.  Bound by HBM: every
 * listed K and V row is read once.  A bad block id or slot range sets
 * PIC_ERR_RANGE in *err_flag and that page is skipped; a bounded wait that runs
 * out sets PIC_ERR_TIMEOUT. */
size_t pic_decode_workspace(int32_t n_req, int32_t Hq, int32_t Hkv, int32_t d, pic_dtype dtype);

pic_status pic_decode_attention(const void* q, const float* q_table, const void* k_pool,
                                const void* v_pool, int64_t num_blocks, pic_dtype dtype,
                                const pic_link_page* pages, const int32_t* page_off,
                                const int32_t* page_tab, const float* rot_table, int64_t n_tab,
                                int32_t n_req, int32_t Hq, int32_t Hkv, int32_t d, float scale, void* out,
                                void* ws, size_t ws_bytes, int32_t* err_flag, pic_stream_t stream);

/* ------------------------------------------------------------------------
 * Linear-layer state composition (HYPIC blog, section 2.1: linear layers).
 * ------------------------------------------------------------------------
 * A hybrid model's linear-attention layer caches, per chunk c and head h, the pair
 * (T_c, S_c): the chunk's cumulative transition operator T_C and its end state from
 * a zero state S(C|0), both d x d.  Linking chunks C1 C2 .. Cn in that order gives
 * the layer's state S = T_n (.. (T_2 S_1 + S_2) ..) + S_n, by the blog's rule
 * S(C1 C2) = T(C2) S(C1) + S(C2); the transition of C1 is never used.
 *
 * The cache keeps T in the form the tensor cores take: two bf16 planes per
 * matrix, hi = bf16(T) and lo = bf16(T - hi) (T = hi + lo to about 2^-16 of |T|,
 * which is all the split product below uses of it).  pic_compose_split_t writes
 * that form from fp32 T once, when a chunk's pair is cached:
 *   T        [n_mats][d][d] fp32 (device)
 *   T_split  [n_mats][2][d][d] bf16 out (device): plane 0 hi, plane 1 lo
 *
 * pic_compose_states:
 *   T_split  [n_pool][H][2][d][d] bf16 (device): the cached transitions
 *   S_pool   [n_pool][H][d][d] fp32 row-major (device): the cached end states
 *   ids        [n_elems] int32 (device): chain of every request, pool entries in
 *              chain order; request r owns ids[chain_off[r] .. chain_off[r+1])
 *   chain_off  [n_req + 1] int32 (device), chain_off[0] = 0, chain_off[n_req] = n_elems
 *   max_chain  host: an upper bound of every chain's length (longer chains are
 *              cut to it and flagged)
 *   seg        0, or the level-0 segment length: chains are cut into segments of
 *              seg elements, folded in parallel (each non-first segment also
 *              forms its transition product), then folded per chain by a second
 *              launch.  0 (or seg >= max_chain) folds every chain in one launch.
 *              pic_compose_segment() gives the choice that fills one wave of `sms`
 *              SMs.  The workspace depends on seg.
 *   out        [n_req][H][d][d] fp32 (device); an empty chain gives zeros
 *   ws         at least pic_compose_workspace() bytes, 256-byte aligned
 * d = 128 only (else PIC_ERR_UNSUPPORTED; 0 from pic_compose_workspace).  Each
 * fold step is a 128 x 128 x 128 tensor-core product of bf16 parts
 * (hi.hi + hi.lo + lo.hi, fp32 accumulate: about 2^-16 relative error per step);
 * S is added in fp32.  One or two launches (one more, a planner, above 352
 * requests).  A pool id outside [0, n_pool) or
 * offsets that disagree with n_elems / max_chain set PIC_ERR_RANGE in *err_flag
 * (pool entry 0 is read in place of a bad id); a bounded wait that runs out sets
 * PIC_ERR_TIMEOUT. */
pic_status pic_compose_split_t(const float* T, int64_t n_mats, int32_t d, void* T_split, pic_stream_t stream);

int32_t pic_compose_segment(int32_t n_req, int64_t n_elems, int32_t max_chain, int32_t H, int32_t sms);

size_t pic_compose_workspace(int32_t n_req, int32_t max_chain, int32_t H, int32_t d, int32_t seg);

pic_status pic_compose_states(const void* T_split, const float* S_pool, int64_t n_pool, const int32_t* ids,
                              const int32_t* chain_off, int32_t n_req, int64_t n_elems, int32_t max_chain,
                              int32_t H, int32_t d, int32_t seg, float* out, void* ws, size_t ws_bytes,
                              int32_t* err_flag, pic_stream_t stream);

/* ------------------------------------------------------------------------
 * Diagnostics.
 * ------------------------------------------------------------------------
 * One 128 x 128 x 128 bf16 tensor-core product through the same shared-memory
 * layouts, descriptors and TMEM read-back the attention kernel uses:
 *   d_kmajor[m][n] = sum_k a[m][k] * b[n][k]    (B K-major, as Q.K^T)
 *   d_mnmajor[m][n] = sum_k a[m][k] * b[k][n]   (B MN-major, as P.V)
 *   d_tmem_a[m][n]  = sum_k a[m][k] * b[k][n]   (A read from TMEM, as P.V)
 * a, b: [128][128] bf16 row-major (device); outputs [128][128] fp32 (device).
 * One launch of one thread block.  Not part of the link step. */
pic_status pic_selftest_umma(const void* a, const void* b, float* d_kmajor, float* d_mnmajor,
                             float* d_tmem_a, int32_t* err_flag, pic_stream_t stream);

/* The CTA-pair products (tcgen05 cta_group::2: two SMs on one M = 256 product, B
 * split along N between them) with the operand layouts of the two-SM attention:
 *   d_s[m][n]  = sum_k a[m][k] * b[n][k]     m < 256, n < 256 (S = Q.K^T: CTA r
 *                holds rows 128r.. of a and keys 128r.. of b)
 *   d_pv[m][n] = sum_j a[m][j] * v[j][n]     m < 256, j, n < 128 (P.V: P from
 *                TMEM, CTA r holds columns 64r.. of v)
 * a, b: [256][128] bf16; v: [128][128] bf16 (device, row-major); d_s [256][256],
 * d_pv [256][128] fp32 (device); info [2] int32: the TMEM base address each CTA
 * was given.  One launch of one cluster of two CTAs.  Not part of the link step. */
pic_status pic_selftest_umma_pair(const void* a, const void* b, const void* v, float* d_s, float* d_pv,
                                  int32_t* info, int32_t* err_flag, pic_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PIC_H_ */
