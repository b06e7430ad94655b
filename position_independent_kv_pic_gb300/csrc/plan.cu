// Link-step metadata on the device: LegoLink row selection, the splice (page
// lists, re-rotation work, fresh-row slots) and the RoPE cos/sin tables.
//
// Row selection follows the EPIC blog review's link_legolink Step 1: chunk 0 is
// never recomputed, every later chunk recomputes its first min(k, L_c) tokens,
// and every query token is recomputed.  The splice follows Step 3: cached K/V
// land at their global positions, the recomputed rows' fresh K/V replace the
// cached head rows (HYPIC's seam window keeps those rows out of the cache), and
// the query's K/V are appended.
#include <algorithm>

#include <cmath>

#include "pic_internal.cuh"

namespace pic {
namespace {

constexpr int kPlanThreads = 256;

// Per-chunk quantities of one request, for chunks processed in groups of
// kPlanThreads.  m = recomputed head rows, np = pages of the chunk,
// kept = cached pages keeping at least one slot, fp = fresh pages.
struct ChunkInfo {
  int L, m, np, kept, fp;
};

__device__ __forceinline__ ChunkInfo chunk_info(int L, int c_local, int k) {
  ChunkInfo ci;
  ci.L = L;
  ci.m = (c_local == 0) ? 0 : min(k, L);
  ci.np = ceil_div(L, PIC_PAGE);
  ci.kept = (ci.m == L) ? 0 : ci.np - ci.m / PIC_PAGE;
  ci.fp = ceil_div(ci.m, PIC_PAGE);
  return ci;
}

__global__ void __launch_bounds__(kPlanThreads)
select_rows_kernel(const int32_t* __restrict__ chunk_lens, const int32_t* __restrict__ chunk_off,
                   const int32_t* __restrict__ q_len, const int32_t* __restrict__ kk,
                   const int32_t* __restrict__ row_off, int32_t* __restrict__ rows,
                   int32_t* __restrict__ chunk_start, int32_t* err) {
  __shared__ int scratch[kPlanThreads / 32 + 1];
  const int r = blockIdx.x;
  const int c0 = chunk_off[r], c1 = chunk_off[r + 1];
  const int q = q_len[r], k = kk[r];
  const int rbeg = row_off[r], rend = row_off[r + 1];
  if (q < 0 || k < 0 || c1 < c0) {
    if (threadIdx.x == 0) set_err(err, PIC_ERR_INVALID);
    return;
  }
  int pos_base = 0, row_base = 0;  // running s_c and running row count
  for (int g = c0; g < c1; g += kPlanThreads) {
    const int c = g + threadIdx.x;
    int L = 0, m = 0;
    if (c < c1) {
      L = chunk_lens[c];
      if (L < 1) {
        set_err(err, PIC_ERR_INVALID);
        L = 1;
      }
      m = (c == c0) ? 0 : min(k, L);
    }
    int totL, totM;
    const int s = pos_base + block_exclusive_scan<kPlanThreads>(L, scratch, &totL);
    const int mo = row_base + block_exclusive_scan<kPlanThreads>(m, scratch, &totM);
    if (c < c1) {
      chunk_start[c] = s;
      for (int j = 0; j < m; ++j) {
        const int idx = rbeg + mo + j;
        if (idx < rend) rows[idx] = s + j;
      }
    }
    pos_base += totL;
    row_base += totM;
  }
  // query rows at T .. T+q-1
  for (int j = threadIdx.x; j < q; j += kPlanThreads) {
    const int idx = rbeg + row_base + j;
    if (idx < rend) rows[idx] = pos_base + j;
  }
  if (threadIdx.x == 0 && row_base + q != rend - rbeg) set_err(err, PIC_ERR_RANGE);
}

// Position of `x` in a non-decreasing prefix array pre[0..n] (pre[0] = 0): the w
// with pre[w] <= x < pre[w+1].
__device__ __forceinline__ int find_owner(const int* pre, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// gridDim.y blocks per request.  Chunks are taken kPlanThreads at a time: block
// scans (repeated by every block of the request, they are cheap) give every
// chunk its first link page, re-rotation entry, fresh page and recomputed row;
// then the request's blocks share the group's pages and row slots, one item per
// thread, so neither a long chunk nor a long request serialises.
__global__ void __launch_bounds__(kPlanThreads)
splice_kernel(const int32_t* __restrict__ chunk_lens, const int32_t* __restrict__ chunk_off,
              const int32_t* __restrict__ q_len, const int32_t* __restrict__ kk,
              const int32_t* __restrict__ chunk_start, const int32_t* __restrict__ chunk_page_off,
              const int32_t* __restrict__ k_src, const int32_t* __restrict__ k_dst,
              const int32_t* __restrict__ v_blk, const int32_t* __restrict__ fresh_off,
              const int32_t* __restrict__ fresh_blocks, const int32_t* __restrict__ row_off,
              const int32_t* __restrict__ page_off, const int32_t* __restrict__ rot_off, int framed,
              pic_link_page* __restrict__ pages, pic_rot_page* __restrict__ rot,
              int32_t* __restrict__ row_block, int32_t* __restrict__ row_slot, int32_t* __restrict__ row_frame_pos,
              int32_t* __restrict__ page_tab, int32_t* err) {
  __shared__ int scratch[kPlanThreads / 32 + 1];
  __shared__ int g_link[kPlanThreads + 1], g_row[kPlanThreads + 1];
  __shared__ int g_rot[kPlanThreads], g_fresh[kPlanThreads];
  __shared__ int g_s[kPlanThreads], g_L[kPlanThreads], g_m[kPlanThreads], g_fp[kPlanThreads], g_j0[kPlanThreads];
  __shared__ int g_run[kPlanThreads];
  const int r = blockIdx.x, tid = threadIdx.x;
  const int c0 = chunk_off[r], c1 = chunk_off[r + 1];
  const int q = q_len[r], k = kk[r];
  if (q < 0 || k < 0 || c1 < c0) {
    if (tid == 0 && blockIdx.y == 0) set_err(err, PIC_ERR_INVALID);
    return;
  }
  const int item0 = blockIdx.y * kPlanThreads + tid, stride = gridDim.y * kPlanThreads;
  const int pbeg = page_off[r], pend = page_off[r + 1];
  const int obeg = rot_off[r], oend = rot_off[r + 1];
  const int fbeg = fresh_off[r], fend = fresh_off[r + 1];
  const int rbeg = row_off[r], rend = row_off[r + 1];

  int link_base = 0, rot_base = 0, fresh_base = 0, row_base = 0, T = 0;
  for (int g = c0; g < c1; g += kPlanThreads) {
    const int c = g + tid;
    const int n_in = min(kPlanThreads, c1 - g);
    ChunkInfo ci = {0, 0, 0, 0, 0};
    if (c < c1) {
      ci = chunk_info(max(chunk_lens[c], 1), c - c0, k);
      if (chunk_page_off[c + 1] - chunk_page_off[c] != ci.np && blockIdx.y == 0) set_err(err, PIC_ERR_RANGE);
    }
    int t_link, t_rot, t_fresh, t_row, t_len;
    // a chunk's link pages: fresh head pages, kept cached pages, and in the framed
    // layout empty entries up to a whole number of key tiles
    const int run = ci.fp + ci.kept;
    const int n_link = (framed && c < c1) ? ceil_div(run, PIC_TILE_PAGES) * PIC_TILE_PAGES : run;
    const int ex_link = block_exclusive_scan<kPlanThreads>(n_link, scratch, &t_link);
    const int ex_rot = block_exclusive_scan<kPlanThreads>((c > c0) ? ci.kept : 0, scratch, &t_rot);
    const int ex_fresh = block_exclusive_scan<kPlanThreads>(ci.fp, scratch, &t_fresh);
    const int ex_row = block_exclusive_scan<kPlanThreads>(ci.m, scratch, &t_row);
    block_exclusive_scan<kPlanThreads>(ci.L, scratch, &t_len);
    g_link[tid] = ex_link;
    g_row[tid] = ex_row;
    g_rot[tid] = ex_rot;
    g_fresh[tid] = ex_fresh;
    g_s[tid] = (c < c1) ? chunk_start[c] : 0;
    g_L[tid] = ci.L;
    g_m[tid] = ci.m;
    g_fp[tid] = ci.fp;
    g_j0[tid] = ci.np - ci.kept;
    g_run[tid] = run;
    if (tid == 0) {
      g_link[kPlanThreads] = t_link;
      g_row[kPlanThreads] = t_row;
    }
    __syncthreads();
    // the group's link pages (and re-rotation entries for chunks after the first)
    for (int P = item0; P < t_link; P += stride) {
      int w = find_owner(g_link, n_in, P);
      while (w + 1 < n_in && g_link[w + 1] <= P) ++w;  // skip chunks without pages
      const int cw = g + w;
      const int f = P - g_link[w];
      const int pi = pbeg + link_base + P;
      if (pi >= pend) { set_err(err, PIC_ERR_RANGE); continue; }
      pic_link_page pg;
      // the frame of the chunk's keys: its offset-table row in the framed layout
      // (chunks after the first), else the global frame
      const int frame = (cw > c0) ? cw : -1;
      if (f < g_fp[w]) {  // fresh head page f of the chunk
        const int fi = fbeg + fresh_base + g_fresh[w] + f;
        if (fi >= fend) { set_err(err, PIC_ERR_RANGE); continue; }
        const int blk = fresh_blocks[fi];
        pg.k_block = blk; pg.v_block = blk; pg.gpos0 = g_s[w] + PIC_PAGE * f;
        pg.lo = 0; pg.hi = (int16_t)min(PIC_PAGE, g_m[w] - PIC_PAGE * f);
        pages[pi] = pg;
        if (page_tab != nullptr) page_tab[pi] = framed ? frame : -1;
      } else if (f >= g_run[w]) {  // framed layout: padding up to the key-tile boundary
        pg.k_block = -1; pg.v_block = -1; pg.gpos0 = g_s[w] + g_L[w];
        pg.lo = 0; pg.hi = 0;
        pages[pi] = pg;
        if (page_tab != nullptr) page_tab[pi] = frame;
      } else {  // cached page j that keeps at least one slot
        const int t = f - g_fp[w];
        const int j = g_j0[w] + t;
        const int cp = chunk_page_off[cw] + j;
        const int src = k_src[cp];
        const int dst = (k_dst != nullptr) ? k_dst[cp] : src;
        pg.k_block = (cw == c0) ? src : dst;  // chunk 0 keeps Delta = 0
        pg.v_block = v_blk[cp];
        pg.gpos0 = g_s[w] + PIC_PAGE * j;
        pg.lo = (int16_t)max(0, g_m[w] - PIC_PAGE * j);
        pg.hi = (int16_t)min(PIC_PAGE, g_L[w] - PIC_PAGE * j);
        pages[pi] = pg;
        if (page_tab != nullptr) page_tab[pi] = frame;
        if (cw > c0) {
          const int oi = obeg + rot_base + g_rot[w] + t;
          if (oi >= oend) { set_err(err, PIC_ERR_RANGE); continue; }
          pic_rot_page rp;
          rp.src_block = src; rp.dst_block = dst; rp.tab = cw; rp.lo = pg.lo; rp.hi = pg.hi;
          rot[oi] = rp;
        }
      }
    }
    // the group's recomputed head rows
    for (int Rr = item0; Rr < t_row; Rr += stride) {
      int w = find_owner(g_row, n_in, Rr);
      while (w + 1 < n_in && g_row[w + 1] <= Rr) ++w;
      const int j = Rr - g_row[w];
      const int ri = rbeg + row_base + Rr, fi = fbeg + fresh_base + g_fresh[w] + j / PIC_PAGE;
      if (ri >= rend || fi >= fend) { set_err(err, PIC_ERR_RANGE); continue; }
      row_block[ri] = fresh_blocks[fi];
      row_slot[ri] = j % PIC_PAGE;
      if (row_frame_pos != nullptr) row_frame_pos[ri] = framed ? j : g_s[w] + j;
    }
    __syncthreads();
    link_base += t_link;
    rot_base += t_rot;
    fresh_base += t_fresh;
    row_base += t_row;
    T += t_len;
  }
  // query pages and rows
  const int qp = ceil_div(q, PIC_PAGE);
  for (int f = item0; f < qp; f += stride) {
    const int fi = fbeg + fresh_base + f, pi = pbeg + link_base + f;
    if (fi >= fend || pi >= pend) { set_err(err, PIC_ERR_RANGE); continue; }
    const int blk = fresh_blocks[fi];
    pic_link_page pg;
    pg.k_block = blk; pg.v_block = blk; pg.gpos0 = T + PIC_PAGE * f;
    pg.lo = 0; pg.hi = (int16_t)min(PIC_PAGE, q - PIC_PAGE * f);
    pages[pi] = pg;
    if (page_tab != nullptr) page_tab[pi] = -1;
  }
  for (int j = item0; j < q; j += stride) {
    const int ri = rbeg + row_base + j, fi = fbeg + fresh_base + j / PIC_PAGE;
    if (ri >= rend || fi >= fend) { set_err(err, PIC_ERR_RANGE); continue; }
    row_block[ri] = fresh_blocks[fi];
    row_slot[ri] = j % PIC_PAGE;
    if (row_frame_pos != nullptr) row_frame_pos[ri] = T + j;  // the query is in the global frame
  }
  if (tid == 0 && blockIdx.y == 0) {
    if (link_base + qp != pend - pbeg || rot_base != oend - obeg ||
        fresh_base + qp != fend - fbeg || row_base + q != rend - rbeg)
      set_err(err, PIC_ERR_RANGE);
  }
}

// table[i][j] = {cos_hi, sin_hi, cos_lo, sin_lo} of pos[i] * theta^(-2j/d): fp64
// math; hi = the value rounded to 16 significant bits (so that a bf16 times hi is
// exact in fp32), lo = fp32(v - hi).
__device__ __forceinline__ float round16(double v) {
  uint32_t u = __float_as_uint((float)v);
  u = (u + 0x7Fu + ((u >> 8) & 1u)) & ~0xFFu;  // ties to even on the 8 dropped bits
  return __uint_as_float(u);
}

// Small blocks: a table of a few thousand entries (the per-chunk offset table, one
// decode row) still spreads over many SMs, whose fp64 units are few.
constexpr int kTabThreads = 64;

// theta^(-2j/d), j < d/2, in fp64 (the host's pow, once per call).
struct InvFreq {
  double w[128];
};

__global__ void __launch_bounds__(kTabThreads)
rope_table_kernel(const int32_t* __restrict__ pos, int64_t n, int half, const __grid_constant__ InvFreq f,
                  float4* __restrict__ table) {
  __shared__ double inv_freq[128];
  for (int j = threadIdx.x; j < half; j += blockDim.x) inv_freq[j] = f.w[j];
  __syncthreads();
  const int64_t total = n * half;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / half;
    const int j = (int)(t - i * half);
    const double ang = (double)__ldg(pos + i) * inv_freq[j];
    double s, c;
    sincos(ang, &s, &c);
    const float ch = round16(c), sh = round16(s);
    table[t] = make_float4(ch, sh, (float)(c - (double)ch), (float)(s - (double)sh));
  }
}

}  // namespace
}  // namespace pic

using namespace pic;

extern "C" {

pic_status pic_select_rows(const int32_t* chunk_lens, const int32_t* chunk_off, const int32_t* q_len,
                           const int32_t* k, const int32_t* row_off, int32_t n_req, int32_t* rows,
                           int32_t* chunk_start, int32_t* err_flag, pic_stream_t stream) {
  if (n_req < 0) return PIC_ERR_INVALID;
  if (n_req == 0) return PIC_OK;
  if (!chunk_off || !q_len || !k || !row_off || !err_flag) return PIC_ERR_INVALID;
  select_rows_kernel<<<n_req, kPlanThreads, 0, (cudaStream_t)stream>>>(
      chunk_lens, chunk_off, q_len, k, row_off, rows, chunk_start, err_flag);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

pic_status pic_splice_pages(const int32_t* chunk_lens, const int32_t* chunk_off, const int32_t* q_len,
                            const int32_t* k, int32_t n_req, const int32_t* chunk_start,
                            const int32_t* chunk_page_off, const int32_t* k_src_blocks,
                            const int32_t* k_dst_blocks, const int32_t* v_blocks,
                            const int32_t* fresh_off, const int32_t* fresh_blocks,
                            const int32_t* row_off, const int32_t* page_off, const int32_t* rot_off,
                            pic_layout layout, pic_link_page* pages, pic_rot_page* rot, int32_t* row_block,
                            int32_t* row_slot, int32_t* row_frame_pos, int32_t* page_tab, int32_t* err_flag,
                            pic_stream_t stream) {
  if (n_req < 0 || (layout != PIC_LAYOUT_SPLICED && layout != PIC_LAYOUT_FRAMED)) return PIC_ERR_INVALID;
  // the framed layout keeps every chunk's K where it is cached
  if (layout == PIC_LAYOUT_FRAMED && k_dst_blocks != nullptr) return PIC_ERR_INVALID;
  if (n_req == 0) return PIC_OK;
  if (!chunk_off || !q_len || !k || !chunk_page_off || !fresh_off || !row_off || !page_off ||
      !rot_off || !err_flag)
    return PIC_ERR_INVALID;
  // enough blocks per request that a long request's pages take about one pass
  const int sms = num_sms_of_current_device();
  const int per_req = std::max(1, std::min(32, (2 * sms + n_req - 1) / n_req));
  splice_kernel<<<dim3((unsigned)n_req, (unsigned)per_req), kPlanThreads, 0, (cudaStream_t)stream>>>(
      chunk_lens, chunk_off, q_len, k, chunk_start, chunk_page_off, k_src_blocks, k_dst_blocks,
      v_blocks, fresh_off, fresh_blocks, row_off, page_off, rot_off, layout == PIC_LAYOUT_FRAMED ? 1 : 0, pages,
      rot, row_block, row_slot, row_frame_pos, page_tab, err_flag);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

pic_status pic_rope_table(const int32_t* pos, int64_t n, int32_t d, double theta, float* table,
                          pic_stream_t stream) {
  if (n < 0 || d < 2 || d > 256 || (d & 1) || !(theta > 0.0)) return PIC_ERR_INVALID;
  if (n == 0) return PIC_OK;
  if (!pos || !table) return PIC_ERR_INVALID;
  InvFreq f;
  for (int j = 0; j < d / 2; ++j) f.w[j] = std::pow(theta, -2.0 * (double)j / (double)d);
  const int64_t total = n * (d / 2);
  const int64_t blocks = (total + kTabThreads - 1) / kTabThreads;
  const int64_t cap = (int64_t)num_sms_of_current_device() * 32;
  rope_table_kernel<<<(unsigned)(blocks < cap ? blocks : cap), kTabThreads, 0, (cudaStream_t)stream>>>(
      pos, n, d / 2, f, reinterpret_cast<float4*>(table));
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

}  // extern "C"
