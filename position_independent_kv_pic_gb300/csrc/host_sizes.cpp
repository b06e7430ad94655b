// Host-side sizing of the link step: closed-form counts that let the caller size
// every buffer without a device round trip (EPIC link_legolink Step 1 gives the
// row count: min(k, L_c) head rows for every chunk but the first, plus the query).
#include <stddef.h>
#include <stdint.h>

#include "pic.h"

namespace {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

pic_status pic_request_sizes_of(const int32_t* lens, int32_t n_chunks, int32_t q, int32_t k,
                                pic_layout layout, pic_request_sizes* out) {
  if (out == nullptr || n_chunks < 0 || q < 0 || k < 0 || (n_chunks > 0 && lens == nullptr))
    return PIC_ERR_INVALID;
  if (layout != PIC_LAYOUT_SPLICED && layout != PIC_LAYOUT_FRAMED) return PIC_ERR_INVALID;
  int64_t T = 0, rows = 0, link = 0, rot = 0, fresh = 0, cpages = 0;
  for (int32_t c = 0; c < n_chunks; ++c) {
    const int64_t L = lens[c];
    if (L < 1) return PIC_ERR_INVALID;
    const int64_t m = (c == 0) ? 0 : (L < k ? L : (int64_t)k);  // recomputed head rows
    const int64_t np = cdiv(L, PIC_PAGE);
    const int64_t kept = (m == L) ? 0 : np - m / PIC_PAGE;      // cached pages keeping a slot
    cpages += np;
    rows += m;
    fresh += cdiv(m, PIC_PAGE);
    const int64_t run = cdiv(m, PIC_PAGE) + kept;  // the chunk's link pages
    link += (layout == PIC_LAYOUT_FRAMED) ? cdiv(run, PIC_TILE_PAGES) * PIC_TILE_PAGES : run;
    if (c > 0) rot += kept;
    T += L;
  }
  const int64_t qp = cdiv(q, PIC_PAGE);
  out->tokens = T + q;
  out->rows = rows + q;
  out->link_pages = link + qp;
  out->rot_pages = rot;
  out->fresh_pages = fresh + qp;
  out->chunk_pages = cpages;
  if (out->tokens > INT32_MAX) return PIC_ERR_INVALID;  // positions are int32
  return PIC_OK;
}

int64_t pic_count_rows(const int32_t* lens, int32_t n_chunks, int32_t q, int32_t k) {
  pic_request_sizes s;
  if (pic_request_sizes_of(lens, n_chunks, q, k, PIC_LAYOUT_SPLICED, &s) != PIC_OK) return -1;
  return s.rows;
}

pic_status pic_plan_offsets(const int32_t* lens, const int32_t* chunk_off, const int32_t* q_len,
                            const int32_t* k, int32_t n_req, pic_layout layout, int32_t* row_off, int32_t* page_off,
                            int32_t* rot_off, int32_t* fresh_off, int32_t* chunk_page_off) {
  if (n_req < 0 || (n_req > 0 && (chunk_off == nullptr || q_len == nullptr || k == nullptr)))
    return PIC_ERR_INVALID;
  if (n_req > 0 && chunk_off[0] != 0) return PIC_ERR_INVALID;
  int64_t acc[4] = {0, 0, 0, 0};
  int64_t cp = 0;
  if (row_off) row_off[0] = 0;
  if (page_off) page_off[0] = 0;
  if (rot_off) rot_off[0] = 0;
  if (fresh_off) fresh_off[0] = 0;
  if (chunk_page_off) chunk_page_off[0] = 0;
  for (int32_t r = 0; r < n_req; ++r) {
    const int32_t c0 = chunk_off[r], c1 = chunk_off[r + 1];
    if (c1 < c0 || (c1 > c0 && lens == nullptr)) return PIC_ERR_INVALID;
    pic_request_sizes s;
    if (pic_request_sizes_of(lens + c0, c1 - c0, q_len[r], k[r], layout, &s) != PIC_OK) return PIC_ERR_INVALID;
    acc[0] += s.rows;
    acc[1] += s.link_pages;
    acc[2] += s.rot_pages;
    acc[3] += s.fresh_pages;
    for (int i = 0; i < 4; ++i)
      if (acc[i] > INT32_MAX) return PIC_ERR_INVALID;
    if (row_off) row_off[r + 1] = (int32_t)acc[0];
    if (page_off) page_off[r + 1] = (int32_t)acc[1];
    if (rot_off) rot_off[r + 1] = (int32_t)acc[2];
    if (fresh_off) fresh_off[r + 1] = (int32_t)acc[3];
    for (int32_t c = c0; c < c1; ++c) {
      cp += cdiv(lens[c], PIC_PAGE);
      if (cp > INT32_MAX) return PIC_ERR_INVALID;
      if (chunk_page_off) chunk_page_off[c + 1] = (int32_t)cp;
    }
  }
  return PIC_OK;
}

const char* pic_strerror(pic_status s) {
  switch (s) {
    case PIC_OK: return "ok";
    case PIC_ERR_INVALID: return "invalid argument or metadata";
    case PIC_ERR_CUDA: return "CUDA call failed";
    case PIC_ERR_UNSUPPORTED: return "unsupported dtype / head dim / GQA group";
    case PIC_ERR_TIMEOUT: return "bounded device wait ran out";
    case PIC_ERR_RANGE: return "block id, slot or count out of range";
    case PIC_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

}  // extern "C"
