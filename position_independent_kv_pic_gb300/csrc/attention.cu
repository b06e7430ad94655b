// Recompute-row link attention on the tensor cores (EPIC blog review,
// link_legolink Step 3: the recomputed rows' Q, roped at their global positions,
// attend over the whole spliced K/V under the causal mask key_pos <= query_pos
// of the KV-cache blog's mask section; scale 1/sqrt(d); a GQA group of
// g = Hq/Hkv query heads shares one KV head).
//
// bf16, d = 128.  One MMA tile is M = 128 rows = g query heads x (128/g)
// recomputed rows of one KV head.  A persistent CTA (one per SM, 640 threads)
// works on a pair of such Q tiles and streams the key tiles (128 keys = 8 pages
// of 16) of one unit through a ring of five 32 KB shared-memory slots (K and V
// tiles alternate), filled by TMA straight from the paged pool, one 4 KB box per
// page.  Per key tile and Q tile i:
//   S_i = Q_i K^T   (tcgen05, fp32 accumulators in TMEM)
//   softmax: S_i -> registers, online softmax in base 2 with lazy rescaling,
//     P_i (bf16) written back over S_i in TMEM
//   O_i += P_i V    (tcgen05 with A from TMEM)
// While Q tile 0's softmax runs the tensor core computes S_1 / P_1 V, and the
// other way round.  Roles: warp 0 issues TMA (K/V pages, Q operands); warp 1
// lane 0 issues the MMAs and warp 1 owns TMEM (S0 | S1 | O0 | O1, 512 columns);
// warps 2-3 wait for each key tile's loads, zero V rows outside a page's valid
// slots (and rotate K in the rotate-on-read instantiation), and release the tile
// to the issuer; warps 4-19 are four softmax warpgroups, one per (Q tile, half of
// the 128 key columns), the two halves of a row exchanging their partial maxima
// through shared memory at a named barrier once per key tile.
//
// Work is cut into units (Q-tile pair, KV head, span of key tiles).  Pairs whose
// key range is longer than the span are split; their partial (O, m, l) are merged
// by the LSE merge kernel.  The planner lists full spans first and tails by
// decreasing length (the LPT greedy rule HYPIC uses to balance segment work);
// CTAs draw units from a global counter while they run.  Key tiles past a pair's
// last row position are never visited (offset-causal tile skipping); keys inside
// boundary tiles are masked per row.  Every mbarrier wait is bounded; a wait that
// runs out sets PIC_ERR_TIMEOUT and the CTA's roles leave together (copies in
// flight drained, TMEM freed).
#include <cudaTypedefs.h>

#include <mutex>

#include "pic_internal.cuh"
#include "tc_ptx.cuh"

namespace pic {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kD = 128;                 // head dim of the tensor-core path
constexpr int kM = 128;                 // rows of one MMA tile
constexpr int kQTiles = 2;              // MMA tiles per CTA
constexpr int kKeys = 128;              // keys per key tile
constexpr int kPagesPerKt = kKeys / PIC_PAGE;
constexpr int kSlots = 5;               // K/V ring slots (32 KB each)
constexpr int kSmWarpgroups = 2 * kQTiles;  // softmax: one warpgroup per (Q tile, half of the key columns)
constexpr int kThreads = 128 * (1 + kSmWarpgroups);
constexpr int kMinSpan = 4;             // key tiles per unit, lower bound
constexpr int kSpanPref = 16;           // ... and while every SM still gets a unit
constexpr int kUnitsPerSm = 7;          // target units per SM when splitting (the cap below binds at 152 SMs)
constexpr int kMaxSplitUnits = 960;     // bound on the units splitting may add
constexpr int kAllSms = 1 << 20;         // split budget: every SM of the device
constexpr int kTailDiv = 3;             // a call with few (tile pair, head) items cuts its tails in 3
constexpr int kTailExtra = 640;         // room for those extra tail pieces (2 per item, < 2 * 160 items)
constexpr int kMaxPlanReqs = 1024;      // requests one planning block handles
constexpr int kMaxPlanTiles = 1024;     // Q-tile pairs planned from shared memory (more: slower path)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may grow up to 2^8 before O is rescaled

constexpr int kHalfBytes = kM * 128;      // one 64-column half of a 128-row operand (16 KB)
constexpr int kOpBytes = 2 * kHalfBytes;  // 128 x 128 bf16 operand (32 KB)
// A K / V slot holds the 8 pages of a key tile, page j at j * kPageBytes, each
// page as [row group g (2)][column half h (2)][8 rows][128 B] with the 128-byte
// swizzle: one TMA box per page.  Rows (keys) 8g' apart then sit kGroupBytes
// apart throughout the tile, so the tile is a K-major operand with an 8-row
// stride of kGroupBytes and each 16-key page is one MN-major k-step.
constexpr int kPageBytes = PIC_PAGE * kD * 2;  // 4 KB
constexpr int kGroupBytes = kPageBytes / 2;    // 8 rows x 2 halves
constexpr int kPageHalfBytes = 1024;           // 8 rows x 64 columns
constexpr int kOffQ = 0;                  // Q tiles 0 and 1
constexpr int kOffSlot = kQTiles * kOpBytes;
constexpr int kOffBar = kOffSlot + kSlots * kOpBytes;
constexpr int kOffXch = kOffBar + 512;  // partial row maxima / sums of the two halves of each Q tile
constexpr int kSmemBytes = kOffXch + kQTiles * 2 * kM * (int)sizeof(float);
static_assert(kSmemBytes <= 232448, "shared memory per block");
constexpr uint32_t kTmemCols = 512;                // S0 | S1 | O0 | O1
constexpr uint32_t kTmemO = 256;
// Register split: the block launches with 640 x 96 registers; warpgroup 0 (TMA
// producer, MMA issuer, V zeroing) gives 32 per thread back, the four softmax
// warpgroups take 8 more each:  4*32*(96-64) == 16*32*(104-96).
constexpr int kLaunchRegs = 96;
constexpr uint32_t kRegsLow = 64, kRegsHigh = 104;
static_assert(4 * 32 * (kLaunchRegs - (int)kRegsLow) == 16 * 32 * ((int)kRegsHigh - kLaunchRegs), "register split");
static_assert(kThreads * kLaunchRegs <= 65536, "register file");

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kM, kKeys, false);
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kM, kD, true);

struct TileMeta {
  int32_t row0, n_rows, page_begin, n_pages;  // rows [row0, row0+n_rows) (<= 2R); pages needed (causal)
  int32_t n_kt, n_spans, part_base, req;      // key tiles; spans per head; partial slots (-1: none)
};
struct Unit {
  int32_t tile, head, kt0, kt1, part, pad0, pad1, pad2;
};
struct WsHeader {
  int32_t n_tiles, n_units, span, total_kt;
  int32_t next_unit;  // run-time unit counter of the attention kernel (zeroed by the planner)
  int32_t pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header size");

struct WsLayout {
  int64_t tiles_cap, units_cap, tail_extra;
  size_t off_tiles, off_units, off_ml, off_o, off_q, total;
};

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace for up to `extra_units` units beyond one per (Q-tile pair, KV head), and
// `tail_extra` more for tails cut into pieces.
WsLayout ws_layout_with(int64_t n_rows, int32_t n_req, int32_t G, int32_t Hkv, int32_t d, int64_t extra_units,
                        int64_t tail_extra) {
  WsLayout L;
  const int R2 = kQTiles * (kM / G);
  L.tiles_cap = n_rows / R2 + n_req + 1;
  L.units_cap = L.tiles_cap * Hkv + extra_units + tail_extra;
  L.tail_extra = tail_extra;
  L.off_tiles = sizeof(WsHeader);
  L.off_units = al256(L.off_tiles + L.tiles_cap * sizeof(TileMeta));
  L.off_ml = al256(L.off_units + L.units_cap * sizeof(Unit));
  L.off_o = al256(L.off_ml + (size_t)L.units_cap * kQTiles * kM * sizeof(float2));
  L.off_q = al256(L.off_o + (size_t)L.units_cap * kQTiles * kM * d * sizeof(float));
  // roped Q of every (Q-tile pair, KV head, Q tile), in the MMA's swizzled layout
  L.total = al256(L.off_q + (size_t)L.tiles_cap * Hkv * kQTiles * kOpBytes);
  return L;
}

WsLayout ws_layout(int64_t n_rows, int32_t n_req, int32_t G, int32_t Hkv, int32_t d) {
  return ws_layout_with(n_rows, n_req, G, Hkv, d, kMaxSplitUnits, kTailExtra);
}

__device__ __forceinline__ bool page_ok(int4 p, int64_t num_blocks) {
  const int lo = (int16_t)(p.w & 0xffff), hi = (int16_t)(p.w >> 16);
  return p.x >= 0 && p.x < num_blocks && p.y >= 0 && p.y < num_blocks && lo >= 0 && hi <= PIC_PAGE && lo < hi;
}

// ------------------------------------------------------------------ planning
// One block.  (1) Q-tile pairs per request and their causal page counts (pages
// are sorted by first valid position: binary search for the last row's
// position).  (2) The span: enough key tiles per unit that at most
// min(kUnitsPerSm * SMs, max_split) extra units appear.  (3) Units: the
// full-length spans first, ordered (request, KV head, span index, tile) so that
// concurrently running units read the same key range, then the shorter tail
// spans by decreasing length.
constexpr int kPlanThreads = 1024;
constexpr int kHist = 2048;

// The tile pairs: each request's rows in pairs of R2 rows, the partial pair (if
// any) first.  s_toff[r] = first tile of request r; returns the number of tiles.
// Block-wide (kPlanThreads threads).
__device__ int plan_tile_offsets(const int32_t* __restrict__ row_off, int n_req, int R2, int* s_toff, int* s_scan) {
  const int tid = threadIdx.x;
  int carry = 0;
  for (int g = 0; g < n_req; g += kPlanThreads) {
    const int r = g + tid;
    const int nt = (r < n_req) ? ceil_div(row_off[r + 1] - row_off[r], R2) : 0;
    int tot;
    const int ex = block_exclusive_scan<kPlanThreads>(nt, s_scan, &tot);
    if (r < n_req) s_toff[r] = carry + ex;
    carry += tot;
  }
  if (tid == 0) s_toff[n_req] = carry;
  __syncthreads();
  return s_toff[n_req];
}
// Request, first row and rows of tile t: the partial pair first, since its rows
// have the smallest positions, so a half-empty tile pair (one Q tile, the MMA
// ping-pong idle) spans the fewest key tiles.
__device__ __forceinline__ void plan_tile_rows(const int32_t* __restrict__ row_off, const int* s_toff, int n_req,
                                               int R2, int t, TileMeta& tm) {
  int lo = 0, hi = n_req;  // request: last r with s_toff[r] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_toff[mid] <= t) lo = mid; else hi = mid;
  }
  const int r = lo;
  tm.req = r;
  const int nr = row_off[r + 1] - row_off[r], rem = nr % R2, k = t - s_toff[r];
  tm.row0 = row_off[r] + (rem > 0 ? (k == 0 ? 0 : rem + (k - 1) * R2) : k * R2);
  tm.n_rows = (rem > 0 && k == 0) ? rem : R2;
}

__device__ __forceinline__ int plan_tile_req(const int* s_toff, int n_req, int t) {
  int lo = 0, hi = n_req;  // last r with s_toff[r] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_toff[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// One block: the tile pairs' rows alone (the first part of the unit plan), so that
// the Q operands can be written before the page list exists.  Writes only the row
// fields of each tile; the unit plan writes the same values and the rest.
__global__ void __launch_bounds__(kPlanThreads)
tile_rows_kernel(const int32_t* __restrict__ row_off, int n_req, int R2, int64_t tiles_cap, WsHeader* hdr,
                 TileMeta* tiles, int32_t* err) {
  __shared__ int s_toff[kMaxPlanReqs + 1];
  __shared__ int s_scan[kPlanThreads / 32 + 1];
  const int n_tiles = plan_tile_offsets(row_off, n_req, R2, s_toff, s_scan);
  if (n_tiles > tiles_cap) {
    if (threadIdx.x == 0) {
      set_err(err, PIC_ERR_RANGE);
      hdr->n_tiles = 0;
    }
    return;
  }
  for (int t = threadIdx.x; t < n_tiles; t += kPlanThreads) {
    TileMeta tm;
    plan_tile_rows(row_off, s_toff, n_req, R2, t, tm);
    tiles[t].req = tm.req;
    tiles[t].row0 = tm.row0;
    tiles[t].n_rows = tm.n_rows;
  }
  if (threadIdx.x == 0) hdr->n_tiles = n_tiles;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_units_kernel(const int32_t* __restrict__ rows, const int32_t* __restrict__ row_off,
                  const pic_link_page* __restrict__ pages, const int32_t* __restrict__ page_off,
                  int n_req, int R2, int Hkv, int num_sms, int max_split, int64_t tiles_cap, int64_t units_cap,
                  int64_t tail_extra, WsHeader* hdr, TileMeta* tiles, Unit* units, int32_t* err) {
  __shared__ int s_toff[kMaxPlanReqs + 1];   // first tile of each request
  __shared__ int s_full[kMaxPlanReqs];       // full spans of one head of each request
  __shared__ int s_fbase[kMaxPlanReqs + 1];  // first full unit of each request
  __shared__ int s_hist[kHist];
  __shared__ int s_scan[kPlanThreads / 32 + 1];
  __shared__ int s_poff[kMaxPlanReqs + 1];   // page offsets of the requests
  __shared__ int s_maxpos[kMaxPlanTiles], s_npages[kMaxPlanTiles], s_nkt[kMaxPlanTiles];
  __shared__ int s_total_kt, s_part;
  const int tid = threadIdx.x;
  // (1) tile offsets over requests
  const int n_tiles = plan_tile_offsets(row_off, n_req, R2, s_toff, s_scan);
  if (tid == 0) {
    s_total_kt = 0;
    s_part = 0;
  }
  for (int r = tid; r < n_req; r += kPlanThreads) s_full[r] = 0;
  for (int i = tid; i < kHist; i += kPlanThreads) s_hist[i] = 0;
  __syncthreads();
  if (n_tiles > tiles_cap) {
    if (tid == 0) {
      set_err(err, PIC_ERR_RANGE);
      hdr->n_units = 0;
      hdr->n_tiles = 0;
      hdr->next_unit = 0;
    }
    return;
  }
  // tiles: rows and last row position; causal page counts from one pass over the pages
  const bool small = n_tiles <= kMaxPlanTiles;
  for (int t = tid; t < n_tiles; t += kPlanThreads) {
    TileMeta tm;
    plan_tile_rows(row_off, s_toff, n_req, R2, t, tm);
    const int r = tm.req;
    const int maxpos = rows[tm.row0 + tm.n_rows - 1];
    tm.page_begin = page_off[r];
    tm.n_pages = 0;
    if (!small) {  // many tiles: binary search per tile
      int a = page_off[r], b = page_off[r + 1];
      while (a < b) {
        const int mid = (a + b) >> 1;
        const pic_link_page p = pages[mid];
        if (p.gpos0 + p.lo <= maxpos) a = mid + 1; else b = mid;
      }
      tm.n_pages = a - page_off[r];
    } else {
      s_maxpos[t] = maxpos;
      s_npages[t] = 0;
    }
    // the row fields (req, row0, n_rows) and the tile count are tile_rows_kernel's:
    // the Q operands are read against them, also while this kernel runs
    TileMeta& out = tiles[t];
    out.page_begin = tm.page_begin;
    out.n_pages = tm.n_pages;
    out.n_kt = 0;
    out.n_spans = 0;
    out.part_base = -1;
  }
  for (int r = tid; r <= n_req; r += kPlanThreads) s_poff[r] = page_off[r];
  __syncthreads();
  if (small) {
    // page p is the last page a tile needs iff first(p) <= maxpos < first(p+1)
    // (pages of a request are sorted by first valid position, tiles by maxpos)
    // four pages per thread and round, their loads issued together, and only the
    // 8 bytes (gpos0, lo | hi) each page's first position needs; the next page's
    // comes from the neighbouring lane (one block reads the whole list, so the bytes
    // it moves set this pass's length on a long list)
    constexpr int kPagesAtOnce = 4;
    const int n_pages_all = s_poff[n_req];
    const int2* pg2 = reinterpret_cast<const int2*>(pages);  // {gpos0, lo | hi << 16} at int2 index 2p + 1
    const int lane = tid & 31;
    for (int p0 = tid; p0 - lane < n_pages_all; p0 += kPagesAtOnce * kPlanThreads) {
      int first[kPagesAtOnce], nextf[kPagesAtOnce];
#pragma unroll
      for (int u = 0; u < kPagesAtOnce; ++u) {
        const int p = p0 + u * kPlanThreads;
        int2 e = make_int2(INT_MAX, 0), en = make_int2(INT_MAX, 0);
        if (p < n_pages_all) e = __ldg(pg2 + 2 * p + 1);
        if (lane == 31 && p + 1 < n_pages_all) en = __ldg(pg2 + 2 * (p + 1) + 1);
        first[u] = e.x == INT_MAX ? INT_MAX : e.x + (int16_t)(e.y & 0xffff);
        const int nb = __shfl_down_sync(0xffffffffu, first[u], 1);
        nextf[u] = lane == 31 ? (en.x == INT_MAX ? INT_MAX : en.x + (int16_t)(en.y & 0xffff)) : nb;
      }
#pragma unroll
      for (int u = 0; u < kPagesAtOnce; ++u) {
        const int p = p0 + u * kPlanThreads;
        if (p >= n_pages_all) break;
        int lo = 0, hi = n_req;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (s_poff[mid] <= p) lo = mid; else hi = mid;
        }
        const int r = lo;
        const int next = (p + 1 < s_poff[r + 1]) ? nextf[u] : INT_MAX;
        int a = s_toff[r], b = s_toff[r + 1];  // first tile with maxpos >= first
        while (a < b) {
          const int mid = (a + b) >> 1;
          if (s_maxpos[mid] < first[u]) a = mid + 1; else b = mid;
        }
        for (int t = a; t < s_toff[r + 1] && s_maxpos[t] < next; ++t) s_npages[t] = p + 1 - s_poff[r];
      }
    }
    __syncthreads();
  }
  for (int t = tid; t < n_tiles; t += kPlanThreads) {
    TileMeta& tm = tiles[t];
    if (small) tm.n_pages = s_npages[t];
    tm.n_kt = ceil_div(tm.n_pages, kPagesPerKt);
    if (small) s_nkt[t] = tm.n_kt;
    atomicAdd(&s_total_kt, tm.n_kt);
  }
  __syncthreads();
  // (2) span
  const int64_t work = (int64_t)s_total_kt * Hkv;
  // six to seven units per SM balance the long calls (long-context call, units in
  // all: 912 -> 897 us, 960 -> 872, 1,000 -> 874, 1,064 -> 900, 1,216 -> 906; fewer
  // left SMs idle at the end, more paid unit overhead and partials); a short
  // call keeps spans of at least 16 tiles as long as every SM still gets a unit,
  // since each unit pays a Q load and a pipeline fill, and a call too short for that
  // spreads over more SMs in spans down to 4 tiles (6-chunk prompt: 46 -> 41 us; 2
  // tiles slowed the 20-chunk call by a tenth)
  const int64_t target = min((int64_t)kUnitsPerSm * num_sms, (int64_t)max_split);
  const int64_t span_fill = min((int64_t)kSpanPref, (work + num_sms - 1) / num_sms);
  const int span = (int)max((int64_t)kMinSpan, max((work + target - 1) / target, span_fill));
  // With few (tile pair, head) items the tails are few and long, and the SMs that
  // draw the last of them finish late: cut each tail into pieces of about a third
  // of a span (long-context call 914 -> 891 us).  Many items already end on many
  // short tails, and more units only add overhead there (16-request batch: slower).
  const int items = n_tiles * Hkv;
  const bool cut = items < 2 * num_sms && (int64_t)(kTailDiv - 1) * items <= tail_extra;
  const int ts = cut ? max(kMinSpan, ceil_div(span, kTailDiv)) : span;  // tail pieces
  for (int t = tid; t < n_tiles; t += kPlanThreads) {
    TileMeta& tm = tiles[t];
    const int len = tm.n_kt % span;
    tm.n_spans = tm.n_kt / span + ceil_div(len, ts);
    if (tm.n_spans > 1) tm.part_base = atomicAdd(&s_part, tm.n_spans * Hkv);
    atomicAdd(&s_full[plan_tile_req(s_toff, n_req, t)], tm.n_kt / span);
    for (int o = 0; o < len; o += ts) atomicAdd(&s_hist[min(min(ts, len - o), kHist - 1)], Hkv);
  }
  __syncthreads();
  // (3) first full unit of every request; tail buckets after all full units, longest first
  int carry = 0;
  for (int g = 0; g < n_req; g += kPlanThreads) {
    const int r = g + tid;
    const int f = (r < n_req) ? s_full[r] * Hkv : 0;
    int tot;
    const int ex = block_exclusive_scan<kPlanThreads>(f, s_scan, &tot);
    if (r < n_req) s_fbase[r] = carry + ex;
    carry += tot;
  }
  const int n_full = carry;
  {  // bucket starts by decreasing length: thread t owns lengths kHist-1-2t and kHist-2-2t
    static_assert(kHist == 2 * kPlanThreads, "two histogram buckets per thread");
    const int l0 = kHist - 1 - 2 * tid, l1 = l0 - 1;
    const int c0 = s_hist[l0], c1 = (l1 >= 1) ? s_hist[l1] : 0;
    int tot;
    const int ex = block_exclusive_scan<kPlanThreads>(c0 + c1, s_scan, &tot);
    s_hist[l0] = n_full + ex;
    if (l1 >= 1) s_hist[l1] = n_full + ex + c0;
    if (tid == 0) s_fbase[n_req] = n_full + tot;  // total units
  }
  __syncthreads();
  const int n_units = s_fbase[n_req];
  if (n_units > units_cap) {
    if (tid == 0) {
      set_err(err, PIC_ERR_RANGE);
      hdr->n_units = 0;
      hdr->n_tiles = 0;
      hdr->next_unit = 0;
    }
    return;
  }
  // full units: index within (request, head) ordered by (span s, tile t).  With the
  // tiles' key-tile counts in shared memory, one thread per (tile, head, span): a
  // thread per (tile, head) writing its spans in turn was the plan's longest chain
  static_assert(kMaxPlanTiles <= kPlanThreads, "one tile per thread in the scan below");
  if (small) {
    int* s_fpre = s_maxpos;  // free again: full units before each tile, over all heads
    int n_full_items;
    const int ex = block_exclusive_scan<kPlanThreads>(tid < n_tiles ? (s_nkt[tid] / span) * Hkv : 0, s_scan,
                                                      &n_full_items);
    if (tid < n_tiles) s_fpre[tid] = ex;
    __syncthreads();
    for (int i = tid; i < n_full_items; i += kPlanThreads) {
      int a = 0, b = n_tiles;  // the last tile with s_fpre[t] <= i (it has units)
      while (b - a > 1) {
        const int mid = (a + b) >> 1;
        if (s_fpre[mid] <= i) a = mid; else b = mid;
      }
      const int t = a, f = s_nkt[t] / span, loc = i - s_fpre[t], h = loc / f, sp = loc % f;
      const int r = plan_tile_req(s_toff, n_req, t), t0 = s_toff[r], t1 = s_toff[r + 1];
      int idx = s_fbase[r] + h * s_full[r];
      for (int t2 = t0; t2 < t1; ++t2) {
        const int f2 = s_nkt[t2] / span;
        idx += min(f2, sp) + ((t2 < t && f2 > sp) ? 1 : 0);
      }
      const int n_spans = tiles[t].n_spans, part_base = tiles[t].part_base;
      Unit un;
      un.tile = t; un.head = h; un.kt0 = sp * span; un.kt1 = (sp + 1) * span;
      un.part = (n_spans > 1) ? part_base + h * n_spans + sp : -1;
      un.pad0 = un.pad1 = un.pad2 = 0;
      units[idx] = un;
    }
  }
  for (int th = tid; th < n_tiles * Hkv; th += kPlanThreads) {
    const int t = th / Hkv, h = th % Hkv;
    // this kernel's fields only (tile_rows_kernel may be writing the others)
    const int n_kt = tiles[t].n_kt, n_spans = tiles[t].n_spans, part_base = tiles[t].part_base;
    const int r = plan_tile_req(s_toff, n_req, t), t0 = s_toff[r], t1 = s_toff[r + 1];
    const int f = n_kt / span;
    for (int s = 0; !small && s < f; ++s) {
      int idx = s_fbase[r] + h * s_full[r];
      for (int t2 = t0; t2 < t1; ++t2) {
        const int f2 = (small ? s_nkt[t2] : tiles[t2].n_kt) / span;
        idx += min(f2, s) + ((t2 < t && f2 > s) ? 1 : 0);
      }
      Unit un;
      un.tile = t; un.head = h; un.kt0 = s * span; un.kt1 = (s + 1) * span;
      un.part = (n_spans > 1) ? part_base + h * n_spans + s : -1;
      un.pad0 = un.pad1 = un.pad2 = 0;
      units[idx] = un;
    }
    const int len = n_kt % span;
    for (int o = 0, j = 0; o < len; o += ts, ++j) {  // the tail, in pieces of at most ts tiles
      const int pl = min(ts, len - o);
      const int idx = atomicAdd(&s_hist[min(pl, kHist - 1)], 1);
      Unit un;
      un.tile = t; un.head = h; un.kt0 = f * span + o; un.kt1 = f * span + o + pl;
      un.part = (n_spans > 1) ? part_base + h * n_spans + f + j : -1;
      un.pad0 = un.pad1 = un.pad2 = 0;
      units[idx] = un;
    }
  }
  if (tid == 0) {
    hdr->n_units = n_units;
    hdr->span = span;
    hdr->next_unit = 0;
    hdr->total_kt = s_total_kt;
  }
}

// ------------------------------------------------------------------ tcgen05 kernel
struct TcArgs {
  const uint8_t* q_tiles;  // [tile][kvh][qt] 32 KB swizzled Q operands
  const bf16* q;
  const float4* row_table;
  const int32_t* rows;
  const pic_link_page* pages;
  bf16* out;
  const WsHeader* hdr;
  int32_t* next_unit;  // &hdr->next_unit
  const TileMeta* tiles;
  const Unit* units;
  float* part_o;
  float2* part_ml;
  int32_t* err;
  int64_t num_blocks;
  int Hq, Hkv, G, R;
  float scale_log2;
  // rotate-on-read (page_tab != nullptr): the keys of page p sit in the frame of
  // offset-table row page_tab[p] (the global frame when negative); all pages of a
  // key tile share one frame (the framed layout), and Q is rotated into it
  const int32_t* page_tab;
  const float4* rot_tab;  // [n_tab][kD / 2] {cos_hi, sin_hi, cos_lo, sin_lo}
  int64_t n_tab;
};

constexpr int kUnitRing = 2;                  // unit indices in flight from the producer
// Slot frees: the MMA issuer commits once per step (a unit's start, then each key
// tile) to kv_step[step % kStepRing]; a step frees the slots its products last read
// (the start the unit's first K, step j V_j and K_(j+1)).  Before load L the producer
// waits for the step that freed load L - kSlots; a later step can complete first only
// if all the loads it reads precede L, i.e. lie among the kSlots loads before it:
// at most three key tiles' worth, each read by at most two steps (a unit's start and
// its first step), so at most five steps run ahead and eight barriers keep every
// awaited phase's parity unambiguous.
constexpr int kStepRing = 8;
constexpr int kUnitReaders = 1 + 2 + 4 * kSmWarpgroups;  // MMA thread, 2 V-zeroing warps, softmax warps

struct Bars {
  uint64_t kv_full[kSlots], kv_step[kStepRing];
  // key tile t (t % kSlots) ready for the MMAs: its K and V landed, K rotated to its
  // global positions when rotating on read, V's invalid rows zeroed
  uint64_t vz_done[kSlots];
  uint64_t q_full[kQTiles], q_free[kQTiles], s_full[kQTiles], p_full[kQTiles], o_done[kQTiles], drain;
  // rotate-on-read: Q tile i written in shared memory for the frame of its next key
  // tiles by its two softmax warpgroups (the MMA issuer waits for it at frame changes)
  uint64_t q_ready[kQTiles];
  uint64_t unit_full[kUnitRing], unit_empty[kUnitRing];
  uint64_t never;  // no thread ever arrives on it (the failure-injection test build waits on it)
  int unit_idx[kUnitRing];
  uint32_t free_step[kSlots];  // producer lane 0 only: the step that frees each slot's load
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier area");

__device__ __forceinline__ uint32_t sw128_off(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void fail(Bars* b, int32_t* err) {
  set_err(err, PIC_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&b->abort) = 1;
}

__device__ __forceinline__ bool wait_bar(Bars* b, uint64_t* bar, uint32_t parity) {
  return tc::mbar_wait(bar, parity, &b->abort, kWaitLimitNs);
}

// ---------------------------------------------------------------- unit schedule
// Units are handed out while the kernel runs: a CTA starts with unit blockIdx.x and
// then draws the next one from a global counter, so CTAs whose units were short take
// more of them (the planner lists long units first).  The producer warp draws; a
// two-entry ring in shared memory passes every index, and finally an index >=
// n_units that ends the loops, to the other warps in the same order.
__device__ __forceinline__ bool publish_unit(Bars* b, uint32_t k, int u) {  // producer lane 0
  const int s = k % kUnitRing;
  if (!wait_bar(b, &b->unit_empty[s], ((k / kUnitRing) & 1) ^ 1)) return false;
  *reinterpret_cast<volatile int*>(&b->unit_idx[s]) = u;
  tc::mbar_arrive(&b->unit_full[s]);
  return true;
}

// The k-th unit of this CTA (one thread per reading warp); -1 if the wait gave up.
__device__ __forceinline__ int read_unit(Bars* b, uint32_t k) {
  const int s = k % kUnitRing;
  if (!wait_bar(b, &b->unit_full[s], (k / kUnitRing) & 1)) return -1;
  const int u = *reinterpret_cast<volatile int*>(&b->unit_idx[s]);
  tc::mbar_arrive(&b->unit_empty[s]);
  return u;
}

// Warp-wide read_unit: lane 0 reads, every lane gets the index.
__device__ __forceinline__ int read_unit_warp(Bars* b, uint32_t k) {
  int u = 0;
  if ((threadIdx.x & 31) == 0) u = read_unit(b, k);
  return __shfl_sync(0xffffffffu, u, 0);
}

// ---------------------------------------------------------------- producer
__device__ __forceinline__ int4 load_page(const pic_link_page* pages, int p, int page_end) {
  if (p < page_end) return __ldg(reinterpret_cast<const int4*>(pages) + p);
  return make_int4(-1, -1, 0, 0);
}

// Rotate-on-read: the frame (offset-table row, -1 = global) of key tile kt of the
// tile pair, read from the tile's first page.  The MMA issuer and the softmax warps
// both derive the frame changes from it, so they agree on them.
__device__ __forceinline__ int tile_frame(const TcArgs& a, const TileMeta& tm, int kt) {
  const int f = __ldg(a.page_tab + tm.page_begin + kt * kPagesPerKt);
  if (f >= a.n_tab) {  // a row past the offset table: flagged, read in the global frame
    set_err(a.err, PIC_ERR_RANGE);
    return -1;
  }
  return f < 0 ? -1 : f;
}

// The whole warp: lane j < 8 owns page j of the key tile (its entry is loaded a
// tile ahead) and issues that page's boxes, so page lookups and box issue run in
// parallel across lanes.  Lane 0 arms each slot's barrier first.
template <bool kRor>
__device__ void producer_loop(const TcArgs& a, const CUtensorMap* kmap, const CUtensorMap* vmap,
                              uint8_t* smem, Bars* b, int n_units) {
  const int lane = threadIdx.x & 31;
  uint32_t ld = 0, uq[kQTiles] = {0, 0};
  // the issuer's step numbering: a unit's start, then one step per key tile; the
  // start frees the unit's first K, step j frees V_j and K_(j+1)
  uint32_t s0 = 0;
  int u = blockIdx.x;
  for (uint32_t k = 0;; ++k) {
    int go = 1;
    if (lane == 0) {
      go = publish_unit(b, k, u < n_units ? u : n_units);
      if (!go) fail(b, a.err);
    }
    if (!__shfl_sync(0xffffffffu, go, 0) || u >= n_units) break;
    // the next unit is drawn now, so the atomic's latency hides behind this unit's loads
    int u_next = 0;
    if (lane == 0) u_next = atomicAdd(a.next_unit, 1) + (int)gridDim.x;
    const Unit un = a.units[u];
    const TileMeta tm = a.tiles[un.tile];
    const int page_end = tm.page_begin + tm.n_pages;
    const int pbase = tm.page_begin + un.kt0 * kPagesPerKt;
    // Q operands of this unit, once the previous unit's last S products have read the buffers
    // (rotating on read, the softmax warps write Q into the buffers themselves)
    if (!kRor && lane == 0) {
      for (int i = 0; i < kQTiles; ++i) {
        if (i == 1 && tm.n_rows <= a.R) break;
        if (!wait_bar(b, &b->q_free[i], (uq[i] & 1) ^ 1)) {
          fail(b, a.err);
          go = 0;
          break;
        }
        ++uq[i];
        tc::mbar_arrive_expect_tx(&b->q_full[i], kOpBytes);
        tc::bulk_load(smem + kOffQ + i * kOpBytes,
                      a.q_tiles + (((int64_t)un.tile * a.Hkv + un.head) * kQTiles + i) * kOpBytes, kOpBytes,
                      &b->q_full[i]);
      }
    }
    if (!__shfl_sync(0xffffffffu, go, 0)) goto drain;
    {
      int4 nxt = load_page(a.pages, lane < kPagesPerKt ? pbase + lane : page_end, page_end);
      for (int kt = un.kt0; kt < un.kt1; ++kt) {
        const int4 pg = nxt;
        if (kt + 1 < un.kt1 && lane < kPagesPerKt)
          nxt = load_page(a.pages, pbase + (kt + 1 - un.kt0) * kPagesPerKt + lane, page_end);
        const bool ok = lane < kPagesPerKt && page_ok(pg, a.num_blocks);
        if (lane < kPagesPerKt && !ok && (int16_t)(pg.w & 0xffff) < (int16_t)(pg.w >> 16))
          set_err(a.err, PIC_ERR_RANGE);
        const uint32_t n_ok = __popc(__ballot_sync(0xffffffffu, ok));
        const uint32_t bytes = n_ok * kPageBytes;  // one box per page
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          const int slot = ld % kSlots;
          if (lane == 0) {
            if (ld >= (uint32_t)kSlots) {
              const uint32_t fs = b->free_step[slot];
              go = wait_bar(b, &b->kv_step[fs % kStepRing], (fs / kStepRing) & 1);
            }
            if (!go) {
              fail(b, a.err);
            } else {
              b->free_step[slot] = s0 + (uint32_t)(kt - un.kt0) + (uint32_t)kv;
              tc::mbar_arrive_expect_tx(&b->kv_full[slot], bytes);
            }
          }
          // a slot is armed only when all its boxes are issued right after
          if (!__shfl_sync(0xffffffffu, go, 0)) goto drain;
          if (ok) {
            uint8_t* dst = smem + kOffSlot + slot * kOpBytes;
            const CUtensorMap* map = kv ? vmap : kmap;
            const int grp = ((kv ? pg.y : pg.x) * a.Hkv + un.head) * (PIC_PAGE / 8);
            tc::tma_load_4d(dst + lane * kPageBytes, map, 0, 0, 0, grp, &b->kv_full[slot]);
          }
          ++ld;
        }
      }
    }
    s0 += (uint32_t)(un.kt1 - un.kt0) + 1u;
    u = __shfl_sync(0xffffffffu, u_next, 0);
  }
drain:
  // no copy may be in flight when the block exits, also after an abort: bounded
  // waits that do not stop at the abort flag, on the last arming of every slot
  if (lane == 0) {
    const int no_abort = 0;
    for (uint32_t k = 0; k < kSlots && k < ld; ++k) {
      const uint32_t t = ld - 1 - k;
      tc::mbar_wait(&b->kv_full[t % kSlots], (t / kSlots) & 1, &no_abort, kWaitLimitNs);
    }
    for (int i = 0; i < kQTiles; ++i)
      if (uq[i] > 0) tc::mbar_wait(&b->q_full[i], (uq[i] - 1) & 1, &no_abort, kWaitLimitNs);
  }
}

// ---------------------------------------------------------------- MMA issuer
template <bool kRor>
__device__ void mma_loop(const TcArgs& a, uint8_t* smem, Bars* b, uint32_t tmem, int n_units) {
  // descriptor words: hi is constant, lo = start address (>> 4) plus the LBO field
  constexpr uint32_t kHi = tc::sw128_desc_hi(1024), kHiKV = tc::sw128_desc_hi(kGroupBytes);
  const uint32_t q_lo = tc::sw128_desc_lo(tc::smem_addr(smem + kOffQ), 16);
  const uint32_t k_lo = tc::sw128_desc_lo(tc::smem_addr(smem + kOffSlot), 16);
  const uint32_t v_lo = tc::sw128_desc_lo(tc::smem_addr(smem + kOffSlot), kPageHalfBytes);
  uint32_t ld = 0, uq[kQTiles] = {0, 0}, c[kQTiles] = {0, 0}, st = 0;
  // Key tile t: its K and V landed (the V-zeroing warps waited for both loads),
  // K rotated when rotating on read, V's invalid rows zeroed.  The issuer waits for
  // this one barrier per tile, before the tile's first S product, and never for the
  // loads themselves: every wait costs issue time between MMA groups, when the
  // tensor pipe runs dry.
  auto wait_tile = [&](uint32_t t) -> bool {
    return wait_bar(b, &b->vz_done[t % kSlots], (t / kSlots) & 1);
  };
  auto issue_s = [&](int i, int slot) {
    const uint32_t qa = q_lo + i * (kOpBytes >> 4), kb = k_lo + slot * (kOpBytes >> 4);
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
      const uint32_t qoff = ((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
      const uint32_t koff = ((ks >> 2) * kPageHalfBytes + (ks & 3) * 32) >> 4;
      tc::mma_bf16_ss(tmem + i * 128, tc::desc_join(qa + qoff, kHi), tc::desc_join(kb + koff, kHiKV), kIdescS,
                      ks > 0 ? 1u : 0u);
    }
  };
  auto issue_pv = [&](int i, int slot, bool acc) {
    const uint32_t vb = v_lo + slot * (kOpBytes >> 4);
#pragma unroll
    for (int ks = 0; ks < kKeys / 16; ++ks)
      tc::mma_bf16_ts(tmem + kTmemO + i * 128, tmem + i * 128 + ks * 8,
                      tc::desc_join(vb + ks * (kPageBytes >> 4), kHiKV), kIdescPV, (acc || ks > 0) ? 1u : 0u);
  };
#ifdef PIC_INJECT_WAIT_TIMEOUT
  // Failure-injection test build only: a bounded wait on a barrier that nothing
  // arrives on runs out, reports PIC_ERR_TIMEOUT and must bring every role of the
  // CTA to a clean exit (copies drained, TMEM freed).
  if (!tc::mbar_wait(&b->never, 0, &b->abort, PIC_INJECT_WAIT_TIMEOUT)) { fail(b, a.err); return; }
#endif
  for (uint32_t k = 0;; ++k) {
    const int u = read_unit(b, k);
    if (u < 0) { fail(b, a.err); return; }
    if (u >= n_units) break;
    const Unit un = a.units[u];
    const TileMeta tm = a.tiles[un.tile];
    const int n = un.kt1 - un.kt0;
    const bool act1 = tm.n_rows > a.R;
    // Q tile i in shared memory: loaded by the producer, or (rotating on read) written
    // for the frame of the unit's first key tile by its softmax warps
    // frames of key tiles j and j + 1, read a tile ahead
    int f_cur = 0, f_nxt = 0;
    if (kRor) {
      f_cur = tile_frame(a, tm, un.kt0);
      f_nxt = n > 1 ? tile_frame(a, tm, un.kt0 + 1) : f_cur;
    }
    uint64_t* const q_in = kRor ? b->q_ready : b->q_full;
    {  // S for the first key tile, each Q tile's as soon as its Q is in shared memory
      const int ks = ld % kSlots;
      if (!wait_bar(b, &q_in[0], uq[0] & 1)) { fail(b, a.err); return; }
      ++uq[0];
      if (!wait_tile(ld / 2)) { fail(b, a.err); return; }
      tc::tc_fence_after();
      issue_s(0, ks);
      tc::mma_commit(&b->s_full[0]);
      if (!kRor && n == 1) tc::mma_commit(&b->q_free[0]);
      if (act1) {
        if (!wait_bar(b, &q_in[1], uq[1] & 1)) { fail(b, a.err); return; }
        ++uq[1];
        tc::tc_fence_after();
        issue_s(1, ks);
        tc::mma_commit(&b->s_full[1]);
        if (!kRor && n == 1) tc::mma_commit(&b->q_free[1]);
      }
      tc::mma_commit(&b->kv_step[st++ % kStepRing]);  // frees the first K
    }
    for (int j = 0; j < n; ++j, ld += 2) {
      const uint32_t vld = ld + 1, nld = ld + 2;
      const int vs = vld % kSlots, ns = nld % kSlots;
      const bool more = j + 1 < n;
      // rotating on read, key tile j + 1 in another frame than tile j needs Q rotated
      // into it: its softmax warps do that once they have written P of tile j
      const bool new_frame = kRor && more && f_nxt != f_cur;
      if (!new_frame) {
#pragma unroll
        for (int i = 0; i < kQTiles; ++i) {
          if (i == 1 && !act1) break;
          if (!wait_bar(b, &b->p_full[i], c[i] & 1)) { fail(b, a.err); return; }
          ++c[i];
          tc::tc_fence_after();
          issue_pv(i, vs, j > 0);
          if (more) {
            if (i == 0 && !wait_tile(nld / 2)) { fail(b, a.err); return; }
            tc::tc_fence_after();
            issue_s(i, ns);
            tc::mma_commit(&b->s_full[i]);
            if (!kRor && j + 2 == n) tc::mma_commit(&b->q_free[i]);  // the unit's last S product of Q tile i
          } else {
            tc::mma_commit(&b->o_done[i]);
          }
        }
      } else {
        // a frame change: both P.V products first, so that the pipe has work while the
        // softmax warps rotate Q into the new frame, then each Q tile's next S product
        // once its Q is written (waiting for Q tile 0's before issuing Q tile 1's P.V
        // left the pipe idle: rotate-on-read call 1.358 -> 1.244 ms)
#pragma unroll
        for (int i = 0; i < kQTiles; ++i) {
          if (i == 1 && !act1) break;
          if (!wait_bar(b, &b->p_full[i], c[i] & 1)) { fail(b, a.err); return; }
          ++c[i];
          tc::tc_fence_after();
          issue_pv(i, vs, j > 0);
        }
        if (!wait_tile(nld / 2)) { fail(b, a.err); return; }
#pragma unroll
        for (int i = 0; i < kQTiles; ++i) {
          if (i == 1 && !act1) break;
          if (!wait_bar(b, &b->q_ready[i], uq[i] & 1)) { fail(b, a.err); return; }
          ++uq[i];
          tc::tc_fence_after();
          issue_s(i, ns);
          tc::mma_commit(&b->s_full[i]);
        }
      }
      tc::mma_commit(&b->kv_step[st++ % kStepRing]);  // frees V_j and K_(j+1)
      if (kRor) {
        f_cur = f_nxt;
        if (j + 2 < n) f_nxt = tile_frame(a, tm, un.kt0 + j + 2);
      }
    }
  }
}

// Q row m, 16-byte chunks cc0 and cc0 + 1 of both 64-column halves: RoPE at the
// row's position, rounded to bf16, stored swizzled.
__device__ __forceinline__ void write_q_row(uint8_t* qs, int m, bool ok, const bf16* __restrict__ src,
                                            const float4* __restrict__ tab, int cc0) {
#pragma unroll
  for (int cc = cc0; cc < cc0 + 2; ++cc) {
    uint4 lo4 = make_uint4(0, 0, 0, 0), hi4 = make_uint4(0, 0, 0, 0);
    if (ok) {
      const uint4 xl = __ldg(reinterpret_cast<const uint4*>(src + 8 * cc));
      const uint4 xh = __ldg(reinterpret_cast<const uint4*>(src + 64 + 8 * cc));
      const __nv_bfloat162* l2 = reinterpret_cast<const __nv_bfloat162*>(&xl);
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&xh);
      uint32_t* lo_w = reinterpret_cast<uint32_t*>(&lo4);
      uint32_t* hi_w = reinterpret_cast<uint32_t*>(&hi4);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(l2[e]);
        const float2 y = __bfloat1622float2(h2[e]);
        float y0, z0, y1, z1;
        rope_rotate_bf16in(x.x, y.x, __ldg(tab + 8 * cc + 2 * e), y0, z0);
        rope_rotate_bf16in(x.y, y.y, __ldg(tab + 8 * cc + 2 * e + 1), y1, z1);
        lo_w[e] = pack_bf16x2(y0, y1);
        hi_w[e] = pack_bf16x2(z0, z1);
      }
    }
    *reinterpret_cast<uint4*>(qs + sw128_off(m, cc)) = lo4;
    *reinterpret_cast<uint4*>(qs + kHalfBytes + sw128_off(m, cc)) = hi4;
  }
}


// Q operands: RoPE at each row's position, rounded to bf16 and laid out exactly as
// the kernel's shared-memory operand (two 64-column halves of 128 swizzled rows),
// so one bulk copy moves a whole Q tile.  One block per (Q-tile pair, KV head,
// quarter of the head dimension pairs).
__global__ void __launch_bounds__(kQTiles * kM)
qprep_kernel(const WsHeader* __restrict__ hdr, const TileMeta* __restrict__ tiles, const bf16* __restrict__ q,
             const float4* __restrict__ row_table, uint8_t* __restrict__ q_tiles, int Hq, int Hkv, int G, int R) {
  const int th = blockIdx.x;
  const int tile = th / Hkv, kvh = th % Hkv;
  if (tile >= hdr->n_tiles) return;
  const int t_row0 = tiles[tile].row0, t_n_rows = tiles[tile].n_rows;  // tile_rows_kernel's fields
  const int qt = threadIdx.x / kM, m = threadIdx.x % kM;
  if (qt == 1 && t_n_rows <= R) return;
  const int hg = m / R, i = m % R;
  const int loc = qt * R + i;
  const bool ok = loc < t_n_rows;
  const int row = t_row0 + (ok ? loc : 0);
  uint8_t* dst = q_tiles + (((int64_t)tile * Hkv + kvh) * kQTiles + qt) * kOpBytes;
  write_q_row(dst, m, ok, q + ((int64_t)row * Hq + kvh * G + hg) * kD, row_table + (int64_t)row * (kD / 2),
              2 * blockIdx.y);
}

// ---------------------------------------------------------------- V-row zeroing (warps 2, 3)
// Masked keys get weight 0 and 0 * V must stay 0 even if a slot outside a page's
// valid range holds stale non-finite bits: once a V tile has landed, the rows of
// slots that hold no valid key are zeroed before the MMA issuer uses the slot.
__device__ void vzero_loop(const TcArgs& a, uint8_t* smem, Bars* b, int n_units) {
  const int lane = threadIdx.x & 31, wz = (threadIdx.x >> 5) - 2;  // 0, 1
  uint32_t ld = 0;
  for (uint32_t k = 0;; ++k) {
    const int u = read_unit_warp(b, k);
    if (u < 0) { fail(b, a.err); return; }
    if (u >= n_units) break;
    const Unit un = a.units[u];
    const TileMeta tm = a.tiles[un.tile];
    const int page_end = tm.page_begin + tm.n_pages;
    for (int kt = un.kt0; kt < un.kt1; ++kt, ld += 2) {
      const int4 pg = load_page(a.pages, lane < kPagesPerKt ? tm.page_begin + kt * kPagesPerKt + lane : page_end,
                                page_end);
      const bool pvalid = lane < kPagesPerKt && page_ok(pg, a.num_blocks);
      const int plo = pvalid ? (int16_t)(pg.w & 0xffff) : 0;
      const int phi = pvalid ? (int16_t)(pg.w >> 16) : 0;
      const bool full = __all_sync(0xffffffffu, lane >= kPagesPerKt || (plo == 0 && phi == PIC_PAGE));
      const uint32_t vld = ld + 1;
      const int vs = vld % kSlots;
      // A slot takes K and V loads in turn, and these warps must see every phase of
      // it in order: a parity wait on the V load's phase while the slot's previous
      // fill (a K load) is still in flight would find that fill's previous phase
      // complete and pass at once.  So the K load is waited for first.  vz_done is the MMA issuer's only sign that the tile's K and V
      // have landed, so it is arrived for every tile (not only partial ones), after
      // both loads were seen; this also keeps these warps at most one phase ahead of
      // the issuer on it: a slot is not refilled before the MMAs that read it, which
      // follow the issuer's wait for vz_done, have completed.
      {
        const bool got = wait_bar(b, &b->kv_full[ld % kSlots], (ld / kSlots) & 1);
        if (!__all_sync(0xffffffffu, got)) { fail(b, a.err); return; }
      }
      const bool vgot = wait_bar(b, &b->kv_full[vs], (vld / kSlots) & 1);
      if (!__all_sync(0xffffffffu, vgot)) { fail(b, a.err); return; }
      if (!full) {
        const int packed = plo | (phi << 16);
        uint8_t* vsm = smem + kOffSlot + vs * kOpBytes;
#pragma unroll
        for (int jj = 0; jj < kPagesPerKt; ++jj) {
          const int lh = __shfl_sync(0xffffffffu, packed, jj);
          if ((jj & 1) != wz) continue;
          const int lo = lh & 0xffff, hi = lh >> 16;
          // 16 slots x 2 halves x 8 chunks of 16 bytes: 8 stores per lane
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const int idx = r * 32 + lane;
            const int cc = idx & 7, h = (idx >> 3) & 1, sl = idx >> 4;
            if (sl < lo || sl >= hi)
              *reinterpret_cast<uint4*>(vsm + jj * kPageBytes + (sl >> 3) * kGroupBytes + h * kPageHalfBytes +
                                        (sl & 7) * 128 + cc * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        tc::fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&b->vz_done[(ld / 2) % kSlots]);
    }
  }
}

// ---------------------------------------------------------------- softmax warpgroups
// Named barrier (ids 1, 2) of the two warpgroups that share Q tile qt, returning
// whether any of its 256 threads passed `failed`.
// A warpgroup whose wait gave up still meets its partner here, and both leave
// together: returning alone would leave the partner at its next barrier forever.
__device__ __forceinline__ bool pair_sync_any(int qt, bool failed) {
  uint32_t any;
  asm volatile(
      "{\n\t.reg .pred f, a;\n\t"
      "setp.ne.u32 f, %1, 0;\n\t"
      "bar.red.or.pred a, %2, 256, f;\n\t"
      "selp.u32 %0, 1, 0, a;\n\t}"
      : "=r"(any)
      : "r"((uint32_t)failed), "r"(1 + qt)
      : "memory");
  return any != 0;
}

// Rotate-on-read: Q tile qt of unit `un` written into shared memory for the key
// frame `frame` (offset-table row, -1 = global).  Since RoPE(q, p) . R(Delta) k =
// R(-Delta) RoPE(q, p) . k, the keys of a chunk can stay at their local positions
// when Q is rotated back by the chunk's offset instead (one Q tile per frame
// instead of one rotation per key tile read).  The 256 threads of the Q tile's two
// warpgroups take the roped operand the Q pre-pass wrote (global memory, already
// in the swizzled shared-memory layout), rotate each dimension pair (i, i + 64) by
// -theta_i * Delta in fp32 (cos / sin = hi + lo parts of the offset table), round
// to bf16 and store it at the same place in shared memory; for the global frame
// they copy.  Then each warp arrives on q_ready[qt].  The caller guarantees that no
// S product still reads the buffer.
__device__ __forceinline__ uint32_t rot_pair_bf16(uint32_t& whi, uint32_t wlo, const float4& t0, const float4& t1) {
  const float c0 = t0.x + t0.z, s0 = t0.y + t0.w, c1 = t1.x + t1.z, s1 = t1.y + t1.w;
  const float a0 = __uint_as_float(wlo << 16), a1 = __uint_as_float(wlo & 0xffff0000u);
  const float b0 = __uint_as_float(whi << 16), b1 = __uint_as_float(whi & 0xffff0000u);
  // R(-phi): (a, b) -> (a cos phi + b sin phi, b cos phi - a sin phi)
  whi = pack_bf16x2(fmaf(b0, c0, -a0 * s0), fmaf(b1, c1, -a1 * s1));
  return pack_bf16x2(fmaf(a0, c0, b0 * s0), fmaf(a1, c1, b1 * s1));
}

__device__ __forceinline__ void prep_q_frame(const TcArgs& a, uint8_t* smem, Bars* b, const Unit& un, int qt, int h,
                                             int t, int frame) {
  const uint8_t* src = a.q_tiles + (((int64_t)un.tile * a.Hkv + un.head) * kQTiles + qt) * kOpBytes;
  uint8_t* dst = smem + kOffQ + qt * kOpBytes;
  // thread (h, t) of the Q tile's 256: column chunk c (dimensions 8c .. 8c + 7 and
  // their partners + 64) of rows r0, r0 + 32, r0 + 64, r0 + 96, so that it needs the
  // cos / sin of only 8 frequencies
  const int tid = h * kM + t, c = tid & 7, r0 = tid >> 3;
  uint4 lo[4], hi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t off = sw128_off(r0 + 32 * k, c);
    lo[k] = *reinterpret_cast<const uint4*>(src + off);
    hi[k] = *reinterpret_cast<const uint4*>(src + kHalfBytes + off);
  }
  if (frame >= 0) {
    const float4* cs = a.rot_tab + (int64_t)frame * (kD / 2) + 8 * c;
    float4 tb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) tb[e] = __ldg(cs + e);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t* lw = reinterpret_cast<uint32_t*>(&lo[k]);
      uint32_t* hw = reinterpret_cast<uint32_t*>(&hi[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) lw[e] = rot_pair_bf16(hw[e], lw[e], tb[2 * e], tb[2 * e + 1]);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t off = sw128_off(r0 + 32 * k, c);
    *reinterpret_cast<uint4*>(dst + off) = lo[k];
    *reinterpret_cast<uint4*>(dst + kHalfBytes + off) = hi[k];
  }
  tc::fence_proxy_async_smem();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&b->q_ready[qt]);
}

// Rotate-on-read: Q tile qt of unit u for the frame of the unit's first key tile,
// if the unit has rows for the Q tile (the MMA issuer waits for it exactly then).
__device__ __forceinline__ void prep_unit_q(const TcArgs& a, uint8_t* smem, Bars* b, int u, int n_units, int qt,
                                            int h, int t) {
  if (u < 0 || u >= n_units) return;
  const Unit un = a.units[u];
  const TileMeta tm = a.tiles[un.tile];
  if (qt == 1 && tm.n_rows <= a.R) return;
  prep_q_frame(a, smem, b, un, qt, h, t, tile_frame(a, tm, un.kt0));
}

// Warpgroup (qt, h) handles key columns 64h .. 64h+63 of every S tile of Q tile qt,
// one row (TMEM lane) per thread.  The two halves of a row exchange their partial
// maxima through shared memory once per key tile (so both take identical lazy
// rescale decisions), write P for their keys into the S columns the MMA reads
// (keys 64h.. -> columns 32h..), keep their own row sums, rescale and store their
// own 64 columns of O.
template <bool kRor>
__device__ void softmax_loop(const TcArgs& a, uint8_t* smem, Bars* b, uint32_t tmem, int n_units, int qt, int h) {
  const int t = (threadIdx.x - 128) & (kM - 1);  // TMEM lane = row of Q tile qt
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = (uint32_t)((t & ~31) << 16);
  const uint32_t tS = tmem + qt * 128 + lane_base;                 // S_qt; P_qt over its first 64 columns
  const uint32_t tO = tmem + kTmemO + qt * 128 + lane_base + 64 * h;  // this half's 64 columns of O_qt
  float* xch = reinterpret_cast<float*>(smem + kOffXch) + qt * 2 * kM;  // [half][row]
  const int hg = t / a.R, i = t % a.R;
  uint32_t c = 0, ou = 0;  // tiles / units this warpgroup worked on
  // Both warpgroups of the Q tile read the same unit sequence and give up together:
  // whether every one of them got unit k + 1 is agreed at the last pair barrier of
  // unit k (the first unit: at a barrier of its own).
  int u = read_unit_warp(b, 0);
  if (pair_sync_any(qt, u < 0)) { fail(b, a.err); return; }
  if (kRor) prep_unit_q(a, smem, b, u, n_units, qt, h, t);
  for (uint32_t k = 0; u < n_units; ++k) {
    const Unit un = a.units[u];
    const TileMeta tm = a.tiles[un.tile];
    const int n = un.kt1 - un.kt0;
    if (qt == 1 && tm.n_rows <= a.R) {  // no rows for this Q tile: only the next unit
      u = read_unit_warp(b, k + 1);
      if (pair_sync_any(qt, u < 0)) { fail(b, a.err); return; }
      if (kRor) prep_unit_q(a, smem, b, u, n_units, qt, h, t);
      continue;
    }
    const int loc = qt * a.R + i;
    const bool row_ok = loc < tm.n_rows;
    const int row = tm.row0 + (row_ok ? loc : 0);
    const int p_row = a.rows[tm.row0 + (row_ok ? loc : tm.n_rows - 1)];
    const int hq = un.head * a.G + hg;
    float m_ref = -INFINITY, l = 0.f;
    const int page_end = tm.page_begin + tm.n_pages;
    const int pbase = tm.page_begin + un.kt0 * kPagesPerKt;
    // lanes 0-3 hold the entries of this half's 4 pages of the key tile (one tile ahead)
    const int my_page = kPagesPerKt / 2 * h + lane;
    int4 pe = load_page(a.pages, lane < kPagesPerKt / 2 ? pbase + my_page : page_end, page_end);
    // rotating on read: frames of key tiles j and j + 1, read a tile ahead
    int f_cur = 0, f_nxt = 0;
    if (kRor) {
      f_cur = tile_frame(a, tm, un.kt0);
      f_nxt = n > 1 ? tile_frame(a, tm, un.kt0 + 1) : f_cur;
    }
    for (int j = 0; j < n; ++j, ++c) {
      const int4 cur = pe;
      if (j + 1 < n && lane < kPagesPerKt / 2)
        pe = load_page(a.pages, pbase + (j + 1) * kPagesPerKt + my_page, page_end);
      const bool pvalid = lane < kPagesPerKt / 2 && page_ok(cur, a.num_blocks);
      const int plo = pvalid ? (int16_t)(cur.w & 0xffff) : 0;
      const int phi = pvalid ? (int16_t)(cur.w >> 16) : 0;
      const bool pfull = plo == 0 && phi == PIC_PAGE;
      const bool half_full = __all_sync(0xffffffffu, lane >= kPagesPerKt / 2 || pfull);
      const int half_last = __reduce_max_sync(0xffffffffu, pvalid ? cur.z + phi - 1 : INT_MIN);

      // masking: key slot sl of page jj is visible to this row iff
      // lo_jj <= sl < min(hi_jj, p_row - gpos0_jj + 1); one 16-bit mask per page.
      // Page entries only, so the bits are ready before S is.
      const bool need_mask = __any_sync(0xffffffffu, !(half_full && half_last <= p_row));
      uint32_t vis[2] = {0, 0};
      if (need_mask) {
        const int packed = plo | (phi << 16);
#pragma unroll
        for (int jj = 0; jj < kPagesPerKt / 2; ++jj) {
          const int g0 = __shfl_sync(0xffffffffu, cur.z, jj);
          const int lh = __shfl_sync(0xffffffffu, packed, jj);
          const int lo = lh & 0xffff;
          const int hi = min(lh >> 16, max(p_row - g0 + 1, 0));
          const uint32_t m16 = hi > lo ? ((1u << hi) - 1u) & ~((1u << lo) - 1u) : 0u;
          vis[jj >> 1] |= m16 << (16 * (jj & 1));
        }
      }

      // A thread whose wait gave up goes on to the pair barrier below (reading S
      // regardless: a stale TMEM read is harmless, and the warp stays converged for
      // the warp-wide load), where both warpgroups of the Q tile learn of it and leave.
      const bool s_ok = wait_bar(b, &b->s_full[qt], c & 1);
      tc::tc_fence_after();
      float s[64];
      {
        uint32_t sr[64];
        tc::tmem_ld32(tS + 64 * h, sr);
        tc::tmem_ld32(tS + 64 * h + 32, sr + 32);
        tc::tmem_ld_wait();
        tc::reg_fence<64>(sr);
#pragma unroll
        for (int k2 = 0; k2 < 64; ++k2) s[k2] = u2f(sr[k2]);
      }
      if (need_mask) {
#pragma unroll
        for (int k2 = 0; k2 < 64; ++k2) s[k2] = (vis[k2 >> 5] & (1u << (k2 & 31))) ? s[k2] : -INFINITY;
      }
      float mx8[8];
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) mx8[q8] = -INFINITY;
#pragma unroll
      for (int k2 = 0; k2 < 64; k2 += 16)
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) mx8[q8] = tc::max3(mx8[q8], s[k2 + 2 * q8], s[k2 + 2 * q8 + 1]);
      const float pmax = tc::max3(tc::max3(mx8[0], mx8[1], mx8[2]), tc::max3(mx8[3], mx8[4], mx8[5]),
                                  fmaxf(mx8[6], mx8[7]));
      // both halves have read their S columns after this barrier, so P may be written;
      // the next write of xch follows s_full of the next tile, i.e. both p_full arrivals
      xch[h * kM + t] = pmax;
      if (pair_sync_any(qt, !s_ok)) { fail(b, a.err); return; }
      const float mt = fmaxf(pmax, xch[(1 - h) * kM + t]) * a.scale_log2;
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_ref + kRescaleThreshold) {
        alpha = tc::ex2(m_ref - mt);
        resc = (m_ref != -INFINITY);
        l *= alpha;
        m_ref = mt;
      }
      const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
      // P for this half's 64 keys in two stores of 16 packed columns; x = s * scale_log2 - mu
      // and the row sum on packed fp32 pairs
      const uint64_t c2 = tc::f2pack(a.scale_log2, a.scale_log2), m2 = tc::f2pack(-mu, -mu);
      uint64_t rs2[2] = {0, 0};
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int k2 = 0; k2 < 16; ++k2) {
          float x0, x1;
          tc::f2unpack(tc::fma2(tc::f2pack(s[32 * cc + 2 * k2], s[32 * cc + 2 * k2 + 1]), c2, m2), x0, x1);
          const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
          rs2[k2 & 1] = tc::add2(rs2[k2 & 1], tc::f2pack(p0, p1));
          pk[k2] = pack_bf16x2(p0, p1);
        }
        tc::tmem_st16(tS + 32 * h + 16 * cc, pk);
      }
      {
        float r0, r1;
        tc::f2unpack(tc::add2(rs2[0], rs2[1]), r0, r1);
        l += r0 + r1;
      }
      // O_qt is stable here (the commit behind s_full covers the previous P.V) and P.V
      // for this tile is not issued before p_full: rescale this half of O after P is stored
      if (__any_sync(0xffffffffu, resc)) {
        const float f = resc ? alpha : 1.f;
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
          uint32_t r[32];
          tc::tmem_ld32(tO + q4 * 32, r);
          tc::tmem_ld_wait();
          tc::reg_fence<32>(r);
#pragma unroll
          for (int x = 0; x < 32; ++x) r[x] = f2u(u2f(r[x]) * f);
          tc::tmem_st32(tO + q4 * 32, r);
        }
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&b->p_full[qt]);
      // the next key tile in another frame: S of this tile has read Q, and the next S
      // product waits for q_ready, so Q is rotated into the new frame now, beside P.V
      if (kRor && j + 1 < n) {
        if (f_nxt != f_cur) prep_q_frame(a, smem, b, un, qt, h, t, f_nxt);
        f_cur = f_nxt;
        if (j + 2 < n) f_nxt = tile_frame(a, tm, un.kt0 + j + 2);
      }
    }
    // The next unit, read now; rotating on read, its first Q tile is written at once
    // (this unit's last S product has completed, so the buffer is free), beside the
    // last P.V, before the epilogue.
    const int u_next = read_unit_warp(b, k + 1);
    if (kRor) prep_unit_q(a, smem, b, u_next, n_units, qt, h, t);
    // epilogue: O / l over both halves' row sums
    const bool o_ok = wait_bar(b, &b->o_done[qt], ou & 1);
    ++ou;
    tc::tc_fence_after();
    xch[h * kM + t] = l;
    if (pair_sync_any(qt, !o_ok)) { fail(b, a.err); return; }
    const float l_all = l + xch[(1 - h) * kM + t];
    // both have read before either writes the next tile's maximum; the next unit agreed
    if (pair_sync_any(qt, u_next < 0)) { fail(b, a.err); return; }
    const float inv = (l_all > 0.f) ? 1.f / l_all : 0.f;
    const int64_t slot = ((int64_t)(un.part < 0 ? 0 : un.part) * kQTiles + qt) * kM + t;
#pragma unroll 1
    for (int q4 = 0; q4 < 2; ++q4) {
      uint32_t r[32];
      tc::tmem_ld32(tO + q4 * 32, r);
      tc::tmem_ld_wait();
      tc::reg_fence<32>(r);
      if (!row_ok) continue;
      const int col = 64 * h + 32 * q4;
      if (un.part < 0) {
        uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)row * a.Hq + hq) * kD + col);
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2)
          dst[k2] = make_uint4(pack_bf16x2(u2f(r[8 * k2]) * inv, u2f(r[8 * k2 + 1]) * inv),
                               pack_bf16x2(u2f(r[8 * k2 + 2]) * inv, u2f(r[8 * k2 + 3]) * inv),
                               pack_bf16x2(u2f(r[8 * k2 + 4]) * inv, u2f(r[8 * k2 + 5]) * inv),
                               pack_bf16x2(u2f(r[8 * k2 + 6]) * inv, u2f(r[8 * k2 + 7]) * inv));
      } else {
        float4* dst = reinterpret_cast<float4*>(a.part_o + slot * kD + col);
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2)
          dst[k2] = make_float4(u2f(r[4 * k2]) * inv, u2f(r[4 * k2 + 1]) * inv, u2f(r[4 * k2 + 2]) * inv,
                                u2f(r[4 * k2 + 3]) * inv);
      }
    }
    tc::tc_fence_before();
    if (h == 0 && row_ok && un.part >= 0) a.part_ml[slot] = make_float2(m_ref, l_all);
    u = u_next;
  }
}

template <bool kRor>
__global__ void __launch_bounds__(kThreads, 1)
link_attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the operand layouts need 1024-byte alignment and there is no room for slack
  if (tc::smem_addr(smem_raw) & 1023u) {
    if (threadIdx.x == 0) set_err(a.err, PIC_ERR_UNSUPPORTED);
    return;
  }
  uint8_t* smem = smem_raw;
  Bars* b = reinterpret_cast<Bars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      tc::mbar_init(&b->kv_full[s], 1);
      tc::mbar_init(&b->vz_done[s], 2);
    }
    for (int s = 0; s < kStepRing; ++s) tc::mbar_init(&b->kv_step[s], 1);
    for (int i = 0; i < kQTiles; ++i) {
      tc::mbar_init(&b->q_full[i], 1);
      tc::mbar_init(&b->q_free[i], 1);
      tc::mbar_init(&b->s_full[i], 1);
      tc::mbar_init(&b->p_full[i], 8);  // every warp of the Q tile's two softmax warpgroups
      tc::mbar_init(&b->o_done[i], 1);
      tc::mbar_init(&b->q_ready[i], 8);  // every warp of the Q tile's two softmax warpgroups
    }
    tc::mbar_init(&b->drain, 1);
    tc::mbar_init(&b->never, 1);
    for (int i = 0; i < kUnitRing; ++i) {
      tc::mbar_init(&b->unit_full[i], 1);
      tc::mbar_init(&b->unit_empty[i], kUnitReaders);
    }
    b->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&kmap);
    tc::tma_prefetch_desc(&vmap);
  }
  if (warp == 1) {
    tc::tmem_alloc(&b->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = b->tmem_base;
  const int n_units = a.hdr->n_units;
  if (warp < 4) {
    tc::regs_dec<kRegsLow>();
    if (warp == 0) {
      producer_loop<kRor>(a, &kmap, &vmap, smem, b, n_units);
    } else if (warp == 1 && lane == 0) {
      mma_loop<kRor>(a, smem, b, tmem, n_units);
      // every MMA this thread issued completes before TMEM is released (also on abort)
      tc::mma_commit(&b->drain);
      const int no_abort = 0;
      tc::mbar_wait(&b->drain, 0, &no_abort, kWaitLimitNs);
    } else if (warp == 2 || warp == 3) {
      vzero_loop(a, smem, b, n_units);
    }
  } else {
    tc::regs_inc<kRegsHigh>();
    const int g = (warp - 4) / 4;  // softmax warpgroup: Q tile g / 2, key columns 64 (g % 2) ..
    softmax_loop<kRor>(a, smem, b, tmem, n_units, g / 2, g % 2);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ CTA-pair self-test
// One pair of CTAs (a cluster of two): the pair products the two-SM attention
// issues, on operands laid out as that kernel lays them out, read back from both
// CTAs' TMEM.  CTA r holds rows 128r.. of A, keys 128r.. of B (K-major pages) and
// columns 64r.. of V (one half page per 16 keys).  Each CTA allocates 256 TMEM
// columns; info[r] receives the base address CTA r was given.
constexpr int kPairTestSmem = 2 * kOpBytes + kOpBytes / 2 + 64;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
selftest_umma_pair_kernel(const bf16* __restrict__ a, const bf16* __restrict__ b, const bf16* __restrict__ v,
                          float* ds, float* dpv, int32_t* info, int32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sa = smem;                 // A: own 128 rows, two 64-column halves
  uint8_t* sb = smem + kOpBytes;      // B: own 128 keys as 8 pages
  uint8_t* sv = smem + 2 * kOpBytes;  // V: own 64 columns of 128 keys, 8 half pages
  uint64_t* done = reinterpret_cast<uint64_t*>(sv + kOpBytes / 2);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
  int* ab = reinterpret_cast<int*>(done + 2);
  const int t = threadIdx.x, warp = t >> 5;
  const uint32_t r = tc::cluster_rank();
  if (t == 0) {
    tc::mbar_init(done, 1);
    *ab = 0;
    tc::fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tc::tmem_alloc2(tslot, 256);
    tc::tmem_relinquish2();
  }
  // operands: thread t fills row / key t
  {
    const int row = 128 * r + t;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<uint4*>(sa + h * kHalfBytes + sw128_off(t, cc)) =
            *reinterpret_cast<const uint4*>(a + row * 128 + h * 64 + cc * 8);
    const int pg = t / PIC_PAGE, sl = t % PIC_PAGE, grp = sl / 8, rr = sl % 8;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<uint4*>(sb + pg * kPageBytes + grp * kGroupBytes + h * kPageHalfBytes + rr * 128 +
                                  ((cc ^ rr) << 4)) = *reinterpret_cast<const uint4*>(b + row * 128 + h * 64 + cc * 8);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc)
      *reinterpret_cast<uint4*>(sv + pg * (kPageBytes / 2) + grp * kPageHalfBytes + rr * 128 + ((cc ^ rr) << 4)) =
          *reinterpret_cast<const uint4*>(v + t * 128 + 64 * r + cc * 8);
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();  // both CTAs' operands and barrier in place
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  if (t == 0) info[r] = (int32_t)tmem;
  const uint32_t lb = (uint32_t)((warp * 32) << 16);
  constexpr uint32_t kIdS2 = tc::idesc_bf16_f32(256, 256, false);
  constexpr uint32_t kIdPV2 = tc::idesc_bf16_f32(256, 128, true);
  // S = A B^T (256 x 256)
  if (r == 0 && t == 0) {
    const uint32_t sa_a = tc::smem_addr(sa), sb_a = tc::smem_addr(sb);
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t aoff = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
      const uint32_t boff = (ks >> 2) * kPageHalfBytes + (ks & 3) * 32;
      tc::mma2_bf16_ss(tmem, tc::sw128_desc(sa_a + aoff, 16, 1024), tc::sw128_desc(sb_a + boff, 16, kGroupBytes),
                       kIdS2, ks > 0);
    }
    tc::mma2_commit(done, 3);
  }
  bool ok = tc::mbar_wait(done, 0, ab, kWaitLimitNs);
  if (!__all_sync(0xffffffffu, ok)) {
    if ((t & 31) == 0) set_err(err, PIC_ERR_TIMEOUT);
  } else {
    tc::tc_fence_after();
    for (int c0 = 0; c0 < 256; c0 += 32) {
      uint32_t x[32];
      tc::tmem_ld32(tmem + lb + c0, x);
      tc::tmem_ld_wait();
      tc::reg_fence<32>(x);
      for (int k = 0; k < 32; ++k) ds[(int64_t)(128 * r + t) * 256 + c0 + k] = u2f(x[k]);
    }
  }
  // P = A's first 128 columns into TMEM columns 128..191 (bf16 pairs), then P V
  {
    uint32_t x[64];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a + (128 * r + t) * 128);
#pragma unroll
    for (int k = 0; k < 64; ++k) x[k] = src[k];
    tc::tmem_st32(tmem + lb + 128, x);
    tc::tmem_st32(tmem + lb + 160, x + 32);
    tc::tmem_st_wait();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();  // both CTAs read S and wrote P
  tc::tc_fence_after();
  if (r == 0 && t == 0) {
    const uint32_t sv_a = tc::smem_addr(sv);
    for (int ks = 0; ks < 8; ++ks)
      tc::mma2_bf16_ts(tmem, tmem + 128 + ks * 8, tc::sw128_desc(sv_a + ks * (kPageBytes / 2), 16, kPageHalfBytes),
                       kIdPV2, ks > 0);
    tc::mma2_commit(done, 3);
  }
  ok = tc::mbar_wait(done, 1, ab, kWaitLimitNs);
  if (!__all_sync(0xffffffffu, ok)) {
    if ((t & 31) == 0) set_err(err, PIC_ERR_TIMEOUT);
  } else {
    tc::tc_fence_after();
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t x[32];
      tc::tmem_ld32(tmem + lb + c0, x);
      tc::tmem_ld_wait();
      tc::reg_fence<32>(x);
      for (int k = 0; k < 32; ++k) dpv[(int64_t)(128 * r + t) * 128 + c0 + k] = u2f(x[k]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();  // no pair product or peer access outstanding
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc2(tmem, 256);
  }
}

// ------------------------------------------------------------------ LSE merge
// Blocks of 8 rows of one (Q-tile pair, KV head) with split spans; one warp per
// row, lane = 4-dim chunk.  Combines the per-span partials (O_s normalised by
// l_s, base-2 max m_s):
//   O = sum_s 2^(m_s - M) l_s O_s / sum_s 2^(m_s - M) l_s.
constexpr int kMergeRows = 8;

__global__ void __launch_bounds__(32 * kMergeRows)
merge_kernel(const WsHeader* __restrict__ hdr, const TileMeta* __restrict__ tiles,
             const float* __restrict__ part_o, const float2* __restrict__ part_ml, bf16* __restrict__ out,
             int Hq, int Hkv, int G, int R) {
  static_assert(kD == 4 * 32, "one float4 per lane");
  const int th = blockIdx.x;
  const int tile = th / Hkv, head = th % Hkv;
  if (tile >= hdr->n_tiles) return;
  const TileMeta tm = tiles[tile];
  if (tm.n_spans <= 1) return;
  const int m2 = blockIdx.y * kMergeRows + (threadIdx.x >> 5), c = threadIdx.x & 31;
  const int qt = m2 / kM, t = m2 % kM;
  const int hg = t / R, i = t % R;
  const int loc = qt * R + i;
  if (loc >= tm.n_rows) return;
  const int base = tm.part_base + head * tm.n_spans;
  // one pass with a running maximum, four spans' loads in flight at a time
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < tm.n_spans; s0 += 4) {
    float2 ml[4];
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ml[k] = make_float2(-INFINITY, 0.f);
      v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s0 + k < tm.n_spans) {
        const int64_t slot = ((int64_t)(base + s0 + k) * kQTiles + qt) * kM + t;
        ml[k] = part_ml[slot];
        v[k] = reinterpret_cast<const float4*>(part_o + slot * kD)[c];
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (!(ml[k].y > 0.f)) continue;  // a span without visible keys contributes nothing
      const float Mn = fmaxf(M, ml[k].x);
      const float a = exp2f(M - Mn), w = ml[k].y * exp2f(ml[k].x - Mn);  // a = 0 while M = -inf
      den = fmaf(den, a, w);
      acc.x = fmaf(acc.x, a, w * v[k].x); acc.y = fmaf(acc.y, a, w * v[k].y);
      acc.z = fmaf(acc.z, a, w * v[k].z); acc.w = fmaf(acc.w, a, w * v[k].w);
      M = Mn;
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(out + ((int64_t)(tm.row0 + loc) * Hq + head * G + hg) * kD) + c;
  *dst = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

// ------------------------------------------------------------------ self-test
// The operand layouts of the attention kernel on one 128 x 128 x 128 product:
// A swizzled in shared memory (as Q), B loaded by TMA with the 128-byte swizzle
// (as a K / V tile), and A written to TMEM by tcgen05.st (as P).
__global__ void __launch_bounds__(128, 1)
selftest_umma_kernel(const __grid_constant__ CUtensorMap bmap, const bf16* __restrict__ a, float* dk,
                     float* dmn, float* dts, int32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sa = smem;
  uint8_t* sbm = smem + kOpBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kOpBytes);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  int* ab = reinterpret_cast<int*>(bars + 3);
  const int t = threadIdx.x, warp = t >> 5;
  if (t == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    *ab = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, 512);
    tc::tmem_relinquish();
  }
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int cc = 0; cc < 8; ++cc)
      *reinterpret_cast<uint4*>(sa + h * kHalfBytes + sw128_off(t, cc)) =
          *reinterpret_cast<const uint4*>(a + t * 128 + h * 64 + cc * 8);
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lb = (uint32_t)((warp * 32) << 16);
  {  // A row t into TMEM columns 384..447 (bf16 pairs)
    uint32_t r[64];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a + t * 128);
#pragma unroll
    for (int x = 0; x < 64; ++x) r[x] = src[x];
    tc::tmem_st32(tmem + lb + 384, r);
    tc::tmem_st32(tmem + lb + 416, r + 32);
    tc::tmem_st_wait();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (t == 0) {
    tc::mbar_arrive_expect_tx(&bars[0], kOpBytes);
    for (int j = 0; j < 8; ++j) tc::tma_load_4d(sbm + j * kPageBytes, &bmap, 0, 0, 0, j * (PIC_PAGE / 8), &bars[0]);
    const bool ok = tc::mbar_wait(&bars[0], 0, ab, kWaitLimitNs);
    if (ok) {
      tc::tc_fence_after();
      const uint32_t sa_a = tc::smem_addr(sa), sb_a = tc::smem_addr(sbm);
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t qoff = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
        const uint32_t koff = (ks >> 2) * kPageHalfBytes + (ks & 3) * 32;
        tc::mma_bf16_ss(tmem, tc::sw128_desc(sa_a + qoff, 16, 1024), tc::sw128_desc(sb_a + koff, 16, kGroupBytes),
                        kIdescS, ks > 0);
      }
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t qoff = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
        tc::mma_bf16_ss(tmem + 128, tc::sw128_desc(sa_a + qoff, 16, 1024),
                        tc::sw128_desc(sb_a + ks * kPageBytes, kPageHalfBytes, kGroupBytes), kIdescPV, ks > 0);
      }
      for (int ks = 0; ks < 8; ++ks)
        tc::mma_bf16_ts(tmem + 256, tmem + 384 + ks * 8,
                        tc::sw128_desc(sb_a + ks * kPageBytes, kPageHalfBytes, kGroupBytes), kIdescPV, ks > 0);
      tc::mma_commit(&bars[1]);
    } else {
      set_err(err, PIC_ERR_TIMEOUT);
      *reinterpret_cast<volatile int*>(ab) = 1;
    }
  }
  __syncthreads();
  if (!*reinterpret_cast<volatile int*>(ab) && tc::mbar_wait(&bars[1], 0, ab, kWaitLimitNs)) {
    tc::tc_fence_after();
    float* outs[3] = {dk, dmn, dts};
    for (int o = 0; o < 3; ++o)
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + lb + o * 128 + c * 32, r);
        tc::tmem_ld_wait();
        for (int x = 0; x < 32; ++x) outs[o][t * 128 + c * 32 + x] = u2f(r[x]);
      }
  } else if (t == 0) {
    set_err(err, PIC_ERR_TIMEOUT);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side
bool tc_shape(pic_dtype dt, int Hq, int Hkv, int d) {
  if (dt != PIC_BF16 || d != kD || Hkv < 1 || Hq % Hkv) return false;
  const int G = Hq / Hkv;
  return G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
}

// The two phases of a tensor-core attention call, with the scratch laid out by L
// in `ws`: the plan (unit list, Q operands — reads no K or V) and the run
// (attention, merge).  The planner may add up to min(kUnitsPerSm * split_sms,
// split_cap) units by splitting key ranges.
// kPhaseQ: the tiles' rows and Q operands (no page list needed); kPhaseUnits: the
// unit plan (reads the page list); kPhaseRun: attention and merge.
enum { kPhaseQ = 1, kPhaseRun = 2, kPhaseUnits = 4, kPhasePlan = kPhaseQ | kPhaseUnits, kPhaseAll = 7 };

pic_status launch_tc(const void* q, const float* row_table, const int32_t* rows, const int32_t* row_off,
                     const void* k_pool, const void* v_pool, int64_t num_blocks, const pic_link_page* pages,
                     const int32_t* page_off, int32_t n_req, int32_t Hq, int32_t Hkv, float scale, void* out,
                     uint8_t* w, const WsLayout& L, int split_sms, int split_cap, int32_t* err_flag, cudaStream_t s,
                     const int32_t* page_tab = nullptr, const float* rot_table = nullptr, int64_t n_tab = 0,
                     int phases = kPhaseAll) {
  const int G = Hq / Hkv;
  if (n_req > kMaxPlanReqs) return PIC_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(row_table) & 15) ||
      (reinterpret_cast<uintptr_t>(pages) & 15))
    return PIC_ERR_INVALID;
  CUtensorMap kmap, vmap;
  if (phases & kPhaseRun) {
    if ((reinterpret_cast<uintptr_t>(k_pool) & 15) || (reinterpret_cast<uintptr_t>(v_pool) & 15) ||
        (reinterpret_cast<uintptr_t>(out) & 15))
      return PIC_ERR_INVALID;
    const uint64_t pool_rows = (uint64_t)num_blocks * Hkv * PIC_PAGE;
    if (pool_rows == 0 || pool_rows > (uint64_t)INT32_MAX) return PIC_ERR_INVALID;
    if (!encode_pages(&kmap, k_pool, pool_rows) || !encode_pages(&vmap, v_pool, pool_rows)) return PIC_ERR_CUDA;
  }
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  TileMeta* tiles = reinterpret_cast<TileMeta*>(w + L.off_tiles);
  Unit* units = reinterpret_cast<Unit*>(w + L.off_units);
  float2* part_ml = reinterpret_cast<float2*>(w + L.off_ml);
  float* part_o = reinterpret_cast<float*>(w + L.off_o);
  const int sms = num_sms_of_current_device();
  const int R = kM / G;
  uint8_t* q_tiles = w + L.off_q;
  if (phases & kPhaseQ) {
    tile_rows_kernel<<<1, kPlanThreads, 0, s>>>(row_off, n_req, kQTiles * R, L.tiles_cap, hdr, tiles, err_flag);
    if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
    qprep_kernel<<<dim3((unsigned)(L.tiles_cap * Hkv), 4), kQTiles * kM, 0, s>>>(
        hdr, tiles, static_cast<const bf16*>(q), reinterpret_cast<const float4*>(row_table), q_tiles, Hq, Hkv, G,
        R);
    if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  }
  if (phases & kPhaseUnits) {
    plan_units_kernel<<<1, kPlanThreads, 0, s>>>(rows, row_off, pages, page_off, n_req, kQTiles * R, Hkv,
                                                  split_sms < sms ? split_sms : sms, split_cap, L.tiles_cap, L.units_cap,
                                                  L.tail_extra, hdr, tiles, units, err_flag);
    if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  }
  if (!(phases & kPhaseRun)) return PIC_OK;
  // rotate-on-read is its own instantiation, so the plain kernel carries none of it
  const auto kern = page_tab != nullptr ? link_attn_tc_kernel<true> : link_attn_tc_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return PIC_ERR_CUDA;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return PIC_ERR_CUDA;
  if (fa.numRegs != kLaunchRegs) return PIC_ERR_UNSUPPORTED;  // the register split assumes this launch size
  TcArgs a;
  a.q_tiles = q_tiles;
  a.q = static_cast<const bf16*>(q);
  a.row_table = reinterpret_cast<const float4*>(row_table);
  a.rows = rows;
  a.pages = pages;
  a.out = static_cast<bf16*>(out);
  a.hdr = hdr;
  a.next_unit = &hdr->next_unit;
  a.tiles = tiles;
  a.units = units;
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.err = err_flag;
  a.num_blocks = num_blocks;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.R = R;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.page_tab = page_tab;
  a.rot_tab = reinterpret_cast<const float4*>(rot_table);
  a.n_tab = n_tab;
  const int64_t grid = L.units_cap < sms ? L.units_cap : sms;
  kern<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(kmap, vmap, a);
  if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  merge_kernel<<<dim3((unsigned)(L.tiles_cap * Hkv), kQTiles * kM / kMergeRows), 32 * kMergeRows, 0, s>>>(
      hdr, tiles, part_o, part_ml, a.out, Hq, Hkv, G, R);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

pic_status check_attention_args(const void* q, const float* row_table, const int32_t* rows, const int32_t* row_off,
                                const void* k_pool, const void* v_pool, int64_t num_blocks, pic_dtype dtype,
                                const pic_link_page* pages, const int32_t* page_off, int32_t n_req, int64_t n_rows,
                                int32_t Hq, int32_t Hkv, int32_t d, float scale, void* out, int32_t* err_flag) {
  if (n_req < 0 || n_rows < 0 || num_blocks < 0 || Hkv < 1 || Hq < 1 || Hq % Hkv || d < 2 || d > 256 ||
      (d & 1) || !(scale > 0.f))
    return PIC_ERR_INVALID;
  if (dtype != PIC_BF16 && dtype != PIC_FP32) return PIC_ERR_INVALID;
  if (n_req == 0 || n_rows == 0) return PIC_OK;
  if (!q || !row_table || !rows || !row_off || !k_pool || !v_pool || !pages || !page_off || !out || !err_flag)
    return PIC_ERR_INVALID;
  return PIC_OK;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Rows of 128 bf16 viewed as [row group][half][row in group][64 columns]: one box of
// 2 x 2 x 8 x 64 moves a whole 16-row page into the [group][half][8 rows] layout.
bool encode_pages(CUtensorMap* map, const void* base, uint64_t rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr || rows % 8) return false;
  cuuint64_t dims[4] = {64, 8, 2, rows / 8};
  cuuint64_t strides[3] = {128 * sizeof(__nv_bfloat16), 64 * sizeof(__nv_bfloat16), 8 * 128 * sizeof(__nv_bfloat16)};
  cuuint32_t box[4] = {64, 8, 2, PIC_PAGE / 8};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pic

using namespace pic;

extern "C" {

size_t pic_link_attention_workspace(int64_t n_rows, int32_t n_req, int32_t Hq, int32_t Hkv, int32_t d,
                                    pic_dtype dtype) {
  if (n_rows < 0 || n_req < 0 || Hkv < 1 || Hq < Hkv || Hq % Hkv) return 0;
  if (!tc_shape(dtype, Hq, Hkv, d)) return 0;
  return ws_layout(n_rows, n_req, Hq / Hkv, Hkv, d).total;
}

pic_status pic_link_attention(const void* q, const float* row_table, const int32_t* rows,
                              const int32_t* row_off, const void* k_pool, const void* v_pool,
                              int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                              const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                              int32_t Hkv, int32_t d, float scale, void* out, void* ws, size_t ws_bytes,
                              int32_t* err_flag, pic_stream_t stream) {
  const pic_status st = check_attention_args(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, dtype, pages,
                                             page_off, n_req, n_rows, Hq, Hkv, d, scale, out, err_flag);
  if (st != PIC_OK || n_req == 0 || n_rows == 0) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (tc_shape(dtype, Hq, Hkv, d)) {
    const WsLayout L = ws_layout(n_rows, n_req, Hq / Hkv, Hkv, d);
    if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PIC_ERR_WORKSPACE;
    return launch_tc(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, pages, page_off, n_req, Hq, Hkv, scale,
                     out, static_cast<uint8_t*>(ws), L, kAllSms, kMaxSplitUnits, err_flag, s);
  }
  return launch_attention_simt(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, dtype, pages, page_off,
                               n_req, n_rows, Hq, Hkv, d, scale, out, s);
}

pic_status pic_link_attention_plan(const void* q, const float* row_table, const int32_t* rows,
                                   const int32_t* row_off, const pic_link_page* pages, const int32_t* page_off,
                                   int32_t n_req, int64_t n_rows, int32_t Hq, int32_t Hkv, int32_t d,
                                   pic_dtype dtype, void* ws, size_t ws_bytes, int32_t* err_flag,
                                   pic_stream_t stream) {
  if (n_req < 0 || n_rows < 0 || Hkv < 1 || Hq < 1 || Hq % Hkv || d < 2 || d > 256 || (d & 1))
    return PIC_ERR_INVALID;
  if (dtype != PIC_BF16 && dtype != PIC_FP32) return PIC_ERR_INVALID;
  if (n_req == 0 || n_rows == 0 || !tc_shape(dtype, Hq, Hkv, d)) return PIC_OK;  // nothing to plan
  if (!q || !row_table || !rows || !row_off || !pages || !page_off || !err_flag) return PIC_ERR_INVALID;
  const WsLayout L = ws_layout(n_rows, n_req, Hq / Hkv, Hkv, d);
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PIC_ERR_WORKSPACE;
  return launch_tc(q, row_table, rows, row_off, nullptr, nullptr, 0, pages, page_off, n_req, Hq, Hkv, 1.f, nullptr,
                   static_cast<uint8_t*>(ws), L, kAllSms, kMaxSplitUnits, err_flag, (cudaStream_t)stream,
                   nullptr, nullptr, 0, kPhasePlan);
}

pic_status pic_link_attention_plan_q(const void* q, const float* row_table, const int32_t* row_off,
                                     int32_t n_req, int64_t n_rows, int32_t Hq, int32_t Hkv, int32_t d,
                                     pic_dtype dtype, void* ws, size_t ws_bytes, int32_t* err_flag,
                                     pic_stream_t stream) {
  if (n_req < 0 || n_rows < 0 || Hkv < 1 || Hq < 1 || Hq % Hkv || d < 2 || d > 256 || (d & 1))
    return PIC_ERR_INVALID;
  if (dtype != PIC_BF16 && dtype != PIC_FP32) return PIC_ERR_INVALID;
  if (n_req == 0 || n_rows == 0 || !tc_shape(dtype, Hq, Hkv, d)) return PIC_OK;  // nothing to plan
  if (!q || !row_table || !row_off || !err_flag) return PIC_ERR_INVALID;
  const WsLayout L = ws_layout(n_rows, n_req, Hq / Hkv, Hkv, d);
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PIC_ERR_WORKSPACE;
  return launch_tc(q, row_table, nullptr, row_off, nullptr, nullptr, 0, nullptr, nullptr, n_req, Hq, Hkv, 1.f,
                   nullptr, static_cast<uint8_t*>(ws), L, kAllSms, kMaxSplitUnits, err_flag, (cudaStream_t)stream,
                   nullptr, nullptr, 0, kPhaseQ);
}

pic_status pic_link_attention_plan_units(const int32_t* rows, const int32_t* row_off, const pic_link_page* pages,
                                         const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                                         int32_t Hkv, int32_t d, pic_dtype dtype, void* ws, size_t ws_bytes,
                                         int32_t* err_flag, pic_stream_t stream) {
  if (n_req < 0 || n_rows < 0 || Hkv < 1 || Hq < 1 || Hq % Hkv || d < 2 || d > 256 || (d & 1))
    return PIC_ERR_INVALID;
  if (dtype != PIC_BF16 && dtype != PIC_FP32) return PIC_ERR_INVALID;
  if (n_req == 0 || n_rows == 0 || !tc_shape(dtype, Hq, Hkv, d)) return PIC_OK;  // nothing to plan
  if (!rows || !row_off || !pages || !page_off || !err_flag) return PIC_ERR_INVALID;
  const WsLayout L = ws_layout(n_rows, n_req, Hq / Hkv, Hkv, d);
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PIC_ERR_WORKSPACE;
  return launch_tc(nullptr, nullptr, rows, row_off, nullptr, nullptr, 0, pages, page_off, n_req, Hq, Hkv, 1.f,
                   nullptr, static_cast<uint8_t*>(ws), L, kAllSms, kMaxSplitUnits, err_flag, (cudaStream_t)stream,
                   nullptr, nullptr, 0, kPhaseUnits);
}

pic_status pic_link_attention_run(const void* q, const float* row_table, const int32_t* rows,
                                  const int32_t* row_off, const void* k_pool, const void* v_pool,
                                  int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                                  const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                                  int32_t Hkv, int32_t d, float scale, void* out, void* ws, size_t ws_bytes,
                                  int32_t* err_flag, pic_stream_t stream) {
  const pic_status st = check_attention_args(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, dtype, pages,
                                             page_off, n_req, n_rows, Hq, Hkv, d, scale, out, err_flag);
  if (st != PIC_OK || n_req == 0 || n_rows == 0) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (tc_shape(dtype, Hq, Hkv, d)) {
    const WsLayout L = ws_layout(n_rows, n_req, Hq / Hkv, Hkv, d);
    if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PIC_ERR_WORKSPACE;
    return launch_tc(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, pages, page_off, n_req, Hq, Hkv, scale,
                     out, static_cast<uint8_t*>(ws), L, kAllSms, kMaxSplitUnits, err_flag, s, nullptr, nullptr,
                     0, kPhaseRun);
  }
  return launch_attention_simt(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, dtype, pages, page_off,
                               n_req, n_rows, Hq, Hkv, d, scale, out, s);
}

pic_status pic_link_attention_ror(const void* q, const float* row_table, const int32_t* rows,
                                  const int32_t* row_off, const void* k_pool, const void* v_pool,
                                  int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                                  const int32_t* page_tab, const float* rot_table, int64_t n_tab,
                                  const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                                  int32_t Hkv, int32_t d, float scale, void* out, void* ws, size_t ws_bytes,
                                  int32_t* err_flag, pic_stream_t stream) {
  const pic_status st = check_attention_args(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, dtype, pages,
                                             page_off, n_req, n_rows, Hq, Hkv, d, scale, out, err_flag);
  if (st != PIC_OK) return st;
  if (n_tab < 0) return PIC_ERR_INVALID;
  if (!tc_shape(dtype, Hq, Hkv, d)) return PIC_ERR_UNSUPPORTED;
  if (n_req == 0 || n_rows == 0) return PIC_OK;
  if (!page_tab || (n_tab > 0 && !rot_table) || (reinterpret_cast<uintptr_t>(rot_table) & 15)) return PIC_ERR_INVALID;
  const WsLayout L = ws_layout(n_rows, n_req, Hq / Hkv, Hkv, d);
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PIC_ERR_WORKSPACE;
  return launch_tc(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, pages, page_off, n_req, Hq, Hkv, scale,
                   out, static_cast<uint8_t*>(ws), L, kAllSms, kMaxSplitUnits, err_flag, (cudaStream_t)stream,
                   page_tab, rot_table, n_tab);
}

pic_status pic_selftest_umma(const void* a, const void* b, float* d_kmajor, float* d_mnmajor, float* d_tmem_a,
                             int32_t* err_flag, pic_stream_t stream) {
  if (!a || !b || !d_kmajor || !d_mnmajor || !d_tmem_a || !err_flag) return PIC_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(a) & 15) || (reinterpret_cast<uintptr_t>(b) & 15)) return PIC_ERR_INVALID;
  CUtensorMap bmap;
  if (!encode_pages(&bmap, b, 128)) return PIC_ERR_CUDA;
  const int smem = 2 * kOpBytes + 64 + 1024;
  if (cudaFuncSetAttribute(selftest_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return PIC_ERR_CUDA;
  selftest_umma_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(bmap, static_cast<const bf16*>(a), d_kmajor,
                                                                d_mnmajor, d_tmem_a, err_flag);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

pic_status pic_selftest_umma_pair(const void* a, const void* b, const void* v, float* d_s, float* d_pv,
                                  int32_t* info, int32_t* err_flag, pic_stream_t stream) {
  if (!a || !b || !v || !d_s || !d_pv || !info || !err_flag) return PIC_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(v)) & 15)
    return PIC_ERR_INVALID;
  const int smem = kPairTestSmem + 1024;
  if (cudaFuncSetAttribute(selftest_umma_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return PIC_ERR_CUDA;
  selftest_umma_pair_kernel<<<2, 128, smem, (cudaStream_t)stream>>>(
      static_cast<const bf16*>(a), static_cast<const bf16*>(b), static_cast<const bf16*>(v), d_s, d_pv, info,
      err_flag);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------------ fixed-scratch variant
// pic_link_attention_noalloc: the tensor-core attention with its planning and
// merge scratch in one statically sized device array instead of a caller
// workspace.  It runs the same kernels as pic_link_attention; it gives the
// planner a smaller split budget (units balanced for kFixedSplitSms SMs, at most
// kFixedSplitUnits = 60 extra units) so that the scratch a call needs stays small.

constexpr size_t kFixedScratchBytes = (size_t)PIC_NOALLOC_SCRATCH_BYTES;

// Held by every GPU that loads this library, until the process exits.
static __device__ __align__(256) uint8_t pic_fixed_scratch[kFixedScratchBytes];

namespace pic {
namespace {

constexpr int kFixedSplitSms = 10;    // the planner balances for 10 SMs' worth of units ...
constexpr int kFixedSplitUnits = 60;  // ... and adds at most 60 to the fixed scratch
static_assert(kFixedSplitUnits == 60 && kFixedSplitUnits <= kUnitsPerSm * kFixedSplitSms, "the split cap pic.h states");
constexpr int kMaxDevices = 256;

std::mutex g_fixed_mu;
void* g_fixed_addr[kMaxDevices];  // device address of pic_fixed_scratch, per device ordinal

// Device address of the scratch on the current device.  Looked up once per
// device (cudaGetSymbolAddress with that device current) and kept for the life of
// the process, so the library must not be used across a cudaDeviceReset (the
// array may move when the device code is loaded again).  The lookup also loads
// this file's device code on the device if that has not happened yet, which is
// when the array is reserved.  Host code must never hand the host-side name
// pic_fixed_scratch to a kernel.
void* fixed_scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_fixed_mu);
  if (g_fixed_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, pic_fixed_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_fixed_addr[dev] = p;
  }
  return g_fixed_addr[dev];
}

WsLayout fixed_layout(int64_t n_rows, int32_t n_req, int32_t G, int32_t Hkv, int32_t d) {
  return ws_layout_with(n_rows, n_req, G, Hkv, d, kFixedSplitUnits, 0);
}

}  // namespace
}  // namespace pic

extern "C" pic_status pic_link_attention_noalloc(const void* q, const float* row_table, const int32_t* rows,
                                                 const int32_t* row_off, const void* k_pool, const void* v_pool,
                                                 int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                                                 const int32_t* page_off, int32_t n_req, int64_t n_rows,
                                                 int32_t Hq, int32_t Hkv, int32_t d, float scale, void* out,
                                                 int32_t* err_flag, pic_stream_t stream) {
  using namespace pic;
  if (n_req < 0 || n_rows < 0 || num_blocks < 0 || Hkv < 1 || Hq < 1 || Hq % Hkv || d < 2 || d > 256 ||
      (d & 1) || !(scale > 0.f))
    return PIC_ERR_INVALID;
  if (dtype != PIC_BF16 && dtype != PIC_FP32) return PIC_ERR_INVALID;
  // A call without rows is the warm-up: it makes the current device load the
  // library's device code (reserving the array) and looks up the array's address,
  // so that neither happens later, after the caller has reserved HBM.
  if (n_req == 0 || n_rows == 0) return fixed_scratch_address() != nullptr ? PIC_OK : PIC_ERR_CUDA;
  const bool tc = tc_shape(dtype, Hq, Hkv, d);
  // size check first: a call that needs more scratch than the array holds is refused before anything else
  if (tc && fixed_layout(n_rows, n_req, Hq / Hkv, Hkv, d).total > kFixedScratchBytes) return PIC_ERR_WORKSPACE;
  const pic_status st = check_attention_args(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, dtype, pages,
                                             page_off, n_req, n_rows, Hq, Hkv, d, scale, out, err_flag);
  if (st != PIC_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  // the SIMT path uses no scratch at all
  if (!tc)
    return launch_attention_simt(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, dtype, pages, page_off,
                                 n_req, n_rows, Hq, Hkv, d, scale, out, s);
  uint8_t* w = static_cast<uint8_t*>(fixed_scratch_address());
  if (w == nullptr) return PIC_ERR_CUDA;
  // Nothing in the scratch has to start at zero: the planner rewrites the header,
  // tile and unit lists on every call, and partials are written before they are read.
  return launch_tc(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, pages, page_off, n_req, Hq, Hkv, scale,
                   out, w, fixed_layout(n_rows, n_req, Hq / Hkv, Hkv, d), kFixedSplitSms, kFixedSplitUnits, err_flag, s);
}
