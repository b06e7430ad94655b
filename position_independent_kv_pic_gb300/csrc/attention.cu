// Recompute-row link attention (EPIC blog review, link_legolink Step 3: the
// recomputed rows' Q, roped at their global positions, attend over the whole
// spliced K/V under the causal mask key_pos <= query_pos of the KV-cache blog's
// mask section; scale 1/sqrt(d); GQA group g = Hq/Hkv shares one KV head).
//
// Tensor-core path (bf16, d = 128): one MMA tile is M = 128 rows = g query heads
// x (128/g) recomputed rows that share KV head `kvh`.  Per 128-key tile (8 pages
// of 16 keys):  S = Q K^T (tcgen05, fp32 in TMEM) -> online softmax in registers
// (one thread per row, base-2, lazy rescale) -> P (bf16) in shared memory ->
// O += P V (tcgen05, fp32 in TMEM).  K/V pages arrive by TMA straight from the
// paged pool.  Warp roles: warp 0 issues TMA, warp 1 issues MMAs and owns TMEM,
// warps 4-7 run the softmax / correction / epilogue for TMEM lanes 0-127.
//
// Work is cut into units (tile, kvh, key-tile span).  Tiles whose key range is
// longer than the span are split; their partial (O, m, l) are merged by the LSE
// merge kernel.  Units are ordered longest first (the LPT greedy rule HYPIC uses
// for balancing segment work) and dealt round-robin to a persistent grid of one
// CTA per SM.  Key tiles beyond a tile's last row position are skipped
// (offset-causal tile skipping); rows inside the boundary tiles are masked per key.
#include <cudaTypedefs.h>

#include <mutex>

#include "pic_internal.cuh"
#include "tc_ptx.cuh"

namespace pic {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kD = 128;                 // head dim of the tensor-core path
constexpr int kM = 128;                 // rows of one MMA tile
constexpr int kKeys = 128;              // keys per key tile
constexpr int kPagesPerKt = kKeys / PIC_PAGE;
constexpr int kStages = 2;
constexpr int kThreads = 256;
constexpr int kMinSpan = 8;             // key tiles per unit, lower bound
constexpr int kUnitsPerSm = 4;          // target units per SM when splitting
constexpr int kMaxSplitUnits = 1024;    // bound on the units splitting may add
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may grow up to 2^8 before O is rescaled

constexpr int kHalfBytes = kM * 128;    // one 64-column half of a 128-row operand (16 KB)
constexpr int kOpBytes = 2 * kHalfBytes;  // 128 x 128 bf16 operand (32 KB)
constexpr int kOffQ = 0;
constexpr int kOffP = kOffQ + kOpBytes;
constexpr int kOffK = kOffP + kOpBytes;
constexpr int kOffV = kOffK + kStages * kOpBytes;
constexpr int kOffBar = kOffV + kStages * kOpBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;  // + barriers + alignment slack
constexpr uint32_t kTmemCols = 512;                // S0 | S1 | O | (unused)

constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kM, kKeys, false);
constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kM, kD, true);

struct TileMeta {
  int32_t row0, n_rows, page_begin, n_pages;  // rows [row0, row0+n_rows); pages needed (causal)
  int32_t n_kt, n_spans, part_base, req;      // key tiles; spans per head; partial slots (-1: none)
};
struct Unit {
  int32_t tile, head, kt0, kt1, part, pad0, pad1, pad2;
};
struct WsHeader {
  int32_t n_tiles, n_units, span, total_kt;
  int32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header size");

struct WsLayout {
  int64_t tiles_cap, units_cap;
  size_t off_tiles, off_units, off_ml, off_o, total;
};

WsLayout ws_layout(int64_t n_rows, int32_t n_req, int32_t G, int32_t Hkv, int32_t d) {
  WsLayout L;
  const int R = kM / G;
  L.tiles_cap = n_rows / R + n_req + 1;
  L.units_cap = L.tiles_cap * Hkv + kMaxSplitUnits;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  L.off_tiles = sizeof(WsHeader);
  L.off_units = al(L.off_tiles + L.tiles_cap * sizeof(TileMeta));
  L.off_ml = al(L.off_units + L.units_cap * sizeof(Unit));
  L.off_o = al(L.off_ml + (size_t)L.units_cap * kM * sizeof(float2));
  L.total = al(L.off_o + (size_t)L.units_cap * kM * d * sizeof(float));
  return L;
}

__device__ __forceinline__ bool page_ok(const pic_link_page& p, int64_t num_blocks) {
  return p.k_block >= 0 && p.k_block < num_blocks && p.v_block >= 0 && p.v_block < num_blocks &&
         p.lo >= 0 && p.hi <= PIC_PAGE && p.lo < p.hi;
}

// ------------------------------------------------------------------ planning
// One block.  Builds tile metadata (causal page count per tile), picks the span,
// and lists the units: full-length spans first, ordered (request, kvh, span,
// tile) so that concurrently running units read the same key range, then the
// shorter tail spans by decreasing length.
constexpr int kPlanThreads = 1024;
constexpr int kHist = 4096;

__global__ void __launch_bounds__(kPlanThreads)
plan_units_kernel(const int32_t* __restrict__ rows, const int32_t* __restrict__ row_off,
                  const pic_link_page* __restrict__ pages, const int32_t* __restrict__ page_off,
                  int n_req, int R, int Hkv, int num_sms, int64_t tiles_cap, int64_t units_cap,
                  WsHeader* hdr, TileMeta* tiles, Unit* units, int32_t* err) {
  __shared__ int s_total_kt, s_ntiles, s_part, s_hist[kHist];
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int r = 0; r < n_req; ++r) acc += ceil_div(row_off[r + 1] - row_off[r], R);
    s_ntiles = acc;
    s_total_kt = 0;
    s_part = 0;
  }
  __syncthreads();
  const int n_tiles = s_ntiles;
  if (n_tiles > tiles_cap) {
    if (threadIdx.x == 0) {
      set_err(err, PIC_ERR_RANGE);
      hdr->n_units = 0;
      hdr->n_tiles = 0;
    }
    return;
  }
  // tile metadata; request of a tile found by walking the per-request tile counts
  for (int t = threadIdx.x; t < n_tiles; t += kPlanThreads) {
    int r = 0, base = 0;
    for (;; ++r) {
      const int nt = ceil_div(row_off[r + 1] - row_off[r], R);
      if (t < base + nt) break;
      base += nt;
    }
    const int lt = t - base;
    TileMeta tm;
    tm.req = r;
    tm.row0 = row_off[r] + lt * R;
    tm.n_rows = min(R, row_off[r + 1] - tm.row0);
    const int maxpos = rows[tm.row0 + tm.n_rows - 1];
    // pages are sorted by first valid position: count those starting at or before maxpos
    int lo = page_off[r], hi = page_off[r + 1];
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      const pic_link_page p = pages[mid];
      if (p.gpos0 + p.lo <= maxpos) lo = mid + 1; else hi = mid;
    }
    tm.page_begin = page_off[r];
    tm.n_pages = lo - page_off[r];
    tm.n_kt = ceil_div(tm.n_pages, kPagesPerKt);
    tm.n_spans = 0;
    tm.part_base = -1;
    tiles[t] = tm;
    atomicAdd(&s_total_kt, tm.n_kt);
  }
  __syncthreads();
  const int64_t work = (int64_t)s_total_kt * Hkv;
  const int64_t target = min((int64_t)kUnitsPerSm * num_sms, (int64_t)kMaxSplitUnits);
  const int span = (int)max((int64_t)kMinSpan, (work + target - 1) / target);
  for (int t = threadIdx.x; t < n_tiles; t += kPlanThreads) {
    TileMeta& tm = tiles[t];
    tm.n_spans = ceil_div(tm.n_kt, span);
    if (tm.n_spans > 1) tm.part_base = atomicAdd(&s_part, tm.n_spans * Hkv);
  }
  for (int i = threadIdx.x; i < kHist; i += kPlanThreads) s_hist[i] = 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    // full spans, (request, head, span, tile) order
    int64_t u = 0;
    int tile_base = 0;
    for (int r = 0; r < n_req; ++r) {
      const int nt = ceil_div(row_off[r + 1] - row_off[r], R);
      for (int h = 0; h < Hkv; ++h) {
        for (int s = 0;; ++s) {
          bool any = false;
          for (int lt = 0; lt < nt; ++lt) {
            const TileMeta tm = tiles[tile_base + lt];
            if (tm.n_kt / span > s) {
              any = true;
              if (u < units_cap) {
                Unit un;
                un.tile = tile_base + lt; un.head = h; un.kt0 = s * span; un.kt1 = (s + 1) * span;
                un.part = (tm.n_spans > 1) ? tm.part_base + h * tm.n_spans + s : -1;
                un.pad0 = un.pad1 = un.pad2 = 0;
                units[u] = un;
              }
              ++u;
            }
          }
          if (!any) break;
        }
      }
      tile_base += nt;
    }
    // tail spans by decreasing length (counting sort on the length)
    for (int t = 0; t < n_tiles; ++t) {
      const int len = tiles[t].n_kt % span;
      if (len > 0) s_hist[min(len, kHist - 1)] += Hkv;
    }
    int64_t pos = u;
    for (int len = kHist - 1; len >= 1; --len) {
      const int c = s_hist[len];
      s_hist[len] = (int)pos;
      pos += c;
    }
    for (int t = 0; t < n_tiles; ++t) {
      const TileMeta tm = tiles[t];
      const int len = tm.n_kt % span;
      if (len == 0) continue;
      const int s = tm.n_kt / span;
      for (int h = 0; h < Hkv; ++h) {
        const int64_t idx = s_hist[min(len, kHist - 1)]++;
        if (idx < units_cap) {
          Unit un;
          un.tile = t; un.head = h; un.kt0 = s * span; un.kt1 = tm.n_kt;
          un.part = (tm.n_spans > 1) ? tm.part_base + h * tm.n_spans + s : -1;
          un.pad0 = un.pad1 = un.pad2 = 0;
          units[idx] = un;
        }
      }
    }
    if (pos > units_cap) {
      set_err(err, PIC_ERR_RANGE);
      pos = units_cap;
    }
    hdr->n_tiles = n_tiles;
    hdr->n_units = (int)pos;
    hdr->span = span;
    hdr->total_kt = s_total_kt;
  }
}

// ------------------------------------------------------------------ tcgen05 kernel
struct TcArgs {
  const bf16* q;
  const float4* row_table;
  const int32_t* rows;
  const pic_link_page* pages;
  bf16* out;
  const WsHeader* hdr;
  const TileMeta* tiles;
  const Unit* units;
  float* part_o;
  float2* part_ml;
  int32_t* err;
  int64_t num_blocks;
  int Hq, Hkv, G, R;
  float scale_log2;
};

struct Bars {
  uint64_t kfull[kStages], vfull[kStages], kvempty[kStages];
  uint64_t sfull[2], sfree[2], pfull, odone, qfull, drain;
  uint32_t tmem_base;
  int abort;
};

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

__device__ void producer_loop(const TcArgs& a, const CUtensorMap* kmap, const CUtensorMap* vmap,
                              uint8_t* smem, Bars* b, int n_units) {
  const volatile int* ab = &b->abort;
  uint32_t it = 0;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const Unit un = a.units[u];
    const TileMeta tm = a.tiles[un.tile];
    const int page_end = tm.page_begin + tm.n_pages;
    for (int kt = un.kt0; kt < un.kt1; ++kt, ++it) {
      const int st = it % kStages;
      const uint32_t ph = (it / kStages) & 1;
      if (!tc::mbar_wait(&b->kvempty[st], ph ^ 1, ab, kWaitLimitNs)) { fail(b, a.err); return; }
      int kb[kPagesPerKt], vb[kPagesPerKt];
      uint32_t bytes = 0;
#pragma unroll
      for (int j = 0; j < kPagesPerKt; ++j) {
        kb[j] = -1;
        vb[j] = -1;
        const int p = tm.page_begin + kt * kPagesPerKt + j;
        if (p < page_end) {
          const pic_link_page pg = a.pages[p];
          if (page_ok(pg, a.num_blocks)) {
            kb[j] = pg.k_block;
            vb[j] = pg.v_block;
            bytes += 2 * PIC_PAGE * 64 * sizeof(bf16);  // two boxes of 16 rows x 64 columns
          } else if (pg.lo < pg.hi) {
            set_err(a.err, PIC_ERR_RANGE);
          }
        }
      }
      uint8_t* ks = smem + kOffK + st * kOpBytes;
      uint8_t* vs = smem + kOffV + st * kOpBytes;
      tc::mbar_arrive_expect_tx(&b->kfull[st], bytes);
#pragma unroll
      for (int j = 0; j < kPagesPerKt; ++j) {
        if (kb[j] < 0) continue;
        const int y = (kb[j] * a.Hkv + un.head) * PIC_PAGE;
        tc::tma_load_2d(ks + j * 2048, kmap, 0, y, &b->kfull[st]);
        tc::tma_load_2d(ks + kHalfBytes + j * 2048, kmap, 64, y, &b->kfull[st]);
      }
      tc::mbar_arrive_expect_tx(&b->vfull[st], bytes);
#pragma unroll
      for (int j = 0; j < kPagesPerKt; ++j) {
        if (vb[j] < 0) continue;
        const int y = (vb[j] * a.Hkv + un.head) * PIC_PAGE;
        tc::tma_load_2d(vs + j * 2048, vmap, 0, y, &b->vfull[st]);
        tc::tma_load_2d(vs + kHalfBytes + j * 2048, vmap, 64, y, &b->vfull[st]);
      }
    }
  }
  // every load issued has been consumed or is awaited below: wait for the last
  // loads of each stage so that no copy is in flight when the block exits
  for (uint32_t k = 0; k < kStages && k < it; ++k) {
    const uint32_t t = it - 1 - k;
    tc::mbar_wait(&b->kfull[t % kStages], (t / kStages) & 1, ab, kWaitLimitNs);
    tc::mbar_wait(&b->vfull[t % kStages], (t / kStages) & 1, ab, kWaitLimitNs);
  }
}

__device__ void mma_loop(const TcArgs& a, uint8_t* smem, Bars* b, uint32_t tmem, int n_units) {
  const volatile int* ab = &b->abort;
  const uint32_t sq = tc::smem_addr(smem + kOffQ);
  const uint32_t sp = tc::smem_addr(smem + kOffP);
  const uint32_t sk = tc::smem_addr(smem + kOffK);
  const uint32_t sv = tc::smem_addr(smem + kOffV);
  const uint32_t tmem_o = tmem + 256;
  uint32_t it = 0, uc = 0;
  auto issue_s = [&](uint32_t t) -> bool {
    const int st = t % kStages;
    const int sb = t & 1;
    if (!tc::mbar_wait(&b->kfull[st], (t / kStages) & 1, ab, kWaitLimitNs)) return false;
    if (!tc::mbar_wait(&b->sfree[sb], ((t >> 1) & 1) ^ 1, ab, kWaitLimitNs)) return false;
    tc::tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
      const uint32_t koff = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
      const uint64_t da = tc::sw128_desc(sq + koff, 16, 1024);
      const uint64_t db = tc::sw128_desc(sk + st * kOpBytes + koff, 16, 1024);
      tc::mma_bf16_ss(tmem + sb * 128, da, db, kIdescS, ks > 0 ? 1u : 0u);
    }
    tc::mma_commit(&b->sfull[sb]);
    return true;
  };
  for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++uc) {
    const Unit un = a.units[u];
    const int n = un.kt1 - un.kt0;
    if (!tc::mbar_wait(&b->qfull, uc & 1, ab, kWaitLimitNs)) { fail(b, a.err); return; }
    tc::tc_fence_after();
    if (!issue_s(it)) { fail(b, a.err); return; }
    for (int j = 0; j < n; ++j, ++it) {
      if (j + 1 < n && !issue_s(it + 1)) { fail(b, a.err); return; }
      const int st = it % kStages;
      if (!tc::mbar_wait(&b->pfull, it & 1, ab, kWaitLimitNs) ||
          !tc::mbar_wait(&b->vfull[st], (it / kStages) & 1, ab, kWaitLimitNs)) {
        fail(b, a.err);
        return;
      }
      tc::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks) {
        const uint64_t da = tc::sw128_desc(sp + (ks >> 2) * kHalfBytes + (ks & 3) * 32, 16, 1024);
        const uint64_t db = tc::sw128_desc(sv + st * kOpBytes + ks * 2048, kHalfBytes, 1024);
        tc::mma_bf16_ss(tmem_o, da, db, kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
      }
      tc::mma_commit(&b->kvempty[st]);
      tc::mma_commit(&b->odone);
    }
  }
}

// Q row m: RoPE at the row's position, rounded to bf16, stored swizzled.
__device__ __forceinline__ void write_q_row(uint8_t* qs, int m, bool ok, const bf16* __restrict__ src,
                                            const float4* __restrict__ tab) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
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
        const float2 a = __bfloat1622float2(l2[e]);
        const float2 bb = __bfloat1622float2(h2[e]);
        float y0, z0, y1, z1;
        rope_rotate(a.x, bb.x, __ldg(tab + 8 * cc + 2 * e), y0, z0);
        rope_rotate(a.y, bb.y, __ldg(tab + 8 * cc + 2 * e + 1), y1, z1);
        lo_w[e] = pack_bf16x2(y0, y1);
        hi_w[e] = pack_bf16x2(z0, z1);
      }
    }
    *reinterpret_cast<uint4*>(qs + sw128_off(m, cc)) = lo4;
    *reinterpret_cast<uint4*>(qs + kHalfBytes + sw128_off(m, cc)) = hi4;
  }
}

__device__ void softmax_loop(const TcArgs& a, uint8_t* smem, Bars* b, uint32_t tmem, int n_units) {
  const volatile int* ab = &b->abort;
  const int t = threadIdx.x - 128;  // 0..127 = TMEM lane = tile row m
  const int m = t;
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = (uint32_t)((t & ~31) << 16);
  const int hg = m / a.R, i = m % a.R;
  uint8_t* qs = smem + kOffQ;
  uint8_t* ps = smem + kOffP;
  uint32_t it = 0;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const Unit un = a.units[u];
    const TileMeta tm = a.tiles[un.tile];
    const int n = un.kt1 - un.kt0;
    const bool row_ok = i < tm.n_rows;
    const int row = tm.row0 + (row_ok ? i : 0);
    const int p_row = a.rows[tm.row0 + (row_ok ? i : tm.n_rows - 1)];
    const int hq = un.head * a.G + hg;
    write_q_row(qs, m, row_ok, a.q + ((int64_t)row * a.Hq + hq) * kD, a.row_table + (int64_t)row * (kD / 2));
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&b->qfull);

    float m_ref = -INFINITY, l = 0.f;
    const int page_end = tm.page_begin + tm.n_pages;
    for (int j = 0; j < n; ++j, ++it) {
      const int sb = it & 1;
      const int st = it % kStages;
      if (!tc::mbar_wait(&b->sfull[sb], (it >> 1) & 1, ab, kWaitLimitNs)) { fail(b, a.err); return; }
      tc::tc_fence_after();
      uint32_t sraw[kKeys];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(tmem + lane_base + sb * 128 + c * 32, sraw + c * 32);
      tc::tmem_ld_wait();
      float s[kKeys];
#pragma unroll
      for (int c = 0; c < kKeys; ++c) s[c] = u2f(sraw[c]);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&b->sfree[sb]);

      // key-tile pages: valid slots and positions
      int g0[kPagesPerKt], plo[kPagesPerKt], phi[kPagesPerKt];
      bool tile_full = true;
      const int pbase = tm.page_begin + (un.kt0 + j) * kPagesPerKt;
#pragma unroll
      for (int jj = 0; jj < kPagesPerKt; ++jj) {
        g0[jj] = 0; plo[jj] = 0; phi[jj] = 0;
        if (pbase + jj < page_end) {
          const pic_link_page pg = a.pages[pbase + jj];
          if (page_ok(pg, a.num_blocks)) { g0[jj] = pg.gpos0; plo[jj] = pg.lo; phi[jj] = pg.hi; }
        }
        tile_full = tile_full && plo[jj] == 0 && phi[jj] == PIC_PAGE;
      }
      const bool row_needs_mask = !(tile_full && g0[kPagesPerKt - 1] + PIC_PAGE - 1 <= p_row);
      if (__any_sync(0xffffffffu, row_needs_mask)) {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          const int jj = c >> 4, sl = c & 15;
          const bool ok = sl >= plo[jj] && sl < phi[jj] && g0[jj] + sl <= p_row;
          s[c] = ok ? s[c] : -INFINITY;
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) mx = fmaxf(mx, s[c]);
      const float mt = mx * a.scale_log2;
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_ref + kRescaleThreshold) {
        alpha = tc::ex2(m_ref - mt);
        resc = (m_ref != -INFINITY);
        l *= alpha;
        m_ref = mt;
      }
      const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
      uint32_t pk[kKeys / 2];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kKeys / 2; ++c) {
        const float p0 = tc::ex2(fmaf(s[2 * c], a.scale_log2, -mu));
        const float p1 = tc::ex2(fmaf(s[2 * c + 1], a.scale_log2, -mu));
        rs += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l += rs;
      // the previous P.V must be done before P is overwritten or O is rescaled
      if (j > 0 && !tc::mbar_wait(&b->odone, (it - 1) & 1, ab, kWaitLimitNs)) { fail(b, a.err); return; }
      tc::tc_fence_after();
      if (__any_sync(0xffffffffu, resc)) {
        const float f = resc ? alpha : 1.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(tmem + 256 + lane_base + c * 32, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) r[x] = f2u(u2f(r[x]) * f);
          tc::tmem_st32(tmem + 256 + lane_base + c * 32, r);
        }
        tc::tmem_st_wait();
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint4 v = make_uint4(pk[h * 32 + cc * 4], pk[h * 32 + cc * 4 + 1], pk[h * 32 + cc * 4 + 2],
                                     pk[h * 32 + cc * 4 + 3]);
          *reinterpret_cast<uint4*>(ps + h * kHalfBytes + sw128_off(m, cc)) = v;
        }
      // V rows of slots that hold no valid key are zeroed (masked keys get
      // weight 0, and 0 * V must stay 0 even if the slot holds stale bits)
      if (!tile_full) {
        if (!tc::mbar_wait(&b->vfull[st], (it / kStages) & 1, ab, kWaitLimitNs)) { fail(b, a.err); return; }
        uint8_t* vs = smem + kOffV + st * kOpBytes;
        for (int idx = t; idx < kPagesPerKt * PIC_PAGE * 2 * 8; idx += 128) {
          const int cc = idx & 7, h = (idx >> 3) & 1, sl = (idx >> 4) & 15, jj = idx >> 8;
          int lo_j = 0, hi_j = 0;
#pragma unroll
          for (int q = 0; q < kPagesPerKt; ++q)
            if (q == jj) { lo_j = plo[q]; hi_j = phi[q]; }
          if (sl < lo_j || sl >= hi_j)
            *reinterpret_cast<uint4*>(vs + h * kHalfBytes + (jj * PIC_PAGE + sl) * 128 + cc * 16) =
                make_uint4(0, 0, 0, 0);
        }
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&b->pfull);
    }
    // epilogue: O / l
    if (!tc::mbar_wait(&b->odone, (it - 1) & 1, ab, kWaitLimitNs)) { fail(b, a.err); return; }
    tc::tc_fence_after();
    uint32_t oraw[kD];
#pragma unroll
    for (int c = 0; c < 4; ++c) tc::tmem_ld32(tmem + 256 + lane_base + c * 32, oraw + c * 32);
    tc::tmem_ld_wait();
    float o[kD];
#pragma unroll
    for (int c = 0; c < kD; ++c) o[c] = u2f(oraw[c]);
    tc::tc_fence_before();
    if (row_ok) {
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      if (un.part < 0) {
        uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)row * a.Hq + hq) * kD);
#pragma unroll
        for (int c = 0; c < kD / 8; ++c)
          dst[c] = make_uint4(pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv),
                              pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                              pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                              pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
      } else {
        float4* dst = reinterpret_cast<float4*>(a.part_o + ((int64_t)un.part * kM + m) * kD);
#pragma unroll
        for (int c = 0; c < kD / 4; ++c)
          dst[c] = make_float4(o[4 * c] * inv, o[4 * c + 1] * inv, o[4 * c + 2] * inv, o[4 * c + 3] * inv);
        a.part_ml[(int64_t)un.part * kM + m] = make_float2(m_ref, l);
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
link_attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const TcArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  Bars* b = reinterpret_cast<Bars*>(smem + kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&b->kfull[s], 1);
      tc::mbar_init(&b->vfull[s], 1);
      tc::mbar_init(&b->kvempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&b->sfull[s], 1);
      tc::mbar_init(&b->sfree[s], 4);
    }
    tc::mbar_init(&b->pfull, 4);
    tc::mbar_init(&b->odone, 1);
    tc::mbar_init(&b->qfull, 4);
    tc::mbar_init(&b->drain, 1);
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

  if (warp == 0) {
    if (lane == 0) producer_loop(a, &kmap, &vmap, smem, b, n_units);
  } else if (warp == 1) {
    if (lane == 0) {
      mma_loop(a, smem, b, tmem, n_units);
      // every MMA this thread issued completes before TMEM is released (also on abort)
      tc::mma_commit(&b->drain);
      const int no_abort = 0;
      tc::mbar_wait(&b->drain, 0, &no_abort, kWaitLimitNs);
    }
  } else if (warp >= 4) {
    softmax_loop(a, smem, b, tmem, n_units);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ LSE merge
// One block per (tile, kvh); threads = rows x 16-dim chunks.  Combines the
// per-span partials (O_s normalised by l_s, base-2 max m_s, l_s):
//   O = sum_s 2^(m_s - M) l_s O_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(256)
merge_kernel(const WsHeader* __restrict__ hdr, const TileMeta* __restrict__ tiles,
             const float* __restrict__ part_o, const float2* __restrict__ part_ml, bf16* __restrict__ out,
             int Hq, int Hkv, int G, int R) {
  const int th = blockIdx.x;
  const int tile = th / Hkv, head = th % Hkv;
  if (tile >= hdr->n_tiles) return;
  const TileMeta tm = tiles[tile];
  if (tm.n_spans <= 1) return;
  for (int idx = threadIdx.x; idx < kM * (kD / 16); idx += blockDim.x) {
    const int m = idx / (kD / 16), c = idx % (kD / 16);
    const int hg = m / R, i = m % R;
    if (i >= tm.n_rows) continue;
    const int base = tm.part_base + head * tm.n_spans;
    float M = -INFINITY;
    for (int s = 0; s < tm.n_spans; ++s) {
      const float2 ml = part_ml[(int64_t)(base + s) * kM + m];
      if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    float acc[16], den = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    for (int s = 0; s < tm.n_spans; ++s) {
      const float2 ml = part_ml[(int64_t)(base + s) * kM + m];
      if (!(ml.y > 0.f)) continue;
      const float w = ml.y * exp2f(ml.x - M);
      den += w;
      const float4* src = reinterpret_cast<const float4*>(part_o + ((int64_t)(base + s) * kM + m) * kD + c * 16);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 v = src[e];
        acc[4 * e] += w * v.x; acc[4 * e + 1] += w * v.y; acc[4 * e + 2] += w * v.z; acc[4 * e + 3] += w * v.w;
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(out + ((int64_t)(tm.row0 + i) * Hq + head * G + hg) * kD + c * 16);
    dst[0] = make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                        pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
    dst[1] = make_uint4(pack_bf16x2(acc[8] * inv, acc[9] * inv), pack_bf16x2(acc[10] * inv, acc[11] * inv),
                        pack_bf16x2(acc[12] * inv, acc[13] * inv), pack_bf16x2(acc[14] * inv, acc[15] * inv));
  }
}

// ------------------------------------------------------------------ SIMT kernel
// fp32 pools and bf16 shapes outside the tensor-core path.  One warp per
// (recomputed row, query head); lanes take 32 key slots (two pages) at a time
// for the scores and then the head dimensions for P.V.  Online softmax in fp32.
constexpr int kSimtMaxDimsPerLane = 8;  // d <= 256

template <typename T>
__global__ void __launch_bounds__(128)
link_attn_simt_kernel(const T* __restrict__ q, const float4* __restrict__ row_table,
                      const int32_t* __restrict__ rows, const int32_t* __restrict__ row_off,
                      const T* __restrict__ kpool, const T* __restrict__ vpool, int64_t num_blocks,
                      const pic_link_page* __restrict__ pages, const int32_t* __restrict__ page_off,
                      int n_req, int Hq, int Hkv, int d, float scale, T* __restrict__ out) {
  extern __shared__ float qs_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t i = blockIdx.x;
  const int h = blockIdx.y * 4 + warp;
  if (h >= Hq) return;
  float* qs = qs_all + warp * d;
  int lo = 0, hi = n_req;  // request of row i: last r with row_off[r] <= i
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (row_off[mid] <= i) lo = mid; else hi = mid;
  }
  const int r = lo;
  const int p = rows[i];
  const int G = Hq / Hkv, kvh = h / G, half = d / 2;
  const T* qrow = q + (i * Hq + h) * (int64_t)d;
  for (int j = lane; j < half; j += 32) {
    float ya, yb;
    rope_rotate(to_f32(qrow[j]), to_f32(qrow[j + half]), row_table[i * half + j], ya, yb);
    qs[j] = to_f32(from_f32<T>(ya));
    qs[j + half] = to_f32(from_f32<T>(yb));
  }
  __syncwarp();
  float acc[kSimtMaxDimsPerLane];
#pragma unroll
  for (int e = 0; e < kSimtMaxDimsPerLane; ++e) acc[e] = 0.f;
  float m_run = -INFINITY, l = 0.f;
  const int pb = page_off[r], pe = page_off[r + 1];
  for (int pp = pb; pp < pe; pp += 2) {
    const pic_link_page first = pages[pp];
    if (first.gpos0 + first.lo > p) break;  // pages are sorted by first valid position
    const int pg = pp + (lane >> 4), sl = lane & 15;
    bool valid = false;
    int kb = 0, vb = 0;
    if (pg < pe) {
      const pic_link_page e = pages[pg];
      valid = e.k_block >= 0 && e.k_block < num_blocks && e.v_block >= 0 && e.v_block < num_blocks &&
              sl >= e.lo && sl < e.hi && e.gpos0 + sl <= p;
      kb = e.k_block;
      vb = e.v_block;
    }
    float sc = -INFINITY;
    if (valid) {
      const T* krow = kpool + (((int64_t)kb * Hkv + kvh) * PIC_PAGE + sl) * d;
      float acc_s = 0.f;
      for (int x = 0; x < d; ++x) acc_s = fmaf(qs[x], to_f32(krow[x]), acc_s);
      sc = acc_s * scale;
    }
    float mx = sc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (mx == -INFINITY) continue;
    const float m_new = fmaxf(m_run, mx);
    const float alpha = (m_run == -INFINITY) ? 0.f : __expf(m_run - m_new);
    const float pl = valid ? __expf(sc - m_new) : 0.f;
    float ps = pl;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    l = l * alpha + ps;
#pragma unroll
    for (int e = 0; e < kSimtMaxDimsPerLane; ++e) acc[e] *= alpha;
    for (int src = 0; src < 32; ++src) {
      const float w = __shfl_sync(0xffffffffu, pl, src);
      const int vbs = __shfl_sync(0xffffffffu, vb, src);
      if (w == 0.f) continue;
      const T* vrow = vpool + (((int64_t)vbs * Hkv + kvh) * PIC_PAGE + (src & 15)) * d;
#pragma unroll
      for (int e = 0; e < kSimtMaxDimsPerLane; ++e) {
        const int x = lane + 32 * e;
        if (x < d) acc[e] = fmaf(w, to_f32(vrow[x]), acc[e]);
      }
    }
    m_run = m_new;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  T* orow = out + (i * Hq + h) * (int64_t)d;
#pragma unroll
  for (int e = 0; e < kSimtMaxDimsPerLane; ++e) {
    const int x = lane + 32 * e;
    if (x < d) orow[x] = from_f32<T>(acc[e] * inv);
  }
}

// ------------------------------------------------------------------ self-test
__global__ void __launch_bounds__(128, 1)
selftest_umma_kernel(const __grid_constant__ CUtensorMap bmap, const bf16* __restrict__ a, float* dk,
                     float* dmn, int32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sa = smem;
  uint8_t* sbm = smem + kOpBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kOpBytes);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  volatile int* ab = reinterpret_cast<volatile int*>(bars + 3);
  const int t = threadIdx.x, warp = t >> 5;
  if (t == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    *ab = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, 256);
    tc::tmem_relinquish();
  }
  // A row t, swizzled, 128-byte rows in two 64-column halves
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
  if (t == 0) {
    tc::mbar_arrive_expect_tx(&bars[0], kOpBytes);
    for (int j = 0; j < 8; ++j) {
      tc::tma_load_2d(sbm + j * 2048, &bmap, 0, j * 16, &bars[0]);
      tc::tma_load_2d(sbm + kHalfBytes + j * 2048, &bmap, 64, j * 16, &bars[0]);
    }
    bool ok = tc::mbar_wait(&bars[0], 0, ab, kWaitLimitNs);
    if (ok) {
      tc::tc_fence_after();
      const uint32_t sa_a = tc::smem_addr(sa), sb_a = tc::smem_addr(sbm);
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
        tc::mma_bf16_ss(tmem, tc::sw128_desc(sa_a + koff, 16, 1024), tc::sw128_desc(sb_a + koff, 16, 1024),
                        kIdescS, ks > 0);
      }
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
        tc::mma_bf16_ss(tmem + 128, tc::sw128_desc(sa_a + koff, 16, 1024),
                        tc::sw128_desc(sb_a + ks * 2048, kHalfBytes, 1024), kIdescPV, ks > 0);
      }
      tc::mma_commit(&bars[1]);
    } else {
      set_err(err, PIC_ERR_TIMEOUT);
      *ab = 1;
    }
  }
  __syncthreads();
  if (!*ab && tc::mbar_wait(&bars[1], 0, ab, kWaitLimitNs)) {
    tc::tc_fence_after();
    const uint32_t lb = (uint32_t)((warp * 32) << 16);
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tc::tmem_ld32(tmem + lb + c * 32, r);
      tc::tmem_ld_wait();
      for (int x = 0; x < 32; ++x) dk[t * 128 + c * 32 + x] = u2f(r[x]);
      tc::tmem_ld32(tmem + 128 + lb + c * 32, r);
      tc::tmem_ld_wait();
      for (int x = 0; x < 32; ++x) dmn[t * 128 + c * 32 + x] = u2f(r[x]);
    }
  } else if (t == 0) {
    set_err(err, PIC_ERR_TIMEOUT);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 256);
  }
}

// ------------------------------------------------------------------ host side
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

// 2-D view [rows][128] bf16 of a buffer, boxes of 16 rows x 64 columns, 128-byte swizzle.
bool encode_rows128(CUtensorMap* map, const void* base, uint64_t rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {128 * sizeof(bf16)};
  cuuint32_t box[2] = {64, PIC_PAGE};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_shape(pic_dtype dt, int Hq, int Hkv, int d) {
  if (dt != PIC_BF16 || d != kD || Hkv < 1 || Hq % Hkv) return false;
  const int G = Hq / Hkv;
  return G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
}

}  // namespace
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
  if (n_req < 0 || n_rows < 0 || num_blocks < 0 || Hkv < 1 || Hq < 1 || Hq % Hkv || d < 2 || d > 256 ||
      (d & 1) || !(scale > 0.f))
    return PIC_ERR_INVALID;
  if (dtype != PIC_BF16 && dtype != PIC_FP32) return PIC_ERR_INVALID;
  if (n_req == 0 || n_rows == 0) return PIC_OK;
  if (!q || !row_table || !rows || !row_off || !k_pool || !v_pool || !pages || !page_off || !out || !err_flag)
    return PIC_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  const int G = Hq / Hkv;
  if (tc_shape(dtype, Hq, Hkv, d)) {
    const WsLayout L = ws_layout(n_rows, n_req, G, Hkv, d);
    if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PIC_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(k_pool) & 15) || (reinterpret_cast<uintptr_t>(v_pool) & 15) ||
        (reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
      return PIC_ERR_INVALID;
    const uint64_t pool_rows = (uint64_t)num_blocks * Hkv * PIC_PAGE;
    if (pool_rows == 0 || pool_rows > (uint64_t)INT32_MAX) return PIC_ERR_INVALID;
    CUtensorMap kmap, vmap;
    if (!encode_rows128(&kmap, k_pool, pool_rows) || !encode_rows128(&vmap, v_pool, pool_rows)) return PIC_ERR_CUDA;
    uint8_t* w = static_cast<uint8_t*>(ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
    TileMeta* tiles = reinterpret_cast<TileMeta*>(w + L.off_tiles);
    Unit* units = reinterpret_cast<Unit*>(w + L.off_units);
    float2* part_ml = reinterpret_cast<float2*>(w + L.off_ml);
    float* part_o = reinterpret_cast<float*>(w + L.off_o);
    const int sms = num_sms_of_current_device();
    plan_units_kernel<<<1, kPlanThreads, 0, s>>>(rows, row_off, pages, page_off, n_req, kM / G, Hkv, sms,
                                                  L.tiles_cap, L.units_cap, hdr, tiles, units, err_flag);
    if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
    if (cudaFuncSetAttribute(link_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return PIC_ERR_CUDA;
    TcArgs a;
    a.q = static_cast<const bf16*>(q);
    a.row_table = reinterpret_cast<const float4*>(row_table);
    a.rows = rows;
    a.pages = pages;
    a.out = static_cast<bf16*>(out);
    a.hdr = hdr;
    a.tiles = tiles;
    a.units = units;
    a.part_o = part_o;
    a.part_ml = part_ml;
    a.err = err_flag;
    a.num_blocks = num_blocks;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = G;
    a.R = kM / G;
    a.scale_log2 = scale * 1.4426950408889634f;
    const int64_t grid = L.units_cap < sms ? L.units_cap : sms;
    link_attn_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(kmap, vmap, a);
    if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
    merge_kernel<<<(unsigned)(L.tiles_cap * Hkv), 256, 0, s>>>(hdr, tiles, part_o, part_ml, a.out, Hq, Hkv, G,
                                                               kM / G);
    return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
  }
  // SIMT path
  const size_t el = (dtype == PIC_BF16) ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(row_table) & 15) || ((size_t)d * el) % 4) return PIC_ERR_INVALID;
  if (n_rows > INT32_MAX) return PIC_ERR_INVALID;
  dim3 grid((unsigned)n_rows, (unsigned)((Hq + 3) / 4));
  const size_t smem = 4 * d * sizeof(float);
  if (dtype == PIC_BF16)
    link_attn_simt_kernel<bf16><<<grid, 128, smem, s>>>(
        static_cast<const bf16*>(q), reinterpret_cast<const float4*>(row_table), rows, row_off,
        static_cast<const bf16*>(k_pool), static_cast<const bf16*>(v_pool), num_blocks, pages, page_off, n_req, Hq,
        Hkv, d, scale, static_cast<bf16*>(out));
  else
    link_attn_simt_kernel<float><<<grid, 128, smem, s>>>(
        static_cast<const float*>(q), reinterpret_cast<const float4*>(row_table), rows, row_off,
        static_cast<const float*>(k_pool), static_cast<const float*>(v_pool), num_blocks, pages, page_off, n_req,
        Hq, Hkv, d, scale, static_cast<float*>(out));
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

pic_status pic_selftest_umma(const void* a, const void* b, float* d_kmajor, float* d_mnmajor, int32_t* err_flag,
                             pic_stream_t stream) {
  if (!a || !b || !d_kmajor || !d_mnmajor || !err_flag) return PIC_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(a) & 15) || (reinterpret_cast<uintptr_t>(b) & 15)) return PIC_ERR_INVALID;
  CUtensorMap bmap;
  if (!encode_rows128(&bmap, b, 128)) return PIC_ERR_CUDA;
  const int smem = 2 * kOpBytes + 64 + 1024;
  if (cudaFuncSetAttribute(selftest_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return PIC_ERR_CUDA;
  selftest_umma_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(bmap, static_cast<const bf16*>(a), d_kmajor,
                                                                d_mnmajor, err_flag);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------------ fixed-scratch variant
// pic_link_attention_noalloc: the tensor-core attention with its planning and
// merge scratch in one statically sized device array instead of a caller
// workspace.  It calls the same kernels as pic_link_attention; it gives the
// planner a smaller split budget (4 extra units per SM for at most 32 SMs) so
// that the scratch a call needs stays small.

constexpr size_t kFixedScratchBytes = (size_t)PIC_NOALLOC_SCRATCH_BYTES;

// Held by every GPU that loads this library, until the process exits.
static __device__ __align__(256) uint8_t pic_fixed_scratch[kFixedScratchBytes];

namespace pic {
namespace {

constexpr int kFixedSplitSms = 32;
constexpr int kMaxDevices = 256;

std::mutex g_fixed_mu;
void* g_fixed_addr[kMaxDevices];  // device address of pic_fixed_scratch, per device ordinal

// Device address of the scratch on the current device.  Looked up once per
// device (cudaGetSymbolAddress with that device current); host code must never
// hand the host-side name pic_fixed_scratch to a kernel.
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
  WsLayout L = ws_layout(n_rows, n_req, G, Hkv, d);
  const int64_t units_cap = L.tiles_cap * Hkv + (int64_t)kUnitsPerSm * kFixedSplitSms;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  L.units_cap = units_cap;
  L.off_ml = al(L.off_units + units_cap * sizeof(Unit));
  L.off_o = al(L.off_ml + (size_t)units_cap * kM * sizeof(float2));
  L.total = al(L.off_o + (size_t)units_cap * kM * d * sizeof(float));
  return L;
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
  if (n_req == 0 || n_rows == 0) return PIC_OK;
  const bool tc = tc_shape(dtype, Hq, Hkv, d);
  const int G = Hq / Hkv;
  // size check first: a call that needs more scratch than the array holds is refused before anything else
  if (tc && fixed_layout(n_rows, n_req, G, Hkv, d).total > kFixedScratchBytes) return PIC_ERR_WORKSPACE;
  if (!q || !row_table || !rows || !row_off || !k_pool || !v_pool || !pages || !page_off || !out || !err_flag)
    return PIC_ERR_INVALID;
  // the SIMT path uses no scratch at all
  if (!tc)
    return pic_link_attention(q, row_table, rows, row_off, k_pool, v_pool, num_blocks, dtype, pages, page_off,
                              n_req, n_rows, Hq, Hkv, d, scale, out, nullptr, 0, err_flag, stream);
  const WsLayout L = fixed_layout(n_rows, n_req, G, Hkv, d);
  if ((reinterpret_cast<uintptr_t>(k_pool) & 15) || (reinterpret_cast<uintptr_t>(v_pool) & 15) ||
      (reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
    return PIC_ERR_INVALID;
  const uint64_t pool_rows = (uint64_t)num_blocks * Hkv * PIC_PAGE;
  if (pool_rows == 0 || pool_rows > (uint64_t)INT32_MAX) return PIC_ERR_INVALID;
  uint8_t* w = static_cast<uint8_t*>(fixed_scratch_address());
  if (w == nullptr) return PIC_ERR_CUDA;
  CUtensorMap kmap, vmap;
  if (!encode_rows128(&kmap, k_pool, pool_rows) || !encode_rows128(&vmap, v_pool, pool_rows)) return PIC_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  // Nothing in the scratch has to start at zero: the planner rewrites the header,
  // tile and unit lists on every call, and partials are written before they are read.
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  TileMeta* tiles = reinterpret_cast<TileMeta*>(w + L.off_tiles);
  Unit* units = reinterpret_cast<Unit*>(w + L.off_units);
  float2* part_ml = reinterpret_cast<float2*>(w + L.off_ml);
  float* part_o = reinterpret_cast<float*>(w + L.off_o);
  const int sms = num_sms_of_current_device();
  const int split_sms = sms < kFixedSplitSms ? sms : kFixedSplitSms;
  plan_units_kernel<<<1, kPlanThreads, 0, s>>>(rows, row_off, pages, page_off, n_req, kM / G, Hkv, split_sms,
                                                L.tiles_cap, L.units_cap, hdr, tiles, units, err_flag);
  if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  if (cudaFuncSetAttribute(link_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess)
    return PIC_ERR_CUDA;
  TcArgs a;
  a.q = static_cast<const bf16*>(q);
  a.row_table = reinterpret_cast<const float4*>(row_table);
  a.rows = rows;
  a.pages = pages;
  a.out = static_cast<bf16*>(out);
  a.hdr = hdr;
  a.tiles = tiles;
  a.units = units;
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.err = err_flag;
  a.num_blocks = num_blocks;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.R = kM / G;
  a.scale_log2 = scale * 1.4426950408889634f;
  const int64_t grid = L.units_cap < sms ? L.units_cap : sms;
  link_attn_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(kmap, vmap, a);
  if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  merge_kernel<<<(unsigned)(L.tiles_cap * Hkv), 256, 0, s>>>(hdr, tiles, part_o, part_ml, a.out, Hq, Hkv, G, kM / G);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}
