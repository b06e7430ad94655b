// Decode after link: one new query row per request attends over the request's
// linked paged cache (EPIC review: the query and the decode tokens are the ones
// that gather information across chunks; "KV cache from scratch": a single-token
// decode reads the whole cache once per step).  The step is bound by HBM: every
// cached K and V row is read once, and g query heads share each row.
//
// Split-KV: CTA (split, KV head, request) walks one span of the request's pages.
// A producer thread moves each page's K and V (4 KB each, one swizzled TMA box
// apiece, the link attention's page layout) into a ring of shared-memory stages;
// four consumer warps take the stages in turn, each keeping an online softmax for
// the g query heads of the KV head.  A page is two small contractions per warp —
// S = Q K^T (g heads x 16 keys x 128) and O += P V (g heads x 16 keys x 128) —
// done with the warp-level bf16 tensor-core MMA (m16n8k16, fp32 accumulate; the g
// heads are rows 0..g-1 of the 16-row operand), operands read with ldmatrix from
// the swizzled page (conflict-free), P kept in registers between the two.  That
// is ~100 instructions per page and warp instead of ~700 on the FMA pipe, so the
// CTA streams pages at the HBM rate.  The CTA combines its warps and writes one
// partial (m, l, unnormalised o); a merge kernel combines the splits.
//
// After a rotate-on-read link (the framed page layout) the keys of a chunk stay in
// the chunk's own frame: the page's frame (its offset-table row) travels with the
// page to the consumer, and a consumer warp whose page is in another frame than the
// last one rebuilds its Q fragments rotated back by that frame's offset (RoPE(q, P)
// . R(Delta) k = R(-Delta) RoPE(q, P) . k).
#include <algorithm>

#include "pic_internal.cuh"
#include "tc_ptx.cuh"

namespace pic {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kDecD = 128;
constexpr int kDecWarps = 4;                     // consumer warps
constexpr int kDecThreads = 32 * (kDecWarps + 1);  // + the producer warp
constexpr int kDecStages = 8;                    // ring stages of one page (K and V), two per consumer warp
// A consumer warp must see every phase of its stages' barriers in order (a parity
// wait two phases ahead would pass on the older phase): warp w takes pages
// w, w + 4, .., so stage i % kDecStages must always belong to warp i % kDecWarps.
static_assert(kDecStages % kDecWarps == 0, "each stage belongs to one consumer warp");
constexpr int kPageHead = PIC_PAGE * kDecD * 2;  // bytes of one page of one KV head
constexpr int kPlanThreads = 1024;  // the planner's one block
constexpr int kMergeGroups = 8;   // thread groups of the merge, each over every 8th split
constexpr uint64_t kDecWaitNs = 2000000000ull;

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

struct DecLayout {
  int64_t ctas;  // upper bound of the decode grid
  size_t off_plan, off_desc, off_ml, off_o, total;
};

// ctas_per_sm: decode CTAs one SM holds at once.  The planner gives request r
// s_r = ceil(np_r / span) splits per KV head, with span chosen so that all splits
// fit in one wave of slots = ctas_per_sm * sms CTAs (never fewer than one split per
// (request, KV head)); so the grid is at most slots + n_req * Hkv.
DecLayout dec_layout(int n_req, int Hq, int Hkv, int sms, int ctas_per_sm) {
  DecLayout L;
  L.ctas = (int64_t)ctas_per_sm * sms + (int64_t)n_req * Hkv;
  const int G = Hq / Hkv;
  L.off_plan = 0;  // int32 [n_req + 1] first CTA of each request, int32 [n_req] splits, int32 span
  L.off_desc = al256((size_t)(2 * n_req + 2) * sizeof(int32_t));  // int4 [ctas] (request, KV head, pages)
  L.off_ml = al256(L.off_desc + (size_t)L.ctas * sizeof(int4));
  L.off_o = al256(L.off_ml + (size_t)L.ctas * G * sizeof(float2));
  L.total = al256(L.off_o + (size_t)L.ctas * G * kDecD * sizeof(float));
  return L;
}

// One block: splits per request and the first CTA of each request.
__global__ void __launch_bounds__(kPlanThreads)
decode_plan_kernel(const int32_t* __restrict__ page_off, int n_req, int Hkv, int slots, int ctas,
                   int32_t* __restrict__ first, int32_t* __restrict__ nsplit, int4* __restrict__ desc) {
  __shared__ int scratch[1024 / 32 + 1];
  __shared__ int s_span;
  const int tid = threadIdx.x;
  if (tid == 0) {
    const int64_t W = (int64_t)Hkv * page_off[n_req];  // page-heads
    const int64_t room = (int64_t)slots - (int64_t)n_req * Hkv;
    const int64_t span = room > 0 ? (W + room - 1) / room : W;
    s_span = (int)(span > 1 ? span : 1);
  }
  __syncthreads();
  const int span = s_span;
  int carry = 0;
  for (int g = 0; g < n_req; g += 1024) {
    const int r = g + tid;
    int sr = 0;
    if (r < n_req) {
      const int np = page_off[r + 1] - page_off[r];
      sr = max(1, (np + span - 1) / span);
      nsplit[r] = sr;
    }
    int tot;
    const int ex = block_exclusive_scan<1024>(sr * Hkv, scratch, &tot);
    if (r < n_req) first[r] = carry + ex;
    carry += tot;
  }
  if (tid == 0) first[n_req] = carry;
  __syncthreads();
  // one descriptor per CTA of the grid, so that a CTA starts from a single load:
  // (request, KV head, first page, end page), request -1 past the last CTA
  for (int c = tid; c < ctas; c += kPlanThreads) {
    int4 d = make_int4(-1, 0, 0, 0);
    if (c < carry) {
      int lo = 0, hi = n_req;  // the last r with first[r] <= c
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (first[mid] <= c) lo = mid; else hi = mid;
      }
      const int splits = nsplit[lo], kvh = (c - first[lo]) / splits, split = (c - first[lo]) % splits;
      const int p0 = page_off[lo], p1 = page_off[lo + 1];
      const int per = (p1 - p0 + splits - 1) / splits;
      const int pb = min(p1, p0 + split * per);
      d = make_int4(lo, kvh, pb, min(p1, pb + per));
    }
    desc[c] = d;
  }
}

// Warp-level bf16 MMA m16n8k16 with fp32 accumulate, rows 8..15 of A zero: d0, d1
// (row g = lane / 4, columns 2 (lane % 4), +1) accumulate in place; the outputs of
// the zero rows are discarded.
__device__ __forceinline__ void mma_rows8(float& d0, float& d1, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  float z0, z1;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d0), "=f"(d1), "=f"(z0), "=f"(z1)
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(d0), "f"(d1), "f"(0.f), "f"(0.f));
  asm volatile("" ::"f"(z0), "f"(z1));  // the zero rows' outputs: read by nothing
}

// Four 8x8 bf16 matrices from shared memory; lane l gives the address of row l % 8
// of matrix l / 8.  trans: each matrix transposed on the way.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset in a swizzled page (see encode_pages) of key row `key`, 16-byte
// chunk `chunk` (0..15 over the 128 columns).
__device__ __forceinline__ uint32_t swz_off(int key, int chunk) {
  const int r = key & 7;
  return (uint32_t)((key >> 3) * 2048 + (chunk >> 3) * 1024 + r * 128 + (((chunk & 7) ^ r) << 4));
}

// Named barrier (id 1) of all the block's warps, met by the producer after its last
// copy has landed and by the consumers after their last page.
__device__ __forceinline__ void ring_drained_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecThreads) : "memory");
}

template <int G>
struct DecSmem {
  // K page, V page per stage (1 KB-aligned swizzle atoms); once every copy has
  // landed and been read, the ring takes the warps' partial outputs
  union {
    uint8_t ring[kDecStages][2][kPageHead];
    float w_o[kDecWarps][G][kDecD];
  };
  uint64_t full[kDecStages], empty[kDecStages];
  uint64_t never;                // no thread ever arrives on it (failure-injection test build)
  int meta[kDecStages];          // the stage's page: valid slots lo | hi << 8, or -1 when skipped
  __nv_bfloat16 qb[G][kDecD];    // Q of the g heads, roped and rounded to bf16
  float w_m[kDecWarps][G], w_l[kDecWarps][G];
  int abort;
};

// Three CTAs per SM (registers capped at 136): the bytes in flight per SM and the
// number of consumer warps both bound the streaming rate (two CTAs were 1.7x slower
// on a 16-request batch).
// Q fragments of row g (head g of the KV head; rows >= G are padding) for the keys of
// frame `frame` (offset-table row; -1: the global frame, Q as roped): lane (g, t)
// holds columns 16 ks + 2t, +1 (qa) and 16 ks + 2t + 8, +9 (qc); column c < 64 and
// c + 64 are a RoPE pair, held by the same lane in fragments ks and ks + 4, so a
// lane rotates its own pairs: (x, y) -> (x cos + y sin, y cos - x sin) for the
// frame's angle, in fp32 (cos / sin = hi + lo parts of the table), rounded to bf16.
template <int G>
__device__ __forceinline__ void q_fragments(const __nv_bfloat16 (*qb)[kDecD], int g, int t, int frame,
                                            const float4* __restrict__ rot_tab, uint32_t* qa, uint32_t* qc) {
  const bool row = g < G;
  const int gg = row ? g : 0;
#pragma unroll
  for (int ks = 0; ks < kDecD / 32; ++ks) {
#pragma unroll
    for (int part = 0; part < 2; ++part) {  // part 0: columns 16 ks + 2t, +1; part 1: + 8
      const int c = 16 * ks + 2 * t + 8 * part;
      float x[2], y[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        x[e] = __bfloat162float(qb[gg][c + e]);
        y[e] = __bfloat162float(qb[gg][c + e + kDecD / 2]);
        if (frame >= 0) {
          const float4 cs = __ldg(rot_tab + (int64_t)frame * (kDecD / 2) + c + e);
          const float co = cs.x + cs.z, si = cs.y + cs.w;
          const float xr = fmaf(x[e], co, y[e] * si);
          y[e] = fmaf(y[e], co, -x[e] * si);
          x[e] = xr;
        }
      }
      __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]), hi = __floats2bfloat162_rn(y[0], y[1]);
      const uint32_t wl = row ? *reinterpret_cast<uint32_t*>(&lo) : 0u;
      const uint32_t wh = row ? *reinterpret_cast<uint32_t*>(&hi) : 0u;
      if (part == 0) {
        qa[ks] = wl;
        qa[ks + kDecD / 32] = wh;
      } else {
        qc[ks] = wl;
        qc[ks + kDecD / 32] = wh;
      }
    }
  }
}

template <int G>
__global__ void __launch_bounds__(kDecThreads, 3)
decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
              const bf16* __restrict__ q, const float4* __restrict__ q_table, int64_t num_blocks,
              const pic_link_page* __restrict__ pages, const int32_t* __restrict__ page_off,
              const int32_t* __restrict__ page_tab, const float4* __restrict__ rot_tab, int64_t n_tab, int n_req, int Hq,
              int Hkv, float scale_log2, const int4* __restrict__ desc, int slots, int32_t* __restrict__ first,
              int32_t* __restrict__ nsplit, float2* __restrict__ part_ml, float* __restrict__ part_o,
              int32_t* err) {
  static_assert(G <= 8, "heads of a KV head: rows 0..7 of the MMA operand");
  extern __shared__ __align__(1024) uint8_t dec_smem_raw[];
  // the swizzled stages need 1024-byte alignment
  if (tc::smem_addr(dec_smem_raw) & 1023u) {
    if (threadIdx.x == 0) set_err(err, PIC_ERR_UNSUPPORTED);
    return;
  }
  DecSmem<G>& sm = *reinterpret_cast<DecSmem<G>*>(dec_smem_raw);
  const int cta = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // (request, KV head, first page, end page) of this CTA: with few requests every
  // CTA takes the planner's split itself (one launch less; CTA 0 writes the split
  // counts the merge reads), else it reads the planner's descriptor
  int4 dsc;
  if (n_req <= kDecThreads) {
    __shared__ int s_scan[kDecThreads / 32 + 1];
    __shared__ int4 s_desc;
    const int64_t W = (int64_t)Hkv * __ldg(page_off + n_req);
    const int64_t room = (int64_t)slots - (int64_t)n_req * Hkv;
    const int span = (int)max((int64_t)1, room > 0 ? (W + room - 1) / room : W);
    const int p0r = tid < n_req ? __ldg(page_off + tid) : 0;
    const int np = tid < n_req ? __ldg(page_off + tid + 1) - p0r : 0;
    const int sr = tid < n_req ? max(1, (np + span - 1) / span) : 0;
    int total;
    const int ex = block_exclusive_scan<kDecThreads>(sr * Hkv, s_scan, &total);
    if (cta == 0 && tid < n_req) {
      first[tid] = ex;
      nsplit[tid] = sr;
    }
    if (cta == 0 && tid == 0) first[n_req] = total;
    if (tid == 0 && cta >= total) s_desc = make_int4(-1, 0, 0, 0);
    if (tid < n_req && cta >= ex && cta < ex + sr * Hkv) {
      const int split = (cta - ex) % sr, per = (np + sr - 1) / sr;
      const int pb0 = min(p0r + np, p0r + split * per);
      s_desc = make_int4(tid, (cta - ex) / sr, pb0, min(p0r + np, pb0 + per));
    }
    __syncthreads();
    dsc = s_desc;
  } else {
    dsc = desc[cta];
  }
  if (dsc.x < 0) return;  // the grid is an upper bound
  const int r = dsc.x, kvh = dsc.y, pb = dsc.z, n = max(dsc.w - dsc.z, 0);
  if (tid == 0) {
    for (int st = 0; st < kDecStages; ++st) {
      tc::mbar_init(&sm.full[st], 1);
      tc::mbar_init(&sm.empty[st], 1);
    }
    tc::mbar_init(&sm.never, 1);
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kDecWarps) {
    // ---- producer: lane 0 streams the span's pages through the ring, reading each
    // page entry one page ahead
    if (lane == 0) {
      int issued = 0;
      int n_go = n;
#ifdef PIC_INJECT_WAIT_TIMEOUT
      // Failure-injection test build only: a bounded wait on a barrier that nothing
      // arrives on runs out and reports PIC_ERR_TIMEOUT; the consumers then give up
      // on their first page and every warp reaches the drained-ring barrier.
      if (!tc::mbar_wait(&sm.never, 0, &sm.abort, PIC_INJECT_WAIT_TIMEOUT)) {
        set_err(err, PIC_ERR_TIMEOUT);
        *reinterpret_cast<volatile int*>(&sm.abort) = 1;
        n_go = 0;
      }
#endif
      int4 nxt = n > 0 ? __ldg(reinterpret_cast<const int4*>(pages) + pb) : make_int4(-1, -1, 0, 0);
      for (int i = 0; i < n_go; ++i) {
        const int st = i % kDecStages;
        const int4 pg = nxt;
        if (i + 1 < n) nxt = __ldg(reinterpret_cast<const int4*>(pages) + pb + i + 1);
        if (!tc::mbar_wait(&sm.empty[st], ((i / kDecStages) & 1) ^ 1, &sm.abort, kDecWaitNs)) {
          set_err(err, PIC_ERR_TIMEOUT);
          *reinterpret_cast<volatile int*>(&sm.abort) = 1;
          break;
        }
        const int lo = (int16_t)(pg.w & 0xffff), hi = (int16_t)(pg.w >> 16);
        const bool ok = pg.x >= 0 && pg.x < num_blocks && pg.y >= 0 && pg.y < num_blocks && lo >= 0 &&
                        hi <= PIC_PAGE && lo < hi;
        if (!ok && !(lo >= hi && lo >= 0 && hi <= PIC_PAGE)) set_err(err, PIC_ERR_RANGE);
        // the consumers read the page's slots and frame from here (published by the
        // arrival below): lo | hi << 5 | (frame + 1) << 10
        int frame = -1;
        if (ok && page_tab != nullptr) {
          frame = __ldg(page_tab + pb + i);
          if (frame >= n_tab) {
            set_err(err, PIC_ERR_RANGE);
            frame = -1;
          }
          frame = frame < 0 ? -1 : frame;
        }
        sm.meta[st] = ok ? (lo | (hi << 5) | ((frame + 1) << 10)) : -1;
        if (ok) {
          tc::mbar_arrive_expect_tx(&sm.full[st], 2 * kPageHead);
          tc::tma_load_4d(sm.ring[st][0], &kmap, 0, 0, 0, (pg.x * Hkv + kvh) * (PIC_PAGE / 8), &sm.full[st]);
          tc::tma_load_4d(sm.ring[st][1], &vmap, 0, 0, 0, (pg.y * Hkv + kvh) * (PIC_PAGE / 8), &sm.full[st]);
        } else {
          tc::mbar_arrive(&sm.full[st]);  // nothing to load: the consumer skips the page
        }
        issued = i + 1;
      }
      // no copy may be in flight when the block exits: the last arming of each stage
      const int no_abort = 0;
      for (int k = 0; k < kDecStages && k < issued; ++k) {
        const int i = issued - 1 - k;
        tc::mbar_wait(&sm.full[i % kDecStages], (i / kDecStages) & 1, &no_abort, kDecWaitNs);
      }
    }
    __syncwarp();
    ring_drained_sync();
  } else {
    // Q of the g heads roped at the row's position and rounded to bf16, as on the
    // link path's tensor-core operand; meanwhile the producer has started the copies
    for (int it = tid; it < G * kDecD / 2; it += 32 * kDecWarps) {
      const int hh = it / (kDecD / 2), i = it % (kDecD / 2);
      const bf16* src = q + ((int64_t)r * Hq + kvh * G + hh) * kDecD;
      float ya, yb;
      rope_rotate_bf16in(to_f32(src[i]), to_f32(src[i + kDecD / 2]), q_table[(int64_t)r * (kDecD / 2) + i], ya, yb);
      sm.qb[hh][i] = from_f32<bf16>(ya);
      sm.qb[hh][i + kDecD / 2] = from_f32<bf16>(yb);
    }
    asm volatile("bar.sync 2, %0;" ::"n"(32 * kDecWarps) : "memory");  // the consumer warps only
    // ---- consumers: warp w takes pages w, w + 4, ..  Lane (g, t) = (lane / 4,
    // lane % 4) holds row g (head g of the KV head; rows >= G are padding) of the
    // MMA fragments: Q at columns 16 ks + 2t, +1 and +8, +9; S at keys 2t, 2t+1 and
    // 8 + 2t, 9 + 2t; O at columns 8 nt + 2t, +1.
    const int g = lane >> 2, t = lane & 3;
    const bool row = g < G;
    uint32_t qa[kDecD / 16], qc[kDecD / 16];
    int q_frame = -1;  // the frame the fragments are in
#pragma unroll
    for (int ks = 0; ks < kDecD / 16; ++ks) {
      qa[ks] = row ? *reinterpret_cast<const uint32_t*>(&sm.qb[row ? g : 0][16 * ks + 2 * t]) : 0u;
      qc[ks] = row ? *reinterpret_cast<const uint32_t*>(&sm.qb[row ? g : 0][16 * ks + 2 * t + 8]) : 0u;
    }
    float o[kDecD / 8][2];
#pragma unroll
    for (int nt = 0; nt < kDecD / 8; ++nt) o[nt][0] = o[nt][1] = 0.f;
    float m_ref = -INFINITY, lsum = 0.f;  // lazy running max (log2 units) and this lane's row-sum share
    // ldmatrix row addresses: lane l gives row l % 8 of matrix l / 8
    const int mr = lane & 7, mi = lane >> 3;
    for (int i = warp; i < n; i += kDecWarps) {
      const int st = i % kDecStages;
      // the outcome is made the same in every lane: the page's work is warp-wide
      // (ldmatrix, mma.sync), so a warp must not go on with some lanes missing
      const bool got = tc::mbar_wait(&sm.full[st], (i / kDecStages) & 1, &sm.abort, kDecWaitNs);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          set_err(err, PIC_ERR_TIMEOUT);
          *reinterpret_cast<volatile int*>(&sm.abort) = 1;
        }
        break;
      }
      const int mt = sm.meta[st];
      if (mt >= 0) {
        const int lo = mt & 31, hi = (mt >> 5) & 31, frame = (mt >> 10) - 1;
        if (frame != q_frame) {  // keys in another frame: Q rotated back by its offset
          q_fragments<G>(sm.qb, g, t, frame, rot_tab, qa, qc);
          q_frame = frame;
        }
        const uint32_t kbase = tc::smem_addr(sm.ring[st][0]), vbase = tc::smem_addr(sm.ring[st][1]);
        // S = Q K^T over the 16 keys: matrices (keys 0-7 | 8-15) x (columns 16ks.. | 16ks+8..)
        float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < kDecD / 16; ++ks) {
          uint32_t b[4];
          ldsm_x4(b, kbase + swz_off(8 * (mi >> 1) + mr, 2 * ks + (mi & 1)));
          mma_rows8(s0[0], s0[1], qa[ks], qc[ks], b[0], b[1]);
          mma_rows8(s1[0], s1[1], qa[ks], qc[ks], b[2], b[3]);
        }
        // online softmax of row g over the page's valid keys [lo, hi)
        const int k0 = 2 * t;
        float sc[4] = {s0[0], s0[1], s1[0], s1[1]};
        const int kk[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
#pragma unroll
        for (int x = 0; x < 4; ++x) sc[x] = (kk[x] >= lo && kk[x] < hi) ? sc[x] * scale_log2 : -INFINITY;
        float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // lazy rescale: P may grow up to 2^8 before O and the sums are rescaled
        const bool up = mx > m_ref + 8.f;
        if (__any_sync(0xffffffffu, up)) {
          const float alpha = up ? tc::ex2(m_ref - mx) : 1.f;  // 0 on the first page (m_ref = -inf)
          lsum *= alpha;
#pragma unroll
          for (int nt = 0; nt < kDecD / 8; ++nt) {
            o[nt][0] *= alpha;
            o[nt][1] *= alpha;
          }
          if (up) m_ref = mx;
        }
        float pv[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) pv[x] = row ? tc::ex2(sc[x] - m_ref) : 0.f;
        lsum += (pv[0] + pv[1]) + (pv[2] + pv[3]);
        const uint32_t pa = pack_bf16x2(pv[0], pv[1]), pc = pack_bf16x2(pv[2], pv[3]);
        // slots outside [lo, hi) may hold anything (NaN): zero them in V so that
        // 0 * V stays 0 (rare: seam pages only)
        if (lo > 0 || hi < PIC_PAGE) {
          uint4* vz = reinterpret_cast<uint4*>(sm.ring[st][1]);
#pragma unroll
          for (int x = 0; x < PIC_PAGE * 2 * 8 / 32; ++x) {  // 16 rows x 2 halves x 8 chunks
            const int c = x * 32 + lane, key = c >> 4;
            if (key < lo || key >= hi) vz[((key >> 3) * 2048 + ((c >> 3) & 1) * 1024 + (key & 7) * 128) / 16 + (c & 7)] =
                make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        // O += P V: matrices (keys 0-7 | 8-15) x columns 8nt.. for nt = 2np, 2np + 1, transposed
#pragma unroll
        for (int np = 0; np < kDecD / 16; ++np) {
          uint32_t b[4];
          ldsm_x4_trans(b, vbase + swz_off(8 * (mi & 1) + mr, 2 * np + (mi >> 1)));
          mma_rows8(o[2 * np][0], o[2 * np][1], pa, pc, b[0], b[1]);
          mma_rows8(o[2 * np + 1][0], o[2 * np + 1][1], pa, pc, b[2], b[3]);
        }
        if (lo > 0 || hi < PIC_PAGE) tc::fence_proxy_async_smem();  // generic writes before the next TMA fill
      }
      __syncwarp();  // the stage is read before it is released
      if (lane == 0) tc::mbar_arrive(&sm.empty[st]);  // the stage may be refilled
    }
    // row sums over the quad; partials kept until the ring is free
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    if (row && t == 0) {
      sm.w_m[warp][g] = m_ref;
      sm.w_l[warp][g] = lsum;
    }
    ring_drained_sync();  // no copy in flight and no consumer reading: the ring takes the partials
    if (row) {
#pragma unroll
      for (int nt = 0; nt < kDecD / 8; ++nt)
        *reinterpret_cast<float2*>(&sm.w_o[warp][row ? g : 0][8 * nt + 2 * t]) = make_float2(o[nt][0], o[nt][1]);
    }
  }
  __syncthreads();
  // the CTA's warps combined into one partial per head
  if (tid < kDecD) {
    const int64_t part = cta;
    for (int hh = 0; hh < G; ++hh) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sm.w_m[w][hh]);
      float Lsum = 0.f, Osum = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = (sm.w_m[w][hh] == -INFINITY) ? 0.f : tc::ex2(sm.w_m[w][hh] - M);
        Lsum += f * sm.w_l[w][hh];
        Osum += f * sm.w_o[w][hh][tid];
      }
      part_o[(part * G + hh) * kDecD + tid] = Osum;
      if (tid == 0) part_ml[part * G + hh] = make_float2(M, Lsum);
    }
  }
}

// out[r][h] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the splits.  One CTA per
// (head, request): thread (group g, lane c) folds splits g, g + 8, .. for columns
// 4c..4c+3, then the groups are combined through shared memory.
__global__ void __launch_bounds__(32 * kMergeGroups)
decode_merge_kernel(const float2* __restrict__ part_ml, const float* __restrict__ part_o, bf16* __restrict__ out,
                    int Hq, int Hkv, const int32_t* __restrict__ first, const int32_t* __restrict__ nsplit) {
  __shared__ float g_m[kMergeGroups], g_l[kMergeGroups];
  __shared__ float4 g_o[kMergeGroups][32];
  const int h = blockIdx.x, r = blockIdx.y, c = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int G = Hq / Hkv, kvh = h / G, hh = h % G;
  const int splits = nsplit[r];
  const int64_t base = first[r] + (int64_t)kvh * splits;  // partials are indexed by CTA
  // one pass with a running maximum, four splits' loads in flight at a time
  float M = -INFINITY, Lsum = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = g; s0 < splits; s0 += 4 * kMergeGroups) {
    float2 ml[4];
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int sp = s0 + k * kMergeGroups;
      ml[k] = make_float2(-INFINITY, 0.f);
      v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (sp < splits) {
        ml[k] = part_ml[(base + sp) * G + hh];
        v[k] = reinterpret_cast<const float4*>(part_o + ((base + sp) * G + hh) * kDecD)[c];
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (ml[k].x == -INFINITY) continue;  // a split without keys
      const float Mn = fmaxf(M, ml[k].x);
      const float a = tc::ex2(M - Mn), f = tc::ex2(ml[k].x - Mn);  // a = 0 while M = -inf
      Lsum = fmaf(Lsum, a, f * ml[k].y);
      O.x = fmaf(O.x, a, f * v[k].x); O.y = fmaf(O.y, a, f * v[k].y);
      O.z = fmaf(O.z, a, f * v[k].z); O.w = fmaf(O.w, a, f * v[k].w);
      M = Mn;
    }
  }
  if (c == 0) {
    g_m[g] = M;
    g_l[g] = Lsum;
  }
  g_o[g][c] = O;
  __syncthreads();
  if (g != 0) return;
  float Mall = -INFINITY;
#pragma unroll
  for (int k = 0; k < kMergeGroups; ++k) Mall = fmaxf(Mall, g_m[k]);
  float Lall = 0.f;
  float4 Oall = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kMergeGroups; ++k) {
    if (g_m[k] == -INFINITY) continue;
    const float f = tc::ex2(g_m[k] - Mall);
    Lall += f * g_l[k];
    Oall.x = fmaf(f, g_o[k][c].x, Oall.x); Oall.y = fmaf(f, g_o[k][c].y, Oall.y);
    Oall.z = fmaf(f, g_o[k][c].z, Oall.z); Oall.w = fmaf(f, g_o[k][c].w, Oall.w);
  }
  const float inv = Lall > 0.f ? 1.f / Lall : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(Oall.x * inv, Oall.y * inv), hi = __floats2bfloat162_rn(Oall.z * inv, Oall.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(out + ((int64_t)r * Hq + h) * kDecD)[c] = pk;
}

template <int G>
cudaError_t occupancy_of(int* n) {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(DecSmem<G>));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, decode_kernel<G>, kDecThreads, sizeof(DecSmem<G>));
}

// Decode CTAs one SM holds at once, for the kernel instance of group size G.
int dec_ctas_per_sm(int G) {
  int n = 0;
  cudaError_t e;
  switch (G) {
    case 1: e = occupancy_of<1>(&n); break;
    case 2: e = occupancy_of<2>(&n); break;
    case 4: e = occupancy_of<4>(&n); break;
    default: e = occupancy_of<8>(&n); break;
  }
  return (e == cudaSuccess && n > 0) ? n : 1;
}

bool dec_shape(pic_dtype dt, int Hq, int Hkv, int d) {
  if (dt != PIC_BF16 || d != kDecD || Hkv < 1 || Hq < Hkv || Hq % Hkv) return false;
  const int G = Hq / Hkv;
  return G == 1 || G == 2 || G == 4 || G == 8;
}

}  // namespace
}  // namespace pic

using namespace pic;

extern "C" {

size_t pic_decode_workspace(int32_t n_req, int32_t Hq, int32_t Hkv, int32_t d, pic_dtype dtype) {
  if (n_req < 0 || !dec_shape(dtype, Hq, Hkv, d)) return 0;
  return dec_layout(n_req, Hq, Hkv, num_sms_of_current_device(), dec_ctas_per_sm(Hq / Hkv)).total;
}

pic_status pic_decode_attention(const void* q, const float* q_table, const void* k_pool, const void* v_pool,
                                int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                                const int32_t* page_off, const int32_t* page_tab, const float* rot_table,
                                int64_t n_tab, int32_t n_req, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                                void* out, void* ws, size_t ws_bytes, int32_t* err_flag, pic_stream_t stream) {
  if (n_req < 0 || num_blocks < 0 || !(scale > 0.f)) return PIC_ERR_INVALID;
  // frames travel with a page in 21 bits
  if (n_tab < 0 || n_tab >= (1 << 21) - 1 || (page_tab != nullptr && n_tab > 0 && rot_table == nullptr) ||
      (reinterpret_cast<uintptr_t>(rot_table) & 15))
    return PIC_ERR_INVALID;
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv || d < 2 || (d & 1)) return PIC_ERR_INVALID;
  if (!dec_shape(dtype, Hq, Hkv, d)) return PIC_ERR_UNSUPPORTED;
  if (n_req == 0) return PIC_OK;
  if (!q || !q_table || !k_pool || !v_pool || !pages || !page_off || !out || !err_flag) return PIC_ERR_INVALID;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(q_table) |
                        reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool) |
                        reinterpret_cast<uintptr_t>(pages) | reinterpret_cast<uintptr_t>(out);
  if (mis & 15) return PIC_ERR_INVALID;
  const DecLayout L = dec_layout(n_req, Hq, Hkv, num_sms_of_current_device(), dec_ctas_per_sm(Hq / Hkv));
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PIC_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* first = reinterpret_cast<int32_t*>(w + L.off_plan);
  int32_t* nsplit = first + (n_req + 1);
  int4* desc = reinterpret_cast<int4*>(w + L.off_desc);
  float2* part_ml = reinterpret_cast<float2*>(w + L.off_ml);
  float* part_o = reinterpret_cast<float*>(w + L.off_o);
  cudaStream_t s = (cudaStream_t)stream;
  const int slots = (int)(L.ctas - (int64_t)n_req * Hkv);
  if (n_req > kDecThreads) {  // else the decode CTAs split the work themselves
    decode_plan_kernel<<<1, kPlanThreads, 0, s>>>(page_off, n_req, Hkv, slots, (int)L.ctas, first, nsplit, desc);
    if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  }
  const uint64_t pool_rows = (uint64_t)num_blocks * Hkv * PIC_PAGE;
  if (pool_rows == 0 || pool_rows > (uint64_t)INT32_MAX) return PIC_ERR_INVALID;
  CUtensorMap kmap, vmap;
  if (!encode_pages(&kmap, k_pool, pool_rows) || !encode_pages(&vmap, v_pool, pool_rows)) return PIC_ERR_CUDA;
  const unsigned grid = (unsigned)L.ctas;
  const float sl2 = scale * 1.4426950408889634f;
  const bf16* qb = static_cast<const bf16*>(q);
  const float4* qt = reinterpret_cast<const float4*>(q_table);
  const float4* rt = reinterpret_cast<const float4*>(rot_table);
  switch (Hq / Hkv) {
    case 1: decode_kernel<1><<<grid, kDecThreads, sizeof(DecSmem<1>), s>>>(kmap, vmap, qb, qt, num_blocks, pages,
        page_off, page_tab, rt, n_tab, n_req, Hq, Hkv, sl2, desc, slots, first, nsplit, part_ml, part_o, err_flag); break;
    case 2: decode_kernel<2><<<grid, kDecThreads, sizeof(DecSmem<2>), s>>>(kmap, vmap, qb, qt, num_blocks, pages,
        page_off, page_tab, rt, n_tab, n_req, Hq, Hkv, sl2, desc, slots, first, nsplit, part_ml, part_o, err_flag); break;
    case 4: decode_kernel<4><<<grid, kDecThreads, sizeof(DecSmem<4>), s>>>(kmap, vmap, qb, qt, num_blocks, pages,
        page_off, page_tab, rt, n_tab, n_req, Hq, Hkv, sl2, desc, slots, first, nsplit, part_ml, part_o, err_flag); break;
    default: decode_kernel<8><<<grid, kDecThreads, sizeof(DecSmem<8>), s>>>(kmap, vmap, qb, qt, num_blocks, pages,
        page_off, page_tab, rt, n_tab, n_req, Hq, Hkv, sl2, desc, slots, first, nsplit, part_ml, part_o, err_flag); break;
  }
  if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  decode_merge_kernel<<<dim3((unsigned)Hq, (unsigned)n_req), 32 * kMergeGroups, 0, s>>>(
      part_ml, part_o, static_cast<bf16*>(out), Hq, Hkv, first, nsplit);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

}  // extern "C"
