// Linear-attention state composition (HYPIC blog, section 2.1).  A linear layer
// caches, per chunk and head, the pair (T_C, S(C|0)): the chunk's cumulative
// transition operator and its end state from a zero state.  Chunks linked in any
// order give the state of the whole chain by S(C1 C2) = T(C2) S(C1) + S(C2),
// applied along the chain; T composes as T(C1 C2) = T(C2) T(C1).
//
// Parallel form: a chain of n elements is cut into segments of `seg` elements; one
// CTA folds a segment into one element (S of the segment and, unless the segment
// starts the chain, its transition product); a second launch folds each chain's
// segment elements in order.  With seg >= n there is one launch and no transition
// product is formed.
//
// One fold step X <- T_i X + S_i (d = 128) is one 128 x 128 x 128 product on the
// tensor cores, taken transposed so that every operand keeps its natural place:
//   D^T = X^T T_i^T,  A = X^T in TMEM (TMEM lane n holds column n of X),
//                     B = T_i in shared memory (row-major T_i is the K-major B).
// Precision: both factors as two bf16 parts, x = x_hi + x_lo with x_hi = bf16(x),
// x_lo = bf16(x - x_hi); the product is hi.hi + hi.lo + lo.hi with fp32
// accumulation (the dropped lo.lo term is below 2^-16 of |x||y|).  The cache keeps
// T in exactly that form (pic_compose_split_t), two bf16 planes, so T_i goes from
// global memory into the B operand by TMA without any conversion; the state is
// split by the epilogue each step.  S_i stays fp32 and is added exactly.
//
// Pipeline (352 threads, one CTA per SM).  Warp 8 lane 0 loads T_i by four 16 KB
// TMA boxes into one of two B buffers; warp 10 lane 0 loads S_i by bulk copies,
// 32 rows at a time, into two rings of three 16 KB slots — ring h holds the rows that epilogue half h
// reads, and only that half consumes it, in order (a slot shared by two consumer
// groups that take turns could be waited on while the other group's earlier fill
// of it is still in flight, and its parity would then report that fill's previous
// phase as complete); warp 9 lane 0 issues the MMAs; warps 0-7 run the epilogue
// (TMEM + S_i -> split -> TMEM).  The S products and the T products are committed
// apart, so that each epilogue overlaps the other's MMAs.  Every wait is bounded.
#include <algorithm>

#include "pic_internal.cuh"
#include "tc_ptx.cuh"

namespace pic {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kCD = 128;                              // d_k = d_v
constexpr int kElt = kCD * kCD;                       // elements per matrix
constexpr int kMatBytes = kElt * 4;                   // 64 KB: one fp32 matrix, or its two bf16 planes
constexpr int kCWorkers = 256;                        // warps 0-7
constexpr int kProdWarp = kCWorkers / 32, kMmaWarp = kProdWarp + 1, kSProdWarp = kMmaWarp + 1;
constexpr int kCThreads = kCWorkers + 96;
constexpr int kBHalf = kCD * 128;                     // one 64-column half of a 128-row bf16 operand
constexpr int kBPart = 2 * kBHalf;                    // 32 KB: one bf16 part of B
constexpr int kBBytes = 2 * kBPart;                   // hi | lo
constexpr int kOffB = 0;                              // two B buffers ([part][k half][128 rows][128 B], SW128)
constexpr int kSRows = 32;                            // rows of S per ring block
constexpr int kSBlk = kSRows * kCD * 4;               // 16 KB
constexpr int kSRing = 3;                             // slots per ring
constexpr int kOffSr = kOffB + 2 * kBBytes;           // ring h at kOffSr + h * kSRing * kSBlk
constexpr int kOffBar = kOffSr + 2 * kSRing * kSBlk;
constexpr int kCSmem = kOffBar + 256;
static_assert(kCSmem <= 232448, "shared memory per CTA");
// TMEM columns: D_S | D_T | A_S hi | A_S lo | A_T hi | A_T lo
constexpr uint32_t kColDS = 0, kColDT = 128, kColAS = 256, kColAT = 384;
constexpr uint64_t kCWaitNs = 2000000000ull;
constexpr uint32_t kCIdesc = tc::idesc_bf16_f32(128, 128, false);

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

struct CBars {
  uint64_t b_full[2], b_empty[2];            // per B buffer: T_i landed / released by the step that read it
  uint64_t s_full[2][kSRing], s_empty[2][kSRing];  // per S ring slot
  uint64_t a_s, a_t;                         // A_S / A_T written for the next step
  uint64_t d_s, d_t;                         // the step's S / T products complete
  uint64_t never;                            // no thread arrives on it (failure-injection test build)
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(CBars) <= 256, "barrier block");

struct Level {
  const bf16* T_in;          // two bf16 planes per matrix: [matrix][part][128][128]
  const float* S_in;
  const int32_t* ids;        // level 0: pool entry of every chain element; else nullptr
  const int32_t* chain_off;  // [n_req + 1] offsets of each request's chain in ids
  const int32_t* first;      // [n_req + 1] first CTA of each request at this level
  int64_t n_pool;            // level 0: entries of the pool
  int64_t in_stride;         // level 1: elements per chain in T_in / S_in
  bf16* T_out;               // level 0 of two: [chain][out_stride][part][128][128]
  float* S_out;              // [chain][out_stride]
  int64_t out_stride;
  int64_t n_elems;           // entries of ids
  int n_req, H, seg, seg_prev;  // seg_prev: level 1 input elements per chain = ceil(n_r / seg_prev)
  int max_chain;             // chain lengths are clamped to it (the planner flags longer ones)
  int level;
  bool last;
  bool self_plan;            // few requests: every CTA finds its own (request, head, segment)
  bool one_level;            // the call folds in one level (an empty chain still gets its CTAs)
  int32_t* err;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, CBars* cb, int32_t* err) {
  if (tc::mbar_wait(bar, parity, &cb->abort, kCWaitNs)) return true;
  set_err(err, PIC_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&cb->abort) = 1;
  return false;
}

// The same for a whole warp that goes on to warp-collective work (TMEM accesses):
// every lane waits, and the outcome is the same in all lanes (a lane that saw the
// phase complete gives up with the others when one of them ran out), so that the
// warp never reaches a .sync.aligned instruction diverged.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, CBars* cb, int32_t* err) {
  const bool ok = tc::mbar_wait(bar, parity, &cb->abort, kCWaitNs);
  if (__all_sync(0xffffffffu, ok)) return true;
  if (!ok) set_err(err, PIC_ERR_TIMEOUT);
  *reinterpret_cast<volatile int*>(&cb->abort) = 1;
  return false;
}

// 16 rows m_first .. +15 of state column nc: the staged S rows (srow[j * kCD], when
// USE_S) plus the accumulator at TMEM column d_col + m_first -> the fp32 output
// (when OUT == 1), the two bf16 planes of a split output (OUT == 2), or the A
// operand (bf16 hi at a_col + m_first / 2, lo 64 columns further).  Warp-collective.
template <bool USE_S, int OUT>
__device__ __forceinline__ void piece16(const float* srow, uint32_t tmem_row, uint32_t d_col, int m_first, int nc,
                                        void* out, uint32_t a_col) {
  float x[16];
  {
    uint32_t rr[16];
    tc::tmem_ld16(tmem_row + d_col + m_first, rr);
    tc::tmem_ld_wait();
    tc::reg_fence<16>(rr);
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = USE_S ? __uint_as_float(rr[j]) + srow[j * kCD] : __uint_as_float(rr[j]);
  }
  if (OUT == 1) {
    float* o = static_cast<float*>(out) + m_first * kCD + nc;
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j * kCD] = x[j];
  } else if (OUT == 2) {
    bf16* o = static_cast<bf16*>(out) + m_first * kCD + nc;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const bf16 h = __float2bfloat16_rn(x[j]);
      o[j * kCD] = h;
      o[kElt + j * kCD] = __float2bfloat16_rn(x[j] - __bfloat162float(h));
    }
  } else {
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bf16 h0 = __float2bfloat16_rn(x[2 * j]), h1 = __float2bfloat16_rn(x[2 * j + 1]);
      hi[j] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      lo[j] = pack_bf16x2(x[2 * j] - __bfloat162float(h0), x[2 * j + 1] - __bfloat162float(h1));
    }
    tc::tmem_st8(tmem_row + a_col + (m_first >> 1), hi);
    tc::tmem_st8(tmem_row + a_col + 64 + (m_first >> 1), lo);
  }
}

__global__ void __launch_bounds__(kCThreads, 1)
compose_kernel(const __grid_constant__ CUtensorMap tmap, const Level lv) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  CBars* cb = reinterpret_cast<CBars*>(sm + kOffBar);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  if (tc::smem_addr(smem_raw) & 1023u) {
    if (tid == 0) set_err(lv.err, PIC_ERR_UNSUPPORTED);
    return;
  }
  int r, first_r;
  if (lv.self_plan) {
    // the planner's CTA counts, found by every CTA itself (one launch less): a scan
    // over the requests; level 0's CTA 0 also checks the chain offsets
    __shared__ int s_scan[kCThreads / 32 + 1];
    __shared__ int s_req[2];
    int w = 0;
    if (tid < lv.n_req) {
      int nr = __ldg(lv.chain_off + tid + 1) - __ldg(lv.chain_off + tid);
      if (lv.level == 0 && cta == 0 &&
          (nr < 0 || nr > lv.max_chain || __ldg(lv.chain_off + tid) < 0 || __ldg(lv.chain_off + tid + 1) > lv.n_elems))
        set_err(lv.err, PIC_ERR_RANGE);
      nr = min(max(nr, 0), lv.max_chain);
      const int segs = nr > 0 ? (nr + lv.seg - 1) / lv.seg : 0;
      w = lv.level == 0 ? lv.H * (lv.one_level ? max(segs, 1) : segs) : lv.H;
    }
    if (lv.level == 0 && cta == 0 && tid == 0 &&
        (__ldg(lv.chain_off) != 0 || __ldg(lv.chain_off + lv.n_req) != lv.n_elems))
      set_err(lv.err, PIC_ERR_RANGE);
    int total;
    const int ex = block_exclusive_scan<kCThreads>(w, s_scan, &total);
    if (tid == 0 && cta >= total) s_req[0] = -1;
    if (tid < lv.n_req && cta >= ex && cta < ex + w) {
      s_req[0] = tid;
      s_req[1] = ex;
    }
    __syncthreads();
    if (s_req[0] < 0) return;  // the grid is an upper bound
    r = s_req[0];
    first_r = s_req[1];
  } else {
    if (cta >= __ldg(lv.first + lv.n_req)) return;
    int lo = 0, hi = lv.n_req;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(lv.first + mid) <= cta) lo = mid; else hi = mid;
    }
    r = lo;
    first_r = __ldg(lv.first + r);
  }
  const int c0 = __ldg(lv.chain_off + r);
  const int n_r = min(max(__ldg(lv.chain_off + r + 1) - c0, 0), lv.max_chain);
  const int n_in = lv.level == 0 ? n_r : (n_r + lv.seg_prev - 1) / lv.seg_prev;
  const int n_segs = max(1, (n_in + lv.seg - 1) / lv.seg);
  const int local = cta - first_r;
  const int h = local / n_segs, g = local % n_segs;
  const int b = g * lv.seg, e = min(n_in, b + lv.seg), n = e - b;
  const bool need_T = !lv.last && g > 0;
  const int64_t chain = (int64_t)r * lv.H + h;
  float* s_out = lv.S_out + (chain * lv.out_stride + g) * kElt;
  bf16* t_out = need_T ? lv.T_out + (chain * lv.out_stride + g) * 2 * kElt : nullptr;

  if (n <= 0) {  // an empty chain: its state is zero
    for (int i = tid; i < kElt / 4; i += kCThreads)
      reinterpret_cast<float4*>(s_out)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  // matrix index of chain element i: its S at S_in + index * kElt, its T planes at
  // T_in + index * 2 kElt (rows 256 index .. of the T tensor map)
  auto mat = [&](int i) -> int64_t {
    if (lv.level == 0) {
      const int64_t at = (int64_t)c0 + i;
      int64_t id = (at >= 0 && at < lv.n_elems) ? __ldg(lv.ids + at) : 0;
      if (id < 0 || id >= lv.n_pool) {  // flagged by the planner, or here when there is none
        if (lv.self_plan) set_err(lv.err, PIC_ERR_RANGE);
        id = 0;
      }
      return id * lv.H + h;
    }
    return chain * lv.in_stride + i;
  };

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&cb->b_full[i], 1);
      tc::mbar_init(&cb->b_empty[i], kCWorkers);
    }
    for (int hh = 0; hh < 2; ++hh)
      for (int sl = 0; sl < kSRing; ++sl) {
        tc::mbar_init(&cb->s_full[hh][sl], 1);
        tc::mbar_init(&cb->s_empty[hh][sl], kCWorkers / 2);
      }
    tc::mbar_init(&cb->a_s, kCWorkers);
    tc::mbar_init(&cb->a_t, kCWorkers);
    tc::mbar_init(&cb->d_s, 1);
    tc::mbar_init(&cb->d_t, 1);
    tc::mbar_init(&cb->never, 1);
    cb->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(&cb->tmem, 512);
    tc::tmem_relinquish();
  }
  if (warp == kProdWarp && lane == 0) tc::tma_prefetch_desc(&tmap);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = cb->tmem;
  const int n_steps = n - 1;

  if (warp == kProdWarp || warp == kSProdWarp) {
    // ---- producers, each its own stream so that neither waits behind the other.
    // T: T(j) = T_{b+1+j} to B buffer j & 1 once the step two before released it.
    // S: S(u) = S_{b+u} as block w = 2u + q (rows 64 h + 32 q ..) to slot w % 3 of
    // ring h once that slot's block w - 3 was read.
    if (lane == 0 && warp == kProdWarp) {
      int t_issued = 0;
      for (int j = 0; j < n_steps; ++j) {
        const int buf = j & 1;
        if (j >= 2 && !wait_bar(&cb->b_empty[buf], ((j >> 1) & 1) ^ 1, cb, lv.err)) break;
        const int32_t y0 = (int32_t)(mat(b + 1 + j) * 2 * kCD);
        uint8_t* dst = sm + kOffB + buf * kBBytes;
        tc::mbar_arrive_expect_tx(&cb->b_full[buf], kBBytes);
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)
            tc::tma_load_2d(dst + p * kBPart + kh * kBHalf, &tmap, 64 * kh, y0 + p * kCD, &cb->b_full[buf]);
        t_issued = j + 1;
      }
      // no copy may be in flight when the block exits
      const int no_abort = 0;
      for (int k = 0; k < 2 && k < t_issued; ++k) {
        const int j = t_issued - 1 - k;
        tc::mbar_wait(&cb->b_full[j & 1], (j >> 1) & 1, &no_abort, kCWaitNs);
      }
    } else if (lane == 0) {
      int w_issued[2] = {0, 0};  // blocks issued per ring
      bool ok = true;
      for (int u = 0; ok && u < n; ++u) {
        const float* src = lv.S_in + mat(b + u) * kElt;
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int w = 2 * u + q, sl = w % kSRing;
            if (ok && !(ok = wait_bar(&cb->s_empty[hh][sl], ((w / kSRing) & 1) ^ 1, cb, lv.err))) break;
            if (!ok) break;
            tc::mbar_arrive_expect_tx(&cb->s_full[hh][sl], kSBlk);
            tc::bulk_load(sm + kOffSr + (hh * kSRing + sl) * kSBlk,
                          reinterpret_cast<const uint8_t*>(src + (64 * hh + kSRows * q) * kCD), kSBlk,
                          &cb->s_full[hh][sl]);
            if (hh == 0) w_issued[0] = w + 1; else w_issued[1] = w + 1;
          }
      }
      // the last fill of every slot (each earlier fill of a slot was read before
      // the slot was filled again)
      const int no_abort = 0;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int wn = hh == 0 ? w_issued[0] : w_issued[1];
        for (int w = wn - 1; w >= 0 && w >= wn - kSRing; --w)
          tc::mbar_wait(&cb->s_full[hh][w % kSRing], (w / kSRing) & 1, &no_abort, kCWaitNs);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---- MMA issue: D_S = A_S B_k, then D_T = A_T B_k, three bf16 part products
    // each, committed apart so that the S epilogue overlaps the T products and the
    // T epilogue the next S products
    if (lane == 0) {
      constexpr uint32_t kHi = tc::sw128_desc_hi(1024);
      const uint32_t b_lo0 = tc::sw128_desc_lo(tc::smem_addr(sm + kOffB), 16);
      auto products = [&](uint32_t d_col, uint32_t a_col, uint32_t b_lo) {
#pragma unroll
        for (int ks = 0; ks < kCD / 16; ++ks) {
          const uint32_t boff = (uint32_t)(((ks >> 2) * kBHalf + (ks & 3) * 32) >> 4);
          const uint64_t bh = tc::desc_join(b_lo + boff, kHi);
          const uint64_t bl = tc::desc_join(b_lo + boff + (kBPart >> 4), kHi);
          tc::mma_bf16_ts(tmem + d_col, tmem + a_col + ks * 8, bh, kCIdesc, ks > 0 ? 1u : 0u);
          tc::mma_bf16_ts(tmem + d_col, tmem + a_col + ks * 8, bl, kCIdesc, 1u);
          tc::mma_bf16_ts(tmem + d_col, tmem + a_col + 64 + ks * 8, bh, kCIdesc, 1u);
        }
      };
      // every commit's arrival lands before the CTA exits: the thread waits for the
      // last phase of each barrier it committed to
      int issued = 0, issued_t = 0;
      int steps = n_steps;
#ifdef PIC_INJECT_WAIT_TIMEOUT
      // Failure-injection test build only: a bounded wait on a barrier that nothing
      // arrives on runs out, reports PIC_ERR_TIMEOUT and stops the CTA cleanly.
      if (!tc::mbar_wait(&cb->never, 0, &cb->abort, PIC_INJECT_WAIT_TIMEOUT)) {
        set_err(lv.err, PIC_ERR_TIMEOUT);
        *reinterpret_cast<volatile int*>(&cb->abort) = 1;
        steps = 0;
      }
#endif
      for (int k = 0; k < steps; ++k) {
        if (!wait_bar(&cb->b_full[k & 1], (k >> 1) & 1, cb, lv.err)) break;
        if (!wait_bar(&cb->a_s, k & 1, cb, lv.err)) break;
        tc::tc_fence_after();
        const uint32_t b_lo = b_lo0 + (uint32_t)((k & 1) * (kBBytes >> 4));
        products(kColDS, kColAS, b_lo);
        tc::mma_commit(&cb->d_s);
        issued = k + 1;
        if (need_T) {
          if (!wait_bar(&cb->a_t, k & 1, cb, lv.err)) break;
          tc::tc_fence_after();
          products(kColDT, kColAT, b_lo);
          tc::mma_commit(&cb->d_t);
          issued_t = k + 1;
        }
      }
      const int no_abort = 0;
      if (issued > 0) tc::mbar_wait(&cb->d_s, (issued - 1) & 1, &no_abort, kCWaitNs);
      if (issued_t > 0) tc::mbar_wait(&cb->d_t, (issued_t - 1) & 1, &no_abort, kCWaitNs);
    }
    __syncwarp();
  } else {
    // ---- epilogue warps: warp w reads TMEM lanes 32 (w % 4) .. +31 (state columns
    // nc = 32 (w % 4) + lane) and accumulator columns m = 64 (w / 4) .. +63
    const int quarter = warp & 3, hf = warp >> 2;
    const int nc = 32 * quarter + lane, m0 = 64 * hf;
    const uint32_t trow = tmem + (uint32_t)((32 * quarter) << 16);
    const float* ring = reinterpret_cast<const float*>(sm + kOffSr) + hf * kSRing * (kSBlk / 4) + nc;
    int su = 0;  // S matrices consumed
    bool ok = true;
    auto signal = [&](uint64_t* bar) {
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(bar);
    };
    // the next S (this half's two ring blocks) plus the accumulator at D_S (when
    // add_d) -> A_S, or the output
    auto s_emit = [&](bool add_d, bool to_out) -> bool {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int w = 2 * su + q, sl = w % kSRing;
        if (!wait_bar_warp(&cb->s_full[hf][sl], (w / kSRing) & 1, cb, lv.err)) return false;
        const float* blk = ring + sl * (kSBlk / 4);  // rows m0 + 32 q .. of S, column nc
        if (!add_d && !to_out) {  // the first element: S_b -> A_S
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int mf = m0 + kSRows * q + 16 * c;
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float x0 = blk[(16 * c + 2 * j) * kCD], x1 = blk[(16 * c + 2 * j + 1) * kCD];
              const bf16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
              hi[j] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
              lo[j] = pack_bf16x2(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
            }
            tc::tmem_st8(trow + kColAS + (mf >> 1), hi);
            tc::tmem_st8(trow + kColAS + 64 + (mf >> 1), lo);
          }
        } else if (!add_d) {  // a one-element segment: S_b is the output
#pragma unroll
          for (int c = 0; c < kSRows; ++c) s_out[(m0 + kSRows * q + c) * kCD + nc] = blk[c * kCD];
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int mf = m0 + kSRows * q + 16 * c;
            if (to_out) piece16<true, 1>(blk + 16 * c * kCD, trow, kColDS, mf, nc, s_out, kColAS);
            else piece16<true, 0>(blk + 16 * c * kCD, trow, kColDS, mf, nc, nullptr, kColAS);
          }
        }
        tc::mbar_arrive(&cb->s_empty[hf][sl]);
      }
      ++su;
      return true;
    };
    auto t_emit = [&](bool to_out) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (to_out) piece16<false, 2>(nullptr, trow, kColDT, m0 + 16 * c, nc, t_out, kColAT);
        else piece16<false, 0>(nullptr, trow, kColDT, m0 + 16 * c, nc, nullptr, kColAT);
      }
    };
    // first element: T_b (its two planes, column nc) -> A_T (or the output)
    if (need_T) {
      const bf16* tb = lv.T_in + mat(b) * 2 * kElt + nc;
      if (n == 1) {
        for (int c = 0; c < 64; ++c) {
          t_out[(m0 + c) * kCD + nc] = tb[(m0 + c) * kCD];
          t_out[kElt + (m0 + c) * kCD + nc] = tb[kElt + (m0 + c) * kCD];
        }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int mf = m0 + 16 * c;
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            hi[j] = (uint32_t)__bfloat16_as_ushort(tb[(mf + 2 * j) * kCD]) |
                    ((uint32_t)__bfloat16_as_ushort(tb[(mf + 2 * j + 1) * kCD]) << 16);
            lo[j] = (uint32_t)__bfloat16_as_ushort(tb[kElt + (mf + 2 * j) * kCD]) |
                    ((uint32_t)__bfloat16_as_ushort(tb[kElt + (mf + 2 * j + 1) * kCD]) << 16);
          }
          tc::tmem_st8(trow + kColAT + (mf >> 1), hi);
          tc::tmem_st8(trow + kColAT + 64 + (mf >> 1), lo);
        }
      }
    }
    ok = s_emit(false, n == 1);
    if (ok && n_steps > 0) {
      signal(&cb->a_s);
      if (need_T) signal(&cb->a_t);
    }
    // steps 0 .. n_steps - 2 feed the next step; the last writes the output
    for (int k = 0; ok && k + 1 < n_steps; ++k) {
      if (!(ok = wait_bar_warp(&cb->d_s, k & 1, cb, lv.err))) break;
      tc::tc_fence_after();
      if (!need_T) tc::mbar_arrive(&cb->b_empty[k & 1]);  // step k's products are complete: B is free
      if (!(ok = s_emit(true, false))) break;
      signal(&cb->a_s);
      if (need_T) {
        if (!(ok = wait_bar_warp(&cb->d_t, k & 1, cb, lv.err))) break;
        tc::tc_fence_after();
        tc::mbar_arrive(&cb->b_empty[k & 1]);
        t_emit(false);
        signal(&cb->a_t);
      }
    }
    if (ok && n_steps > 0 && wait_bar_warp(&cb->d_s, (n_steps - 1) & 1, cb, lv.err)) {
      tc::tc_fence_after();
      if (s_emit(true, true) && need_T && wait_bar_warp(&cb->d_t, (n_steps - 1) & 1, cb, lv.err)) {
        tc::tc_fence_after();
        t_emit(true);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// T in the cached form: hi = bf16(T), lo = bf16(T - hi), two planes per matrix.
__global__ void __launch_bounds__(256) split_t_kernel(const float* __restrict__ T, int64_t n, bf16* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(T) + i);
    const int64_t m = i / (kElt / 4), w = i % (kElt / 4);
    const bf16 h0 = __float2bfloat16_rn(v.x), h1 = __float2bfloat16_rn(v.y);
    const bf16 h2 = __float2bfloat16_rn(v.z), h3 = __float2bfloat16_rn(v.w);
    uint2 hv, lv;
    hv.x = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
    hv.y = (uint32_t)__bfloat16_as_ushort(h2) | ((uint32_t)__bfloat16_as_ushort(h3) << 16);
    lv.x = pack_bf16x2(v.x - __bfloat162float(h0), v.y - __bfloat162float(h1));
    lv.y = pack_bf16x2(v.z - __bfloat162float(h2), v.w - __bfloat162float(h3));
    reinterpret_cast<uint2*>(out + m * 2 * kElt)[w] = hv;
    reinterpret_cast<uint2*>(out + m * 2 * kElt + kElt)[w] = lv;
  }
}

// 2-D view [rows][128] bf16 of a split-T array (rows = 256 per matrix), boxes of
// 128 rows x 64 columns with the 128-byte swizzle: one box is one k half of one
// plane of a B operand.
bool encode_t(CUtensorMap* map, const void* base, uint64_t rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr || rows == 0 || rows > (uint64_t)INT32_MAX) return false;
  cuuint64_t dims[2] = {kCD, rows};
  cuuint64_t strides[1] = {kCD * sizeof(bf16)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One block: the first CTA of every request at both levels, and a check of the
// chain offsets and of every chain element id.  Level 0 gives request r
// H * ceil(n_r / seg0) CTAs (H at least, for an empty chain's zero state, when
// level 0 is the last); level 1 gives H.
__global__ void __launch_bounds__(1024)
compose_plan_kernel(const int32_t* __restrict__ ids, const int32_t* __restrict__ chain_off, int n_req, int H,
                    int64_t n_pool, int64_t n_elems, int max_chain, int seg0, bool one_level,
                    int32_t* __restrict__ first0, int32_t* __restrict__ first1, int32_t* err) {
  __shared__ int scratch[1024 / 32 + 1];
  int carry0 = 0, carry1 = 0;
  for (int base = 0; base < n_req; base += 1024) {
    const int r = base + threadIdx.x;
    int w0 = 0, w1 = 0;
    if (r < n_req) {
      int n_r = chain_off[r + 1] - chain_off[r];
      if (n_r < 0 || n_r > max_chain || chain_off[r] < 0 || chain_off[r + 1] > n_elems) set_err(err, PIC_ERR_RANGE);
      n_r = min(max(n_r, 0), max_chain);
      const int segs = n_r > 0 ? (n_r + seg0 - 1) / seg0 : 0;
      w0 = H * (one_level ? max(segs, 1) : segs);
      w1 = H;
    }
    int tot;
    const int ex0 = block_exclusive_scan<1024>(w0, scratch, &tot);
    if (r < n_req) first0[r] = carry0 + ex0;
    carry0 += tot;
    const int ex1 = block_exclusive_scan<1024>(w1, scratch, &tot);
    if (r < n_req) first1[r] = carry1 + ex1;
    carry1 += tot;
  }
  if (threadIdx.x == 0) {
    first0[n_req] = carry0;
    first1[n_req] = carry1;
  }
  if (threadIdx.x == 0 && (chain_off[0] != 0 || chain_off[n_req] != n_elems)) set_err(err, PIC_ERR_RANGE);
  for (int64_t i = threadIdx.x; i < n_elems; i += blockDim.x)
    if (ids[i] < 0 || (int64_t)ids[i] >= n_pool) set_err(err, PIC_ERR_RANGE);
}

struct CLayout {
  bool one_level;
  int seg0;
  int64_t n_out0;  // level-0 outputs per chain when there are two levels
  size_t off_first0, off_first1, off_T, off_S, total;
};

CLayout c_layout(int n_req, int max_chain, int H, int seg) {
  CLayout L;
  L.one_level = seg <= 1 || seg >= max_chain;
  L.seg0 = L.one_level ? std::max(max_chain, 1) : seg;
  L.n_out0 = L.one_level ? 0 : (max_chain + seg - 1) / seg;
  const size_t inter = (size_t)n_req * H * L.n_out0 * (size_t)kMatBytes;
  L.off_first0 = 0;
  L.off_first1 = al256((size_t)(n_req + 1) * 4);
  L.off_T = L.off_first1 + al256((size_t)(n_req + 1) * 4);
  L.off_S = L.off_T + al256(inter);
  L.total = L.off_S + al256(inter);
  return L;
}

}  // namespace
}  // namespace pic

using namespace pic;

extern "C" {

int32_t pic_compose_segment(int32_t n_req, int64_t n_elems, int32_t max_chain, int32_t H, int32_t sms) {
  if (n_req < 1 || H < 1 || max_chain < 1 || sms < 1 || n_elems < max_chain) return 0;
  // one level when the chains alone fill the SMs; else the shortest segment whose
  // level-0 CTAs (at most H * (ceil(n_elems / seg) + n_req - 1)) fit in one wave
  if ((int64_t)n_req * H >= sms) return 0;
  for (int seg = 2; seg < max_chain; ++seg)
    if ((int64_t)H * ((n_elems + seg - 1) / seg + n_req - 1) <= sms) return seg;
  return 0;
}

size_t pic_compose_workspace(int32_t n_req, int32_t max_chain, int32_t H, int32_t d, int32_t seg) {
  if (n_req < 0 || max_chain < 0 || H < 1 || d != kCD || seg < 0) return 0;
  return c_layout(n_req, max_chain, H, seg).total;
}

pic_status pic_compose_split_t(const float* T, int64_t n_mats, int32_t d, void* T_split, pic_stream_t stream) {
  if (n_mats < 0) return PIC_ERR_INVALID;
  if (d != kCD) return PIC_ERR_UNSUPPORTED;
  if (n_mats == 0) return PIC_OK;
  if (!T || !T_split || (reinterpret_cast<uintptr_t>(T) & 15) || (reinterpret_cast<uintptr_t>(T_split) & 15))
    return PIC_ERR_INVALID;
  const int64_t n = n_mats * (kElt / 4);
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)num_sms_of_current_device() * 16);
  split_t_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(T, n, static_cast<bf16*>(T_split));
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

pic_status pic_compose_states(const void* T_split, const float* S_pool, int64_t n_pool, const int32_t* ids,
                              const int32_t* chain_off, int32_t n_req, int64_t n_elems, int32_t max_chain,
                              int32_t H, int32_t d, int32_t seg, float* out, void* ws, size_t ws_bytes,
                              int32_t* err_flag, pic_stream_t stream) {
  if (n_req < 0 || n_elems < 0 || H < 1 || max_chain < 0 || max_chain > n_elems || n_pool < 0 || seg < 0)
    return PIC_ERR_INVALID;
  if (d != kCD) return PIC_ERR_UNSUPPORTED;
  if (n_req == 0) return PIC_OK;
  if (n_elems > 0 && n_pool < 1) return PIC_ERR_INVALID;
  if (!T_split || !S_pool || !ids || !chain_off || !out || !err_flag) return PIC_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(T_split) | reinterpret_cast<uintptr_t>(S_pool) |
       reinterpret_cast<uintptr_t>(out)) & 15)
    return PIC_ERR_INVALID;
  const CLayout L = c_layout(n_req, max_chain, H, seg);
  if (ws == nullptr || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PIC_ERR_WORKSPACE;
  const int64_t grid0 = (int64_t)H * ((n_elems + L.seg0 - 1) / L.seg0 + n_req);
  if (grid0 > 0x7fffffff || (int64_t)n_req * H > 0x7fffffff) return PIC_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaFuncSetAttribute(compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCSmem) != cudaSuccess)
    return PIC_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* first0 = reinterpret_cast<int32_t*>(w + L.off_first0);
  int32_t* first1 = reinterpret_cast<int32_t*>(w + L.off_first1);
  CUtensorMap t0map;
  if (!encode_t(&t0map, T_split, (uint64_t)n_pool * H * 2 * kCD)) return PIC_ERR_CUDA;
  const bool self_plan = n_req <= kCThreads;  // else a one-block planner writes the CTA counts
  if (!self_plan) {
    compose_plan_kernel<<<1, 1024, 0, s>>>(ids, chain_off, n_req, H, n_pool, n_elems, max_chain, L.seg0,
                                           L.one_level, first0, first1, err_flag);
    if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  }

  Level l0{};
  l0.T_in = static_cast<const bf16*>(T_split);
  l0.S_in = S_pool;
  l0.ids = ids;
  l0.chain_off = chain_off;
  l0.first = first0;
  l0.n_pool = n_pool;
  l0.n_elems = n_elems;
  l0.n_req = n_req;
  l0.H = H;
  l0.max_chain = max_chain;
  l0.seg = L.seg0;
  l0.seg_prev = 1;
  l0.level = 0;
  l0.last = L.one_level;
  l0.err = err_flag;
  l0.self_plan = self_plan;
  l0.one_level = L.one_level;
  if (L.one_level) {
    l0.S_out = out;
    l0.out_stride = 1;
  } else {
    l0.T_out = reinterpret_cast<bf16*>(w + L.off_T);
    l0.S_out = reinterpret_cast<float*>(w + L.off_S);
    l0.out_stride = L.n_out0;
  }
  // level-0 CTAs: at most H * (ceil(n_elems / seg0) + n_req) (one more per chain
  // for rounding, and one for an empty chain's zero state); the rest exit at once
  compose_kernel<<<(unsigned)std::max<int64_t>(grid0, 1), kCThreads, kCSmem, s>>>(t0map, l0);
  if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  if (L.one_level) return PIC_OK;

  CUtensorMap t1map;
  if (!encode_t(&t1map, w + L.off_T, (uint64_t)n_req * H * L.n_out0 * 2 * kCD)) return PIC_ERR_CUDA;
  Level l1 = l0;
  l1.T_in = l0.T_out;
  l1.S_in = l0.S_out;
  l1.ids = nullptr;
  l1.first = first1;
  l1.in_stride = L.n_out0;
  l1.T_out = nullptr;
  l1.S_out = out;
  l1.out_stride = 1;
  l1.seg = (int)std::max<int64_t>(L.n_out0, 1);
  l1.seg_prev = L.seg0;
  l1.level = 1;
  l1.last = true;
  compose_kernel<<<(unsigned)((int64_t)n_req * H), kCThreads, kCSmem, s>>>(t1map, l1);
  if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  return PIC_OK;
}

}  // extern "C"
