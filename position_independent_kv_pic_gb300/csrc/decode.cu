// Decode after link: one new query row per request attends over the request's
// linked paged cache (EPIC review: the query and the decode tokens are the ones
// that gather information across chunks; "KV cache from scratch": a single-token
// decode reads the whole cache once per step).  The step is bound by HBM: every
// cached K and V row is read once, and g query heads share each row.
//
// Split-KV: CTA (split, KV head, request) walks one span of the request's pages.
// A producer thread streams each page's K and V (4 KB each, one bulk copy apiece)
// into a ring of shared-memory stages; four consumer warps take the stages in
// turn, each keeping an online softmax for the g query heads of the KV head.  In a
// page, lane l scores key l % 16 over half l / 16 of the head dimension for all g
// heads (reading its 16-byte chunks in an order rotated by the key, so a warp's
// reads hit distinct banks), the two halves add up, and P.V runs with lane l
// owning columns 4l..4l+3.  The CTA combines its warps and writes one partial
// (m, l, unnormalised o); a merge kernel combines the splits.
#include <algorithm>

#include "pic_internal.cuh"
#include "tc_ptx.cuh"

namespace pic {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kDecD = 128;
constexpr int kDecWarps = 4;                     // consumer warps
constexpr int kDecThreads = 32 * (kDecWarps + 1);  // + the producer warp
constexpr int kDecStages = 4;                    // ring stages of one page (K and V): one per consumer warp
constexpr int kPageHead = PIC_PAGE * kDecD * 2;  // bytes of one page of one KV head
constexpr int kQPad = 12;                        // floats per 8-column chunk of Q in shared memory
constexpr int kMergeGroups = 8;   // thread groups of the merge, each over every 8th split
constexpr uint64_t kDecWaitNs = 2000000000ull;

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

struct DecLayout {
  int64_t ctas;  // upper bound of the decode grid
  size_t off_plan, off_ml, off_o, total;
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
  L.off_ml = al256((size_t)(2 * n_req + 2) * sizeof(int32_t));
  L.off_o = al256(L.off_ml + (size_t)L.ctas * G * sizeof(float2));
  L.total = al256(L.off_o + (size_t)L.ctas * G * kDecD * sizeof(float));
  return L;
}

// One block: splits per request and the first CTA of each request.
__global__ void __launch_bounds__(1024)
decode_plan_kernel(const int32_t* __restrict__ page_off, int n_req, int Hkv, int slots, int32_t* __restrict__ first,
                   int32_t* __restrict__ nsplit) {
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
}

// Two bf16 (low, high half of w) as a packed fp32 pair: a bf16 is the top half of
// the fp32 with the same value.
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
  return (uint64_t)(w << 16) | ((uint64_t)(w & 0xffff0000u) << 32);
}

// Named barrier (id 1) of all the block's warps, met by the producer after its last
// copy has landed and by the consumers after their last page.
__device__ __forceinline__ void ring_drained_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecThreads) : "memory");
}

template <int G>
struct DecSmem {
  // K page, V page per stage; once every copy has landed and been read, the ring
  // takes the warps' partial outputs
  union {
    uint8_t ring[kDecStages][2][kPageHead];
    float w_o[kDecWarps][G][kDecD];
  };
  uint64_t full[kDecStages], empty[kDecStages];
  float q[G][2][8][kQPad];                 // [head][half][chunk][8 + pad]
  float p[kDecWarps][G][PIC_PAGE];         // a page's weights, per consumer warp
  float w_m[kDecWarps][G], w_l[kDecWarps][G];
  int abort;
};

template <int G>
__global__ void __launch_bounds__(kDecThreads)
decode_kernel(const bf16* __restrict__ q, const float4* __restrict__ q_table, const bf16* __restrict__ kp,
              const bf16* __restrict__ vp, int64_t num_blocks, const pic_link_page* __restrict__ pages,
              const int32_t* __restrict__ page_off, int n_req, int Hq, int Hkv, float scale_log2,
              const int32_t* __restrict__ first, const int32_t* __restrict__ nsplit, float2* __restrict__ part_ml,
              float* __restrict__ part_o, int32_t* err) {
  extern __shared__ __align__(128) uint8_t dec_smem_raw[];
  DecSmem<G>& sm = *reinterpret_cast<DecSmem<G>*>(dec_smem_raw);
  const int cta = blockIdx.x;
  if (cta >= first[n_req]) return;  // the grid is an upper bound
  int r;
  {  // request of this CTA: the last r with first[r] <= cta
    int lo = 0, hi = n_req;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (first[mid] <= cta) lo = mid; else hi = mid;
    }
    r = lo;
  }
  const int splits = nsplit[r];
  const int kvh = (cta - first[r]) / splits, split = (cta - first[r]) % splits;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int st = 0; st < kDecStages; ++st) {
      tc::mbar_init(&sm.full[st], 1);
      tc::mbar_init(&sm.empty[st], 1);
    }
    sm.abort = 0;
    tc::fence_mbar_init();
  }
  // Q of the g heads roped at the row's position and rounded to bf16, as on the
  // link path's tensor-core operand
  for (int it = tid; it < G * kDecD / 2; it += kDecThreads) {
    const int hh = it / (kDecD / 2), i = it % (kDecD / 2);
    const bf16* src = q + ((int64_t)r * Hq + kvh * G + hh) * kDecD;
    float ya, yb;
    rope_rotate_bf16in(to_f32(src[i]), to_f32(src[i + kDecD / 2]), q_table[(int64_t)r * (kDecD / 2) + i], ya, yb);
    sm.q[hh][0][i >> 3][i & 7] = to_f32(from_f32<bf16>(ya));
    sm.q[hh][1][i >> 3][i & 7] = to_f32(from_f32<bf16>(yb));
  }
  __syncthreads();

  const int p0 = page_off[r], p1 = page_off[r + 1];
  const int per = (p1 - p0 + splits - 1) / splits;
  const int pb = p0 + split * per, pe = min(p1, pb + per);
  const int n = max(pe - pb, 0);

  if (warp == kDecWarps) {
    // ---- producer: lane 0 streams the span's pages through the ring
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % kDecStages;
        if (!tc::mbar_wait(&sm.empty[st], ((i / kDecStages) & 1) ^ 1, &sm.abort, kDecWaitNs)) {
          set_err(err, PIC_ERR_TIMEOUT);
          *reinterpret_cast<volatile int*>(&sm.abort) = 1;
          break;
        }
        const int4 pg = __ldg(reinterpret_cast<const int4*>(pages) + pb + i);
        const int lo = (int16_t)(pg.w & 0xffff), hi = (int16_t)(pg.w >> 16);
        const bool ok = pg.x >= 0 && pg.x < num_blocks && pg.y >= 0 && pg.y < num_blocks && lo >= 0 &&
                        hi <= PIC_PAGE && lo < hi;
        if (ok) {
          tc::mbar_arrive_expect_tx(&sm.full[st], 2 * kPageHead);
          tc::bulk_load(sm.ring[st][0], kp + ((int64_t)pg.x * Hkv + kvh) * PIC_PAGE * kDecD, kPageHead, &sm.full[st]);
          tc::bulk_load(sm.ring[st][1], vp + ((int64_t)pg.y * Hkv + kvh) * PIC_PAGE * kDecD, kPageHead, &sm.full[st]);
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
    // ---- consumers: warp w takes pages w, w + 4, ..
    const int key = lane & 15, half = lane >> 4;
    // o: columns 4 lane .. +3 of every head as two packed pairs; lsum: this lane's
    // share of the row sums (its key, counted in the half-0 lane only)
    float m[G], lsum[G];
    uint64_t o01[G], o23[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      m[hh] = -INFINITY;
      lsum[hh] = 0.f;
      o01[hh] = o23[hh] = 0;
    }
    for (int i = warp; i < n; i += kDecWarps) {
      const int st = i % kDecStages;
      if (!tc::mbar_wait(&sm.full[st], (i / kDecStages) & 1, &sm.abort, kDecWaitNs)) {
        if (lane == 0) {
          set_err(err, PIC_ERR_TIMEOUT);
          *reinterpret_cast<volatile int*>(&sm.abort) = 1;
        }
        break;
      }
      const int4 pg = __ldg(reinterpret_cast<const int4*>(pages) + pb + i);
      const int lo = (int16_t)(pg.w & 0xffff), hi = (int16_t)(pg.w >> 16);
      const bool ok = pg.x >= 0 && pg.x < num_blocks && pg.y >= 0 && pg.y < num_blocks && lo >= 0 &&
                      hi <= PIC_PAGE && lo < hi;
      if (!ok) {
        if (lane == 0 && !(lo >= hi && lo >= 0 && hi <= PIC_PAGE)) set_err(err, PIC_ERR_RANGE);
      } else {
        const uint8_t* kpage = sm.ring[st][0];
        const uint8_t* vpage = sm.ring[st][1];
        // scores on packed pairs (even, odd columns)
        uint64_t s2[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) s2[hh] = 0;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const int cc = (c8 + key) & 7;
          const uint4 kr = *reinterpret_cast<const uint4*>(kpage + key * (2 * kDecD) + half * kDecD + cc * 16);
          const uint64_t k2[4] = {bf16x2_to_f32x2(kr.x), bf16x2_to_f32x2(kr.y), bf16x2_to_f32x2(kr.z),
                                  bf16x2_to_f32x2(kr.w)};
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(&sm.q[hh][half][cc][0]);
            const ulonglong2 qb = *reinterpret_cast<const ulonglong2*>(&sm.q[hh][half][cc][4]);
            s2[hh] = tc::fma2(k2[0], qa.x, s2[hh]);
            s2[hh] = tc::fma2(k2[1], qa.y, s2[hh]);
            s2[hh] = tc::fma2(k2[2], qb.x, s2[hh]);
            s2[hh] = tc::fma2(k2[3], qb.y, s2[hh]);
          }
        }
        const bool valid = key >= lo && key < hi;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          float se, so;
          tc::f2unpack(s2[hh], se, so);
          float sv = se + so;
          sv += __shfl_xor_sync(0xffffffffu, sv, 16);
          sv = valid ? sv * scale_log2 : -INFINITY;
          float mx = sv;
#pragma unroll
          for (int x = 1; x < 16; x <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, x));
          const float mn = fmaxf(m[hh], mx);  // finite: the page has a valid key
          const float alpha = tc::ex2(m[hh] - mn);
          const float pv = valid ? tc::ex2(sv - mn) : 0.f;
          lsum[hh] = lsum[hh] * alpha + (half ? 0.f : pv);
          m[hh] = mn;
          const uint64_t a2 = tc::f2pack(alpha, alpha), z2 = 0;
          o01[hh] = tc::fma2(o01[hh], a2, z2);
          o23[hh] = tc::fma2(o23[hh], a2, z2);
          if (half == 0) sm.p[warp][hh][key] = pv;
        }
        __syncwarp();
#pragma unroll
        for (int k4 = 0; k4 < PIC_PAGE / 4; ++k4) {
          float4 w4[G];
#pragma unroll
          for (int hh = 0; hh < G; ++hh) w4[hh] = *reinterpret_cast<const float4*>(&sm.p[warp][hh][4 * k4]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int k2 = 4 * k4 + j;
            if (k2 < lo || k2 >= hi) continue;  // masked slots may hold anything
            const uint2 vv = *reinterpret_cast<const uint2*>(vpage + k2 * (2 * kDecD) + 8 * lane);
            const uint64_t v01 = bf16x2_to_f32x2(vv.x), v23 = bf16x2_to_f32x2(vv.y);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
              const float w = j == 0 ? w4[hh].x : j == 1 ? w4[hh].y : j == 2 ? w4[hh].z : w4[hh].w;
              const uint64_t w2 = tc::f2pack(w, w);
              o01[hh] = tc::fma2(w2, v01, o01[hh]);
              o23[hh] = tc::fma2(w2, v23, o23[hh]);
            }
          }
        }
      }
      __syncwarp();  // the weights are read before the next page writes them
      if (lane == 0) tc::mbar_arrive(&sm.empty[st]);  // the stage may be refilled
    }
    // row sums over the lanes; partials kept until the ring is free
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
#pragma unroll
      for (int x = 1; x < 32; x <<= 1) lsum[hh] += __shfl_xor_sync(0xffffffffu, lsum[hh], x);
      if (lane == 0) {
        sm.w_m[warp][hh] = m[hh];
        sm.w_l[warp][hh] = lsum[hh];
      }
    }
    ring_drained_sync();  // no copy in flight and no consumer reading: the ring takes the partials
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float a0, a1, a2v, a3;
      tc::f2unpack(o01[hh], a0, a1);
      tc::f2unpack(o23[hh], a2v, a3);
      *reinterpret_cast<float4*>(&sm.w_o[warp][hh][4 * lane]) = make_float4(a0, a1, a2v, a3);
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
  float M = -INFINITY;
  for (int s = g; s < splits; s += kMergeGroups) M = fmaxf(M, part_ml[(base + s) * G + hh].x);
  float Lsum = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = g; s < splits; s += kMergeGroups) {
    const float2 ml = part_ml[(base + s) * G + hh];
    const float4 v = reinterpret_cast<const float4*>(part_o + ((base + s) * G + hh) * kDecD)[c];
    if (ml.x == -INFINITY) continue;  // a split without keys
    const float f = tc::ex2(ml.x - M);
    Lsum += f * ml.y;
    O.x = fmaf(f, v.x, O.x); O.y = fmaf(f, v.y, O.y); O.z = fmaf(f, v.z, O.z); O.w = fmaf(f, v.w, O.w);
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
                                const int32_t* page_off, int32_t n_req, int32_t Hq, int32_t Hkv, int32_t d,
                                float scale, void* out, void* ws, size_t ws_bytes, int32_t* err_flag,
                                pic_stream_t stream) {
  if (n_req < 0 || num_blocks < 0 || !(scale > 0.f)) return PIC_ERR_INVALID;
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
  float2* part_ml = reinterpret_cast<float2*>(w + L.off_ml);
  float* part_o = reinterpret_cast<float*>(w + L.off_o);
  cudaStream_t s = (cudaStream_t)stream;
  const int slots = (int)(L.ctas - (int64_t)n_req * Hkv);
  decode_plan_kernel<<<1, 1024, 0, s>>>(page_off, n_req, Hkv, slots, first, nsplit);
  if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  const unsigned grid = (unsigned)L.ctas;
  const float sl2 = scale * 1.4426950408889634f;
  const bf16* qb = static_cast<const bf16*>(q);
  const float4* qt = reinterpret_cast<const float4*>(q_table);
  const bf16* kb = static_cast<const bf16*>(k_pool);
  const bf16* vb = static_cast<const bf16*>(v_pool);
  switch (Hq / Hkv) {
    case 1: decode_kernel<1><<<grid, kDecThreads, sizeof(DecSmem<1>), s>>>(qb, qt, kb, vb, num_blocks, pages, page_off,
        n_req, Hq, Hkv, sl2, first, nsplit, part_ml, part_o, err_flag); break;
    case 2: decode_kernel<2><<<grid, kDecThreads, sizeof(DecSmem<2>), s>>>(qb, qt, kb, vb, num_blocks, pages, page_off,
        n_req, Hq, Hkv, sl2, first, nsplit, part_ml, part_o, err_flag); break;
    case 4: decode_kernel<4><<<grid, kDecThreads, sizeof(DecSmem<4>), s>>>(qb, qt, kb, vb, num_blocks, pages, page_off,
        n_req, Hq, Hkv, sl2, first, nsplit, part_ml, part_o, err_flag); break;
    default: decode_kernel<8><<<grid, kDecThreads, sizeof(DecSmem<8>), s>>>(qb, qt, kb, vb, num_blocks, pages,
        page_off, n_req, Hq, Hkv, sl2, first, nsplit, part_ml, part_o, err_flag); break;
  }
  if (cudaGetLastError() != cudaSuccess) return PIC_ERR_CUDA;
  decode_merge_kernel<<<dim3((unsigned)Hq, (unsigned)n_req), 32 * kMergeGroups, 0, s>>>(
      part_ml, part_o, static_cast<bf16*>(out), Hq, Hkv, first, nsplit);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

}  // extern "C"
