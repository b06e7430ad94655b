// SIMT link attention for fp32 pools and bf16 shapes outside the tensor-core
// path (EPIC blog review, link_legolink Step 3; offset causal mask of the
// KV-cache blog).  Same inputs and semantics as the tensor-core kernel.
#include "pic_internal.cuh"

namespace pic {
namespace {

using bf16 = __nv_bfloat16;

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

}  // namespace

pic_status launch_attention_simt(const void* q, const float* row_table, const int32_t* rows,
                                 const int32_t* row_off, const void* k_pool, const void* v_pool,
                                 int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                                 const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                                 int32_t Hkv, int32_t d, float scale, void* out, cudaStream_t s) {
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

}  // namespace pic
