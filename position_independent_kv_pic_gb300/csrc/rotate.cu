// Rotary correction of cached K (article on RoPE and prefix caching, section
// 3.3): a K cached at local position j is moved to global position j + Delta by
// ONE rotation R(theta * Delta) of every dimension pair (i, i + d/2), with
// cos/sin taken from a per-offset table.  Also the fresh K/V writer of the
// recomputed rows (EPIC link_legolink Step 3).
//
// Both are HBM-bound streaming passes.  One work item is one 16-byte vector of
// the low half of a key row plus the matching vector of its high half (the
// pair partners), so every warp access is a run of full 32-byte sectors; the
// cos/sin vectors come from a small table that stays in L1/L2.
#include "pic_internal.cuh"

namespace pic {
namespace {

constexpr int kRotThreads = 128;
constexpr int kRotUnroll = 4;  // independent items in flight per thread

template <typename T> struct Vec16;
template <> struct Vec16<__nv_bfloat16> { static constexpr int N = 8; };
template <> struct Vec16<float> { static constexpr int N = 4; };

template <typename T>
__device__ __forceinline__ void unpack(const uint4& v, float* f) {
  if constexpr (sizeof(T) == 2) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  } else {
    const float* s = reinterpret_cast<const float*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = s[i];
  }
}

template <typename T>
__device__ __forceinline__ uint4 pack(const float* f) {
  uint4 v;
  if constexpr (sizeof(T) == 2) {
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  } else {
    float* s = reinterpret_cast<float*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] = f[i];
  }
  return v;
}

template <int N>
__device__ __forceinline__ void rotate(float* lo, float* hi, const float4* cs) {
#pragma unroll
  for (int i = 0; i < N; ++i) rope_rotate(lo[i], hi[i], cs[i], lo[i], hi[i]);
}

// Rotate one 16-byte vector of low-half elements against the matching vector of
// high-half elements, word by word (keeps few values live).
template <typename T>
__device__ __forceinline__ void rotate_vec(const uint4& xl, const uint4& xh, const float4* cs, uint4& ol,
                                           uint4& oh) {
  const uint32_t* wl = reinterpret_cast<const uint32_t*>(&xl);
  const uint32_t* wh = reinterpret_cast<const uint32_t*>(&xh);
  uint32_t* vl = reinterpret_cast<uint32_t*>(&ol);
  uint32_t* vh = reinterpret_cast<uint32_t*>(&oh);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    if constexpr (sizeof(T) == 2) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wl[w]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wh[w]));
      float y0, z0, y1, z1;
      rope_rotate_bf16in(a.x, b.x, cs[2 * w], y0, z0);
      rope_rotate_bf16in(a.y, b.y, cs[2 * w + 1], y1, z1);
      __nv_bfloat162 p = __floats2bfloat162_rn(y0, y1), q = __floats2bfloat162_rn(z0, z1);
      vl[w] = *reinterpret_cast<uint32_t*>(&p);
      vh[w] = *reinterpret_cast<uint32_t*>(&q);
    } else {
      float y, z;
      rope_rotate(__uint_as_float(wl[w]), __uint_as_float(wh[w]), cs[w], y, z);
      vl[w] = __float_as_uint(y);
      vh[w] = __float_as_uint(z);
    }
  }
}

template <int N>
__device__ __forceinline__ void load_cs(const float4* __restrict__ p, float4* cs) {
#pragma unroll
  for (int i = 0; i < N; ++i) cs[i] = __ldg(p + i);
}

// One block per page entry at a time (grid-stride over entries).  Within an
// entry, item = (head h, slot s, vector v), v fastest, so a warp covers four
// 256-byte key rows with full sectors.  The entry record is read once per block
// (uniform), there is no 64-bit index division, and each thread keeps the cos/sin
// of its vector while the vector index stays the same.
template <typename T>
__global__ void __launch_bounds__(kRotThreads, 4)
rerotate_kernel(T* __restrict__ pool, int64_t num_blocks, int Hkv, int d,
                const pic_rot_page* __restrict__ rot, int64_t n_rot, const float4* __restrict__ table,
                int64_t n_tab, int32_t* err) {
  constexpr int N = Vec16<T>::N;
  const int half = d / 2;
  const int G = half / N;
  const int per_entry = Hkv * PIC_PAGE * G;
  const int hs = d * PIC_PAGE;  // elements of one (block, head) slice
  // the next entry's record is loaded while this one streams, so the record's
  // latency is not paid in front of every entry's data loads
  pic_rot_page rp_next = {0, 0, 0, 0, 0};
  if (blockIdx.x < n_rot) rp_next = rot[blockIdx.x];
  for (int64_t e = blockIdx.x; e < n_rot; e += gridDim.x) {
    const pic_rot_page rp = rp_next;
    if (e + gridDim.x < n_rot) rp_next = rot[e + gridDim.x];
    if (rp.src_block < 0 || rp.src_block >= num_blocks || rp.dst_block < 0 || rp.dst_block >= num_blocks ||
        rp.tab < 0 || rp.tab >= n_tab || rp.lo < 0 || rp.hi > PIC_PAGE) {
      if (threadIdx.x == 0) set_err(err, PIC_ERR_RANGE);
      continue;
    }
    const T* src_base = pool + (int64_t)rp.src_block * Hkv * hs;
    T* dst_base = pool + (int64_t)rp.dst_block * Hkv * hs;
    const float4* tab = table + (int64_t)rp.tab * half;
    int v_have = -1;
    float4 cs[N];
    for (int base = 0; base < per_entry; base += kRotThreads * kRotUnroll) {
      uint4 xl[kRotUnroll], xh[kRotUnroll];
      int off[kRotUnroll], vv[kRotUnroll];
      bool act[kRotUnroll];
#pragma unroll
      for (int u = 0; u < kRotUnroll; ++u) {
        const int it = base + u * kRotThreads + threadIdx.x;
        const int v = it % G;
        const int sl = (it / G) % PIC_PAGE;
        const int h = it / (G * PIC_PAGE);
        act[u] = it < per_entry && sl >= rp.lo && sl < rp.hi;
        off[u] = h * hs + sl * d + v * N;
        vv[u] = v;
        if (act[u]) {
          xl[u] = __ldcs(reinterpret_cast<const uint4*>(src_base + off[u]));
          xh[u] = __ldcs(reinterpret_cast<const uint4*>(src_base + off[u] + half));
        }
      }
#pragma unroll
      for (int u = 0; u < kRotUnroll; ++u) {
        if (!act[u]) continue;
        if (vv[u] != v_have) {
          load_cs<N>(tab + vv[u] * N, cs);
          v_have = vv[u];
        }
        uint4 ol, oh;
        rotate_vec<T>(xl[u], xh[u], cs, ol, oh);
        __stcs(reinterpret_cast<uint4*>(dst_base + off[u]), ol);
        __stcs(reinterpret_cast<uint4*>(dst_base + off[u] + half), oh);
      }
    }
  }
}

// Scheme B (article on RoPE and prefix caching, section 3.2): a chunk's K cached
// without its position encoding is encoded on link at its global positions: slot
// s of page j of chunk c gets RoPE at s_c + 16 j + s, from a table with one row
// per position (a per-model table; composing each angle from a chunk-offset row
// and a chunk-local row instead, by compensated angle addition, kept HBM to K
// alone but made the pass slower: 105 vs 89 us on the long-context link).  The
// work items are the rotation kernel's; the page's chunk and request come from
// binary searches over the page and chunk offsets, and the kept slots are those
// not recomputed (the first min(k, L_c) rows of every chunk after the first are
// replaced by fresh rows).  Out of place (every chunk, the first too, encoded into
// private pages) when chunks are shared by requests.
template <typename T>
__global__ void __launch_bounds__(kRotThreads, 4)
rope_cached_kernel(T* __restrict__ pool, int64_t num_blocks, int Hkv, int d, const int32_t* __restrict__ chunk_lens,
                   const int32_t* __restrict__ chunk_off, const int32_t* __restrict__ kk, int n_req,
                   const int32_t* __restrict__ chunk_start, const int32_t* __restrict__ chunk_page_off,
                   int n_chunks, int64_t n_cpages, const int32_t* __restrict__ k_src,
                   const int32_t* __restrict__ k_dst, const float4* __restrict__ table, int64_t n_pos,
                   int32_t* err) {
  constexpr int N = Vec16<T>::N;
  const int half = d / 2;
  const int G = half / N;
  const int per_entry = Hkv * PIC_PAGE * G;
  const int hs = d * PIC_PAGE;
  __shared__ int s_c, s_r;
  for (int64_t cp = blockIdx.x; cp < n_cpages; cp += gridDim.x) {
    if (threadIdx.x == 0) {
      int lo = 0, hi = n_chunks;  // last c with chunk_page_off[c] <= cp
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (chunk_page_off[mid] <= cp) lo = mid; else hi = mid;
      }
      s_c = lo;
      int a = 0, b = n_req;  // last r with chunk_off[r] <= c
      while (b - a > 1) {
        const int mid = (a + b) >> 1;
        if (chunk_off[mid] <= lo) a = mid; else b = mid;
      }
      s_r = a;
    }
    __syncthreads();
    const int c = s_c, r = s_r;
    __syncthreads();  // read before the next page's search writes them
    const int j = (int)(cp - chunk_page_off[c]);
    const int L = chunk_lens[c];
    const int m = (c == chunk_off[r]) ? 0 : min(kk[r], L);
    const int slo = max(0, m - PIC_PAGE * j), shi = min(PIC_PAGE, L - PIC_PAGE * j);
    if (slo >= shi) continue;
    const int64_t pos0 = (int64_t)chunk_start[c] + PIC_PAGE * j;
    const int src = k_src[cp], dst = (k_dst != nullptr) ? k_dst[cp] : src;
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || pos0 < 0 || pos0 + shi > n_pos) {
      if (threadIdx.x == 0) set_err(err, PIC_ERR_RANGE);
      continue;
    }
    const T* src_base = pool + (int64_t)src * Hkv * hs;
    T* dst_base = pool + (int64_t)dst * Hkv * hs;
    int key_have = -1;  // (slot, vector) whose cos/sin the thread holds
    float4 cs[N];
    for (int base = 0; base < per_entry; base += kRotThreads * kRotUnroll) {
      uint4 xl[kRotUnroll], xh[kRotUnroll];
      int off[kRotUnroll], key[kRotUnroll];
      bool act[kRotUnroll];
#pragma unroll
      for (int u = 0; u < kRotUnroll; ++u) {
        const int it = base + u * kRotThreads + threadIdx.x;
        const int v = it % G;
        const int sl = (it / G) % PIC_PAGE;
        const int h = it / (G * PIC_PAGE);
        act[u] = it < per_entry && sl >= slo && sl < shi;
        off[u] = h * hs + sl * d + v * N;
        key[u] = sl * G + v;
        if (act[u]) {
          xl[u] = __ldcs(reinterpret_cast<const uint4*>(src_base + off[u]));
          xh[u] = __ldcs(reinterpret_cast<const uint4*>(src_base + off[u] + half));
        }
      }
#pragma unroll
      for (int u = 0; u < kRotUnroll; ++u) {
        if (!act[u]) continue;
        if (key[u] != key_have) {
          const int sl = key[u] / G, v = key[u] % G;
          load_cs<N>(table + (pos0 + sl) * half + v * N, cs);
          key_have = key[u];
        }
        uint4 ol, oh;
        rotate_vec<T>(xl[u], xh[u], cs, ol, oh);
        __stcs(reinterpret_cast<uint4*>(dst_base + off[u]), ol);
        __stcs(reinterpret_cast<uint4*>(dst_base + off[u] + half), oh);
      }
    }
  }
}

// Fresh rows: item = (row i, head h, vector v).  K is roped at the row's global
// position (row table), V is copied.
template <typename T>
__global__ void __launch_bounds__(kRotThreads)
write_fresh_kernel(T* __restrict__ kpool, T* __restrict__ vpool, int64_t num_blocks, int Hkv, int d,
                   const T* __restrict__ k_raw, const T* __restrict__ v_raw,
                   const float4* __restrict__ row_table, const int32_t* __restrict__ row_block,
                   const int32_t* __restrict__ row_slot, int64_t n_rows, int32_t* err) {
  constexpr int N = Vec16<T>::N;
  const int half = d / 2;
  const int G = half / N;
  const int64_t per_row = (int64_t)Hkv * G;
  const int64_t total = n_rows * per_row;
  for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < total;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = it / per_row;
    const int rem = (int)(it - i * per_row);
    const int v = rem % G;
    const int h = rem / G;
    const int b = row_block[i], s = row_slot[i];
    if (b < 0 || b >= num_blocks || s < 0 || s >= PIC_PAGE) {
      set_err(err, PIC_ERR_RANGE);
      continue;
    }
    const int64_t src = (i * Hkv + h) * (int64_t)d + v * N;
    const int64_t dst = (((int64_t)b * Hkv + h) * PIC_PAGE + s) * d + v * N;
    const uint4 kl = *reinterpret_cast<const uint4*>(k_raw + src);
    const uint4 kh = *reinterpret_cast<const uint4*>(k_raw + src + half);
    const uint4 vl = *reinterpret_cast<const uint4*>(v_raw + src);
    const uint4 vh = *reinterpret_cast<const uint4*>(v_raw + src + half);
    float4 cs[N];
    load_cs<N>(row_table + i * half + v * N, cs);
    uint4 ol, oh;
    rotate_vec<T>(kl, kh, cs, ol, oh);
    *reinterpret_cast<uint4*>(kpool + dst) = ol;
    *reinterpret_cast<uint4*>(kpool + dst + half) = oh;
    *reinterpret_cast<uint4*>(vpool + dst) = vl;
    *reinterpret_cast<uint4*>(vpool + dst + half) = vh;
  }
}

int grid_for(int64_t items) {
  const int sms = num_sms_of_current_device();
  const int64_t want = (items + kRotThreads * kRotUnroll - 1) / (kRotThreads * kRotUnroll);
  const int64_t cap = (int64_t)sms * 8;  // 8 blocks of 256 threads fill an SM
  return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

bool shape_ok(pic_dtype dt, int Hkv, int d) {
  if (Hkv < 1 || d < 2 || d > 256 || (d & 1)) return false;
  const int n = (dt == PIC_BF16) ? 8 : 4;
  return (d / 2) % n == 0;
}

}  // namespace

int num_sms_of_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

}  // namespace pic

using namespace pic;

extern "C" {

pic_status pic_rerotate_k(void* k_pool, int64_t num_blocks, pic_dtype dtype, int32_t Hkv, int32_t d,
                          const pic_rot_page* rot, int64_t n_rot, const float* table, int64_t n_tab,
                          int32_t* err_flag, pic_stream_t stream) {
  if (n_rot < 0 || num_blocks < 0 || n_tab < 0) return PIC_ERR_INVALID;
  if (dtype != PIC_BF16 && dtype != PIC_FP32) return PIC_ERR_INVALID;
  if (!shape_ok(dtype, Hkv, d)) return (d > 0 && !(d & 1)) ? PIC_ERR_UNSUPPORTED : PIC_ERR_INVALID;
  if (n_rot == 0) return PIC_OK;
  if (!k_pool || !rot || !table || !err_flag) return PIC_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(k_pool) & 15) || (reinterpret_cast<uintptr_t>(table) & 15))
    return PIC_ERR_INVALID;
  const int sms = num_sms_of_current_device();
  const int64_t cap = (int64_t)sms * 4;  // one wave: 4 resident blocks of 128 threads per SM
  const int grid = (int)(n_rot < cap ? n_rot : cap);
  if (dtype == PIC_BF16)
    rerotate_kernel<__nv_bfloat16><<<grid, kRotThreads, 0, (cudaStream_t)stream>>>(
        static_cast<__nv_bfloat16*>(k_pool), num_blocks, Hkv, d, rot, n_rot,
        reinterpret_cast<const float4*>(table), n_tab, err_flag);
  else
    rerotate_kernel<float><<<grid, kRotThreads, 0, (cudaStream_t)stream>>>(
        static_cast<float*>(k_pool), num_blocks, Hkv, d, rot, n_rot,
        reinterpret_cast<const float4*>(table), n_tab, err_flag);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

pic_status pic_rope_cached_k(void* k_pool, int64_t num_blocks, pic_dtype dtype, int32_t Hkv, int32_t d,
                             const int32_t* chunk_lens, const int32_t* chunk_off, const int32_t* k, int32_t n_req,
                             const int32_t* chunk_start, const int32_t* chunk_page_off, int32_t n_chunks,
                             int64_t n_chunk_pages, const int32_t* k_src_blocks, const int32_t* k_dst_blocks,
                             const float* pos_table, int64_t n_pos, int32_t* err_flag, pic_stream_t stream) {
  if (n_req < 0 || n_chunks < 0 || n_chunk_pages < 0 || num_blocks < 0 || n_pos < 0) return PIC_ERR_INVALID;
  if (dtype != PIC_BF16 && dtype != PIC_FP32) return PIC_ERR_INVALID;
  if (!shape_ok(dtype, Hkv, d)) return (d > 0 && !(d & 1)) ? PIC_ERR_UNSUPPORTED : PIC_ERR_INVALID;
  if (n_req == 0 || n_chunk_pages == 0) return PIC_OK;
  if (!k_pool || !chunk_lens || !chunk_off || !k || !chunk_start || !chunk_page_off || !k_src_blocks ||
      !pos_table || !err_flag)
    return PIC_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(k_pool) & 15) || (reinterpret_cast<uintptr_t>(pos_table) & 15))
    return PIC_ERR_INVALID;
  const int64_t cap = (int64_t)num_sms_of_current_device() * 4;
  const int grid = (int)(n_chunk_pages < cap ? n_chunk_pages : cap);
  if (dtype == PIC_BF16)
    rope_cached_kernel<__nv_bfloat16><<<grid, kRotThreads, 0, (cudaStream_t)stream>>>(
        static_cast<__nv_bfloat16*>(k_pool), num_blocks, Hkv, d, chunk_lens, chunk_off, k, n_req, chunk_start,
        chunk_page_off, n_chunks, n_chunk_pages, k_src_blocks, k_dst_blocks,
        reinterpret_cast<const float4*>(pos_table), n_pos, err_flag);
  else
    rope_cached_kernel<float><<<grid, kRotThreads, 0, (cudaStream_t)stream>>>(
        static_cast<float*>(k_pool), num_blocks, Hkv, d, chunk_lens, chunk_off, k, n_req, chunk_start,
        chunk_page_off, n_chunks, n_chunk_pages, k_src_blocks, k_dst_blocks,
        reinterpret_cast<const float4*>(pos_table), n_pos, err_flag);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

pic_status pic_write_fresh_kv(void* k_pool, void* v_pool, int64_t num_blocks, pic_dtype dtype,
                              int32_t Hkv, int32_t d, const void* k_raw, const void* v_raw,
                              const float* row_table, const int32_t* row_block,
                              const int32_t* row_slot, int64_t n_rows, int32_t* err_flag,
                              pic_stream_t stream) {
  if (n_rows < 0 || num_blocks < 0) return PIC_ERR_INVALID;
  if (dtype != PIC_BF16 && dtype != PIC_FP32) return PIC_ERR_INVALID;
  if (!shape_ok(dtype, Hkv, d)) return (d > 0 && !(d & 1)) ? PIC_ERR_UNSUPPORTED : PIC_ERR_INVALID;
  if (n_rows == 0) return PIC_OK;
  if (!k_pool || !v_pool || !k_raw || !v_raw || !row_table || !row_block || !row_slot || !err_flag)
    return PIC_ERR_INVALID;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool) |
                        reinterpret_cast<uintptr_t>(k_raw) | reinterpret_cast<uintptr_t>(v_raw) |
                        reinterpret_cast<uintptr_t>(row_table);
  if (mis & 15) return PIC_ERR_INVALID;
  const int n = (dtype == PIC_BF16) ? 8 : 4;
  const int64_t items = n_rows * Hkv * (d / 2 / n);
  const int grid = grid_for(items * kRotUnroll);
  if (dtype == PIC_BF16)
    write_fresh_kernel<__nv_bfloat16><<<grid, kRotThreads, 0, (cudaStream_t)stream>>>(
        static_cast<__nv_bfloat16*>(k_pool), static_cast<__nv_bfloat16*>(v_pool), num_blocks, Hkv, d,
        static_cast<const __nv_bfloat16*>(k_raw), static_cast<const __nv_bfloat16*>(v_raw),
        reinterpret_cast<const float4*>(row_table), row_block, row_slot, n_rows, err_flag);
  else
    write_fresh_kernel<float><<<grid, kRotThreads, 0, (cudaStream_t)stream>>>(
        static_cast<float*>(k_pool), static_cast<float*>(v_pool), num_blocks, Hkv, d,
        static_cast<const float*>(k_raw), static_cast<const float*>(v_raw),
        reinterpret_cast<const float4*>(row_table), row_block, row_slot, n_rows, err_flag);
  return cudaGetLastError() == cudaSuccess ? PIC_OK : PIC_ERR_CUDA;
}

}  // extern "C"
