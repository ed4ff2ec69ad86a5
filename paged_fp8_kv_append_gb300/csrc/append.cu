// append.cu -- kv_append_quantize: page allocation with tag stamping, then
// quantise-on-write of the new K/V rows into the paged cache.
//
// "Smaller, faster, safer: running Kimi and GLM at scale":
//   section "Quantizing the KV cache"   -- the cache holds FP8 e4m3;
//   section "Protecting a shared KV cache" -- each physical page's tag
//   changes whenever the page is reallocated.
//
// Two launches:
//  1. append_plan (one CTA): requests are served in index order.  A block-wide
//     scan of the pages each request needs gives every request its slice of
//     the free list, so pops come out exactly as a sequential walk would.  The
//     first request that cannot be served stops the call; it and all later
//     requests are untouched.  Popped pages get tag += 1; page_table,
//     exp_tags and seq_lens are updated; ctl gets the new free head, the stop
//     index and the error code.
//  2. append_data (one CTA per (request, touched page, kv head, K|V)): reads
//     the request's rows for that page, computes the amax of a fresh page
//     (K and V separately), scale = amax/448 (IEEE division; 1 when 0), and stores
//     e4m3(x / scale) with round-to-nearest-even and saturation; a page that
//     already held rows keeps its scale.  bf16 pools copy the bits.
#include "common.cuh"
#include "internal.h"

namespace kvfp8 {

namespace {

constexpr int kPlanThreads = 1024;

// Inclusive block scan of a 64-bit value over kPlanThreads threads.
__device__ long long block_incl_scan(long long v, long long* warp_sums) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  if (wid == 0) {
    long long w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  long long r = v + (wid > 0 ? warp_sums[wid - 1] : 0);
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kPlanThreads) append_plan_kernel(AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ long long warp_sums[32];
  __shared__ int s_stop, s_code;
  __shared__ long long s_consumed_at_stop, s_chunk_total;
  const kv_pool_desc& d = a.d;
  const long long P = d.page_size;
  const long long head0 = a.d.ctl[KV_CTL_FREE_HEAD];
  long long consumed = 0;
  int stop = a.B, stop_code = 0;
  if (head0 < 0 || head0 > d.num_pages) {  // corrupt control block: serve nothing
    if (threadIdx.x == 0) {
      d.ctl[KV_CTL_APPEND_STOP] = 0;
      set_error(d.ctl, KV_ERR_INVALID_ARG);
    }
    return;
  }

  for (int base = 0; base < a.B; base += kPlanThreads) {
    const int r = base + threadIdx.x;
    long long need = 0, L = 0, n = 0, first = 0;
    int code = 0;
    if (r < a.B) {
      L = a.seq_lens[r];
      n = (long long)a.new_indptr[r + 1] - a.new_indptr[r];
      if (n < 0 || L < 0 || n > a.max_new || L + n > (long long)a.max_pages * P) {
        code = KV_ERR_INVALID_ARG;
      } else {
        if (n > 0 && L % P != 0) {
          // rows go into the partly filled last page: check its mapping like
          // a read, so a page reallocated since is never written
          const long long jl = L / P;
          const int p = a.page_table[(long long)r * a.max_pages + jl];
          if (p < 0 || p >= d.num_pages)
            code = KV_ERR_BAD_PAGE_ID;
          else if (d.tags[p] != a.exp_tags[(long long)r * a.max_pages + jl])
            code = KV_ERR_TAG_MISMATCH;
        }
        first = (L + P - 1) / P;
        need = (L + n + P - 1) / P - first;
      }
    }
    const long long incl = block_incl_scan(need, warp_sums);
    const long long excl = incl - need;
    const long long pos0 = head0 + consumed + excl;  // this request's free-list slice
    if (r < a.B && code == 0) {
      if (pos0 + need > d.num_pages) {
        code = KV_ERR_OUT_OF_PAGES;
      } else {
        for (long long j = 0; j < need; ++j) {
          const int p = d.free_list[pos0 + j];
          if (p < 0 || p >= d.num_pages) {
            code = KV_ERR_BAD_PAGE_ID;
            break;
          }
        }
      }
    }
    if (threadIdx.x == 0) {
      s_stop = a.B;
      s_code = 0;
    }
    __syncthreads();
    if (code != 0) atomicMin(&s_stop, r);
    __syncthreads();
    const int chunk_stop = s_stop;
    if (r == chunk_stop) {
      s_code = code;
      s_consumed_at_stop = excl;
    }
    if (threadIdx.x == kPlanThreads - 1) s_chunk_total = incl;
    __syncthreads();
    if (r < a.B && r < chunk_stop) {
      for (long long j = 0; j < need; ++j) {
        const int p = d.free_list[pos0 + j];
        const uint32_t t = d.tags[p] + 1u;  // wraps mod 2^32
        d.tags[p] = t;
        a.page_table[(long long)r * a.max_pages + first + j] = p;
        a.exp_tags[(long long)r * a.max_pages + first + j] = t;
      }
      a.seq_lens[r] = (int32_t)(L + n);
    }
    if (chunk_stop < a.B) {
      consumed += s_consumed_at_stop;
      stop = chunk_stop;
      stop_code = s_code;
      break;
    }
    consumed += s_chunk_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    d.ctl[KV_CTL_FREE_HEAD] = (int32_t)(head0 + consumed);
    d.ctl[KV_CTL_APPEND_STOP] = stop;
    if (stop_code != 0) set_error(d.ctl, stop_code);
  }
}

constexpr int kDataThreads = 256;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) {
  return __uint_as_float((b & 0xFFFFu) << 16);
}

__device__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) red[wid] = v;
  __syncthreads();
  if (wid == 0) {
    float w = lane < (kDataThreads / 32) ? red[lane] : 0.0f;
    w = warp_max(w);
    if (lane == 0) red[8] = w;
  }
  __syncthreads();
  float r = red[8];
  __syncthreads();
  return r;
}

// e4m3 codes of x / scale for two values (x0 -> low byte): IEEE fp32
// division, then the hardware round-to-nearest-even saturating conversion.
__device__ __forceinline__ uint32_t quant2(float x0, float x1, float scale) {
  const float2 q = make_float2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale));
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3)) & 0xFFFFu;
}

// Scale of a fresh block: amax / 448 in fp32; 1 when that is 0.
__device__ __forceinline__ float scale_from_amax(float amax) {
  const float s = __fdiv_rn(amax, 448.0f);
  return s > 0.0f ? s : 1.0f;
}

__device__ __forceinline__ float amax8(uint4 v) {
  float m = 0.0f;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    m = fmaxf(m, fabsf(bf16_bits_to_f32(w[k])));
    m = fmaxf(m, fabsf(bf16_bits_to_f32(w[k] >> 16)));
  }
  return m;
}

// 8 bf16 values -> 8 e4m3 codes (byte k = element k)
__device__ __forceinline__ uint2 quant8(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = quant2(bf16_bits_to_f32(w[k]), bf16_bits_to_f32(w[k] >> 16), s);
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// One block of rows for one (page, kv head, K-or-V): `nrows` source rows of
// D bf16 values, row i at src + i * src_stride (elements).  Pass 1 finds the
// amax (fresh e4m3 blocks only), pass 2 quantises (or copies) and stores.
// Token-major destination (K, latent): row i at dst + (slot0 + i) * D.
// Dim-major destination (GQA V): element (i, dd) at dst + dd * P + slot0 + i,
// assembled in shared memory and written one dim row at a time.
__device__ void append_block(const uint16_t* src, long long src_stride, int nrows, int D,
                             bool fp8, bool fresh, float* scale_slot, void* dst,
                             bool dim_major, int P, int slot0, uint8_t* tile, float* red) {
  const int tpr = D / 8;                       // threads per row (16-byte loads)
  const int rpp = kDataThreads / tpr;          // rows per pass
  const int c = threadIdx.x % tpr, i_off = threadIdx.x / tpr;
  const bool active = i_off < rpp;
  float s = 1.0f;
  if (fp8) {
    if (fresh) {
      float m = 0.0f;
      for (int i0 = 0; i0 < nrows; i0 += rpp) {
        const int i = i0 + i_off;
        if (active && i < nrows)
          m = fmaxf(m, amax8(*reinterpret_cast<const uint4*>(src + i * src_stride + 8 * c)));
      }
      m = block_max(m, red);
      s = scale_from_amax(m);
      if (threadIdx.x == 0) *scale_slot = s;
    } else {
      s = *scale_slot;
    }
  }
  for (int i0 = 0; i0 < nrows; i0 += rpp) {
    const int i = i0 + i_off;
    if (!(active && i < nrows)) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(src + i * src_stride + 8 * c);
    if (!dim_major) {
      if (fp8)
        *reinterpret_cast<uint2*>(static_cast<uint8_t*>(dst) + (long long)(slot0 + i) * D + 8 * c) =
            quant8(v, s);
      else
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst) + (long long)(slot0 + i) * D + 8 * c) = v;
    } else {
      const int slot = slot0 + i;
      if (fp8) {
        const uint2 q = quant8(v, s);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tile[(8 * c + k) * P + slot] = (uint8_t)(((k < 4 ? q.x : q.y) >> (8 * (k & 3))) & 0xFFu);
      } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint16_t* t16 = reinterpret_cast<uint16_t*>(tile);
#pragma unroll
        for (int k = 0; k < 8; ++k) t16[(8 * c + k) * P + slot] = (uint16_t)(w[k >> 1] >> (16 * (k & 1)));
      }
    }
  }
  if (dim_major) {
    __syncthreads();
    const int es = fp8 ? 1 : 2;
    if (nrows == P && (P * es) % 16 == 0) {
      // whole page: copy the tile out in 16-byte chunks
      const int chunks = D * P * es / 16;
      for (int k = threadIdx.x; k < chunks; k += kDataThreads)
        reinterpret_cast<uint4*>(dst)[k] = reinterpret_cast<const uint4*>(tile)[k];
    } else {
      const int nel = D * nrows;
      for (int e = threadIdx.x; e < nel; e += kDataThreads) {
        const int dd = e / nrows, i = e - dd * nrows;
        const int o = dd * P + slot0 + i;
        if (fp8)
          static_cast<uint8_t*>(dst)[o] = tile[o];
        else
          static_cast<uint16_t*>(dst)[o] = reinterpret_cast<const uint16_t*>(tile)[o];
      }
    }
    __syncthreads();
  }
}

// One (request, touched page, kv head, K|V) per CTA (blockIdx.z = 2 * head +
// {0: K, 1: V}; latent pools use z = 0 only), so a decode-step append of one
// row per request is a short chain of memory round trips.
__global__ void __launch_bounds__(kDataThreads) append_data_kernel(AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[9];
  extern __shared__ __align__(16) uint8_t tile[];
  const kv_pool_desc& d = a.d;
  const int r = blockIdx.x;
  if (r >= d.ctl[KV_CTL_APPEND_STOP]) return;
  const long long n = (long long)a.new_indptr[r + 1] - a.new_indptr[r];
  if (n <= 0) return;
  const long long P = d.page_size;
  const long long Lnew = a.seq_lens[r];
  const long long L0 = Lnew - n;
  const bool fp8 = d.dtype == KV_DTYPE_E4M3;
  const int H = d.num_kv_heads, Dk = d.head_dim_k, Dv = d.head_dim_v;
  const int h = blockIdx.z >> 1;
  const bool is_v = (blockIdx.z & 1) != 0;
  for (long long jp = L0 / P + blockIdx.y; jp * P < Lnew; jp += gridDim.y) {
    const long long pos_lo = max(jp * P, L0), pos_hi = min((jp + 1) * P, Lnew);
    const int nrows = (int)(pos_hi - pos_lo);
    const int slot0 = (int)(pos_lo - jp * P);
    const long long row0 = a.new_indptr[r] + (pos_lo - L0);
    const int p = a.page_table[(long long)r * a.max_pages + jp];
    if (p < 0 || p >= d.num_pages) {
      if (threadIdx.x == 0) set_error(d.ctl, KV_ERR_BAD_PAGE_ID);
      return;  // uniform across the block
    }
    const bool fresh = jp * P >= L0;  // popped by this call
    if (d.layout == KV_LAYOUT_LATENT) {
      append_block(a.k_new + row0 * Dk, Dk, nrows, Dk, true, fresh, d.k_scale + p,
                   static_cast<uint8_t*>(d.k_cache) + (long long)p * P * Dk, false, (int)P,
                   slot0, tile, red);
      continue;
    }
    const int es = fp8 ? 1 : 2;
    if (!is_v) {
      const long long kp = (((long long)p * H + h) * P) * Dk;
      append_block(a.k_new + (row0 * H + h) * Dk, (long long)H * Dk, nrows, Dk, fp8, fresh,
                   fp8 ? d.k_scale + (long long)p * H + h : nullptr,
                   static_cast<uint8_t*>(d.k_cache) + kp * es, false, (int)P, slot0, tile, red);
    } else {
      const long long vp = ((long long)p * H + h) * (long long)Dv * P;
      append_block(a.v_new + (row0 * H + h) * Dv, (long long)H * Dv, nrows, Dv, fp8, fresh,
                   fp8 ? d.v_scale + (long long)p * H + h : nullptr,
                   static_cast<uint8_t*>(d.v_cache) + vp * es, true, (int)P, slot0, tile, red);
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s, int* launches) {
  cudaError_t e = launch_pdl(append_plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  ++*launches;
  // pages a request can touch in one call: ceil((max_new + P - 1) / P)
  const long long P = a.d.page_size;
  long long pieces = (a.max_new + 2 * P - 2) / P;
  if (pieces <= 0 || a.B <= 0) return cudaSuccess;
  if (pieces > 65535) pieces = 65535;  // the kernel strides over the rest
  const size_t tile_bytes = a.d.layout == KV_LAYOUT_GQA
                                ? (size_t)a.d.head_dim_v * a.d.page_size *
                                      (a.d.dtype == KV_DTYPE_E4M3 ? 1 : 2)
                                : 0;
  if (tile_bytes > 48 * 1024) {
    e = cudaFuncSetAttribute(append_data_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tile_bytes);
    if (e != cudaSuccess) return e;
  }
  const unsigned items = a.d.layout == KV_LAYOUT_GQA ? 2u * (unsigned)a.d.num_kv_heads : 1u;
  dim3 grid((unsigned)a.B, (unsigned)pieces, items);
  e = launch_pdl(append_data_kernel, grid, dim3(kDataThreads), tile_bytes, s, a);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace kvfp8
