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
//     already held rows keeps its scale.  bf16 pools copy the bits.  A partly
//     filled page whose tag this call changed (a later request popped it) is
//     not written through the stale mapping.
#include <climits>

#include "common.cuh"
#include "decode_plan.cuh"
#include "internal.h"
#include "quant.cuh"

namespace kvfp8 {

namespace {

constexpr int kPlanThreads = 1024;
static_assert(kPlanThreads == kDecodePlanThreads, "the fused attention plan runs on this block");

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

// Index of the request whose popped-page range [incl[r] - need[r], incl[r])
// holds flattened page g of the chunk: the first r with incl[r] > g.
__device__ __forceinline__ int owner_of(const long long* incl, int n, long long g) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (incl[mid] > g) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Rows request r appends in this call (none when the step mask drops it).
__device__ __forceinline__ long long req_rows(const AppendArgs& a, int r) {
  if (a.step_mask != nullptr && a.step_mask[r] != 0) return 0;
  if (a.from_pool) return a.src_lens[r];
  return (long long)a.new_indptr[r + 1] - a.new_indptr[r];
}

// With a step mask, every request at or after `stop` is marked unserved.
__device__ void mark_unserved(const AppendArgs& a, int stop) {
  if (a.step_mask == nullptr) return;
  for (int r = stop + threadIdx.x; r < a.B; r += blockDim.x) a.step_mask[r] |= KV_ABORT_UNSERVED;
}

// Open-addressing table of the chunk's partly filled pages (at most one per
// request, so at most half full).
constexpr int kPartialSlots = 2 * kPlanThreads;

__device__ __forceinline__ int partial_slot(int p) {
  return (int)(((uint32_t)p * 2654435761u) >> 21) & (kPartialSlots - 1);
}

__global__ void __launch_bounds__(kPlanThreads) append_plan_kernel(AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ long long warp_sums[32];
  __shared__ long long s_incl[kPlanThreads];  // inclusive prefix of pages popped in the chunk
  __shared__ long long s_first[kPlanThreads]; // first new logical page of each request
  __shared__ int s_pkey[kPartialSlots];       // partly filled page ids (-1: empty slot)
  __shared__ short s_preq[kPartialSlots];     // chunk-local request checking that page
  __shared__ unsigned char s_tagfail[kPlanThreads];
  __shared__ int s_stop, s_code;
  __shared__ long long s_badg;
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
    mark_unserved(a, 0);
    if (a.fuse_plan) {
      __syncthreads();  // every abort bit is set
      decode_plan_block(a.plan);
    }
    return;
  }

  for (int base = 0; base < a.B; base += kPlanThreads) {
    const int r = base + threadIdx.x;
    const int nreq = min(kPlanThreads, a.B - base);
    long long need = 0, L = 0, n = 0, first = 0;
    int code = 0, plast = -1;
    if (r < a.B) {
      L = a.seq_lens[r];
      n = req_rows(a, r);
      // the new length must fit the page table and stay an int32 length; a
      // handoff fills empty requests from rows its source table maps
      if (n < 0 || L < 0 || n > a.max_new || L + n > (long long)a.max_pages * P ||
          L + n > INT_MAX ||
          (a.from_pool && n > 0 && (L != 0 || n > (long long)a.src_max_pages * P))) {
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
          else
            plast = p;
        }
        first = (L + P - 1) / P;
        need = (L + n + P - 1) / P - first;
      }
    }
    const long long incl = block_incl_scan(need, warp_sums);
    const long long pool0 = head0 + consumed;  // free-list position of the chunk's first pop
    s_incl[threadIdx.x] = incl;
    s_first[threadIdx.x] = first;
    s_tagfail[threadIdx.x] = 0;
    for (int i = threadIdx.x; i < kPartialSlots; i += kPlanThreads) s_pkey[i] = -1;
    if (threadIdx.x == 0) {
      s_stop = a.B;
      s_code = 0;
      s_badg = LLONG_MAX;
    }
    __syncthreads();
    // The tags read above are those before this call's pops.  Requests are
    // served in order, so a partly filled page that an earlier request of the
    // chunk pops (its tag is bumped first) fails the later request's check:
    // the partly filled pages go into a table that the pop scan looks up.
    if (plast >= 0) {
      for (int h = partial_slot(plast);; h = (h + 1) & (kPartialSlots - 1)) {
        if (atomicCAS(&s_pkey[h], -1, plast) == -1) {
          s_preq[h] = (short)threadIdx.x;
          break;
        }
      }
    }
    __syncthreads();
    const long long chunk_total = s_incl[nreq - 1];
    // every entry the chunk would pop, all threads at once: the first one
    // that is not a page id marks its request; one that is the partly filled
    // page of a later request fails that request's tag check
    for (long long g = threadIdx.x; g < chunk_total && pool0 + g < d.num_pages; g += kPlanThreads) {
      const int p = d.free_list[pool0 + g];
      if (p < 0 || p >= d.num_pages) {
        atomicMin(reinterpret_cast<unsigned long long*>(&s_badg), (unsigned long long)g);
        continue;
      }
      for (int h = partial_slot(p); s_pkey[h] != -1; h = (h + 1) & (kPartialSlots - 1)) {
        if (s_pkey[h] == p) {
          const int rr = s_preq[h];
          if (owner_of(s_incl, nreq, g) < rr) s_tagfail[rr] = 1;
        }
      }
    }
    __syncthreads();
    if (r < a.B && code == 0 && s_tagfail[threadIdx.x]) code = KV_ERR_TAG_MISMATCH;
    if (r < a.B && code == 0 && pool0 + incl > d.num_pages) code = KV_ERR_OUT_OF_PAGES;
    if (s_badg != LLONG_MAX && r < a.B && code == 0 &&
        threadIdx.x == owner_of(s_incl, nreq, s_badg))
      code = KV_ERR_BAD_PAGE_ID;
    if (code != 0) atomicMin(&s_stop, r);
    __syncthreads();
    const int chunk_stop = s_stop;
    if (r == chunk_stop) s_code = code;
    __syncthreads();
    // pages popped by the requests before the stopping one
    const int si = chunk_stop - base;
    const long long served =
        chunk_stop < a.B ? (si > 0 ? s_incl[si - 1] : 0) : chunk_total;
    for (long long g = threadIdx.x; g < served; g += kPlanThreads) {
      const int i = owner_of(s_incl, nreq, g);
      const long long j = s_first[i] + g - (i > 0 ? s_incl[i - 1] : 0);
      const int p = d.free_list[pool0 + g];
      const uint32_t t = d.tags[p] + 1u;  // wraps mod 2^32
      d.tags[p] = t;
      a.page_table[(long long)(base + i) * a.max_pages + j] = p;
      a.exp_tags[(long long)(base + i) * a.max_pages + j] = t;
    }
    if (r < a.B && r < chunk_stop) a.seq_lens[r] = (int32_t)(L + n);
    consumed += served;
    if (chunk_stop < a.B) {
      stop = chunk_stop;
      stop_code = s_code;
      break;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    d.ctl[KV_CTL_FREE_HEAD] = (int32_t)(head0 + consumed);
    d.ctl[KV_CTL_APPEND_STOP] = stop;
    if (stop_code != 0) set_error(d.ctl, stop_code);
  }
  __syncthreads();  // every thread has read its own mask entry
  mark_unserved(a, stop);
  if (a.fuse_plan) {
    __syncthreads();  // final lengths and abort bits are written
    decode_plan_block(a.plan);
  }
}

constexpr int kDataThreads = 256;

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

// KV_SCALE_REQUANTIZE: the code c of a block whose scale grows from s_old
// to s_new becomes e4m3(fp32(decode(c) * s_old) / s_new) (IEEE divide).
__device__ __forceinline__ uint8_t requant_code(uint8_t c, float s_old, float s_new) {
  const float v = __fmul_rn(__half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3))), s_old);
  return (uint8_t)(e4m3x2(__fdiv_rn(v, s_new), 0.0f) & 0xFFu);
}

// Re-encode the n_old slots already written in a block (token-major: rows of
// D codes; dim-major: D rows of P slots), threads tid, tid + nthreads, ...
__device__ void requant_block(uint8_t* dst, int n_old, int D, bool dim_major, int P, float s_old,
                              float s_new, int tid, int nthreads) {
  for (int e = tid; e < n_old * D; e += nthreads) {
    const int o = dim_major ? (e / n_old) * P + e % n_old : e;
    dst[o] = requant_code(dst[o], s_old, s_new);
  }
}

// One block of rows for one (page, kv head, K-or-V): `nrows` source rows of
// D bf16 values, row i at src + i * src_stride (elements).  Pass 1 finds the
// amax (fresh e4m3 blocks only), pass 2 quantises (or copies) and stores.
// Token-major destination (K, latent): row i at dst + (slot0 + i) * D.
// Dim-major destination (GQA V): element (i, dd) at dst + dd * P + slot0 + i,
// assembled in shared memory and written one dim row at a time.
__device__ void append_block(const uint16_t* src, long long src_stride, int nrows, int D,
                             bool fp8, bool fresh, float* scale_slot, void* dst,
                             bool dim_major, int P, int slot0, uint8_t* tile, float* red,
                             bool requant) {
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
      if (requant) {  // a larger scale for the new rows: re-encode the old ones
        float m = 0.0f;
        for (int i0 = 0; i0 < nrows; i0 += rpp) {
          const int i = i0 + i_off;
          if (active && i < nrows)
            m = fmaxf(m, amax8(*reinterpret_cast<const uint4*>(src + i * src_stride + 8 * c)));
        }
        const float s_new = scale_from_amax(block_max(m, red));
        if (s_new > s) {
          requant_block(static_cast<uint8_t*>(dst), slot0, D, dim_major, P, s, s_new,
                        threadIdx.x, kDataThreads);
          __syncthreads();  // every thread has read the old scale
          if (threadIdx.x == 0) *scale_slot = s_new;
          s = s_new;
        }
      }
    }
  }
  const float rs = __frcp_rn(s);
  for (int i0 = 0; i0 < nrows; i0 += rpp) {
    const int i = i0 + i_off;
    if (!(active && i < nrows)) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(src + i * src_stride + 8 * c);
    if (!dim_major) {
      if (fp8)
        *reinterpret_cast<uint2*>(static_cast<uint8_t*>(dst) + (long long)(slot0 + i) * D + 8 * c) =
            quant8_rs(v, s, rs);
      else
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst) + (long long)(slot0 + i) * D + 8 * c) = v;
    } else {
      const int slot = slot0 + i;
      if (fp8) {
        const uint2 q = quant8_rs(v, s, rs);
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
  const long long n = req_rows(a, r);
  if (n <= 0) return;
  const long long P = d.page_size;
  const long long Lnew = a.seq_lens[r];
  const long long L0 = Lnew - n;
  const bool fp8 = d.dtype == KV_DTYPE_E4M3;
  const bool requant = fp8 && d.scale_mode == KV_SCALE_REQUANTIZE;
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
    // a partly filled page that this call's pops handed to a later request
    // (its tag changed after the plan's check) is not written through the
    // stale mapping
    if (!fresh && d.tags[p] != a.exp_tags[(long long)r * a.max_pages + jp]) continue;
    const int es = fp8 ? 1 : 2;
    if (d.layout == KV_LAYOUT_LATENT) {
      append_block(a.k_new + row0 * Dk, Dk, nrows, Dk, fp8, fresh, fp8 ? d.k_scale + p : nullptr,
                   static_cast<uint8_t*>(d.k_cache) + (long long)p * P * Dk * es, false, (int)P,
                   slot0, tile, red, requant);
      continue;
    }
    if (!is_v) {
      const long long kp = (((long long)p * H + h) * P) * Dk;
      append_block(a.k_new + (row0 * H + h) * Dk, (long long)H * Dk, nrows, Dk, fp8, fresh,
                   fp8 ? d.k_scale + (long long)p * H + h : nullptr,
                   static_cast<uint8_t*>(d.k_cache) + kp * es, false, (int)P, slot0, tile, red,
                   requant);
    } else {
      const long long vp = ((long long)p * H + h) * (long long)Dv * P;
      append_block(a.v_new + (row0 * H + h) * Dv, (long long)H * Dv, nrows, Dv, fp8, fresh,
                   fp8 ? d.v_scale + (long long)p * H + h : nullptr,
                   static_cast<uint8_t*>(d.v_cache) + vp * es, true, (int)P, slot0, tile, red,
                   requant);
    }
  }
}

// ---- register-resident paths (the common shapes) ----------------------------
//
// Bulk appends (a prefill handed to the decode cache) touch every page of a
// request; these paths read each source byte once.  A GQA (page, kv head,
// K|V) tile of up to 2048 values sits in one warp's registers: amax by a warp
// reduction, then quantise and store from the registers.  A latent page (up
// to 64 rows of up to 576 values) is split over a CTA's 8 warps by row, with
// a block-wide amax.  Both kernels are persistent (two CTAs per SM).

constexpr int kTileWarps = 8;
constexpr int kTileChunks = 8;   // 16-byte source chunks per lane (P * D <= 2048)
constexpr int kLatChunks = 18;   // per lane: ceil(8 rows * 72 chunks / 32)

// A whole 16 x 128 page whose scale is below 2^-90, element by element with
// the IEEE divide (kept out of line: it is rare and its code is long).
__device__ __noinline__ void page_ieee(const uint16_t* src, long long src_stride, bool dim_major,
                                       float s, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < 16 * 128; e += 32) {
    const int i = e >> 7, dd = e & 127;
    const float x = bf16_bits_to_f32(src[i * src_stride + dd]);
    dst[dim_major ? dd * 16 + i : i * 128 + dd] =
        (uint8_t)(e4m3x2(__fdiv_rn(x, s), 0.0f) & 0xFFu);
  }
}

// A whole 16-token page of a 128-dim V tile, transposed in registers: lane l
// loads dims 4l..4l+3 of every row and writes those 4 dim rows of 16 slots.
__device__ void v_page_16x128(const uint16_t* src, long long src_stride, bool fp8,
                              float* scale_slot, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
  uint2 x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    x[i] = *reinterpret_cast<const uint2*>(src + i * src_stride + 4 * lane);
  if (!fp8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t a = k < 2 ? x[2 * j].x : x[2 * j].y, b = k < 2 ? x[2 * j + 1].x
                                                                      : x[2 * j + 1].y;
        w[j] = (k & 1) ? __byte_perm(a, b, 0x7632) : __byte_perm(a, b, 0x5410);
      }
      uint4* o = reinterpret_cast<uint4*>(dst + (4 * lane + k) * 32);
      o[0] = make_uint4(w[0], w[1], w[2], w[3]);
      o[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    return;
  }
  uint32_t mb = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) mb = absbits_max2(absbits_max2(mb, x[i].x), x[i].y);
  mb = absbits_warp_max(mb);
  float amax = __uint_as_float(mb << 16);
  if (mb > 0x7F80u) {  // a NaN: the float maximum skips it
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fmaxf(amax2(x[i].x), amax2(x[i].y)));
    amax = warp_max(m);
  }
  const float s = scale_from_amax(amax), rs = __frcp_rn(s);
  if (lane == 0) *scale_slot = s;
  if (!scale_fast_ok(s)) {
    page_ieee(src, src_stride, true, s, dst);
    return;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t a = k < 2 ? x[2 * j].x : x[2 * j].y, b = k < 2 ? x[2 * j + 1].x
                                                                    : x[2 * j + 1].y;
      c[j] = (k & 1) ? e4m3x2(div_fresh(bf16_hi(a), s, rs), div_fresh(bf16_hi(b), s, rs))
                     : e4m3x2(div_fresh(bf16_lo(a), s, rs), div_fresh(bf16_lo(b), s, rs));
    }
    *reinterpret_cast<uint4*>(dst + (4 * lane + k) * 16) =
        make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16),
                   c[6] | (c[7] << 16));
  }
}

// A whole 16-token page of a 128-dim K tile (token-major): lane l holds
// dims 8 (l % 16) .. +7 of rows l / 16, l / 16 + 2, ...
__device__ void k_page_16x128(const uint16_t* src, long long src_stride, bool fp8,
                              float* scale_slot, uint8_t* dst) {
  const int lane = threadIdx.x & 31, c = lane & 15, i0 = lane >> 4;
  uint4 x[8];
#pragma unroll
  for (int t = 0; t < 8; ++t)
    x[t] = *reinterpret_cast<const uint4*>(src + (2 * t + i0) * src_stride + 8 * c);
  if (!fp8) {
#pragma unroll
    for (int t = 0; t < 8; ++t)
      *reinterpret_cast<uint4*>(dst + ((2 * t + i0) * 128 + 8 * c) * 2) = x[t];
    return;
  }
  uint32_t mb = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) mb = absbits_max8(mb, x[t]);
  mb = absbits_warp_max(mb);
  float amax = __uint_as_float(mb << 16);
  if (mb > 0x7F80u) {  // a NaN: the float maximum skips it
    float m = 0.0f;
#pragma unroll
    for (int t = 0; t < 8; ++t) m = fmaxf(m, amax8(x[t]));
    amax = warp_max(m);
  }
  const float s = scale_from_amax(amax), rs = __frcp_rn(s);
  if (lane == 0) *scale_slot = s;
  if (!scale_fast_ok(s)) {
    page_ieee(src, src_stride, false, s, dst);
    return;
  }
#pragma unroll
  for (int t = 0; t < 8; ++t)
    *reinterpret_cast<uint2*>(dst + (2 * t + i0) * 128 + 8 * c) =
        make_uint2(quant_word_fresh(x[t].x, s, rs) | (quant_word_fresh(x[t].y, s, rs) << 16),
                   quant_word_fresh(x[t].z, s, rs) | (quant_word_fresh(x[t].w, s, rs) << 16));
}

// Any other tile: part of a page, another page shape, or the re-quantising
// mode's re-encoding (kept out of line so the whole-page code stays small).
__device__ __noinline__ void tile_warp_generic(const uint16_t* src, long long src_stride,
                                               int nrows, int D, bool fp8, bool fresh,
                                               float* scale_slot, uint8_t* dst, bool dim_major,
                                               int P, int slot0, uint8_t* wtile, bool requant) {
  const int lane = threadIdx.x & 31;
  const int cpr = D / 8, total = nrows * cpr;
  uint4 v[kTileChunks];
#pragma unroll
  for (int t = 0; t < kTileChunks; ++t) {
    const int q = lane + 32 * t;
    v[t] = q < total ? *reinterpret_cast<const uint4*>(src + (q / cpr) * src_stride + 8 * (q % cpr))
                     : make_uint4(0, 0, 0, 0);
  }
  float s = 1.0f;
  if (fp8) {
    if (fresh) {
      float m = 0.0f;
#pragma unroll
      for (int t = 0; t < kTileChunks; ++t) m = fmaxf(m, amax8(v[t]));
      s = scale_from_amax(warp_max(m));
      if (lane == 0) *scale_slot = s;
    } else {
      s = *scale_slot;
      if (requant) {  // a larger scale for the new rows: re-encode the old ones
        float m = 0.0f;
#pragma unroll
        for (int t = 0; t < kTileChunks; ++t) m = fmaxf(m, amax8(v[t]));
        const float s_new = scale_from_amax(warp_max(m));
        if (s_new > s) {
          requant_block(dst, slot0, D, dim_major, P, s, s_new, lane, 32);
          __syncwarp();
          if (lane == 0) *scale_slot = s_new;
          s = s_new;
        }
      }
    }
  }
  const float rs = __frcp_rn(s);
  if (!dim_major) {
#pragma unroll
    for (int t = 0; t < kTileChunks; ++t) {
      const int q = lane + 32 * t;
      if (q < total) {
        const long long o = (long long)(slot0 + q / cpr) * D + 8 * (q % cpr);
        if (fp8)
          *reinterpret_cast<uint2*>(dst + o) = quant8_rs(v[t], s, rs);
        else
          *reinterpret_cast<uint4*>(dst + 2 * o) = v[t];
      }
    }
    return;
  }
  // dim-major destination: element (row i, dim dd) at (dd * P + slot0 + i),
  // assembled in this warp's shared tile, or without one (wtile null)
  // stored element by element
  if (wtile == nullptr) {
#pragma unroll
    for (int t = 0; t < kTileChunks; ++t) {
      const int q = lane + 32 * t;
      if (q < total) {
        const int o = 8 * (q % cpr) * P + slot0 + q / cpr;
        if (fp8) {
          const uint2 c8 = quant8_rs(v[t], s, rs);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[o + k * P] = (uint8_t)(((k < 4 ? c8.x : c8.y) >> (8 * (k & 3))) & 0xFFu);
        } else {
          const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
          uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
          for (int k = 0; k < 8; ++k) d16[o + k * P] = (uint16_t)(w[k >> 1] >> (16 * (k & 1)));
        }
      }
    }
    return;
  }
#pragma unroll
  for (int t = 0; t < kTileChunks; ++t) {
    const int q = lane + 32 * t;
    if (q < total) {
      const int i = q / cpr, c = q % cpr;
      const int o = 8 * c * P + slot0 + i;
      if (fp8) {
        const uint2 c8 = quant8_rs(v[t], s, rs);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          wtile[o + k * P] = (uint8_t)(((k < 4 ? c8.x : c8.y) >> (8 * (k & 3))) & 0xFFu);
      } else {
        const uint32_t w[4] = {v[t].x, v[t].y, v[t].z, v[t].w};
        uint16_t* t16 = reinterpret_cast<uint16_t*>(wtile);
#pragma unroll
        for (int k = 0; k < 8; ++k) t16[o + k * P] = (uint16_t)(w[k >> 1] >> (16 * (k & 1)));
      }
    }
  }
  __syncwarp();
  const int es = fp8 ? 1 : 2;
  if (nrows == P && (D * P * es) % 16 == 0) {
    for (int k = lane; k < D * P * es / 16; k += 32)
      reinterpret_cast<uint4*>(dst)[k] = reinterpret_cast<const uint4*>(wtile)[k];
  } else {
    for (int e = lane; e < D * nrows; e += 32) {
      const int o = (e / nrows) * P + slot0 + e % nrows;
      if (fp8)
        dst[o] = wtile[o];
      else
        reinterpret_cast<uint16_t*>(dst)[o] = reinterpret_cast<const uint16_t*>(wtile)[o];
    }
  }
  __syncwarp();
}

__device__ __forceinline__ void tile_warp(const uint16_t* src, long long src_stride, int nrows,
                                          int D, bool fp8, bool fresh, float* scale_slot,
                                          uint8_t* dst, bool dim_major, int P, int slot0,
                                          uint8_t* wtile, bool requant) {
  if (nrows == 16 && P == 16 && D == 128) {  // a whole page (fresh by construction)
    if (dim_major)
      v_page_16x128(src, src_stride, fp8, scale_slot, dst);
    else
      k_page_16x128(src, src_stride, fp8, scale_slot, dst);
    return;
  }
  tile_warp_generic(src, src_stride, nrows, D, fp8, fresh, scale_slot, dst, dim_major, P, slot0,
                    wtile, requant);
}

// A V tile of a pool-to-pool handoff: read from a bf16 pool's dim-major tile
// (element (slot, dd) at src[dd * P + slot]) into this pool's dim-major tile
// at dst.  Only the first nrows slots (the source request's rows) are read
// and written; the page is fresh, so e4m3 codes take the scale of their own
// amax (the same division as every other path), and bf16 copies the bits.
// One warp; a whole 16-slot page takes 16-byte loads (lane l: dims l,
// l + 32, ...), anything else goes element by element.
__device__ __forceinline__ void v_tile_from_dim_major(const uint16_t* src, int nrows, int D, int P,
                                                   bool fp8, float* scale_slot, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
  const bool whole = nrows == P && P == 16;
  if (!fp8) {
    uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
    if (whole) {
      for (int k = lane; k < D * 2; k += 32)
        reinterpret_cast<uint4*>(d16)[k] = reinterpret_cast<const uint4*>(src)[k];
    } else {
      for (int e = lane; e < D * nrows; e += 32) {
        const int dd = e / nrows, i = e - dd * nrows;
        d16[dd * P + i] = src[dd * P + i];
      }
    }
    return;
  }
  float m = 0.0f;  // fmaxf skips a NaN, as the amax of every other path does
  if (whole) {
    for (int dd = lane; dd < D; dd += 32) {
      const uint4* row = reinterpret_cast<const uint4*>(src + dd * 16);
      m = fmaxf(m, fmaxf(amax8(row[0]), amax8(row[1])));
    }
  } else {
    for (int e = lane; e < D * nrows; e += 32) {
      const int dd = e / nrows, i = e - dd * nrows;
      m = fmaxf(m, fabsf(bf16_bits_to_f32(src[dd * P + i])));
    }
  }
  const float s = scale_from_amax(warp_max(m));
  if (lane == 0) *scale_slot = s;
  const float rs = __frcp_rn(s);
  const bool fast = scale_fast_ok(s);
  if (whole && fast) {
    for (int dd = lane; dd < D; dd += 32) {
      const uint4* row = reinterpret_cast<const uint4*>(src + dd * 16);
      const uint4 a = row[0], b = row[1];
      *reinterpret_cast<uint4*>(dst + dd * 16) = make_uint4(
          quant_word_fresh(a.x, s, rs) | (quant_word_fresh(a.y, s, rs) << 16),
          quant_word_fresh(a.z, s, rs) | (quant_word_fresh(a.w, s, rs) << 16),
          quant_word_fresh(b.x, s, rs) | (quant_word_fresh(b.y, s, rs) << 16),
          quant_word_fresh(b.z, s, rs) | (quant_word_fresh(b.w, s, rs) << 16));
    }
    return;
  }
  for (int e = lane; e < D * nrows; e += 32) {
    const int dd = e / nrows, i = e - dd * nrows;
    const float x = bf16_bits_to_f32(src[dd * P + i]);
    dst[dd * P + i] = (uint8_t)(e4m3x2(fast ? div_fresh(x, s, rs) : __fdiv_rn(x, s), 0.0f) & 0xFFu);
  }
}

// Work items of a bulk append: every (request, page this call touches),
// times per_page (tiles per page for GQA, 1 for latent), in request order.
// The CTA's threads build the inclusive prefix pre[0..B] in shared memory, so
// a persistent grid visits only real work however few requests have rows.
constexpr int kMaxPersistB = 16384;

__device__ int bulk_items_prefix(const AppendArgs& a, int B, int per_page, int* pre, int* wsum) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const long long P = a.d.page_size;
  int carry = 0;
  if (threadIdx.x == 0) pre[0] = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int r = base + threadIdx.x;
    int v = 0;
    if (r < B) {
      const long long n = req_rows(a, r);
      if (n > 0) {
        const long long Lnew = a.seq_lens[r], L0 = Lnew - n;
        v = (int)((Lnew - 1) / P - L0 / P + 1) * per_page;
      }
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) wsum[wid] = v;
    __syncthreads();
    int before = carry;
    for (int k = 0; k < wid; ++k) before += wsum[k];
    if (r < B) pre[r + 1] = before + v;
    int chunk = 0;
    for (int k = 0; k < nw; ++k) chunk += wsum[k];
    carry += chunk;
    __syncthreads();
  }
  return carry;
}

// request owning item i: the r with pre[r] <= i < pre[r + 1]
__device__ __forceinline__ int item_owner(const int* pre, int B, int i) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// GQA: persistent CTAs; each warp takes (request, page, tile) items in turn.
// FROM_POOL: the pool-to-pool handoff (its own instance, so that the source
// addressing does not change the register allocation of the common append).
template <bool FROM_POOL>
__global__ void __launch_bounds__(kTileWarps * 32) append_gqa_kernel(AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int wsum[kTileWarps];
  const kv_pool_desc& d = a.d;
  const long long P = d.page_size;
  const bool fp8 = d.dtype == KV_DTYPE_E4M3;
  const bool requant = fp8 && d.scale_mode == KV_SCALE_REQUANTIZE;
  const int es = fp8 ? 1 : 2;
  const int H = d.num_kv_heads, Dk = d.head_dim_k, Dv = d.head_dim_v;
  const int warp = threadIdx.x >> 5;
  const int B = min(a.B, (int)d.ctl[KV_CTL_APPEND_STOP]);
  uint8_t* wtile = smem + (size_t)warp * Dv * P * es;
  int* pre = reinterpret_cast<int*>(smem + (size_t)kTileWarps * Dv * P * es);
  const int tiles = 2 * H;
  const int total = B > 0 ? bulk_items_prefix(a, B, tiles, pre, wsum) : 0;
  for (int it = blockIdx.x * kTileWarps + warp; it < total; it += gridDim.x * kTileWarps) {
    const int r = item_owner(pre, B, it);
    const int local = it - pre[r], t = local % tiles;
    const long long n = req_rows(a, r);
    const long long Lnew = a.seq_lens[r], L0 = Lnew - n;
    const long long jp = L0 / P + local / tiles;
    const long long pos_lo = max(jp * P, L0), pos_hi = min((jp + 1) * P, Lnew);
    const int nrows = (int)(pos_hi - pos_lo);
    const int slot0 = (int)(pos_lo - jp * P);
    const long long row0 = FROM_POOL ? 0 : a.new_indptr[r] + (pos_lo - L0);
    const int p = a.page_table[(long long)r * a.max_pages + jp];
    if (p < 0 || p >= d.num_pages) {  // uniform across the warp
      if ((threadIdx.x & 31) == 0) set_error(d.ctl, KV_ERR_BAD_PAGE_ID);
      continue;
    }
    // rows of this tile: the caller's (row0 of k_new / v_new) or, in a
    // handoff, source page jp of the request (the destination was empty, so
    // every page is fresh and takes source page j whole)
    const int h = t >> 1;
    long long src_tile = -1;
    if constexpr (FROM_POOL) {
      const int sp = a.src_page_table[(long long)r * a.src_max_pages + jp];
      if (sp < 0 || sp >= a.src.num_pages) {  // uniform across the warp
        if ((threadIdx.x & 31) == 0) set_error(d.ctl, KV_ERR_BAD_PAGE_ID);
        continue;
      }
      src_tile = (long long)sp * H + h;
    }
    const bool fresh = jp * P >= L0;  // popped by this call
    // not through a stale mapping (see append_data_kernel)
    if (!fresh && d.tags[p] != a.exp_tags[(long long)r * a.max_pages + jp]) continue;
    if ((t & 1) == 0) {
      const uint16_t* src = FROM_POOL
                                ? static_cast<const uint16_t*>(a.src.k_cache) + src_tile * P * Dk
                                : a.k_new + (row0 * H + h) * Dk;
      tile_warp(src, FROM_POOL ? (long long)Dk : (long long)H * Dk, nrows, Dk, fp8, fresh,
                fp8 ? d.k_scale + (long long)p * H + h : nullptr,
                static_cast<uint8_t*>(d.k_cache) + (((long long)p * H + h) * P * Dk) * es, false,
                (int)P, slot0, wtile, requant);
    } else if (FROM_POOL) {  // the source V tile is dim-major already
      v_tile_from_dim_major(static_cast<const uint16_t*>(a.src.v_cache) + src_tile * Dv * P,
                            nrows, Dv, (int)P, fp8, fp8 ? d.v_scale + (long long)p * H + h : nullptr,
                            static_cast<uint8_t*>(d.v_cache) + (((long long)p * H + h) * Dv * P) * es);
    } else {
      tile_warp(a.v_new + (row0 * H + h) * Dv, (long long)H * Dv, nrows, Dv, fp8, fresh,
                fp8 ? d.v_scale + (long long)p * H + h : nullptr,
                static_cast<uint8_t*>(d.v_cache) + (((long long)p * H + h) * Dv * P) * es, true,
                (int)P, slot0, wtile, requant);
    }
  }
}

// ---- staged bulk append (GQA) ----------------------------------------------
//
// The same work as append_gqa_kernel, organised per page so that loads stay in
// flight: one CTA per SM takes (request, page) items in turn; a producer warp
// moves an item's rows into a ring of shared-memory stages with bulk
// asynchronous copies, up to S items ahead -- the page's K rows and V rows,
// two contiguous runs of k_new / v_new (a handoff: the source page's K tiles
// and V tiles, also two contiguous runs) -- and 12 consumer warps quantise (or
// copy) the page's 2 H tiles from there with the register-resident tile code.
// The producer also does each item's bookkeeping (owner, rows, page ids, tag
// check), so the consumers read nothing from global memory but the rows.
// The one-tile-per-warp kernel had at most one tile's loads in flight per
// warp and spent its time waiting on them.  For 16-row, 128-wide pages the V
// tiles of partly filled pages (a few per request) are stored element by
// element rather than through per-warp shared tiles, which leaves that shared
// memory to the ring (a third stage for bf16 pages).
constexpr int kStgWarps = 12;
constexpr int kStgThreads = (kStgWarps + 1) * 32;
constexpr int kStgMaxStages = 4;
constexpr int kStgMaxB = 4096;  // requests whose item prefix fits shared memory

// whether the staged kernel keeps per-warp shared tiles for the V tiles of
// partly filled pages
__host__ __device__ constexpr bool stg_wtiles(long long P, int Dv) {
  return !(P == 16 && Dv == 128);
}

// bytes of shared memory after the stages: item metadata, full / empty
// barriers, abort flag, warp sums, item prefix
__host__ __device__ constexpr size_t stg_ring_bytes(int B) {
  return kStgMaxStages * 16 + 2 * kStgMaxStages * 8 + 16 + 16 * 4 + (size_t)(B + 1) * 4;
}
// GQA: besides the stages, also the per-warp V tiles
__host__ __device__ constexpr size_t stg_fixed_bytes(int Dv, int P, int es, int B) {
  return (stg_wtiles(P, Dv) ? (size_t)kStgWarps * Dv * P * es : 0) + stg_ring_bytes(B);
}

// The producer warp of the staged bulk-append kernels: items (request, page)
// of this CTA, each one stage -- the page's K rows (latent: its rows) and V
// rows, copied in bulk from k_new / v_new (a handoff: the source pool's page)
// -- with the item's metadata (destination page, rows, first slot, flags:
// 1 fresh page, 2 skip) in meta[stage].
template <bool FROM_POOL, bool LATENT>
__device__ __forceinline__ void stg_produce(const AppendArgs& a, int B, int total, const int* pre,
                                            int S, int stage_bytes, uint8_t* stages, int4* meta,
                                            uint64_t* full, uint64_t* empty,
                                            volatile int* abort_flag) {
  const kv_pool_desc& d = a.d;
  const long long P = d.page_size;
  const int H = d.num_kv_heads, Dk = d.head_dim_k, Dv = d.head_dim_v;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kbytes = (int)(P * H * Dk * 2);  // the K part of a stage
  // The warp works out 32 items' bookkeeping at a time (one lane per item),
  // then lane 0 issues each item's bulk copies as its stage frees up.  The
  // bookkeeping is a chain of dependent loads (owner's lengths; then source
  // and destination page ids; then the destination's tag), so the next
  // batch's loads are issued while the current batch's copies go out: its
  // lengths before the first copy, its page ids half way.
  struct Item {
    const uint16_t *ks, *vs;
    uint32_t kb, vb, et;
    int p, nrows, slot0, flags;  // flags: 1 fresh page, 2 skip
    bool live, bad;
  };
  const uint64_t policy = l2_evict_first_policy();
  const long long cnt =
      (long long)blockIdx.x < total ? (total - (long long)blockIdx.x + gridDim.x - 1) / gridDim.x
                                    : 0;
  // phase A: the item's owner and its lengths
  auto phase_a = [&](long long kk, int& r, long long& n, long long& Lnew, long long& ind0) {
    r = -1;
    if (kk < cnt) {
      r = item_owner(pre, B, (int)(blockIdx.x + kk * gridDim.x));
      n = req_rows(a, r);
      Lnew = a.seq_lens[r];
      ind0 = FROM_POOL ? 0 : a.new_indptr[r];
    }
  };
  // phase B: rows and source; loads of the page ids and the expected tag
  auto phase_b = [&](long long kk, int r, long long n, long long Lnew, long long ind0, Item& m) {
    m.live = r >= 0;
    m.bad = false;
    m.kb = m.vb = 0;
    m.ks = m.vs = nullptr;
    m.p = -1;
    m.nrows = m.slot0 = m.flags = 0;
    m.et = 0;
    if (!m.live) return;
    const int it = (int)(blockIdx.x + kk * gridDim.x);
    const long long L0 = Lnew - n;
    const long long jp = L0 / P + (it - pre[r]);
    const long long pos_lo = max(jp * P, L0), pos_hi = min((jp + 1) * P, Lnew);
    m.nrows = (int)(pos_hi - pos_lo);
    m.slot0 = (int)(pos_lo - jp * P);
    if constexpr (FROM_POOL) {  // the destination request was empty: source page jp
      const int sp = a.src_page_table[(long long)r * a.src_max_pages + jp];
      if (sp >= 0 && sp < a.src.num_pages) {
        m.ks = static_cast<const uint16_t*>(a.src.k_cache) + (long long)sp * H * P * Dk;
        m.kb = (uint32_t)kbytes;
        if constexpr (!LATENT) {
          m.vs = static_cast<const uint16_t*>(a.src.v_cache) + (long long)sp * H * Dv * P;
          m.vb = (uint32_t)(P * H * Dv * 2);
        }
      } else {
        m.bad = true;
      }
    } else {
      const long long row0 = ind0 + (pos_lo - L0);
      m.ks = a.k_new + row0 * H * Dk;
      m.kb = (uint32_t)(m.nrows * H * Dk * 2);
      if constexpr (!LATENT) {
        m.vs = a.v_new + row0 * H * Dv;
        m.vb = (uint32_t)(m.nrows * H * Dv * 2);
      }
    }
    m.p = a.page_table[(long long)r * a.max_pages + jp];
    m.flags = jp * P >= L0 ? 1 : 0;  // popped by this call
    if (m.flags == 0) m.et = a.exp_tags[(long long)r * a.max_pages + jp];
  };
  // phase C: checks on the destination page
  auto phase_c = [&](Item& m) {
    if (!m.live) return;
    if (m.bad || m.p < 0 || m.p >= d.num_pages) {
      set_error(d.ctl, KV_ERR_BAD_PAGE_ID);
      m.flags = 2;
    } else if (m.flags == 0 && d.tags[m.p] != m.et) {
      m.flags = 2;  // not through a stale mapping (see append_data_kernel)
    }
    if (m.flags & 2) m.kb = m.vb = 0;  // nothing to read for an item that is skipped
  };
  int ar = -1;
  long long an = 0, aL = 0, ai = 0;
  Item cur, nxt;
  phase_a(lane, ar, an, aL, ai);
  phase_b(lane, ar, an, aL, ai, cur);
  phase_c(cur);
  long long issued = 0;
  bool go = true;
  for (long long k0 = 0; go && k0 < cnt; k0 += 32) {
    const int nb = (int)min(32ll, cnt - k0);
    const bool more = k0 + 32 < cnt;
    if (more) phase_a(k0 + 32 + lane, ar, an, aL, ai);
    for (int j = 0; j < nb; ++j) {
      const long long k = k0 + j;
      const int stage = (int)(k % S);
      bool ok = true;
      if (lane == 0 && k >= S)
        ok = mbar_wait(&empty[stage], (uint32_t)(((k / S) - 1) & 1), abort_flag, d.ctl,
                       wait_info(warp, 1, stage));
      if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
        go = false;
        break;
      }
      const int jp_ = __shfl_sync(0xffffffffu, cur.p, j);
      const int jn = __shfl_sync(0xffffffffu, cur.nrows, j);
      const int js = __shfl_sync(0xffffffffu, cur.slot0, j);
      const int jf = __shfl_sync(0xffffffffu, cur.flags, j);
      const uint32_t jkb = __shfl_sync(0xffffffffu, cur.kb, j);
      const uint32_t jvb = __shfl_sync(0xffffffffu, cur.vb, j);
      const uint16_t* jks = reinterpret_cast<const uint16_t*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(cur.ks), j));
      const uint16_t* jvs = reinterpret_cast<const uint16_t*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(cur.vs), j));
      if (lane == 0) {
        meta[stage] = make_int4(jp_, jn, js, jf);
        uint8_t* dst = stages + (size_t)stage * stage_bytes;
        if (jkb + jvb > 0) {
          mbar_arrive_expect_tx(&full[stage], jkb + jvb);
          bulk_g2s(dst, jks, jkb, &full[stage], policy);
          if (jvb > 0) bulk_g2s(dst + kbytes, jvs, jvb, &full[stage], policy);
        } else {
          mbar_arrive(&full[stage]);
        }
      }
      issued = k + 1;
      if (more && j == (nb >> 1)) phase_b(k0 + 32 + lane, ar, an, aL, ai, nxt);
    }
    if (go && more) {
      phase_c(nxt);
      cur = nxt;
    }
  }
  // after a wait gave up, copies already issued may still be landing
  if (lane == 0 && *abort_flag) {
    for (long long q = max(0ll, issued - S); q < issued; ++q) {
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(&full[q % S], (uint32_t)((q / S) & 1)) &&
             global_ns() - t0 < 100000000ull) {
      }
    }
  }
}

template <bool FROM_POOL>
__global__ void __launch_bounds__(kStgThreads, 1)
    append_gqa_staged_kernel(AppendArgs a, int S, int stage_bytes) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  const kv_pool_desc& d = a.d;
  const long long P = d.page_size;
  const bool fp8 = d.dtype == KV_DTYPE_E4M3;
  const bool requant = fp8 && d.scale_mode == KV_SCALE_REQUANTIZE;
  const int es = fp8 ? 1 : 2;
  const int H = d.num_kv_heads, Dk = d.head_dim_k, Dv = d.head_dim_v;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* stages = smem;
  uint8_t* wtiles = stages + (size_t)S * stage_bytes;
  const bool use_wtiles = stg_wtiles(P, Dv);
  int4* meta =
      reinterpret_cast<int4*>(wtiles + (use_wtiles ? (size_t)kStgWarps * Dv * P * es : 0));
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + kStgMaxStages);
  uint64_t* empty = full + kStgMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStgMaxStages);
  int* wsum = reinterpret_cast<int*>(empty + kStgMaxStages) + 4;
  int* pre = wsum + 16;
  const int B = min(a.B, (int)d.ctl[KV_CTL_APPEND_STOP]);
  if (S < 2 || S > kStgMaxStages) {  // the host chose a bad ring
    if (threadIdx.x == 0) set_error(d.ctl, KV_ERR_INTERNAL);
    return;
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kStgWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  const int total = B > 0 ? bulk_items_prefix(a, B, 1, pre, wsum) : 0;
  __syncthreads();
  const int kbytes = (int)(P * H * Dk * 2);  // the K part of a stage

  if (warp == kStgWarps) {
    stg_produce<FROM_POOL, false>(a, B, total, pre, S, stage_bytes, stages, meta, full, empty,
                                  abort_flag);
    return;
  }

  // ---- consumers: the page's 2 H tiles (even: K of head t / 2, odd: V) are
  // dealt round-robin over the warps, continuing from one page to the next,
  // so every warp gets the same share of the work over a few pages
  uint8_t* wtile = use_wtiles ? wtiles + (size_t)warp * Dv * P * es : nullptr;
  const int T = 2 * H;
  int first = warp;  // this warp's first tile of the current page
  long long k = 0;
  for (int it = blockIdx.x; it < total; it += gridDim.x, ++k) {
    const int stage = (int)(k % S);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], (uint32_t)((k / S) & 1),
                                                      abort_flag, d.ctl,
                                                      wait_info(warp, 0, stage)));
    if (!ok) break;
    const int4 m = meta[stage];
    const int p = m.x, nrows = m.y, slot0 = m.z;
    const bool fresh = (m.w & 1) != 0;
    const uint8_t* src = stages + (size_t)stage * stage_bytes;
    int t = first;
    if ((m.w & 2) == 0) {
      for (; t < T; t += kStgWarps) {
        const int h = t >> 1;
        const long long tile = (long long)p * H + h;
        if ((t & 1) == 0) {
          const uint16_t* ks = reinterpret_cast<const uint16_t*>(src) +
                               (FROM_POOL ? (long long)h * P * Dk : (long long)h * Dk);
          tile_warp(ks, FROM_POOL ? (long long)Dk : (long long)H * Dk, nrows, Dk, fp8, fresh,
                    fp8 ? d.k_scale + tile : nullptr,
                    static_cast<uint8_t*>(d.k_cache) + tile * P * Dk * es, false, (int)P, slot0,
                    wtile, requant);
        } else if constexpr (FROM_POOL) {  // the source V tile is dim-major already
          v_tile_from_dim_major(reinterpret_cast<const uint16_t*>(src + kbytes) +
                                    (long long)h * Dv * P,
                                nrows, Dv, (int)P, fp8, fp8 ? d.v_scale + tile : nullptr,
                                static_cast<uint8_t*>(d.v_cache) + tile * Dv * P * es);
        } else {
          tile_warp(reinterpret_cast<const uint16_t*>(src + kbytes) + (long long)h * Dv,
                    (long long)H * Dv, nrows, Dv, fp8, fresh, fp8 ? d.v_scale + tile : nullptr,
                    static_cast<uint8_t*>(d.v_cache) + tile * Dv * P * es, true, (int)P, slot0,
                    wtile, requant);
        }
      }
    } else {
      while (t < T) t += kStgWarps;
    }
    first = t - T;  // where this warp's turn falls on the next page
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
}

// The latent layout's staged kernel: one stage per page (its rows, one row of
// head_dim_k values per token, contiguous in k_new or in the source pool), and
// the 12 consumer warps share each page: thread t holds 16-byte chunks
// t, t + 384, ... of the page's rows, the page's amax is reduced over the 12
// warps, and every thread quantises and stores its chunks -- consecutive
// threads, consecutive chunks.  The consumers meet on an mbarrier (bounded
// waits, so a consumer that gave up cannot leave the others waiting), and the
// reduction words alternate between two rows by meeting number: a row is
// rewritten two meetings later, after every warp has read it.
constexpr int kLatStgThreads = kStgWarps * 32;
constexpr int kLatStgChunks = 12;  // per thread: 64 rows x 72 chunks / 384

// meeting number n of the consumer warps; false when a wait gave up
__device__ __forceinline__ bool lat_meet(uint64_t* cbar, uint32_t& n, volatile int* abort_flag,
                                         int32_t* ctl) {
  const int warp = threadIdx.x >> 5;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(cbar);
  const bool ok = __all_sync(0xffffffffu, mbar_wait(cbar, n & 1u, abort_flag, ctl,
                                                    wait_info(warp, 0, 63)));
  ++n;
  return ok;
}

// largest magnitude of the page's rows over the consumer warps (bit-pattern
// maximum; a NaN falls back to the float maximum, which skips it); false when
// a meeting gave up
__device__ bool lat_stg_amax(const uint4 (&v)[kLatStgChunks], uint32_t (*red)[kStgWarps],
                             uint64_t* cbar, uint32_t& n, volatile int* abort_flag, int32_t* ctl,
                             float& amax) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t mb = 0;
#pragma unroll
  for (int t = 0; t < kLatStgChunks; ++t) mb = absbits_max8(mb, v[t]);
  mb = absbits_warp_max(mb);
  uint32_t* row = red[n & 1u];
  if (lane == 0) row[warp] = mb;
  if (!lat_meet(cbar, n, abort_flag, ctl)) return false;
  mb = __reduce_max_sync(0xffffffffu, lane < kStgWarps ? row[lane] : 0u);
  amax = __uint_as_float(mb << 16);
  if (mb > 0x7F80u) {  // a NaN (uniform): the float maximum over the same chunks
    float m = 0.0f;
#pragma unroll
    for (int t = 0; t < kLatStgChunks; ++t) m = fmaxf(m, amax8(v[t]));
    m = warp_max(m);
    float* frow = reinterpret_cast<float*>(red[n & 1u]);
    if (lane == 0) frow[warp] = m;
    if (!lat_meet(cbar, n, abort_flag, ctl)) return false;
    amax = warp_max(lane < kStgWarps ? frow[lane] : 0.0f);
  }
  return true;
}

template <bool FROM_POOL>
__global__ void __launch_bounds__(kStgThreads, 1)
    append_latent_staged_kernel(AppendArgs a, int S, int stage_bytes) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t red[2][kStgWarps];
  __shared__ __align__(8) uint64_t cbar;  // the consumers' meetings
  const kv_pool_desc& d = a.d;
  const long long P = d.page_size;
  const int Dk = d.head_dim_k;
  const bool fp8 = d.dtype == KV_DTYPE_E4M3;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* stages = smem;
  int4* meta = reinterpret_cast<int4*>(stages + (size_t)S * stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + kStgMaxStages);
  uint64_t* empty = full + kStgMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStgMaxStages);
  int* wsum = reinterpret_cast<int*>(empty + kStgMaxStages) + 4;
  int* pre = wsum + 16;
  const int B = min(a.B, (int)d.ctl[KV_CTL_APPEND_STOP]);
  if (S < 2 || S > kStgMaxStages || P * Dk > 8LL * kLatStgThreads * kLatStgChunks) {
    if (threadIdx.x == 0) set_error(d.ctl, KV_ERR_INTERNAL);  // the host chose a bad ring
    return;
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kStgWarps);
    }
    mbar_init(&cbar, kStgWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  const int total = B > 0 ? bulk_items_prefix(a, B, 1, pre, wsum) : 0;
  __syncthreads();
  if (warp == kStgWarps) {
    stg_produce<FROM_POOL, true>(a, B, total, pre, S, stage_bytes, stages, meta, full, empty,
                                 abort_flag);
    return;
  }

  // ---- consumers
  const int tid = threadIdx.x;
  uint32_t meets = 0;
  long long k = 0;
  for (int it = blockIdx.x; it < total; it += gridDim.x, ++k) {
    const int stage = (int)(k % S);
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], (uint32_t)((k / S) & 1),
                                                      abort_flag, d.ctl,
                                                      wait_info(warp, 0, stage)));
    if (!ok) return;
    const int4 m = meta[stage];
    const int p = m.x, nrows = m.y, slot0 = m.z;
    if ((m.w & 2) == 0) {
      const bool fresh = (m.w & 1) != 0;
      const int nch = nrows * (Dk / 8);  // 16-byte chunks of this call's rows
      const uint4* src = reinterpret_cast<const uint4*>(stages + (size_t)stage * stage_bytes);
      uint4 v[kLatStgChunks];
#pragma unroll
      for (int t = 0; t < kLatStgChunks; ++t) {
        const int c = tid + kLatStgThreads * t;
        v[t] = c < nch ? src[c] : make_uint4(0, 0, 0, 0);
      }
      const long long row_base = (long long)p * P + slot0;  // destination row of chunk row 0
      if (!fp8) {  // a bf16 latent pool: the rows' bits
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(d.k_cache) + row_base * Dk);
#pragma unroll
        for (int t = 0; t < kLatStgChunks; ++t) {
          const int c = tid + kLatStgThreads * t;
          if (c < nch) dst[c] = v[t];
        }
      } else {
        float s, amax;
        bool own_rows = false;  // the scale is the amax of exactly these rows
        if (fresh) {
          if (!lat_stg_amax(v, red, &cbar, meets, abort_flag, d.ctl, amax)) return;
          s = scale_from_amax(amax);
          if (tid == 0) d.k_scale[p] = s;
          own_rows = true;
        } else {
          s = d.k_scale[p];
          if (d.scale_mode == KV_SCALE_REQUANTIZE) {  // re-encode the rows already written
            // (every thread has read the old scale before the reduction's meeting)
            if (!lat_stg_amax(v, red, &cbar, meets, abort_flag, d.ctl, amax)) return;
            const float s_new = scale_from_amax(amax);
            if (s_new > s) {
              requant_block(static_cast<uint8_t*>(d.k_cache) + (long long)p * P * Dk, slot0, Dk,
                            false, (int)P, s, s_new, tid, kLatStgThreads);
              if (tid == 0) d.k_scale[p] = s_new;
              s = s_new;
              own_rows = true;
            }
          }
        }
        const float rs = __frcp_rn(s);
        uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(d.k_cache) + row_base * Dk);
        if (own_rows && scale_fast_ok(s)) {  // uniform across the consumers
#pragma unroll
          for (int t = 0; t < kLatStgChunks; ++t) {
            const int c = tid + kLatStgThreads * t;
            if (c < nch)
              dst[c] = make_uint2(
                  quant_word_fresh(v[t].x, s, rs) | (quant_word_fresh(v[t].y, s, rs) << 16),
                  quant_word_fresh(v[t].z, s, rs) | (quant_word_fresh(v[t].w, s, rs) << 16));
          }
        } else {
#pragma unroll
          for (int t = 0; t < kLatStgChunks; ++t) {
            const int c = tid + kLatStgThreads * t;
            if (c < nch) dst[c] = quant8_rs(v[t], s, rs);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
}

// Block-wide largest magnitude of the latent rows a CTA holds (bit-pattern
// maximum; a NaN falls back to the float maximum, which skips it).
__device__ float latent_block_amax(const uint4 (&v)[kLatChunks], uint32_t* redu) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t mb = 0;
#pragma unroll
  for (int t = 0; t < kLatChunks; ++t) mb = absbits_max8(mb, v[t]);
  mb = absbits_warp_max(mb);
  if (lane == 0) redu[warp] = mb;
  __syncthreads();
  mb = __reduce_max_sync(0xffffffffu, lane < kTileWarps ? redu[lane] : 0u);
  float amax = __uint_as_float(mb << 16);
  if (mb > 0x7F80u) {  // uniform across the block
    float m = 0.0f;
#pragma unroll
    for (int t = 0; t < kLatChunks; ++t) m = fmaxf(m, amax8(v[t]));
    m = warp_max(m);
    __syncthreads();
    if (lane == 0) reinterpret_cast<float*>(redu)[warp] = m;
    __syncthreads();
    amax = warp_max(lane < kTileWarps ? reinterpret_cast<float*>(redu)[lane] : 0.0f);
  }
  __syncthreads();  // redu is reused by the next page
  return amax;
}

// Rows of a latent page quantised against a scale they did not set (a partly
// filled page) or a scale below 2^-90: the guarded division (out of line).
__device__ __noinline__ void latent_rows_slow(const uint4 (&v)[kLatChunks], int my_rows, int cpr,
                                              int Dk, float s, float rs, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < kLatChunks; ++t) {
    const int q = lane + 32 * t, qd = q / cpr, qm = q - qd * cpr;
    if (qd < my_rows)
      *reinterpret_cast<uint2*>(dst + (long long)qd * kTileWarps * Dk + 8 * qm) =
          quant8_rs(v[t], s, rs);
  }
}

// Latent: persistent CTAs; each CTA takes (request, page) items in turn.
// kCpr: 16-byte chunks per row when known at compile time (72 for 576-wide
// rows), 0 to take it from the pool.
template <int kCpr>
__global__ void __launch_bounds__(kTileWarps * 32) append_latent_kernel(AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint32_t redu[kTileWarps];
  __shared__ int wsum[kTileWarps];
  const kv_pool_desc& d = a.d;
  const long long P = d.page_size;
  const int Dk = kCpr > 0 ? 8 * kCpr : d.head_dim_k, cpr = kCpr > 0 ? kCpr : Dk / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = min(a.B, (int)d.ctl[KV_CTL_APPEND_STOP]);
  int* pre = reinterpret_cast<int*>(smem);
  const int total = B > 0 ? bulk_items_prefix(a, B, 1, pre, wsum) : 0;
  for (int it = blockIdx.x; it < total; it += gridDim.x) {
    const int r = item_owner(pre, B, it);
    const long long n = req_rows(a, r);
    const long long Lnew = a.seq_lens[r], L0 = Lnew - n;
    const long long jp = L0 / P + (it - pre[r]);
    const long long pos_lo = max(jp * P, L0), pos_hi = min((jp + 1) * P, Lnew);
    const int nrows = (int)(pos_hi - pos_lo);
    const int slot0 = (int)(pos_lo - jp * P);
    const long long row0 = a.from_pool ? 0 : a.new_indptr[r] + (pos_lo - L0);
    const int p = a.page_table[(long long)r * a.max_pages + jp];
    if (p < 0 || p >= d.num_pages) {  // uniform across the block
      if (threadIdx.x == 0) set_error(d.ctl, KV_ERR_BAD_PAGE_ID);
      continue;
    }
    int sp = 0;  // handoff: source page jp (the destination request was empty)
    if (a.from_pool) {
      sp = a.src_page_table[(long long)r * a.src_max_pages + jp];
      if (sp < 0 || sp >= a.src.num_pages) {  // uniform across the block
        if (threadIdx.x == 0) set_error(d.ctl, KV_ERR_BAD_PAGE_ID);
        continue;
      }
    }
    const bool fresh = jp * P >= L0;
    // not through a stale mapping (see append_data_kernel)
    if (!fresh && d.tags[p] != a.exp_tags[(long long)r * a.max_pages + jp]) continue;
    // warp w takes rows w, w + 8, ... of this call's rows in the page
    const int my_rows = nrows > warp ? (nrows - warp + kTileWarps - 1) / kTileWarps : 0;
    const uint16_t* src = a.from_pool ? static_cast<const uint16_t*>(a.src.k_cache) +
                                            ((long long)sp * P + warp) * Dk
                                      : a.k_new + (row0 + warp) * Dk;
    // chunk t of this lane: q = lane + 32 t, row q / cpr of the warp's rows
    uint4 v[kLatChunks];
#pragma unroll
    for (int t = 0; t < kLatChunks; ++t) {
      const int q = lane + 32 * t, qd = q / cpr, qm = q - qd * cpr;
      v[t] = qd < my_rows
                 ? *reinterpret_cast<const uint4*>(src + (long long)qd * kTileWarps * Dk + 8 * qm)
                 : make_uint4(0, 0, 0, 0);
    }
    if (d.dtype != KV_DTYPE_E4M3) {  // a bf16 latent pool: the rows' bits
      uint16_t* dst16 = static_cast<uint16_t*>(d.k_cache) + (long long)(p * P + slot0 + warp) * Dk;
#pragma unroll
      for (int t = 0; t < kLatChunks; ++t) {
        const int q = lane + 32 * t, qd = q / cpr, qm = q - qd * cpr;
        if (qd < my_rows)
          *reinterpret_cast<uint4*>(dst16 + (long long)qd * kTileWarps * Dk + 8 * qm) = v[t];
      }
      continue;
    }
    float s;
    bool own_rows = false;  // every row of the page's block is in this call
    if (fresh) {
      s = scale_from_amax(latent_block_amax(v, redu));
      if (threadIdx.x == 0) d.k_scale[p] = s;
      own_rows = true;
    } else {
      s = d.k_scale[p];
      if (d.scale_mode == KV_SCALE_REQUANTIZE) {  // re-encode the rows already written
        const float s_new = scale_from_amax(latent_block_amax(v, redu));
        if (s_new > s) {
          requant_block(static_cast<uint8_t*>(d.k_cache) + (long long)p * P * Dk, slot0, Dk,
                        false, (int)P, s, s_new, threadIdx.x, kTileWarps * 32);
          s = s_new;
          own_rows = true;  // the new scale is the amax of exactly these rows
        }
        __syncthreads();  // the old scale is read by every thread
        if (threadIdx.x == 0 && s_new > d.k_scale[p]) d.k_scale[p] = s_new;
      }
    }
    const float rs = __frcp_rn(s);
    uint8_t* dst = static_cast<uint8_t*>(d.k_cache) + (long long)(p * P + slot0 + warp) * Dk;
    if (own_rows && scale_fast_ok(s)) {  // uniform across the block
#pragma unroll
      for (int t = 0; t < kLatChunks; ++t) {
        const int q = lane + 32 * t, qd = q / cpr, qm = q - qd * cpr;
        if (qd < my_rows)
          *reinterpret_cast<uint2*>(dst + (long long)qd * kTileWarps * Dk + 8 * qm) = make_uint2(
              quant_word_fresh(v[t].x, s, rs) | (quant_word_fresh(v[t].y, s, rs) << 16),
              quant_word_fresh(v[t].z, s, rs) | (quant_word_fresh(v[t].w, s, rs) << 16));
      }
    } else {
      latent_rows_slow(v, my_rows, cpr, Dk, s, rs, dst);
    }
  }
}

}  // namespace

namespace {

// the persistent kernels' shape limits (a GQA tile in one warp's registers;
// a latent page over one CTA's warps)
bool gqa_tile_fits(const kv_pool_desc& d) {
  return (long long)d.page_size * d.head_dim_k <= 32 * 8 * kTileChunks &&
         (long long)d.page_size * d.head_dim_v <= 32 * 8 * kTileChunks;
}
bool latent_page_fits(const kv_pool_desc& d) {
  return d.page_size <= 8 * kTileWarps &&
         (long long)((d.page_size + kTileWarps - 1) / kTileWarps) * (d.head_dim_k / 8) <=
             32 * kLatChunks;
}

}  // namespace

bool append_handoff_supported(const kv_pool_desc& d, int B, int src_max_pages) {
  const long long per_page = d.layout == KV_LAYOUT_GQA ? 2LL * d.num_kv_heads : 1LL;
  if (B > kMaxPersistB || (long long)B * src_max_pages * per_page > INT_MAX) return false;
  return d.layout == KV_LAYOUT_GQA ? gqa_tile_fits(d) : latent_page_fits(d);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s, int* launches) {
  cudaError_t e = launch_pdl(append_plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  ++*launches;
  // pages a request can touch in one call: ceil((max_new + P - 1) / P)
  const long long P = a.d.page_size;
  long long pieces = a.from_pool ? (long long)a.src_max_pages : (a.max_new + 2 * P - 2) / P;
  if (pieces <= 0 || a.B <= 0) return cudaSuccess;
  const long long pages_per_req = pieces;
  if (pieces > 65535) pieces = 65535;  // the kernel strides over the rest
  const long long Pl = a.d.page_size;
  const int es = a.d.dtype == KV_DTYPE_E4M3 ? 1 : 2;
  // The register-resident kernels are large: a decode-size append (a few
  // rows per request, a handful of CTAs) spends its time fetching their
  // instructions, so it takes the compact per-tile kernel below.
  // (a handoff always takes them: the host checked its shape fits)
  const bool bulk = a.from_pool || a.max_new >= 2 * Pl;
  static int sms = 0;
  if (sms == 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess)
    sms = 0;
  const size_t pre_bytes = sizeof(int) * ((size_t)a.B + 1);
  // the work-item count is held in an int
  const long long per_page = a.d.layout == KV_LAYOUT_GQA ? 2LL * a.d.num_kv_heads : 1LL;
  const bool persist = bulk && sms > 0 && a.B <= kMaxPersistB &&
                       (long long)a.B * pages_per_req * per_page <= INT_MAX;
  if (a.from_pool && !persist) return cudaErrorNotSupported;
  if (persist && a.d.layout == KV_LAYOUT_GQA && gqa_tile_fits(a.d) && a.B <= kStgMaxB) {
    // the staged kernel: a page's K and V rows per stage, 2..4 stages
    const long long stage = (Pl * a.d.num_kv_heads * (a.d.head_dim_k + a.d.head_dim_v) * 2 + 127) /
                            128 * 128;
    const size_t fixed = stg_fixed_bytes(a.d.head_dim_v, (int)Pl, es, a.B);
    const long long room = 227LL * 1024 - (long long)fixed;
    const int S = (int)min((long long)kStgMaxStages, room > 0 ? room / stage : 0);
    if (S >= 2) {
      const size_t smem = (size_t)S * stage + fixed;
      e = a.from_pool ? cudaFuncSetAttribute(append_gqa_staged_kernel<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                      : cudaFuncSetAttribute(append_gqa_staged_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      e = a.from_pool ? launch_pdl(append_gqa_staged_kernel<true>, dim3((unsigned)sms),
                                   dim3(kStgThreads), smem, s, a, S, (int)stage)
                      : launch_pdl(append_gqa_staged_kernel<false>, dim3((unsigned)sms),
                                   dim3(kStgThreads), smem, s, a, S, (int)stage);
      if (e == cudaSuccess) ++*launches;
      return e;
    }
  }
  if (persist && a.d.layout == KV_LAYOUT_GQA && gqa_tile_fits(a.d)) {
    const size_t smem = (size_t)kTileWarps * a.d.head_dim_v * Pl * es + pre_bytes;
    if (smem > 48 * 1024) {
      e = a.from_pool ? cudaFuncSetAttribute(append_gqa_kernel<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                      : cudaFuncSetAttribute(append_gqa_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    e = a.from_pool ? launch_pdl(append_gqa_kernel<true>, dim3((unsigned)(2 * sms)),
                                 dim3(kTileWarps * 32), smem, s, a)
                    : launch_pdl(append_gqa_kernel<false>, dim3((unsigned)(2 * sms)),
                                 dim3(kTileWarps * 32), smem, s, a);
    if (e == cudaSuccess) ++*launches;
    return e;
  }
  if (persist && a.d.layout == KV_LAYOUT_LATENT && latent_page_fits(a.d) && a.B <= kStgMaxB &&
      Pl * a.d.head_dim_k <= 8LL * kLatStgThreads * kLatStgChunks) {
    // the staged kernel: one page's rows per stage, 2..4 stages
    const long long stage = (Pl * a.d.head_dim_k * 2 + 127) / 128 * 128;
    // (256 bytes left for the kernel's static shared memory)
    const long long room = 227LL * 1024 - 256 - (long long)stg_ring_bytes(a.B);
    const int S = (int)min((long long)kStgMaxStages, room > 0 ? room / stage : 0);
    if (S >= 2) {
      const size_t smem = (size_t)S * stage + stg_ring_bytes(a.B);
      e = a.from_pool ? cudaFuncSetAttribute(append_latent_staged_kernel<true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                      : cudaFuncSetAttribute(append_latent_staged_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      e = a.from_pool ? launch_pdl(append_latent_staged_kernel<true>, dim3((unsigned)sms),
                                   dim3(kStgThreads), smem, s, a, S, (int)stage)
                      : launch_pdl(append_latent_staged_kernel<false>, dim3((unsigned)sms),
                                   dim3(kStgThreads), smem, s, a, S, (int)stage);
      if (e == cudaSuccess) ++*launches;
      return e;
    }
  }
  if (persist && a.d.layout == KV_LAYOUT_LATENT && latent_page_fits(a.d)) {
    const bool k72 = a.d.head_dim_k == 576;
    if (pre_bytes > 48 * 1024) {
      e = k72 ? cudaFuncSetAttribute(append_latent_kernel<72>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pre_bytes)
              : cudaFuncSetAttribute(append_latent_kernel<0>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pre_bytes);
      if (e != cudaSuccess) return e;
    }
    e = k72 ? launch_pdl(append_latent_kernel<72>, dim3((unsigned)(2 * sms)),
                         dim3(kTileWarps * 32), pre_bytes, s, a)
            : launch_pdl(append_latent_kernel<0>, dim3((unsigned)(2 * sms)),
                         dim3(kTileWarps * 32), pre_bytes, s, a);
    if (e == cudaSuccess) ++*launches;
    return e;
  }
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
