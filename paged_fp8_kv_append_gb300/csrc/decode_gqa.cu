// decode_gqa.cu -- split-K paged decode attention over a GQA cache (e4m3 or
// bf16), the batch plan it runs on, and the combine step.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": decode attention reads the FP8 e4m3 cache and
// converts values as it reads them; BF16 is the baseline cache format.
// Section "Protecting a shared KV cache": aborted requests read nothing and
// return nothing.
//
// Work decomposition.  The unit of work is one page of one request for a
// group of Hs kv heads.  Units are laid out request-major, head-group-minor
// ("segments" of ceil(L_r/P) pages each; aborted requests have none) and cut
// into gridDim.x equal contiguous ranges, one per persistent CTA, so every
// CTA streams the same number of bytes whatever the length mix.  A CTA range
// crosses segment boundaries; each (CTA, segment) piece yields one partial
// (o, running max, sum) in slot segment + cta (injective because both are
// sorted along the range), and the combine kernel merges the pieces of a
// segment.
//
// CTA layout: the last warp is the producer: it reads page ids and scales
// and moves each unit's K tiles and V tiles into a shared-memory ring with
// bulk async copies (cp.async.bulk, completion on an mbarrier).  The other
// warps are consumers, each serving one (kv head, block of query rows) of
// every few units; it keeps its own online-softmax state and merges with the
// warps that share its rows at the end of a piece.
//
// Per page a consumer computes S^T = K Q^T (M = 16 tokens, N = 8 query rows,
// K = 128 dims) and O^T += V^T P^T (M = 128 dims, N = 8 rows, K = 16 tokens)
// with mma.sync m16n8k16.  With more than 8 query rows per kv head the
// consumers take 16 rows as the M dimension instead (gqa_split_wide_kernel,
// gqa_split_wide_bf16_kernel), so each K/V byte is read and converted once
// for all the rows of its kv head.  At 8 query rows per kv head the work is
// 16 flop per cache byte, beyond what the fp32 CUDA cores sustain at HBM
// speed, so the tensor pipe carries the dot products and the CUDA cores only
// convert and run the softmax.  e4m3 codes convert exactly to f16; the per-page K scale
// multiplies the scores and the V scale enters P as an exponent bias.
#include <float.h>

#include "common.cuh"
#include "decode_plan.cuh"
#include "internal.h"

namespace kvfp8 {
namespace {

// ----------------------------------------------------------- batch plan

constexpr int kPlanThreads = kDecodePlanThreads;

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(DecodeArgs a) {
  pdl_wait();
  pdl_trigger();
  decode_plan_block(a);
}

// ------------------------------------------------- segment cursor

// Walks segments (request r, head group h) of the flattened unit sequence;
// `groups` is the number of head groups per request.  pfx may live in shared
// or global memory.
struct Cursor {
  int r, h, np;
  long long seg_start;
};

__device__ __forceinline__ Cursor cursor_at(const int32_t* pfx, int B, int groups, long long x) {
  // last r with pfx[r] <= x / groups; that request has pages (pfx[r+1] > x/groups)
  const long long v = x / groups;
  int lo = 0, hi = B;  // invariant: pfx[lo] <= v < pfx[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pfx[mid] <= v)
      lo = mid;
    else
      hi = mid;
  }
  Cursor c;
  c.r = lo;
  c.np = pfx[lo + 1] - pfx[lo];
  c.h = (int)((x - (long long)groups * pfx[lo]) / c.np);
  c.seg_start = (long long)groups * pfx[lo] + (long long)c.h * c.np;
  return c;
}

__device__ __forceinline__ void cursor_next(Cursor& c, const int32_t* pfx, int B, int groups) {
  if (++c.h == groups) {
    c.h = 0;
    do {
      ++c.r;
    } while (c.r < B && pfx[c.r + 1] == pfx[c.r]);
    if (c.r < B) c.np = pfx[c.r + 1] - pfx[c.r];
  }
  if (c.r < B) {
    c.seg_start = (long long)groups * pfx[c.r] + (long long)c.h * c.np;
  } else {  // past the last request (cannot happen inside a CTA range): end every loop
    c.seg_start = (long long)groups * pfx[B];
    c.np = 1;
  }
}

// ------------------------------------------------- tensor-core helpers


// Four e4m3 codes (bytes 0..3 of w) -> two f16x2 words, lo = (b0, b1) and
// hi = (b2, b3); exact (every e4m3 value is an f16 value).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// 2^x on the special-function unit (flushes denormal results to zero, which
// only drops softmax weights below 2^-126).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The e4m3 paths multiply the bf16 query in f16.  Each query row is first
// scaled by an exact power of two 2^e that puts its largest magnitude in
// [2^15, 2^16): inside f16's range (below 65504) with all of its bits, and
// small elements stay clear of f16's subnormals.  The row's scores are then
// 2^e times the true ones and its score scale takes 2^-e.  For a row whose
// elements are all normal f16 values either way, scores are bit-identical to
// the unscaled ones (a power-of-two factor commutes with rounding).
// Largest magnitude of 8 bf16 values as a bit pattern with the sign cleared
// (bit-pattern order is magnitude order for finite values).
__device__ __forceinline__ uint32_t bf16_absbits_max8(const uint4& v) {
  const uint32_t a = max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu);
  const uint32_t b = max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu);
  const uint32_t c = max(v.z & 0x7FFFu, (v.z >> 16) & 0x7FFFu);
  const uint32_t d = max(v.w & 0x7FFFu, (v.w >> 16) & 0x7FFFu);
  return max(max(a, b), max(c, d));
}
// e for a row whose largest magnitude has bf16 bits mb: 15 - floor(log2),
// within [-112, 112] so that 2^e and 2^-e times the score scale stay normal
// fp32 numbers (all-zero or subnormal rows take 112).
__device__ __forceinline__ int q_row_exp(uint32_t mb) {
  const int E = (int)(mb >> 7);
  return E == 0 ? 112 : min(112, max(-112, 142 - E));
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float pw) {
  const float lo = __uint_as_float(w << 16) * pw, hi = __uint_as_float(w & 0xFFFF0000u) * pw;
  return f32x2_to_f16x2(lo, hi);
}

template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ uint32_t lds32(const void* p) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ uint32_t w_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// ------------------------------------------------- split kernel

// A unit of work is one page of one request for Hs kv heads (a "head
// group"; Hs = the largest power of two <= 8 that divides Hkv, <= 4 for
// bf16).  The Hs K tiles of a page are contiguous in the cache, and so are
// its Hs V tiles, so one unit is two bulk copies of Hs * P * D elements.
// One CTA per SM: a producer warp and CONSUMERS consumer warps.  A kv head's
// R = T * G query rows come in RB = ceil(R / 8) blocks of 8 (one mma N tile);
// a (kv head, row block) pair is a "virtual head", Hv = Hs * RB of them per
// unit.  Consumer w serves virtual head w % Hv of every (w / Hv)-th unit, so
// each unit is consumed by exactly Hv warps, which share its K and V tiles.
// The ring holds kRingBytes of units in flight.
#ifndef KV_GQA_FP8_CONSUMERS
#define KV_GQA_FP8_CONSUMERS 12
#endif
#ifndef KV_GQA_BF16_CONSUMERS
#define KV_GQA_BF16_CONSUMERS 8
#endif
#ifndef KV_GQA_RING_KB
#define KV_GQA_RING_KB 160
#endif

constexpr int kMaxStages = 40;

template <bool FP8>
struct GqaCfg {
  static constexpr int P = 16;                      // tokens per page
  static constexpr int D = 128;                     // head dim (K and V)
  static constexpr int ES = FP8 ? 1 : 2;            // cache element bytes
  static constexpr int TILE = P * D * ES;           // bytes of one head's K or V tile
  static constexpr int RING = KV_GQA_RING_KB * 1024;
  // consumer warps: e4m3 pages carry half the bytes of bf16 ones, so each
  // byte needs twice the consumer work; measured best at 12 (e4m3) and 8 (bf16)
  static constexpr int CONSUMERS = FP8 ? KV_GQA_FP8_CONSUMERS : KV_GQA_BF16_CONSUMERS;
  static constexpr int THREADS = (CONSUMERS + 1) * 32;
  static constexpr int R8 = 8;                      // query rows per kv head (padded)
  static constexpr int PFX_CACHE = 1024;            // pfx entries cached in smem
  static constexpr int PBUF = FP8 ? R8 * P * 2 : R8 * P * 4;  // per-warp P transpose
  // shared memory carve-up (byte offsets)
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_MERGE_O = OFF_RING + RING;                         // [W][R8][D] f32
  static constexpr int OFF_MERGE_ML = OFF_MERGE_O + CONSUMERS * R8 * D * 4;  // [W][R8][2] f32
  static constexpr int OFF_PBUF = OFF_MERGE_ML + CONSUMERS * R8 * 2 * 4;
  static constexpr int OFF_META = OFF_PBUF + CONSUMERS * PBUF;               // [S] StageMeta
  static constexpr int OFF_BAR = OFF_META + kMaxStages * 80;                  // full, empty
  static constexpr int OFF_PFX = OFF_BAR + 2 * kMaxStages * 8;
  static constexpr int OFF_FLAG = OFF_PFX + PFX_CACHE * 4;  // abort flag, piece-bad flag
  static constexpr int OFF_WSUM = OFF_FLAG + 16;              // [32] plan scan warp sums
  static constexpr int SMEM = OFF_WSUM + 32 * 4;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Most units a producer warp issues per warp instruction (one per lane; at most
// a quarter of the ring depth so most stages stay in flight while a group waits).
constexpr int kIssueGroup = 8;

struct StageMeta {
  int n_valid;    // tokens of this page below the request length; -1: a page
                  // that must not be read (id out of range or stale tag)
  int pos0;       // position of the page's first token
  float ks[8];    // K scales of the unit's heads (1 for bf16)
  float vs[8];    // V scales
  int unit;       // stage sequence number (low 32 bits): consumers check it
  int pad;
};
static_assert(sizeof(StageMeta) == 80, "StageMeta layout");

// End of a piece: merges the online-softmax states of the WPH warps that
// share each of the Hv virtual heads (8 rows each) into the piece's partial.
// merge_ml[(w * 8 + nw) * 2 + {0, 1}] holds warp w's running max and sum of
// row nw, merge_o[(w * 8 + nw) * 128 + dd] its unnormalised output.  Pass 1,
// one thread per row: the row's max M over the warps, each warp's weight
// 2^(m_w - M) (written over m_w) and the weighted sum, stored with M (a
// piece that met a page it must not read stores the sum -1 instead).  Pass
// 2, every consumer thread: the weighted outputs, four dims at a time.
// row_of(v, nw) is the partial row of virtual head v's row nw.  Starts and
// ends with the consumer warps synchronised.
template <class C, class RowOf>
__device__ __forceinline__ void merge_piece(float* merge_o, float* merge_ml, int Hv, int WPH,
                                            const DecodeArgs& a, RowOf row_of,
                                            volatile int* piece_bad, bool reset_bad) {
  constexpr int R8 = C::R8, D = C::D, NT = C::CONSUMERS * 32;
  static_assert(R8 == 8 && D == 128, "index shifts");
  const int tid = threadIdx.x;
  named_bar_sync(1, NT);  // every warp's state is in the merge buffers
  if (tid < Hv * R8) {
    const int v = tid >> 3, nw = tid & 7;
    float M = -INFINITY;
    for (int q = 0; q < WPH; ++q) M = fmaxf(M, merge_ml[((q * Hv + v) * R8 + nw) * 2]);
    float lsum = 0.0f;
    for (int q = 0; q < WPH; ++q) {
      float* ml = merge_ml + ((q * Hv + v) * R8 + nw) * 2;
      const float w = (ml[0] == -INFINITY) ? 0.0f : exp2f(ml[0] - M);
      lsum += ml[1] * w;
      ml[0] = w;
    }
    const long long row = row_of(v, nw);
    a.ws.ml_part[row * 2 + 0] = M;
    a.ws.ml_part[row * 2 + 1] = *piece_bad ? -1.0f : lsum;
  }
  named_bar_sync(1, NT);
  if (reset_bad && tid == 0) *piece_bad = 0;
  for (int e = tid; e < Hv * R8 * (D / 4); e += NT) {
    const int d4 = e & 31, rr = e >> 5, v = rr >> 3, nw = rr & 7;
    float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int q = 0; q < WPH; ++q) {
      const int w = (q * Hv + v) * R8 + nw;
      const float wt = merge_ml[w * 2];
      const float4 x = *reinterpret_cast<const float4*>(merge_o + w * D + 4 * d4);
      o.x = fmaf(wt, x.x, o.x);
      o.y = fmaf(wt, x.y, o.y);
      o.z = fmaf(wt, x.z, o.z);
      o.w = fmaf(wt, x.w, o.w);
    }
    *reinterpret_cast<float4*>(a.ws.o_part + row_of(v, nw) * D + 4 * d4) = o;
  }
  named_bar_sync(1, NT);
}

// WIDE: a consumer warp takes 16 query rows of its kv head instead of 8 (see
// the wide consumer below); the producer and the ring are the same.
template <bool FP8, bool WIDE>
__device__ __forceinline__ void gqa_split_body(const DecodeArgs& a) {
  using C = GqaCfg<FP8>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem + C::OFF_RING;
  float* merge_o = reinterpret_cast<float*>(smem + C::OFF_MERGE_O);
  float* merge_ml = reinterpret_cast<float*>(smem + C::OFF_MERGE_ML);
  uint8_t* pbuf_all = smem + C::OFF_PBUF;
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + C::OFF_META);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + kMaxStages;
  int32_t* pfx_s = reinterpret_cast<int32_t*>(smem + C::OFF_PFX);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  volatile int* piece_bad = abort_flag + 1;
  int* wsum_s = reinterpret_cast<int*>(smem + C::OFF_WSUM);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.B, Hkv = a.d.num_kv_heads;
  const int Hs = a.Hs, HG = a.HG;              // heads per unit, head groups
  // query rows of a kv head come in blocks of 8 (16 for WIDE), one block per
  // consumer warp: a unit is consumed by Hv = Hs * RBW warps ("virtual heads")
  const int RB = a.R8 / C::R8;
  const int RBW = WIDE ? (RB + 1) / 2 : RB, Hv = Hs * RBW;
  const int rb_mul = (256 + RB - 1) / RB;  // v / RB == (v * rb_mul) >> 8 for v < 12
  const int S = a.stages;                      // ring stages (<= kMaxStages)
  const int stage_bytes = 2 * Hs * C::TILE;
  // 8-row consumers: exactly ceil(R / 8) row blocks (at most 4); 16-row
  // consumers: an even count of at most 8, which may include whole padding
  // blocks (the host pads so that the warps divide evenly)
  const bool rows_ok = WIDE ? (RB % 2 == 0 && RB <= 8 && a.R >= 1 && a.R <= C::R8 * RB)
                            : (RB <= 4 && (a.R + C::R8 - 1) / C::R8 == RB);
  // (not in the 16-row e4m3 kernel: at its 128-register cap the plan code
  // made it spill)
  constexpr bool kCanSelfPlan = !(FP8 && WIDE);
  if (Hs < 1 || RB < 1 || !rows_ok || RB * C::R8 != a.R8 ||
      C::CONSUMERS % Hv != 0 || S < 2 || S > kMaxStages || S % (C::CONSUMERS / Hv) != 0 ||
      stage_bytes * S > C::RING ||
      (a.self_plan && (B + 1 > C::PFX_CACHE || !kCanSelfPlan))) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) set_error(a.d.ctl, KV_ERR_INTERNAL);  // host chose a bad configuration
    return;
  }
  // Before the wait for the kernels ahead of this one: only this CTA's shared
  // memory (the ring barriers), so the set-up overlaps their tail.
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // two arrivals: the copies' expected bytes, then the stage metadata
      mbar_init(&full[s], 2);
      mbar_init(&empty[s], Hv);
    }
    *abort_flag = 0;
    *piece_bad = 0;
    fence_mbar_init();
  }
  pdl_wait();
  pdl_trigger();  // the combine's CTAs may wait resident in what this kernel leaves free
  // the batch plan: built here (self_plan; CTA 0 stores it for the combine)
  // or read from the plan kernel's output, cached in shared memory
  const int32_t* pfx_g = a.ws.pfx;
  const bool cached = B + 1 <= C::PFX_CACHE;
  if (kCanSelfPlan && a.self_plan) {
    const bool refused = decode_plan_shared(a, pfx_s, wsum_s);
    if (blockIdx.x == 0) decode_plan_store(a, pfx_s, refused);
  } else if (cached) {
    for (int i = threadIdx.x; i <= B; i += C::THREADS) pfx_s[i] = pfx_g[i];
  }
  __syncthreads();  // the plan and the barrier set-up are visible to every warp
  const int32_t* pfx = cached ? pfx_s : pfx_g;
  const long long total = (long long)pfx[B] * HG;
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  const long long x_begin = (long long)blockIdx.x * per;
  const long long x_end = min(total, x_begin + per);
  if (x_begin >= x_end) return;
  const Cursor start = cursor_at(pfx, B, HG, x_begin);
  const int P = C::P, D = C::D;

  if (warp == C::CONSUMERS) {
    // ======================= producer warp =======================
    // Lane l owns unit x0 + l of each batch of 32 consecutive units.  Page
    // ids (and lengths) are loaded two batches ahead and scales one batch
    // ahead, so the dependent page-id -> scale loads never hold up the copy
    // issue; each lane then issues its own unit's two copies.
    const uint64_t policy = l2_evict_first_policy();
    const int maxp = a.max_pages;
    Cursor lc = start;  // per-lane cursor, only moves forward
    struct Unit {
      int r, hg, j, p, L;
    };
    auto locate_load = [&](long long xu) {
      Unit u;
      u.r = 0;
      u.hg = 0;
      u.j = 0;
      u.p = -1;
      u.L = 0;
      if (xu < x_end) {
        while (xu >= lc.seg_start + lc.np) cursor_next(lc, pfx, B, HG);
        u.r = lc.r;
        u.hg = lc.h;
        u.j = (int)(xu - lc.seg_start);
        u.p = a.page_table[(long long)u.r * maxp + u.j];
        u.L = a.seq_lens[u.r];
      }
      return u;
    };
    // a page may be read only if its id is in range and, with the fused
    // check, its tag is the expected one; the tag and the scales are loaded
    // together (both depend only on the page id)
    auto scales = [&](const Unit& u, long long xu, float (&ks)[8], float (&vs)[8], bool& ok) {
      ok = false;
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) ks[hh] = vs[hh] = 1.0f;
      if (xu < x_end) {
        const bool in_range = u.p >= 0 && u.p < a.d.num_pages;
        uint32_t tag = 0, et = 0;
        if (in_range) {
          if (a.exp_tags != nullptr) {
            tag = a.d.tags[u.p];
            et = a.exp_tags[(long long)u.r * maxp + u.j];
          }
          if (FP8) {
            const long long base = (long long)u.p * Hkv + (long long)u.hg * Hs;
#pragma unroll
            for (int hh = 0; hh < 8; ++hh) {
              if (hh < Hs) {
                ks[hh] = a.d.k_scale[base + hh];
                vs[hh] = a.d.v_scale[base + hh];
              }
            }
          }
        }
        // without the fused check `ok` must not wait for any load
        ok = in_range && (a.exp_tags == nullptr || tag == et);
        if (!in_range) set_error(a.d.ctl, KV_ERR_BAD_PAGE_ID);
      }
    };
    Unit u0 = locate_load(x_begin + lane);
    Unit u1 = locate_load(x_begin + 32 + lane);
    float ks0[8], vs0[8], ks1[8], vs1[8];
    bool ok0, ok1;
    scales(u0, x_begin + lane, ks0, vs0, ok0);
    // issue group: a group waits for the stages of the units S earlier, so it
    // must stay small next to S or the ring drains before it refills; large
    // units (S small) need few issues per byte anyway
    const int grp = max(1, min(kIssueGroup, S / 4));
    long long k = 0;       // stage sequence number of the batch's first unit
    long long issued = 0;  // units whose copies have been issued
    for (long long xb = x_begin; xb < x_end && !*abort_flag; xb += 32) {
      scales(u1, xb + 32 + lane, ks1, vs1, ok1);
      const Unit u2 = locate_load(xb + 64 + lane);
      const int cnt = (int)min(32ll, x_end - xb);
      bool go = true;
      for (int g0 = 0; g0 < cnt && go; g0 += grp) {
        const bool mine = lane >= g0 && lane < min(g0 + grp, cnt);
        // stage numbers stay below 2^31 (the plan refuses larger batches), so
        // 32-bit arithmetic suffices
        const uint32_t kl = (uint32_t)(k + lane), us = (uint32_t)S;
        const int stage = (int)(kl % us);
        bool ok = true;
        if (mine && kl >= us)
          ok = mbar_wait(&empty[stage], ((kl / us) - 1u) & 1u, abort_flag, a.d.ctl,
                         wait_info(warp, 1, stage));
        go = __all_sync(0xffffffffu, ok);
        if (!go) break;
        if (mine) {
          // the copies first (they need only the page id), then the metadata
          // (scales), whose arrival completes the stage with the copies' bytes
          if (ok0) {
            uint8_t* dst = ring + (size_t)stage * stage_bytes;
            const long long ph = (long long)u0.p * Hkv + (long long)u0.hg * Hs;
            mbar_arrive_expect_tx(&full[stage], (uint32_t)stage_bytes);
            bulk_g2s(dst, static_cast<const uint8_t*>(a.d.k_cache) + ph * C::TILE,
                     (uint32_t)(Hs * C::TILE), &full[stage], policy);
            bulk_g2s(dst + Hs * C::TILE, static_cast<const uint8_t*>(a.d.v_cache) + ph * C::TILE,
                     (uint32_t)(Hs * C::TILE), &full[stage], policy);
          } else {
            mbar_arrive(&full[stage]);
          }
          StageMeta m;
          m.n_valid = ok0 ? min(P, u0.L - u0.j * P) : -1;
          m.pos0 = u0.j * P;
#pragma unroll
          for (int hh = 0; hh < 8; ++hh) {
            m.ks[hh] = ks0[hh];
            m.vs[hh] = vs0[hh];
          }
          m.unit = (int)kl;
          m.pad = 0;
          meta[stage] = m;
          mbar_arrive(&full[stage]);
        }
        __syncwarp();
        issued = k + min(g0 + grp, cnt);
      }
      if (!go) break;
      k += cnt;
      u0 = u1;
#pragma unroll
      for (int hh = 0; hh < 8; ++hh) {
        ks0[hh] = ks1[hh];
        vs0[hh] = vs1[hh];
      }
      ok0 = ok1;
      u1 = u2;
    }
    // On abort, copies already issued may still be landing: wait for them
    // (bounded) before this CTA's shared memory goes away.
    if (*abort_flag && lane == 0) {
      for (long long q = max(0ll, issued - S); q < issued; ++q) {
        const int stage = (int)(q % S);
        const uint32_t par = (uint32_t)((q / S) & 1);
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(&full[stage], par) && global_ns() - t0 < 100000000ull) {
        }
      }
    }
    return;
  }

  if constexpr (WIDE) {
    // ================= consumer warps, 16 query rows each =================
    // Rows are the mma M dimension: S = Q K^T (M = 16 rows, N = 8 tokens,
    // two N tiles per page) and O += P V (M = 16 rows, N = 8 dims, 16 dim
    // tiles, K = the page's 16 tokens).  The S accumulators are already in
    // the A-fragment layout of P, so P never leaves registers, and each K/V
    // byte of a kv head is read (and, e4m3, converted) once for all its rows.
    // A kv head's rows take up to 4 such warps (RBW); rows past R are
    // padding.
    //   k-slot order: in k-step j of S, thread t's slots 2t, 2t+1, 2t+8,
    //   2t+9 are dims 32t + 4j + 0..3 (its 32 dims are contiguous: two
    //   16-byte loads of an e4m3 K row, four of a bf16 one); column c of S's
    //   N tile nt is token 2c - (c & 1) + 2 nt, so P's slots 2t, 2t+1 (tile 0)
    //   and 2t+8, 2t+9 (tile 1) are tokens 4t .. 4t+3: one 4-byte (e4m3) or
    //   8-byte (bf16) load of the dim-major V tile gives both B registers of
    //   a PV dim tile.
    const int g = lane >> 2, t = lane & 3;
    const int G = a.G, T = a.T, R = a.R;
    const int WPH = C::CONSUMERS / Hv;      // warps per virtual head
    const int vh = warp % Hv, lg = warp / Hv;
    const int hw = vh / RBW;                // kv head within the group
    const int n0 = (vh - hw * RBW) * 16;    // this warp's first query row of the head
    Cursor cur = start;
    long long x = x_begin;
    long long k_base = 0;
    const float ssl = a.sm_scale_log2;
    const int tok0 = 2 * g - (g & 1);       // token of S column g in tile 0 (tile 1: +2)

    while (x < x_end) {
      const long long seg_end = cur.seg_start + cur.np;
      const long long piece_end = min(seg_end, x_end);
      const int npages = (int)(piece_end - x);
      const int r = cur.r, h = cur.h * Hs + hw;
      const int L = a.seq_lens[r];

      // ---- Q as A fragments {a0, a1, a2, a3} of k-step j = rows g, g+8 x
      // dims 32t+4j+0..1, +2..3, staged in this warp's merge buffer (4 KB,
      // idle until the piece ends) as [j][lane] 16-byte words: registers
      // hold the 16 x 128 output instead
      uint32_t* qs = reinterpret_cast<uint32_t*>(merge_o + warp * C::R8 * D);
      // score scales of rows g and g+8 (with the row's 2^-e for e4m3 pools)
      float qscA = ssl, qscB = ssl;
      {
        uint32_t qa[8][4];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int row = n0 + g + 8 * hr;
          const bool live = row < R;
          const int tq = live ? row / G : 0, hq = live ? h * G + row % G : 0;
          const uint16_t* qrow = a.q + (((long long)r * T + tq) * a.Hq + hq) * D + 32 * t;
          uint4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)  // dims 32t + 8u .. +7: k-steps 2u and 2u+1
            v[u] = live ? *reinterpret_cast<const uint4*>(qrow + 8 * u) : make_uint4(0, 0, 0, 0);
          float pw = 1.0f;
          if constexpr (FP8) {  // the row's 128 dims are spread over the 4 threads t
            uint32_t mb = max(max(bf16_absbits_max8(v[0]), bf16_absbits_max8(v[1])),
                              max(bf16_absbits_max8(v[2]), bf16_absbits_max8(v[3])));
            mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            const int e = q_row_exp(mb);
            pw = pow2f(e);
            if (hr == 0) qscA = ssl * pow2f(-e); else qscB = ssl * pow2f(-e);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            // f16 for e4m3 pools (the codes convert exactly to f16), bf16 as is
            qa[2 * u][hr] = FP8 ? bf16x2_to_f16x2_scaled(v[u].x, pw) : v[u].x;
            qa[2 * u][2 + hr] = FP8 ? bf16x2_to_f16x2_scaled(v[u].y, pw) : v[u].y;
            qa[2 * u + 1][hr] = FP8 ? bf16x2_to_f16x2_scaled(v[u].z, pw) : v[u].z;
            qa[2 * u + 1][2 + hr] = FP8 ? bf16x2_to_f16x2_scaled(v[u].w, pw) : v[u].w;
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(qs + (j * 32 + lane) * 4) =
              make_uint4(qa[j][0], qa[j][1], qa[j][2], qa[j][3]);
        __syncwarp();
      }
      // visibility limits (inclusive) of rows g and g+8
      const int limA = L - T + min((n0 + g) / G, T - 1);
      const int limB = L - T + min((n0 + g + 8) / G, T - 1);

      float mA = -INFINITY, mB = -INFINITY, lA = 0.0f, lB = 0.0f;
      float acc[16][4];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

      const long long kfirst = k_base + (long long)((lg - (int)(k_base % WPH) + WPH) % WPH);
      // stage and phase of unit kk, advanced without a division per page (a
      // step of WPH <= S wraps the ring at most once; S is a multiple of WPH)
      int stage = (int)(kfirst % S);
      uint32_t phase = (uint32_t)((kfirst / S) & 1);
      for (long long kk = kfirst; kk < k_base + npages; kk += WPH) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase,
                                                          abort_flag, a.d.ctl,
                                                          wait_info(warp, 0, stage)));
        const StageMeta& mt = meta[stage];
        if (ok && mt.unit != (int)kk) {  // would mean a stale stage: report, never compute on it
          if (lane == 0) set_error(a.d.ctl, KV_ERR_INTERNAL);
          *abort_flag = 1;
        }
        // (a plain store on the rare path: a register here made this kernel
        // spill; the merge reads the flag after a barrier)
        if (mt.n_valid < 0 && lane == 0) *const_cast<int*>(piece_bad) = 1;
        if (ok && mt.unit == (int)kk && mt.n_valid > 0) {
          const uint8_t* Kt = ring + (size_t)stage * stage_bytes + hw * C::TILE;
          const uint8_t* Vt = ring + (size_t)stage * stage_bytes + (Hs + hw) * C::TILE;
          // ---------------- S = Q K^T: N tile nt, column g = token tok0 + 2 nt
          float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          if constexpr (FP8) {
#pragma unroll
            for (int kh = 0; kh < 2; ++kh) {  // dims 32t + 16 kh .. +15: k-steps 4kh .. 4kh+3
              const uint4 k0 = lds128(Kt + tok0 * 128 + 32 * t + 16 * kh);
              const uint4 k1 = lds128(Kt + (tok0 + 2) * 128 + 32 * t + 16 * kh);
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const uint4 qa = lds128(qs + ((4 * kh + jj) * 32 + lane) * 4);
                uint32_t b0, b1;
                e4m3x4_to_f16(w_of(k0, jj), b0, b1);
                mma16816<true>(s[0], qa.x, qa.y, qa.z, qa.w, b0, b1);
                e4m3x4_to_f16(w_of(k1, jj), b0, b1);
                mma16816<true>(s[1], qa.x, qa.y, qa.z, qa.w, b0, b1);
              }
            }
          } else {
            // bf16 rows of 256 bytes: thread t's 32 dims are 64 bytes, each
            // 16-byte load two k-steps' B registers
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {  // dims 32t + 8 kq .. +7: k-steps 2kq, 2kq+1
              const uint4 k0 = lds128(Kt + tok0 * 256 + 64 * t + 16 * kq);
              const uint4 k1 = lds128(Kt + (tok0 + 2) * 256 + 64 * t + 16 * kq);
#pragma unroll
              for (int jj = 0; jj < 2; ++jj) {
                const uint4 qa = lds128(qs + ((2 * kq + jj) * 32 + lane) * 4);
                mma16816<false>(s[0], qa.x, qa.y, qa.z, qa.w, jj ? k0.z : k0.x,
                                jj ? k0.w : k0.y);
                mma16816<false>(s[1], qa.x, qa.y, qa.z, qa.w, jj ? k1.z : k1.x,
                                jj ? k1.w : k1.y);
              }
            }
          }
          // s[nt][e]: row g (e < 2) or g+8, token 4t + 2 nt + (e & 1); log2 domain
          const float ksc = FP8 ? mt.ks[hw] : 1.0f;
          const float scA = ksc * qscA, scB = ksc * qscB;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[nt][e] *= e < 2 ? scA : scB;
          const int nv = mt.n_valid;
          const bool full_page = nv == P;
          if (!full_page || mt.pos0 + P - 1 > min(limA, limB)) {
            // partial page or causal edge: mask invisible positions
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int tk = 4 * t + 2 * nt + (e & 1);
                const int lim = e < 2 ? limA : limB;
                s[nt][e] = (tk < nv && mt.pos0 + tk <= lim) ? s[nt][e] : -INFINITY;
              }
          }
          float mxA = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
          float mxB = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
#pragma unroll
          for (int o = 1; o < 4; o <<= 1) {
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, o));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, o));
          }
          // the page's V scale as an exponent bias, as in the 8-row consumer
          const float bias = FP8 ? __log2f(mt.vs[hw]) : 0.0f;
          const float unbias = FP8 ? fast_exp2(-bias) : 1.0f;
          const float nA = fmaxf(mA, mxA + bias), nB = fmaxf(mB, mxB + bias);
          const float alA = (nA == -INFINITY) ? 1.0f : fast_exp2(mA - nA);
          const float alB = (nB == -INFINITY) ? 1.0f : fast_exp2(mB - nB);
          const float cA = bias - nA, cB = bias - nB;
          float p[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            p[nt][0] = (nA == -INFINITY) ? 0.0f : fast_exp2(s[nt][0] + cA);
            p[nt][1] = (nA == -INFINITY) ? 0.0f : fast_exp2(s[nt][1] + cA);
            p[nt][2] = (nB == -INFINITY) ? 0.0f : fast_exp2(s[nt][2] + cB);
            p[nt][3] = (nB == -INFINITY) ? 0.0f : fast_exp2(s[nt][3] + cB);
          }
          mA = nA;
          mB = nB;
          // per-thread partial row sums (this thread's tokens); summed over t at the end
          lA = lA * alA + (p[0][0] + p[0][1] + p[1][0] + p[1][1]) * unbias;
          lB = lB * alB + (p[0][2] + p[0][3] + p[1][2] + p[1][3]) * unbias;
          if (__any_sync(0xffffffffu, alA != 1.0f || alB != 1.0f)) {  // a running max moved
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              acc[i][0] *= alA;
              acc[i][1] *= alA;
              acc[i][2] *= alB;
              acc[i][3] *= alB;
            }
          }
          // ---------------- O += P V: P from registers, V tile dim-major;
          // tokens beyond the length are zeroed in V (stale bytes could be NaN)
          const int keep = min(max(nv - 4 * t, 0), 4);
          if constexpr (FP8) {
            const uint32_t pa0 = f32x2_to_f16x2(p[0][0], p[0][1]);
            const uint32_t pa1 = f32x2_to_f16x2(p[0][2], p[0][3]);
            const uint32_t pa2 = f32x2_to_f16x2(p[1][0], p[1][1]);
            const uint32_t pa3 = f32x2_to_f16x2(p[1][2], p[1][3]);
            const uint32_t vmask = keep >= 4 ? 0xFFFFFFFFu : ((1u << (8 * keep)) - 1u);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              uint32_t b0, b1;
              e4m3x4_to_f16(lds32(Vt + (8 * i + g) * 16 + 4 * t) & vmask, b0, b1);
              mma16816<true>(acc[i], pa0, pa1, pa2, pa3, b0, b1);
            }
          } else {
            // P = hi + lo in bf16 keeps ~16 bits of the weights (two MMAs)
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float f0 = p[e >> 1][2 * (e & 1)], f1 = p[e >> 1][2 * (e & 1) + 1];
              ph[e] = f32x2_to_bf16x2(f0, f1);
              pl[e] = f32x2_to_bf16x2(f0 - __uint_as_float(ph[e] << 16),
                                      f1 - __uint_as_float(ph[e] & 0xFFFF0000u));
            }
            // tokens (4t, 4t+1) and (4t+2, 4t+3) of a dim: one 8-byte load
            const uint32_t mlo = keep >= 2 ? 0xFFFFFFFFu : (keep == 1 ? 0x0000FFFFu : 0u);
            const uint32_t mhi = keep >= 4 ? 0xFFFFFFFFu : (keep == 3 ? 0x0000FFFFu : 0u);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint2 vv = lds64(Vt + (8 * i + g) * 32 + 8 * t);
              const uint32_t b0 = vv.x & mlo, b1 = vv.y & mhi;
              mma16816<false>(acc[i], ph[0], ph[1], ph[2], ph[3], b0, b1);
              mma16816<false>(acc[i], pl[0], pl[1], pl[2], pl[3], b0, b1);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        stage += WPH;
        if (stage >= S) {
          stage -= S;
          phase ^= 1u;
        }
      }

      // ---- merge the states of the warps that share a virtual head, 8 rows
      // at a time (rows g, then g + 8) through the 8-row merge buffers
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        lA += __shfl_xor_sync(0xffffffffu, lA, o);
        lB += __shfl_xor_sync(0xffffffffu, lB, o);
      }
      const long long slot = (long long)r * HG + cur.h + blockIdx.x;
      const int rbw_mul = (256 + RBW - 1) / RBW;  // v / RBW == (v * rbw_mul) >> 8 for v < 12
      __syncwarp();  // the warp's last reads of its staged Q come before the merge data
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float* mo = merge_o + warp * C::R8 * D + g * D;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          *reinterpret_cast<float2*>(mo + 8 * i + 2 * t) =
              half ? make_float2(acc[i][2], acc[i][3]) : make_float2(acc[i][0], acc[i][1]);
        if (t == 0) {
          float* ml = merge_ml + (warp * C::R8 + g) * 2;
          ml[0] = half ? mB : mA;
          ml[1] = half ? lB : lA;
        }
        // row nw of virtual head v (kv head hh, row block v - hh RBW) is row
        // 16 (v - hh RBW) + 8 half + nw of the kv head
        merge_piece<C>(merge_o, merge_ml, Hv, WPH, a,
                       [&](int v, int nw) -> long long {
                         const int hh = (v * rbw_mul) >> 8;  // v / RBW (v < 12)
                         const int n = (v - hh * RBW) * 16 + 8 * half + nw;
                         return (slot * Hs + hh) * a.R8 + n;
                       },
                       piece_bad, half == 1);
      }

      k_base += npages;
      x = piece_end;
      if (x == seg_end) cursor_next(cur, pfx, B, HG);
    }
    return;
  }

  // ========================= consumer warps =========================
  const int g = lane >> 2, t = lane & 3;
  uint8_t* pbuf = pbuf_all + warp * C::PBUF;
  const int G = a.G, T = a.T, R = a.R;
  const int WPH = C::CONSUMERS / Hv;          // warps per virtual head
  const int vh = warp % Hv, lg = warp / Hv;  // virtual head, page lane
  const int hw = vh / RB;                    // kv head within the group
  const int n0 = (vh % RB) * C::R8;          // this warp's first query row of the head
  Cursor cur = start;
  long long x = x_begin;
  long long k_base = 0;
  const float ssl = a.sm_scale_log2;

  while (x < x_end) {
    const long long seg_end = cur.seg_start + cur.np;
    const long long piece_end = min(seg_end, x_end);
    const int npages = (int)(piece_end - x);
    const int r = cur.r, h = cur.h * Hs + hw;  // request, kv head of this warp
    const int L = a.seq_lens[r];

    // ---- query fragments for row n = g (zero for padding rows)
    // dims of k-step j: chunk c = t + 4*(j/4) (fp8) -- 16 dims per chunk --
    // or chunk c = t + 4*(j/2) (bf16) -- 8 dims per chunk.
    uint32_t qf[8][2];
    // score scales of rows 2t and 2t+1 (with the row's 2^-e for e4m3 pools)
    float qsc0 = ssl, qsc1 = ssl;
    {
      const int row = n0 + g;
      const bool live = row < R;
      const int tq = live ? row / G : 0, hq = live ? h * G + row % G : 0;
      const uint16_t* qrow = a.q + (((long long)r * T + tq) * a.Hq + hq) * D;
      if constexpr (FP8) {
        uint4 v[2][2];
#pragma unroll
        for (int half = 0; half < 2; ++half)  // chunk t + 4 half: 16 dims = 2 uint4
#pragma unroll
          for (int u = 0; u < 2; ++u)
            v[half][u] = live ? *reinterpret_cast<const uint4*>(qrow + 16 * (t + 4 * half) + 8 * u)
                              : make_uint4(0, 0, 0, 0);
        // the row's 128 dims are spread over the 4 threads t of group g
        uint32_t mb = max(max(bf16_absbits_max8(v[0][0]), bf16_absbits_max8(v[0][1])),
                          max(bf16_absbits_max8(v[1][0]), bf16_absbits_max8(v[1][1])));
        mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
        mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
        const int e = q_row_exp(mb);
        const float pw = pow2f(e);
        // rows 2t and 2t+1 are held by groups 2t and 2t+1
        qsc0 = ssl * pow2f(-__shfl_sync(0xffffffffu, e, 8 * t));
        qsc1 = ssl * pow2f(-__shfl_sync(0xffffffffu, e, 8 * t + 4));
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            // words of v: dims 16c + 8u + {0,1}, {2,3}, {4,5}, {6,7}
            const int j0 = 4 * half + 2 * u;
            qf[j0][0] = bf16x2_to_f16x2_scaled(v[half][u].x, pw);
            qf[j0][1] = bf16x2_to_f16x2_scaled(v[half][u].y, pw);
            qf[j0 + 1][0] = bf16x2_to_f16x2_scaled(v[half][u].z, pw);
            qf[j0 + 1][1] = bf16x2_to_f16x2_scaled(v[half][u].w, pw);
          }
        }
      } else {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (live) v = *reinterpret_cast<const uint4*>(qrow + 8 * (t + 4 * m));
          qf[2 * m][0] = v.x;
          qf[2 * m][1] = v.y;
          qf[2 * m + 1][0] = v.z;
          qf[2 * m + 1][1] = v.w;
        }
      }
    }
    // visibility limit (inclusive) of rows 2t and 2t+1
    const int lim0 = L - T + min((n0 + 2 * t) / G, T - 1);
    const int lim1 = L - T + min((n0 + 2 * t + 1) / G, T - 1);

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    int bad_units = 0;  // OR of the units' n_valid: negative if one must not be read
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

    // this warp's units of the piece: stage numbers kk == lg (mod WPH)
    const long long kfirst = k_base + (long long)((lg - (int)(k_base % WPH) + WPH) % WPH);
    // stage and phase of unit kk, advanced without a division per page (a
    // step of WPH <= S wraps the ring at most once; S is a multiple of WPH)
    int stage = (int)(kfirst % S);
    uint32_t phase = (uint32_t)((kfirst / S) & 1);
    for (long long kk = kfirst; kk < k_base + npages; kk += WPH) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase,
                                                        abort_flag, a.d.ctl,
                                                        wait_info(warp, 0, stage)));
      const StageMeta& mt = meta[stage];
      if (ok && mt.unit != (int)kk) {  // would mean a stale stage: report, never compute on it
        if (lane == 0) set_error(a.d.ctl, KV_ERR_INTERNAL);
        *abort_flag = 1;
      }
      bad_units |= mt.n_valid;  // sign bit: a page that must not be read
      if (ok && mt.unit == (int)kk && mt.n_valid > 0) {
        const uint8_t* Kt = ring + (size_t)stage * stage_bytes + hw * C::TILE;
        const uint8_t* Vt = ring + (size_t)stage * stage_bytes + (Hs + hw) * C::TILE;
        // ---------------- S^T = K Q^T  (two accumulator chains for ILP)
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (FP8) {
          // row g (and g+8): dims 16t..16t+15 and 64+16t..64+16t+15
          const uint4 kA = lds128(Kt + g * 128 + 16 * t);
          const uint4 kB = lds128(Kt + g * 128 + 64 + 16 * t);
          const uint4 hA = lds128(Kt + (g + 8) * 128 + 16 * t);
          const uint4 hB = lds128(Kt + (g + 8) * 128 + 64 + 16 * t);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t a0, a1, a2, a3;
            e4m3x4_to_f16(w_of(j < 4 ? kA : kB, j & 3), a0, a2);
            e4m3x4_to_f16(w_of(j < 4 ? hA : hB, j & 3), a1, a3);
            if (j & 1)
              mma16816<true>(sb, a0, a1, a2, a3, qf[j][0], qf[j][1]);
            else
              mma16816<true>(sa, a0, a1, a2, a3, qf[j][0], qf[j][1]);
          }
        } else {
          // row g (and g+8): chunks t, t+4, t+8, t+12 (8 dims each)
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint4 vg = lds128(Kt + g * 256 + 16 * (t + 4 * m));
            const uint4 v8 = lds128(Kt + (g + 8) * 256 + 16 * (t + 4 * m));
            mma16816<false>(sa, vg.x, v8.x, vg.y, v8.y, qf[2 * m][0], qf[2 * m][1]);
            mma16816<false>(sb, vg.z, v8.z, vg.w, v8.w, qf[2 * m + 1][0], qf[2 * m + 1][1]);
          }
        }
        // scores (log2 domain) for (token g | g+8, row 2t | 2t+1)
        const float ksc = FP8 ? mt.ks[hw] : 1.0f;
        const float sc0 = ksc * qsc0, sc1 = ksc * qsc1;
        float s[4] = {(sa[0] + sb[0]) * sc0, (sa[1] + sb[1]) * sc1, (sa[2] + sb[2]) * sc0,
                      (sa[3] + sb[3]) * sc1};
        const int nv = mt.n_valid;
        const bool full_page = nv == P;
        if (!full_page || mt.pos0 + P - 1 > min(lim0, lim1)) {
          // partial page or causal edge: mask invisible positions
          const int pA = mt.pos0 + g, pB = mt.pos0 + g + 8;
          const bool vA = g < nv, vB = g + 8 < nv;
          s[0] = (vA && pA <= lim0) ? s[0] : -INFINITY;
          s[1] = (vA && pA <= lim1) ? s[1] : -INFINITY;
          s[2] = (vB && pB <= lim0) ? s[2] : -INFINITY;
          s[3] = (vB && pB <= lim1) ? s[3] : -INFINITY;
        }
        float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        // e4m3: the page's V scale enters the weights as a bias log2(v_scale)
        // on the exponent and the running max m tracks max(score + bias), so
        // the f16 weights P = 2^(s + bias - m) stay <= 1 and a small scale
        // cannot push them into f16's subnormal range; the row sum l takes
        // the bias back out (bf16 KV has no scale: bias 0)
        const float bias = FP8 ? __log2f(mt.vs[hw]) : 0.0f;
        const float unbias = FP8 ? fast_exp2(-bias) : 1.0f;
        const float n0 = fmaxf(m0, mx0 + bias), n1 = fmaxf(m1, mx1 + bias);
        // rows with nothing visible yet keep m = -inf and contribute nothing
        const float al0 = (n0 == -INFINITY) ? 1.0f : fast_exp2(m0 - n0);
        const float al1 = (n1 == -INFINITY) ? 1.0f : fast_exp2(m1 - n1);
        const float c0 = bias - n0, c1 = bias - n1;
        const float p0 = (n0 == -INFINITY) ? 0.0f : fast_exp2(s[0] + c0);
        const float p1 = (n1 == -INFINITY) ? 0.0f : fast_exp2(s[1] + c1);
        const float p2 = (n0 == -INFINITY) ? 0.0f : fast_exp2(s[2] + c0);
        const float p3 = (n1 == -INFINITY) ? 0.0f : fast_exp2(s[3] + c1);
        m0 = n0;
        m1 = n1;
        l0 = l0 * al0 + (p0 + p2) * unbias;
        l1 = l1 * al1 + (p1 + p3) * unbias;
        if (__any_sync(0xffffffffu, al0 != 1.0f || al1 != 1.0f)) {  // a running max moved
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            acc[i][0] *= al0;
            acc[i][2] *= al0;
            acc[i][1] *= al1;
            acc[i][3] *= al1;
          }
        }
        // ---------------- P^T to the B-fragment layout via shared memory;
        // tokens beyond the request length are zeroed in V (stale cache bytes
        // could be NaN patterns; 0 * NaN would poison the sum)
        if constexpr (FP8) {
          __half* pb = reinterpret_cast<__half*>(pbuf);  // [8 rows][16 tokens]
          pb[(2 * t) * 16 + g] = __float2half_rn(p0);
          pb[(2 * t + 1) * 16 + g] = __float2half_rn(p1);
          pb[(2 * t) * 16 + g + 8] = __float2half_rn(p2);
          pb[(2 * t + 1) * 16 + g + 8] = __float2half_rn(p3);
          __syncwarp();
          const uint2 bq = lds64(pbuf + g * 32 + 8 * t);  // row g, tokens 4t..4t+3
          __syncwarp();
          if (full_page) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint32_t a0, a1, a2, a3;
              e4m3x4_to_f16(lds32(Vt + (16 * i + g) * 16 + 4 * t), a0, a2);
              e4m3x4_to_f16(lds32(Vt + (16 * i + g + 8) * 16 + 4 * t), a1, a3);
              mma16816<true>(acc[i], a0, a1, a2, a3, bq.x, bq.y);
            }
          } else {
            const int keep = min(max(nv - 4 * t, 0), 4);  // bytes of tokens 4t.. kept
            const uint32_t vmask = keep >= 4 ? 0xFFFFFFFFu : ((1u << (8 * keep)) - 1u);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint32_t a0, a1, a2, a3;
              e4m3x4_to_f16(lds32(Vt + (16 * i + g) * 16 + 4 * t) & vmask, a0, a2);
              e4m3x4_to_f16(lds32(Vt + (16 * i + g + 8) * 16 + 4 * t) & vmask, a1, a3);
              mma16816<true>(acc[i], a0, a1, a2, a3, bq.x, bq.y);
            }
          }
        } else {
          float* pb = reinterpret_cast<float*>(pbuf);  // [8 rows][16 tokens] f32
          pb[(2 * t) * 16 + g] = p0;
          pb[(2 * t + 1) * 16 + g] = p1;
          pb[(2 * t) * 16 + g + 8] = p2;
          pb[(2 * t + 1) * 16 + g + 8] = p3;
          __syncwarp();
          const uint4 pq = lds128(pbuf + g * 64 + 16 * t);  // row g, tokens 4t..4t+3
          __syncwarp();
          const float f0 = __uint_as_float(pq.x), f1 = __uint_as_float(pq.y);
          const float f2 = __uint_as_float(pq.z), f3 = __uint_as_float(pq.w);
          // P = hi + lo in bf16 keeps ~16 bits of the weights
          const uint32_t h01 = f32x2_to_bf16x2(f0, f1), h23 = f32x2_to_bf16x2(f2, f3);
          const uint32_t l01 = f32x2_to_bf16x2(f0 - __uint_as_float(h01 << 16),
                                               f1 - __uint_as_float(h01 & 0xFFFF0000u));
          const uint32_t l23 = f32x2_to_bf16x2(f2 - __uint_as_float(h23 << 16),
                                               f3 - __uint_as_float(h23 & 0xFFFF0000u));
          uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;  // tokens (4t,4t+1) and (4t+2,4t+3)
          if (!full_page) {
            const int keep = min(max(nv - 4 * t, 0), 4);
            mlo = keep >= 2 ? 0xFFFFFFFFu : (keep == 1 ? 0x0000FFFFu : 0u);
            mhi = keep >= 4 ? 0xFFFFFFFFu : (keep == 3 ? 0x0000FFFFu : 0u);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint2 vl = lds64(Vt + (16 * i + g) * 32 + 8 * t);
            const uint2 vh = lds64(Vt + (16 * i + g + 8) * 32 + 8 * t);
            const uint32_t a0 = vl.x & mlo, a2 = vl.y & mhi, a1 = vh.x & mlo, a3 = vh.y & mhi;
            mma16816<false>(acc[i], a0, a1, a2, a3, h01, h23);
            mma16816<false>(acc[i], a0, a1, a2, a3, l01, l23);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      stage += WPH;
      if (stage >= S) {
        stage -= S;
        phase ^= 1u;
      }
    }

    // ---- merge the states of the warps that share a head into one partial
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    float* mo = merge_o + warp * C::R8 * D;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      mo[(2 * t) * D + 16 * i + g] = acc[i][0];
      mo[(2 * t + 1) * D + 16 * i + g] = acc[i][1];
      mo[(2 * t) * D + 16 * i + g + 8] = acc[i][2];
      mo[(2 * t + 1) * D + 16 * i + g + 8] = acc[i][3];
    }
    if (bad_units < 0 && lane == 0) *piece_bad = 1;  // read after the merge's first barrier
    if (g == 0) {
      float* ml = merge_ml + warp * C::R8 * 2;
      ml[(2 * t) * 2 + 0] = m0;
      ml[(2 * t) * 2 + 1] = l0;
      ml[(2 * t + 1) * 2 + 0] = m1;
      ml[(2 * t + 1) * 2 + 1] = l1;
    }
    {
      // slot of this (CTA, segment) piece; row nw of virtual head v (kv head
      // hh's row block j) is row 8 j + nw of the kv head.  v < Hv <= 12,
      // where (v * ceil(256 / RB)) >> 8 is exactly v / RB for RB <= 4.
      const long long slot = (long long)r * HG + cur.h + blockIdx.x;
      merge_piece<C>(merge_o, merge_ml, Hv, WPH, a,
                     [&](int v, int nw) -> long long {
                       const int hh = (v * rb_mul) >> 8, n = (v - hh * RB) * C::R8 + nw;
                       return (slot * Hs + hh) * a.R8 + n;
                     },
                     piece_bad, true);
    }

    k_base += npages;
    x = piece_end;
    if (x == seg_end) cursor_next(cur, pfx, B, HG);
  }
}

template <bool FP8>
__global__ void __launch_bounds__(GqaCfg<FP8>::THREADS, 1)
    gqa_split_kernel(const DecodeArgs a) {
  gqa_split_body<FP8, false>(a);
}

__global__ void __launch_bounds__(GqaCfg<true>::THREADS, 1)
    gqa_split_wide_kernel(const DecodeArgs a) {
  gqa_split_body<true, true>(a);
}

__global__ void __launch_bounds__(GqaCfg<false>::THREADS, 1)
    gqa_split_wide_bf16_kernel(const DecodeArgs a) {
  gqa_split_body<false, true>(a);
}

// ------------------------------------------------- combine

constexpr int kCombineWarps = 8;

// One warp per (segment, query row): merges the pieces of the segment,
// O = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c, with a running max so a
// single pass over the pieces suffices; lane l owns dims [4l, 4l+4) of every
// 128-dim group.  Written as bf16 (RNE).
// S warps per output row (S = 1, 2, 4 or 8): warp k of a row merges the row's
// partials k, k + S, ..., then the S running states are merged through
// shared memory.  S > 1 when a segment has many partials (few long requests),
// so the merge of one row is no long serial chain.
// NG: 128-dim groups of a row (Dv / 128: 1 or 4).
template <int NG>
__global__ void __launch_bounds__(kCombineWarps * 32, 2)
    combine_kernel(const DecodeArgs a, int S) {
  __shared__ float st_o[kCombineWarps][512];
  __shared__ float st_ml[kCombineWarps][2];
  __shared__ int st_bad[kCombineWarps];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = warp % S;
  const long long item = (long long)blockIdx.x * (kCombineWarps / S) + warp / S;
  const int Hkv = a.d.num_kv_heads;
  const long long nitems = (long long)a.B * Hkv * a.R;
  const int Dv = 128 * NG;
  constexpr int ngroups = NG;
  float acc[4][4];
  float M = -INFINITY, L = 0.0f;
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.0f;
  // every warp reaches the block barrier below, so no early return
  bool skip = item >= nitems;
  int r = 0, h = 0, n = 0;
  int pfx_r = 0, pfx_r1 = 0, pfx_B = 0;
  if (!skip) {
    n = (int)(item % a.R);
    const long long rh = item / a.R;
    r = (int)(rh / Hkv);
    h = (int)(rh % Hkv);
    // the plan's prefix and the skip flag are independent loads
    pfx_r = a.ws.pfx[r];
    pfx_r1 = a.ws.pfx[r + 1];
    pfx_B = a.ws.pfx[a.B];
    skip = a.ws.rq_skip[r];  // aborted or invalid length: output left untouched
  }
  // a piece whose sum is -1 met a page it must not read: no output either
  bool bad = false;
  if (!skip) {
    const int Hs = a.Hs, HG = a.HG;
    // segment (request, head group | row block) and row inside its partials
    const bool latent = a.d.layout == KV_LAYOUT_LATENT;
    const int hg = latent ? n / a.R8 : h / Hs, hw = latent ? 0 : h % Hs;
    const int nl = latent ? n % a.R8 : n;
    const long long seg = (long long)r * HG + hg;
    const int np = pfx_r1 - pfx_r;
    if (np > 0) {
      const long long total = (long long)pfx_B * HG;
      const long long per = (total + a.grid - 1) / a.grid;
      const long long start = (long long)HG * pfx_r + (long long)hg * np;
      const int c0 = (int)(start / per), c1 = (int)((start + np - 1) / per);
      const long long slot0 = seg + c0;
      const int R8 = a.R8;
      // partial row of this warp's piece jj (pieces c = sub + S jj)
      auto row_of = [&](int jj) -> long long {
        return ((slot0 + sub + (long long)S * jj) * Hs + hw) * R8 + nl;
      };
      auto load_o = [&](long long row, int q) -> float4 {
        return *reinterpret_cast<const float4*>(a.ws.o_part + row * Dv + 128 * q + 4 * lane);
      };
      constexpr int kU = 8 / NG;  // pieces whose output loads are in flight together
      auto accumulate = [&](const float4 (&o)[kU][NG], const float (&wk)[kU]) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          // a piece that saw nothing has weight 0 and adds nothing
          const bool use = wk[u] != 0.0f;
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            acc[q][0] = use ? __fmaf_rn(o[u][q].x, wk[u], acc[q][0]) : acc[q][0];
            acc[q][1] = use ? __fmaf_rn(o[u][q].y, wk[u], acc[q][1]) : acc[q][1];
            acc[q][2] = use ? __fmaf_rn(o[u][q].z, wk[u], acc[q][2]) : acc[q][2];
            acc[q][3] = use ? __fmaf_rn(o[u][q].w, wk[u], acc[q][3]) : acc[q][3];
          }
        }
      };
      // this warp's pieces, merged 32 at a time: each lane reads one piece's
      // (max, sum) while the outputs of the chunk's first kU pieces are
      // already loading; the chunk's max and weights come from warp
      // reductions, then the weighted outputs are summed with independent
      // loads (no chain through a running max)
      const int cnt = (c1 - c0 + 1 - sub + S - 1) / S;
      for (int j0 = 0; j0 < cnt; j0 += 32) {
        const int nj = min(32, cnt - j0);
        float4 o[kU][NG];
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int q = 0; q < NG; ++q)
            o[u][q] = u < nj ? load_o(row_of(j0 + u), q) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        const int j = j0 + lane;
        float mj = -INFINITY, lj = 0.0f;
        if (j < cnt) {
          const float2 ml = *reinterpret_cast<const float2*>(a.ws.ml_part + row_of(j) * 2);
          mj = ml.x;
          lj = ml.y;
        }
        bad = bad || __any_sync(0xffffffffu, lj < 0.0f);
        const float Mc = warp_max(mj);
        if (Mc == -INFINITY) continue;  // no piece of the chunk saw anything visible
        const float Mn = fmaxf(M, Mc);
        const float sa = exp2f(M - Mn);  // 0 while nothing is accumulated (M = -inf)
        const float wj = (mj == -INFINITY) ? 0.0f : exp2f(mj - Mn);
        L = L * sa + warp_sum(lj * wj);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          acc[q][0] *= sa, acc[q][1] *= sa, acc[q][2] *= sa, acc[q][3] *= sa;
        float wk[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const float wu = __shfl_sync(0xffffffffu, wj, u);
          wk[u] = u < nj ? wu : 0.0f;
        }
        accumulate(o, wk);
        for (int k0 = kU; k0 < nj; k0 += kU) {
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const bool ok = k0 + u < nj;  // uniform across the warp
            const float wu = __shfl_sync(0xffffffffu, wj, ok ? k0 + u : 0);
            wk[u] = ok ? wu : 0.0f;
#pragma unroll
            for (int q = 0; q < NG; ++q)
              o[u][q] = ok ? load_o(row_of(j0 + k0 + u), q) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          }
          accumulate(o, wk);
        }
        M = Mn;
      }
    }
  }
  if (S > 1) {
    if (lane == 0) {
      st_ml[warp][0] = M;
      st_ml[warp][1] = L;
      st_bad[warp] = bad ? 1 : 0;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q < ngroups)
        *reinterpret_cast<float4*>(&st_o[warp][128 * q + 4 * lane]) =
            make_float4(acc[q][0], acc[q][1], acc[q][2], acc[q][3]);
    __syncthreads();
    if (sub == 0 && !skip) {
      for (int k = 1; k < S; ++k) bad = bad || st_bad[warp + k] != 0;
      for (int k = 1; k < S; ++k) {
        const float Mk = st_ml[warp + k][0], Lk = st_ml[warp + k][1];
        if (Mk == -INFINITY) continue;
        const float Mn = fmaxf(M, Mk);
        const float sa = exp2f(M - Mn), sb = exp2f(Mk - Mn);
        L = L * sa + Lk * sb;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q < ngroups) {
            const float4 ok = *reinterpret_cast<const float4*>(&st_o[warp + k][128 * q + 4 * lane]);
            acc[q][0] = acc[q][0] * sa + ok.x * sb;
            acc[q][1] = acc[q][1] * sa + ok.y * sb;
            acc[q][2] = acc[q][2] * sa + ok.z * sb;
            acc[q][3] = acc[q][3] * sa + ok.w * sb;
          }
        }
        M = Mn;
      }
    }
  }
  // fused tag check: the warp of the request's first row writes its abort
  // bit (every segment and row of a request meets the same pages)
  if (a.abort_out != nullptr && sub == 0 && item < nitems && h == 0 && n == 0)
    a.abort_out[r] = (skip || bad) ? 1 : 0;
  if (sub != 0 || skip || bad) return;
  const int tq = n / a.G, hq = h * a.G + n % a.G;
  uint16_t* out = a.out + (((long long)r * a.T + tq) * a.Hq + hq) * Dv;
  const float inv = (M == -INFINITY) ? 0.0f : 1.0f / L;  // nothing visible: zeros
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (q < ngroups) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[q][0] * inv, acc[q][1] * inv);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[q][2] * inv, acc[q][3] * inv);
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t*>(&lo);
      w.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(out + 128 * q + 4 * lane) = w;
    }
  }
}


}  // namespace

// ------------------------------------------------- host side

// kinds: 0 = e4m3 (8-row consumers), 1 = bf16, 3 = e4m3 with 16-row consumers,
// 4 = bf16 with 16-row consumers
int gqa_ring_bytes(int kind) {
  return (kind == 1 || kind == 4) ? GqaCfg<false>::RING : GqaCfg<true>::RING;
}
int gqa_max_stages() { return kMaxStages; }
bool gqa_kind_self_plans(int kind) { return kind == 0 || kind == 1 || kind == 4; }
int gqa_self_plan_max_batch() {
  static_assert(GqaCfg<true>::PFX_CACHE == GqaCfg<false>::PFX_CACHE, "one prefix cache size");
  return GqaCfg<true>::PFX_CACHE - 1;
}
int gqa_consumer_warps(int kind) {
  return (kind == 1 || kind == 4) ? GqaCfg<false>::CONSUMERS : GqaCfg<true>::CONSUMERS;
}

int gqa_split_ctas_per_sm(int kind) {
  static int cache[5] = {-1, -1, -1, -1, -1};
  if (kind < 0 || kind > 4 || kind == 2) return 0;
  if (cache[kind] >= 0) return cache[kind];
  int n = 0;
  cudaError_t e;
  if (kind == 4) {
    cudaFuncSetAttribute(gqa_split_wide_bf16_kernel,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, GqaCfg<false>::SMEM);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_split_wide_bf16_kernel,
                                                      GqaCfg<false>::THREADS, GqaCfg<false>::SMEM);
  } else if (kind == 3) {
    cudaFuncSetAttribute(gqa_split_wide_kernel,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, GqaCfg<true>::SMEM);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_split_wide_kernel,
                                                      GqaCfg<true>::THREADS, GqaCfg<true>::SMEM);
  } else if (kind == 0) {
    cudaFuncSetAttribute(gqa_split_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         GqaCfg<true>::SMEM);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_split_kernel<true>,
                                                      GqaCfg<true>::THREADS, GqaCfg<true>::SMEM);
  } else {
    cudaFuncSetAttribute(gqa_split_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         GqaCfg<false>::SMEM);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_split_kernel<false>,
                                                      GqaCfg<false>::THREADS, GqaCfg<false>::SMEM);
  }
  if (e != cudaSuccess || n <= 0) return 0;
  cache[kind] = n;
  return n;
}

cudaError_t launch_decode_plan(const DecodeArgs& a, cudaStream_t s, int* launches) {
  const cudaError_t e = launch_pdl(decode_plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, a);
  if (e == cudaSuccess) ++*launches;
  return e;
}

cudaError_t launch_gqa_split(const DecodeArgs& a, int kind, cudaStream_t s, int* launches) {
  const cudaError_t e =
      kind == 4   ? launch_pdl(gqa_split_wide_bf16_kernel, dim3(a.grid),
                               dim3(GqaCfg<false>::THREADS), GqaCfg<false>::SMEM, s, a)
      : kind == 3 ? launch_pdl(gqa_split_wide_kernel, dim3(a.grid),
                               dim3(GqaCfg<true>::THREADS), GqaCfg<true>::SMEM, s, a)
      : kind == 0 ? launch_pdl(gqa_split_kernel<true>, dim3(a.grid),
                               dim3(GqaCfg<true>::THREADS), GqaCfg<true>::SMEM, s, a)
                  : launch_pdl(gqa_split_kernel<false>, dim3(a.grid),
                               dim3(GqaCfg<false>::THREADS), GqaCfg<false>::SMEM, s, a);
  if (e == cudaSuccess) ++*launches;
  return e;
}

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t s, int* launches) {
  const long long items = (long long)a.B * a.d.num_kv_heads * a.R;
  if (items <= 0) return cudaSuccess;
  // partials of one segment: about 1 + grid / segments; give each merging
  // warp at least two of them
  const double pieces = 1.0 + (double)a.grid / ((double)a.B * a.HG);
  int S = 1;
  while (S < kCombineWarps && 4.0 * S <= pieces) S *= 2;
  const long long per_cta = kCombineWarps / S;
  const long long blocks = (items + per_cta - 1) / per_cta;
  const cudaError_t e =
      a.d.head_dim_v == 128
          ? launch_pdl(combine_kernel<1>, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s,
                       a, S)
          : launch_pdl(combine_kernel<4>, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s,
                       a, S);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace kvfp8
