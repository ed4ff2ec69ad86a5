// decode_latent.cu -- split-K decode attention over a latent (MLA-style) e4m3
// cache on the tcgen05 tensor cores: the speculative-verify shape, where many
// query rows (T draft tokens x Hq heads) share one 576-wide cache row per
// token and QK^T / PV are real dense contractions.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": the attention reads the e4m3 cache and converts
// values as it reads them.  Speculative decoding (Cloudflare's post on
// serving extra-large LLMs, section on speculative decoding) scores several
// draft tokens in one forward pass: query token i sees positions
// 0 .. L - T + i.
//
// Work decomposition: a segment is (request, block of 64 query rows); a unit
// is 32 tokens (half a 64-token page).  Units are laid out segment-major and
// cut into equal ranges, one per CTA (one CTA per SM); each (CTA, segment)
// piece leaves a partial (o, running max, sum) for the combine kernel.
//
// Per unit:
//   converter warps load the unit's 32 x 576 e4m3 bytes (the next unit's
//                   loads in flight while this one converts) and convert them
//                   exactly to f16 into one of three 128B-swizzled K-major
//                   tiles (the same tile is the MN-major V^T operand);
//   MMA warp        S = Q K^T   (tcgen05, M = 64 rows, N = 32 tokens, K = 576,
//                   f16 x f16 -> f32 into one of four tensor-memory buffers),
//                   and two units later O^T += V^T P^T (M = 128 dims x 4
//                   blocks, N = 64 rows, K = 32 tokens) accumulating in tensor
//                   memory, so the tensor pipe never waits for the softmax;
//   softmax warps   read S from tensor memory (one row per thread), apply the
//                   page scale, the causal mask and the online softmax with a
//                   lazily updated reference max (the output is rescaled only
//                   when a row's max grows by more than 2^8), and write P (f16,
//                   V scale folded in) as the swizzled B operand.
// Every wait is bounded; on timeout the kernel records KV_ERR_TIMEOUT, lets
// the asynchronous work it issued finish (bounded) and frees its tensor
// memory before returning.
#include "common.cuh"
#include "internal.h"

namespace kvfp8 {
namespace {

constexpr int kUT = 32;        // tokens per unit
constexpr int kPage = 64;      // tokens per page
constexpr int kDK = 576, kDV = 512, kNKB = kDK / 64;  // K blocks of 64 dims
constexpr int kRB = 64;        // query rows per segment
constexpr int kNKV = 3;        // f16 KV tiles (converted units)
constexpr int kNS = 4;         // S buffers in tensor memory
constexpr int kLag = 2;        // PV(u) is issued right after S(u + kLag)
constexpr int kUnitBytes = kUT * kDK;  // 18432

// warps: 0-3 softmax (tensor-memory lane quarters 0-3), 4-7 converters
// (global e4m3 -> swizzled f16 tiles), 8 MMA issuer
constexpr int kThreads = 288;
constexpr int kSoftmaxWarps = 4, kConvWarps = 4;
constexpr int kMmaWarp = 8;

// shared memory (bytes); tiles 1024-byte aligned for the 128B swizzle
constexpr int OFF_Q = 0;                                   // 9 x [64 rows][128 B]
constexpr int OFF_KV = OFF_Q + kNKB * kRB * 128;           // 3 x 9 x [32 tokens][128 B]
constexpr int KV_BYTES = kNKB * kUT * 128;                 // 36864
constexpr int OFF_P = OFF_KV + kNKV * KV_BYTES;            // 2 x [64 rows][128 B]
constexpr int P_BYTES = kRB * 128;
constexpr int OFF_ALPHA = OFF_P + 2 * P_BYTES;             // 2 x 64 floats
constexpr int OFF_FLAG = OFF_ALPHA + 2 * kRB * 4;          // 2 ints (+pad)
constexpr int OFF_META = OFF_FLAG + 16;                    // unit meta [3]
constexpr int OFF_BAR = OFF_META + kNKV * 16;
constexpr int NBAR = 2 * kNKV + 2 * kNS + 2 + 2 + 4;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM = OFF_MISC + 64;
static_assert(OFF_KV % 1024 == 0 && OFF_P % 1024 == 0 && OFF_BAR % 8 == 0, "alignment");
static_assert(SMEM <= 227 * 1024, "shared memory budget");

// tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;     // O^T: 4 blocks x 64 columns
constexpr uint32_t kTmemS = 256;   // S: 4 buffers x 32 columns

struct UnitMeta {
  int n_valid;  // valid tokens of the unit (0: skip)
  int pos0;     // position of its first token
  float scale;  // page scale (K and V share the row)
  int unit;     // unit sequence number (checked by consumers)
};

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: f32 accumulate, f16 operands
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc_f16(64, kUT, 0, 0);   // S = Q K^T
constexpr uint32_t kIdescPV = idesc_f16(128, kRB, 1, 0); // O^T += V^T P^T

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive columns of this warp's 32 lanes
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// byte offset of 16-byte chunk c (0..7) of row r inside a 128B-swizzled block
__device__ __forceinline__ uint32_t swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// segment cursor over (request, row block), `groups` row blocks per request
struct Seg {
  int r, rb, np;
  long long start;
};
__device__ Seg seg_at(const int32_t* pfx, int B, int groups, long long x) {
  const long long v = x / groups;
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pfx[mid] <= v) lo = mid; else hi = mid;
  }
  Seg s;
  s.r = lo;
  s.np = pfx[lo + 1] - pfx[lo];
  s.rb = (int)((x - (long long)groups * pfx[lo]) / s.np);
  s.start = (long long)groups * pfx[lo] + (long long)s.rb * s.np;
  return s;
}
__device__ void seg_next(Seg& s, const int32_t* pfx, int B, int groups) {
  if (++s.rb == groups) {
    s.rb = 0;
    do { ++s.r; } while (s.r < B && pfx[s.r + 1] == pfx[s.r]);
    if (s.r < B) s.np = pfx[s.r + 1] - pfx[s.r];
  }
  if (s.r < B) {
    s.start = (long long)groups * pfx[s.r] + (long long)s.rb * s.np;
  } else {  // past the last request (cannot happen inside a CTA range): end every loop
    s.start = (long long)groups * pfx[B];
    s.np = 1;
  }
}

__global__ void __launch_bounds__(kThreads, 1) latent_split_kernel(const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* q_s = smem + OFF_Q;
  uint8_t* kv_s = smem + OFF_KV;
  uint8_t* p_s = smem + OFF_P;
  float* alpha_s = reinterpret_cast<float*>(smem + OFF_ALPHA);    // [2][64]
  volatile int* flag_s = reinterpret_cast<volatile int*>(smem + OFF_FLAG);  // [2]
  UnitMeta* kv_meta = reinterpret_cast<UnitMeta*>(smem + OFF_META);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* kv_ready = bars;                    // [3] converters
  uint64_t* kv_free = kv_ready + kNKV;          // [3] MMA commit after PV
  uint64_t* s_full = kv_free + kNKV;            // [4] MMA commit after S
  uint64_t* s_free = s_full + kNS;              // [4] softmax
  uint64_t* p_ready = s_free + kNS;             // [2] softmax
  uint64_t* p_free = p_ready + 2;               // [2] MMA commit after PV
  uint64_t* q_ready = p_free + 2;               // converters
  uint64_t* q_free = q_ready + 1;               // MMA commit after a piece's last S
  uint64_t* epi_done = q_free + 1;              // softmax
  uint64_t* drain = epi_done + 1;               // MMA commit at exit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.B, NRB = a.HG;  // row blocks per request
  const int32_t* pfx = a.ws.pfx;
  const long long total = (long long)pfx[B] * NRB;
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  const long long x_begin = (long long)blockIdx.x * per;
  const long long x_end = min(total, x_begin + per);
  if (x_begin >= x_end) return;

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < kNKV; ++i) {
      mbar_init(&kv_ready[i], kConvWarps);
      mbar_init(&kv_free[i], 1);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], kSoftmaxWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_ready[i], kSoftmaxWarps);
      mbar_init(&p_free[i], 1);
      flag_s[i] = -1;
    }
    mbar_init(q_ready, kConvWarps);
    mbar_init(q_free, 1);
    mbar_init(epi_done, kSoftmaxWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int32_t* ctl = a.d.ctl;
  const Seg start = seg_at(pfx, B, NRB, x_begin);
  const uint8_t* cache = static_cast<const uint8_t*>(a.d.k_cache);

  if (warp >= kSoftmaxWarps && warp < kSoftmaxWarps + kConvWarps) {
    // ============================ converters ============================
    // thread ct handles 16-byte pieces g = ct + 128 i (i < 9) of a unit's
    // 32 x 576 e4m3 bytes: token g / 36, dims 16 (g % 36) .. +15
    const int ct = threadIdx.x - kSoftmaxWarps * 32;
    const int maxp = a.max_pages;
    struct Pre {
      uint4 d[9];
      UnitMeta m;
    };
    auto fetch = [&](const Seg& sg, long long xu, long long uu, Pre& pr) {
      const int j = (int)(xu - sg.start);
      const int p = a.page_table[(long long)sg.r * maxp + (j >> 1)];
      const bool ok = p >= 0 && p < a.d.num_pages;
      const int L = a.seq_lens[sg.r];
      pr.m.n_valid = ok ? min(kUT, L - j * kUT) : 0;
      pr.m.pos0 = j * kUT;
      pr.m.scale = ok ? a.d.k_scale[p] : 1.0f;
      pr.m.unit = (int)uu;
      if (!ok && ct == 0) {
        a.ws.rq_bad[sg.r] = 1;
        set_error(ctl, KV_ERR_BAD_PAGE_ID);
      }
      const uint8_t* src = cache + (long long)(ok ? p : 0) * kPage * kDK + (long long)(j & 1) * kUnitBytes;
#pragma unroll
      for (int i = 0; i < 9; ++i) {
        const int g = ct + 128 * i, t = g / 36;
        pr.d[i] = (ok && t < pr.m.n_valid)
                      ? __ldg(reinterpret_cast<const uint4*>(src + t * kDK + (g % 36) * 16))
                      : make_uint4(0, 0, 0, 0);
      }
    };
    Seg s = start;
    long long x = x_begin, u = 0;
    int piece = 0;
    bool go = true;
    while (x < x_end && go) {
      const long long seg_end = s.start + s.np, piece_end = min(seg_end, x_end);
      // ---- Q block of this segment: rows rb*64 .. +63 of the request's T*Hq rows
      if (piece > 0 &&
          !mbar_wait(q_free, (uint32_t)((piece - 1) & 1), abort_flag, ctl, wait_info(warp, 1, 60))) {
        go = false;
        break;
      }
      {
        const uint16_t* qbase = a.q + ((long long)s.r * a.T * a.Hq + (long long)s.rb * kRB) * kDK;
        for (int c = ct; c < kRB * (kDK / 8); c += kConvWarps * 32) {
          const int n = c / (kDK / 8), ck = c % (kDK / 8);
          const uint4 v = *reinterpret_cast<const uint4*>(qbase + (long long)n * kDK + ck * 8);
          uint4 o;
          o.x = bf16x2_to_f16x2(v.x);
          o.y = bf16x2_to_f16x2(v.y);
          o.z = bf16x2_to_f16x2(v.z);
          o.w = bf16x2_to_f16x2(v.w);
          *reinterpret_cast<uint4*>(q_s + (ck >> 3) * (kRB * 128) + swz(n, ck & 7)) = o;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready);
      }
      // ---- units, the next one's loads in flight while this one converts
      Pre cur, nxt;
      fetch(s, x, u, cur);
      for (long long xu = x; xu < piece_end; ++xu, ++u) {
        if (xu + 1 < piece_end) fetch(s, xu + 1, u + 1, nxt);
        const int kb = (int)(u % kNKV);
        if (u >= kNKV && !mbar_wait(&kv_free[kb], (uint32_t)(((u / kNKV) - 1) & 1), abort_flag,
                                    ctl, wait_info(warp, 1, 32 + kb))) {
          go = false;
          break;
        }
        uint8_t* dst = kv_s + kb * KV_BYTES;
#pragma unroll
        for (int i = 0; i < 9; ++i) {
          const int g = ct + 128 * i, t = g / 36, c16 = g % 36;
          uint4 lo, hi;
          e4m3x4_to_f16(cur.d[i].x, lo.x, lo.y);
          e4m3x4_to_f16(cur.d[i].y, lo.z, lo.w);
          e4m3x4_to_f16(cur.d[i].z, hi.x, hi.y);
          e4m3x4_to_f16(cur.d[i].w, hi.z, hi.w);
          uint8_t* blk = dst + (c16 >> 2) * (kUT * 128);
          *reinterpret_cast<uint4*>(blk + swz(t, (c16 & 3) * 2)) = lo;
          *reinterpret_cast<uint4*>(blk + swz(t, (c16 & 3) * 2 + 1)) = hi;
        }
        if (ct == 0) kv_meta[kb] = cur.m;
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_ready[kb]);
        cur = nxt;
      }
      ++piece;
      x = piece_end;
      if (x == seg_end) seg_next(s, pfx, B, NRB);
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ============================
    Seg s = start;
    long long x = x_begin, u = 0;
    int piece = 0;
    bool go = true;
    const uint32_t q_base = smem_u32(q_s), kv_base = smem_u32(kv_s), p_base = smem_u32(p_s);
    while (x < x_end && go) {
      const long long seg_end = s.start + s.np, piece_end = min(seg_end, x_end);
      const long long u0 = u, n = piece_end - x;
      if (!mbar_wait(q_ready, (uint32_t)(piece & 1), abort_flag, ctl, wait_info(warp, 0, 62))) {
        go = false;
        break;
      }
      for (long long i = 0; i < n + kLag && go; ++i) {
        if (i < n) {  // ---- S(u0 + i) = Q K^T into S buffer (u0+i) % 4
          const long long uu = u0 + i;
          const int kb = (int)(uu % kNKV), sb = (int)(uu % kNS);
          go = mbar_wait(&kv_ready[kb], (uint32_t)((uu / kNKV) & 1), abort_flag, ctl,
                         wait_info(warp, 0, 40 + kb));
          go = go && (uu < kNS || mbar_wait(&s_free[sb], (uint32_t)(((uu / kNS) - 1) & 1),
                                            abort_flag, ctl, wait_info(warp, 1, 44 + sb)));
          go = __all_sync(0xffffffffu, go);
          if (!go) break;
          tc_fence_after();
          if (lane == 0) {
            for (int st = 0; st < kDK / 16; ++st) {
              const uint64_t ad =
                  sw128_desc(q_base + (st >> 2) * (kRB * 128) + (st & 3) * 32, 16, 1024);
              const uint64_t bd = sw128_desc(
                  kv_base + kb * KV_BYTES + (st >> 2) * (kUT * 128) + (st & 3) * 32, 16, 1024);
              mma_f16(tmem + kTmemS + 32 * sb, ad, bd, kIdescS, st > 0);
            }
            mma_commit(&s_full[sb]);
            if (i == n - 1) mma_commit(q_free);  // every S of this piece is issued
          }
          __syncwarp();
        }
        if (i >= kLag) {  // ---- PV(u0 + i - kLag): O^T += V^T P^T
          const long long v = u0 + i - kLag;
          const int kb = (int)(v % kNKV), pb = (int)(v & 1);
          // the first PV of a piece overwrites O: the previous piece's
          // epilogue must have read it (its S products already ran ahead)
          if (v == u0 && piece > 0) {
            go = __all_sync(0xffffffffu, mbar_wait(epi_done, (uint32_t)((piece - 1) & 1),
                                                   abort_flag, ctl, wait_info(warp, 1, 61)));
            if (!go) break;
          }
          go = __all_sync(0xffffffffu, mbar_wait(&p_ready[pb], (uint32_t)((v >> 1) & 1),
                                                 abort_flag, ctl, wait_info(warp, 0, 48 + pb)));
          if (!go) break;
          tc_fence_after();
          if (lane == 0) {
            for (int db = 0; db < kDV / 128; ++db) {
              for (int st = 0; st < kUT / 16; ++st) {
                // V^T: dims 128db.. (two 64-dim blocks, LBO apart), tokens 16st..
                const uint64_t ad = sw128_desc(kv_base + kb * KV_BYTES +
                                                   (2 * db) * (kUT * 128) + st * 2048,
                                               kUT * 128, 1024);
                const uint64_t bd = sw128_desc(p_base + pb * P_BYTES + st * 32, 16, 1024);
                mma_f16(tmem + kTmemO + 64 * db, ad, bd, kIdescPV, !(v == u0 && st == 0));
              }
            }
            mma_commit(&kv_free[kb]);
            mma_commit(&p_free[pb]);
          }
          __syncwarp();
        }
      }
      u = u0 + n;
      ++piece;
      x = piece_end;
      if (x == seg_end) seg_next(s, pfx, B, NRB);
    }
    // let every tensor-core operation issued here finish (bounded) before
    // tensor memory is freed: a commit tracks all earlier ones
    if (lane == 0) {
      mma_commit(drain);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(drain, 0) && global_ns() - t0 < 100000000ull) {
      }
    }
    __syncwarp();
  } else if (warp < kSoftmaxWarps) {
    // ============================ softmax (warps 0-3) ============================
    const int q4 = warp;                 // tensor-memory lane quarter
    const bool owner = lane < 16;        // S rows live in lanes 0-15 of each quarter
    const int n = 16 * q4 + lane;        // query row within the block (owners)
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float ssl = a.sm_scale_log2;
    Seg s = start;
    long long x = x_begin, u = 0;
    bool go = true;
    while (x < x_end) {
      const long long seg_end = s.start + s.np, piece_end = min(seg_end, x_end);
      const int L = a.seq_lens[s.r];
      // row rb*64 + n of the request's (t, hq) rows: draft token t = row / Hq
      const int tq = (s.rb * kRB + n) / a.Hq;
      const int lim = L - a.T + min(tq, a.T - 1);  // last visible position (inclusive)
      float m_ref = -INFINITY, l = 0.0f;
      const long long u0 = u;
      // every softmax warp runs every unit (and every named barrier), even
      // after a wait gave up, so the barrier sequence never diverges
      for (long long xu = x; xu < piece_end; ++xu, ++u) {
        const int sb = (int)(u % kNS), kb = (int)(u % kNKV), pb = (int)(u & 1);
        go = go && mbar_wait(&s_full[sb], (uint32_t)((u / kNS) & 1), abort_flag, ctl,
                             wait_info(warp, 0, 52 + sb));
        go = go && mbar_wait(&kv_ready[kb], (uint32_t)((u / kNKV) & 1), abort_flag, ctl,
                             wait_info(warp, 0, 40 + kb));
        go = __all_sync(0xffffffffu, go);  // tensor-memory loads are warp-collective
        float v[32];
        if (go) {
          tc_fence_after();
          tmem_ld32(tmem + kTmemS + 32 * sb + lane_off, v);
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[sb]);
        const UnitMeta m = kv_meta[kb];
        if (go && m.unit != (int)u) {
          if (lane == 0) set_error(ctl, KV_ERR_INTERNAL);
          *abort_flag = 1;
          go = false;
        }
        // P buffer pb is free once PV(u-2) has completed
        go = go && (u < 2 || mbar_wait(&p_free[pb], (uint32_t)(((u >> 1) - 1) & 1), abort_flag,
                                       ctl, wait_info(warp, 1, 56 + pb)));
        go = __all_sync(0xffffffffu, go);
        float alpha = 1.0f;
        if (owner && go) {
          const float sc = m.scale * ssl;
          float mx = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const bool vis = i < m.n_valid && m.pos0 + i <= lim;
            v[i] = vis ? v[i] * sc : -INFINITY;
            mx = fmaxf(mx, v[i]);
          }
          // lazy reference max: only move it (and rescale O) when the tile's
          // max exceeds it by more than 2^8
          if (mx > m_ref + 8.0f) {
            alpha = (m_ref == -INFINITY) ? 0.0f : ex2(m_ref - mx);
            l *= alpha;
            m_ref = mx;
          }
          float sum = 0.0f;
          const float vs = m.scale;
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float p0 = (v[i] == -INFINITY) ? 0.0f : ex2(v[i] - m_ref);
            const float p1 = (v[i + 1] == -INFINITY) ? 0.0f : ex2(v[i + 1] - m_ref);
            sum += p0 + p1;
            pk[i >> 1] = pack_f16(p0 * vs, p1 * vs);
          }
          l += sum;
          // P row n: tokens 0..31 = chunks 0..3 of a 128B-swizzled row
          uint8_t* prow = p_s + pb * P_BYTES;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(prow + swz(n, c)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          if (alpha != 1.0f) flag_s[pb] = (int)u;  // unit number: never stale
        }
        if (owner) alpha_s[pb * kRB + n] = alpha;
        fence_async_smem();
        named_bar_sync(2, kSoftmaxWarps * 32);
        if (flag_s[pb] == (int)u && u > u0) {
          // O^T columns are query rows: column n *= alpha[n], after PV(u-1)
          const long long pu = u - 1;
          go = go && mbar_wait(&p_free[pu & 1], (uint32_t)((pu >> 1) & 1), abort_flag, ctl,
                               wait_info(warp, 1, 58));
          go = __all_sync(0xffffffffu, go);
          if (go) {
            tc_fence_after();
            for (int db = 0; db < kDV / 128; ++db) {
              for (int half = 0; half < 2; ++half) {
                float o[32];
                const uint32_t ta = tmem + kTmemO + 64 * db + 32 * half + lane_off;
                tmem_ld32(ta, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] *= alpha_s[pb * kRB + 32 * half + i];
                tmem_st32(ta, o);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_ready[pb]);
      }
      // ---- epilogue: partial (o, m, l) of this piece
      if (u > u0) {
        const long long last = u - 1;
        go = go && mbar_wait(&p_free[last & 1], (uint32_t)((last >> 1) & 1), abort_flag, ctl,
                             wait_info(warp, 0, 59));
      }
      go = __all_sync(0xffffffffu, go);
      tc_fence_after();
      const long long slot = (long long)s.r * NRB + s.rb + blockIdx.x;
      // (after a failed wait the loop still runs, so every softmax warp keeps
      // the same named-barrier sequence; the partial is then not written)
      for (int db = 0; db < kDV / 128 && go; ++db) {
        for (int half = 0; half < 2; ++half) {
          float o[32];
          tmem_ld32(tmem + kTmemO + 64 * db + 32 * half + lane_off, o);
          const int dv = 128 * db + 32 * q4 + lane;
          for (int i = 0; i < 32; ++i)
            a.ws.o_part[(slot * kRB + 32 * half + i) * kDV + dv] = o[i];
        }
      }
      if (owner && go) {
        a.ws.ml_part[(slot * kRB + n) * 2 + 0] = m_ref;
        a.ws.ml_part[(slot * kRB + n) * 2 + 1] = l;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(epi_done);
      x = piece_end;
      if (x == seg_end) seg_next(s, pfx, B, NRB);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

}  // namespace

int latent_split_ctas_per_sm() {
  static int cached = -1;
  if (cached >= 0) return cached;
  int n = 0;
  if (cudaFuncSetAttribute(latent_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SMEM) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, latent_split_kernel, kThreads, SMEM) !=
          cudaSuccess)
    n = 0;
  cached = n > 1 ? 1 : n;  // one CTA per SM: each holds all 512 tensor-memory columns
  return cached;
}

int latent_unit_tokens() { return kUT; }
int latent_row_block() { return kRB; }

cudaError_t launch_latent_split(const DecodeArgs& a, cudaStream_t s, int* launches) {
  latent_split_kernel<<<a.grid, kThreads, SMEM, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace kvfp8
