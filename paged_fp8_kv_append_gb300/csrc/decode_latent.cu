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
// is one 64-token page.  Units are laid out segment-major and cut into equal
// ranges, one per CTA (one CTA per SM); each (CTA, segment) piece leaves a
// partial (o, running max, sum) for the combine kernel.
//
// Per unit:
//   converter warps load the page's 64 x 576 e4m3 bytes (each half's loads a
//                   half ahead; the page two units ahead is prefetched into
//                   L2) and convert them exactly to f16 into one of two
//                   128B-swizzled K-major tiles (the same tile is the
//                   MN-major V^T operand);
//   MMA warp        S = Q K^T   (tcgen05, M = 64 rows, N = 64 tokens, K = 576,
//                   f16 x f16 -> f32 into one of two tensor-memory buffers;
//                   Q's first 256 dims are read from tensor memory, where
//                   the converters put them when a segment starts, the rest
//                   from shared memory)
//                   and O^T += V^T P^T (M = 128 dims x 4 blocks, N = 64 rows,
//                   K = 64 tokens) accumulating in tensor memory, each issued
//                   as soon as its inputs are ready, S up to one unit ahead;
//   softmax warps   read S from tensor memory (all 32 lanes: two threads per
//                   row), apply the page scale, the causal mask and the online
//                   softmax with a lazily updated reference max (the output is
//                   rescaled only when a row's max grows by more than 2^8),
//                   and write P (f16; the page's scale enters as an exponent
//                   bias) into the tile's last 64-dim block, which V does not
//                   use, as the swizzled B operand.
// Every wait is bounded; on timeout the kernel records KV_ERR_TIMEOUT, lets
// the asynchronous work it issued finish (bounded) and frees its tensor
// memory before returning.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace kvfp8 {
namespace {

constexpr int kUT = 64;        // tokens per unit: one page
constexpr int kDK = 576, kDV = 512, kNKB = kDK / 64;  // K blocks of 64 dims
constexpr int kRB = 64;        // query rows per segment
constexpr int kNKV = 2;        // f16 KV tiles (converted units)
constexpr int kUnitBytes = kUT * kDK;            // 36864 e4m3 bytes per unit
constexpr int kHalfPieces = kUnitBytes / 16 / 256;  // 16-byte pieces per thread per half unit
static_assert(kHalfPieces == 9, "converter mapping");

// warps: 0-3 softmax (tensor-memory lane quarters 0-3), 4-7 converters
// (global e4m3 -> swizzled f16 tiles), 8 MMA issuer
constexpr int kThreads = 288;
constexpr int kSoftmaxWarps = 4, kConvWarps = 4;
constexpr int kMmaWarp = 8;

// shared memory (bytes); tiles 1024-byte aligned for the 128B swizzle.  A KV
// tile is 9 blocks of [64 tokens][128 B]; once S has read it, its last block
// (dims 512..575, not part of V) holds the unit's P tile [64 rows][128 B].
constexpr int BLK = kUT * 128;                             // 8192
constexpr int OFF_Q = 0;                                   // 9 x [64 rows][128 B]
constexpr int OFF_KV = OFF_Q + kNKB * kRB * 128;
constexpr int KV_BYTES = kNKB * BLK;                       // 73728
constexpr int OFF_P_IN_KV = (kNKB - 1) * BLK;              // block 8
constexpr int OFF_ALPHA = OFF_KV + kNKV * KV_BYTES;        // 2 x 64 floats
constexpr int OFF_FLAG = OFF_ALPHA + 2 * kRB * 4;          // 2 ints (+pad)
constexpr int OFF_META = OFF_FLAG + 16;                    // unit meta [2]
constexpr int OFF_BAR = OFF_META + kNKV * 16;
constexpr int NBAR = 4 * kNKV + 4;
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int OFF_QEXP = OFF_MISC + 64;                    // [64] query row exponents
constexpr int SMEM = OFF_QEXP + kRB * 4;
static_assert(OFF_KV % 1024 == 0 && KV_BYTES % 1024 == 0 && OFF_BAR % 8 == 0, "alignment");
static_assert(SMEM <= 227 * 1024, "shared memory budget");

// tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;     // O^T: 4 blocks x 64 columns
constexpr uint32_t kTmemS = 256;   // S: 2 buffers x 64 columns
// Q dims 0..255 as the A operand of S (f16, two dims per column; row r of the
// M = 64 block in lane 32 (r / 16) + r % 16, as the M = 64 accumulator): the
// first kQTmemSlices of S's 16-dim K slices read A from here instead of
// shared memory, so shared memory serves only their B (K) operand.
constexpr uint32_t kTmemQ = 384;
constexpr int kQTmemDims = 256, kQTmemSlices = kQTmemDims / 16;

// page id standing for a page whose tag failed the fused check
constexpr int kStaleTag = INT_MIN;

struct UnitMeta {
  int n_valid;  // valid tokens of the unit; -1: a page that must not be read
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
constexpr uint32_t kIdescS = idesc_f16(kRB, kUT, 0, 0);  // S = Q K^T
constexpr uint32_t kIdescPV = idesc_f16(128, kRB, 1, 0); // O^T += V^T P^T

// issued by the elected lane of a converged warp (cheaper than a lone lane)
__device__ __forceinline__ void mma_f16_if(uint32_t leader, uint32_t d_tmem, uint64_t a,
                                           uint64_t b, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0), "r"(leader)
      : "memory");
}

// the same with the A operand read from tensor memory at column address a_tmem
__device__ __forceinline__ void mma_f16_ts_if(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem,
                                              uint64_t b, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0), "r"(leader)
      : "memory");
}

__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred;
}

// non-blocking phase test
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// whole page into L2 ahead of the converters' loads (16-byte aligned, size a
// multiple of 16)
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
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

// M = 64 accumulator rows live in lanes 0..15 of each lane quarter: threads
// 0..15 read lane t at columns c..c+31, threads 16..31 lane t-16 at c+32..c+63
__device__ __forceinline__ void tmem_ld16x2(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], 32;"
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

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
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

// The bf16 query is multiplied in f16.  Each query row is first scaled by an
// exact power of two 2^e that puts its largest magnitude in [2^15, 2^16):
// inside f16's range (below 65504) with all of its bits, and small elements
// clear of f16's subnormals; the row's score scale takes 2^-e.  For a row
// whose elements are normal f16 values either way the scores are
// bit-identical to unscaled ones (a power-of-two factor commutes with
// rounding).  Largest magnitude of 8 bf16 values, sign cleared:
__device__ __forceinline__ uint32_t bf16_absbits_max8(const uint4& v) {
  const uint32_t a = max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu);
  const uint32_t b = max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu);
  const uint32_t c = max(v.z & 0x7FFFu, (v.z >> 16) & 0x7FFFu);
  const uint32_t d = max(v.w & 0x7FFFu, (v.w >> 16) & 0x7FFFu);
  return max(max(a, b), max(c, d));
}
// e = 15 - floor(log2 max), within [-112, 112] (all-zero or subnormal rows: 112)
__device__ __forceinline__ int q_row_exp(uint32_t mb) {
  const int E = (int)(mb >> 7);
  return E == 0 ? 112 : min(112, max(-112, 142 - E));
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }
// exponent of query row `row` of a 576-dim block: two threads per row (the
// pair differ in lane bit `pair_bit`), each taking 288 dims
__device__ __forceinline__ int q_row_exp_pair(const uint16_t* qrow, int half, int pair_bit) {
  constexpr int kN = kDK / 16, kG = 12;  // 36 loads per thread, 12 in flight at a time
  static_assert(kN % kG == 0, "load groups");
  const uint16_t* base = qrow + half * (kDK / 2);
  uint32_t mb = 0;
#pragma unroll
  for (int k0 = 0; k0 < kN; k0 += kG) {
    uint4 v[kG];
#pragma unroll
    for (int k = 0; k < kG; ++k) v[k] = *reinterpret_cast<const uint4*>(base + 8 * (k0 + k));
#pragma unroll
    for (int k = 0; k < kG; ++k) mb = max(mb, bf16_absbits_max8(v[k]));
  }
  mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, pair_bit));
  return q_row_exp(mb);
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float pw) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * pw,
                                      __uint_as_float(w & 0xFFFF0000u) * pw);
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
  pdl_wait();
  pdl_trigger();  // the combine's CTAs may wait resident in what this kernel leaves free
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* q_s = smem + OFF_Q;
  uint8_t* kv_s = smem + OFF_KV;
  float* alpha_s = reinterpret_cast<float*>(smem + OFF_ALPHA);    // [2][64]
  volatile int* flag_s = reinterpret_cast<volatile int*>(smem + OFF_FLAG);  // [2]
  UnitMeta* kv_meta = reinterpret_cast<UnitMeta*>(smem + OFF_META);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* kv_ready = bars;               // [2] converters (tile + meta written)
  uint64_t* kv_free = kv_ready + kNKV;     // [2] MMA commit after PV: tile and P free
  uint64_t* s_full = kv_free + kNKV;       // [2] MMA commit after S
  uint64_t* p_ready = s_full + kNKV;       // [2] softmax: P written, O rescaled
  uint64_t* q_ready = p_ready + kNKV;      // converters
  uint64_t* q_free = q_ready + 1;          // MMA commit after a piece's last S
  uint64_t* epi_done = q_free + 1;         // softmax: O of the piece read out
  uint64_t* drain = epi_done + 1;          // MMA commit at exit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  int* qexp_s = reinterpret_cast<int*>(smem + OFF_QEXP);
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
      mbar_init(&s_full[i], 1);
      mbar_init(&p_ready[i], kSoftmaxWarps);
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
    // A unit's 64 x 576 e4m3 bytes are converted in two halves of 32 tokens,
    // 9 16-byte pieces per thread each; each half's loads are issued one half
    // ahead, and the page two units ahead is pulled into L2.
    const int ct = threadIdx.x - kSoftmaxWarps * 32;
    const int maxp = a.max_pages;
    Seg s = start;
    long long x = x_begin, u = 0;
    int piece = 0;
    bool go = true;
    while (x < x_end && go) {
      const long long seg_end = s.start + s.np, piece_end = min(seg_end, x_end);
      const int32_t* prow = a.page_table + (long long)s.r * maxp;
      const int L = a.seq_lens[s.r];
      // ---- Q block of this segment: rows rb*64 .. +63 of the request's T*Hq rows
      if (piece > 0 &&
          !mbar_wait(q_free, (uint32_t)((piece - 1) & 1), abort_flag, ctl, wait_info(warp, 1, 60))) {
        go = false;
        break;
      }
      tc_fence_after();  // the previous piece's S MMAs have read Q's tensor memory
      {
        const uint16_t* qbase = a.q + ((long long)s.r * a.T * a.Hq + (long long)s.rb * kRB) * kDK;
        // this warp stages the 16 rows of its tensor-memory lane quarter qq:
        // first their exponents (lanes i and i + 16 take the two halves of
        // row 16 qq + i), so that no other warp's rows are involved
        const int qq = warp & 3;
        {
          const int e = q_row_exp_pair(qbase + (long long)(16 * qq + (lane & 15)) * kDK,
                                       lane >> 4, 16);
          if (lane < 16) qexp_s[16 * qq + lane] = e;
          __syncwarp();
        }
        // dims kQTmemDims.. of these rows to shared memory, 128B-swizzled
        // (the A operand of S's remaining slices; the blocks below them stay
        // unused)
        constexpr int kCk0 = kQTmemDims / 8, kCkN = kDK / 8 - kCk0;
        for (int c = lane; c < 16 * kCkN; c += 32) {
          const int n = 16 * qq + c / kCkN, ck = kCk0 + c % kCkN;
          const uint4 v = *reinterpret_cast<const uint4*>(qbase + (long long)n * kDK + ck * 8);
          const float pw = pow2f(qexp_s[n]);
          uint4 o;
          o.x = bf16x2_to_f16x2_scaled(v.x, pw);
          o.y = bf16x2_to_f16x2_scaled(v.y, pw);
          o.z = bf16x2_to_f16x2_scaled(v.z, pw);
          o.w = bf16x2_to_f16x2_scaled(v.w, pw);
          *reinterpret_cast<uint4*>(q_s + (ck >> 3) * (kRB * 128) + swz(n, ck & 7)) = o;
        }
        // dims 0..kQTmemDims-1 to tensor memory: converter warp w writes lane
        // quarter w % 4; its lane i < 16 holds row 16 (w % 4) + i of the block
        // (lanes 16..31 write zeros to columns nothing else uses)
        {
          const int row = 16 * qq + (lane & 15);
          const uint16_t* qrow = qbase + (long long)row * kDK;
          const uint32_t q_lanes = (uint32_t)(32 * qq) << 16;
          const float pw = pow2f(qexp_s[row]);
#pragma unroll 1
          for (int k = 0; k < kQTmemDims / 64; ++k) {  // 64 dims = 32 columns per store
            uint32_t w[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint4 v = lane < 16
                                  ? *reinterpret_cast<const uint4*>(qrow + 64 * k + 8 * j)
                                  : make_uint4(0, 0, 0, 0);
              w[4 * j + 0] = bf16x2_to_f16x2_scaled(v.x, pw);
              w[4 * j + 1] = bf16x2_to_f16x2_scaled(v.y, pw);
              w[4 * j + 2] = bf16x2_to_f16x2_scaled(v.z, pw);
              w[4 * j + 3] = bf16x2_to_f16x2_scaled(v.w, pw);
            }
            tmem_st32u(tmem + kTmemQ + 32 * k + q_lanes, w);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        tc_fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready);
      }
      auto page_ok = [&](int pg) { return pg >= 0 && pg < a.d.num_pages; };
      // unit j of the request is page j; with the fused tag check a page
      // whose tag is not the expected one becomes kStaleTag here, before
      // anything (the L2 prefetch included) reads it
      // (without the check nothing here may depend on the loaded id: the
      // id of the unit three ahead is only used a unit later)
      auto page_of = [&](long long xu) -> int {
        if (xu >= piece_end) return -1;
        const int pg = prow[xu - s.start];
        if (a.exp_tags == nullptr) return pg;
        if (!page_ok(pg)) return pg;
        return a.d.tags[pg] == a.exp_tags[(long long)s.r * maxp + (xu - s.start)] ? pg
                                                                                  : kStaleTag;
      };
      auto src_of = [&](int pg) -> const uint8_t* {
        return cache + (long long)(page_ok(pg) ? pg : 0) * kUnitBytes;
      };
      // half h = tokens 32h..32h+31; piece k of this thread is token
      // 32h + ct / 4, dims 64k + 16 (ct % 4) .. +15 (dim block k), so a warp
      // stores 8 rows of one block and the 128B swizzle spreads its 16-byte
      // stores over all banks
      auto load_half = [&](int pg, long long xu, int h, uint4 (&d)[kHalfPieces]) {
        const int nv = page_ok(pg) ? min(kUT, L - (int)(xu - s.start) * kUT) : 0;
        const int t = 32 * h + (ct >> 2);
        const uint8_t* src = src_of(pg) + t * kDK + (ct & 3) * 16;
#pragma unroll
        for (int k = 0; k < kHalfPieces; ++k)
          d[k] = (t < nv) ? __ldg(reinterpret_cast<const uint4*>(src + k * 64))
                          : make_uint4(0, 0, 0, 0);
      };
      auto convert_half = [&](uint8_t* dst, int h, const uint4 (&d)[kHalfPieces]) {
        const int t = 32 * h + (ct >> 2), j = ct & 3;
        const uint32_t o_lo = swz(t, 2 * j), o_hi = swz(t, 2 * j + 1);
#pragma unroll
        for (int k = 0; k < kHalfPieces; ++k) {
          uint4 lo, hi;
          e4m3x4_to_f16(d[k].x, lo.x, lo.y);
          e4m3x4_to_f16(d[k].y, lo.z, lo.w);
          e4m3x4_to_f16(d[k].z, hi.x, hi.y);
          e4m3x4_to_f16(d[k].w, hi.z, hi.w);
          *reinterpret_cast<uint4*>(dst + k * BLK + o_lo) = lo;
          *reinterpret_cast<uint4*>(dst + k * BLK + o_hi) = hi;
        }
      };
      int pg0 = page_of(x), pg1 = page_of(x + 1), pg2 = page_of(x + 2);
      if (ct == 0) {
        if (page_ok(pg0)) prefetch_l2(src_of(pg0), kUnitBytes);
        if (page_ok(pg1)) prefetch_l2(src_of(pg1), kUnitBytes);
      }
      uint4 d0[kHalfPieces], d1[kHalfPieces];
      load_half(pg0, x, 0, d0);
      for (long long xu = x; xu < piece_end; ++xu, ++u) {
        const int b = (int)(u & 1);
        load_half(pg0, xu, 1, d1);
        if (ct == 0 && page_ok(pg2)) prefetch_l2(src_of(pg2), kUnitBytes);
        const int pg3 = page_of(xu + 3);
        // meta of this unit (its scale load is the only dependent one)
        UnitMeta m;
        const bool ok = page_ok(pg0);
        m.n_valid = ok ? min(kUT, L - (int)(xu - s.start) * kUT) : -1;
        m.pos0 = (int)(xu - s.start) * kUT;
        m.scale = ok ? a.d.k_scale[pg0] : 1.0f;
        m.unit = (int)u;
        if (!ok && pg0 != kStaleTag && ct == 0) set_error(ctl, KV_ERR_BAD_PAGE_ID);
        // tile b is free once PV(u - 2) has completed
        if (u >= kNKV && !mbar_wait(&kv_free[b], (uint32_t)(((u >> 1) - 1) & 1), abort_flag, ctl,
                                    wait_info(warp, 1, 32 + b))) {
          go = false;
          break;
        }
        uint8_t* dst = kv_s + b * KV_BYTES;
        convert_half(dst, 0, d0);
        if (xu + 1 < piece_end) load_half(pg1, xu + 1, 0, d0);
        convert_half(dst, 1, d1);
        if (ct == 0) kv_meta[b] = m;
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_ready[b]);
        pg0 = pg1;
        pg1 = pg2;
        pg2 = pg3;
      }
      ++piece;
      x = piece_end;
      if (x == seg_end) seg_next(s, pfx, B, NRB);
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ============================
    // Per piece, S(u) and PV(u) are issued as soon as their inputs are ready
    // (PV first when both are): S(u) needs tile u converted and at most one
    // unit ahead of PV; PV(u) needs P(u) (and, for the piece's first unit, the
    // previous piece's output read out).
    const uint32_t leader = elect_one();
    Seg s = start;
    long long x = x_begin, u = 0;
    int piece = 0;
    bool go = true;
    const uint32_t q_base = smem_u32(q_s), kv_base = smem_u32(kv_s);
    const uint64_t dq0 = sw128_desc(q_base, 16, 1024);
    const uint64_t dk0 = sw128_desc(kv_base, 16, 1024);
    const uint64_t dv0 = sw128_desc(kv_base, BLK, 1024);
    const uint64_t dp0 = sw128_desc(kv_base + OFF_P_IN_KV, 16, 1024);
    while (x < x_end && go) {
      const long long seg_end = s.start + s.np, piece_end = min(seg_end, x_end);
      const long long u0 = u, ue = u0 + (piece_end - x);
      go = __all_sync(0xffffffffu, mbar_wait(q_ready, (uint32_t)(piece & 1), abort_flag, ctl,
                                             wait_info(warp, 0, 62)));
      if (!go) break;
      tc_fence_after();  // Q's tensor-memory stores are ordered before the S MMAs
      long long ns = u0, np = u0;
      bool epi_ok = piece == 0;
      uint32_t idle = 0;
      uint64_t t_idle = global_ns();
      while (np < ue) {
        bool did = false;
        if (np < ns) {  // ---- PV(np): O^T += V^T P^T
          const int b = (int)(np & 1);
          if (!epi_ok)
            epi_ok = __all_sync(0xffffffffu, mbar_test(epi_done, (uint32_t)((piece - 1) & 1)));
          if (epi_ok &&
              __all_sync(0xffffffffu, mbar_test(&p_ready[b], (uint32_t)((np >> 1) & 1)))) {
            tc_fence_after();
            const uint32_t kvo = (uint32_t)(b * KV_BYTES) >> 4;
#pragma unroll
            for (int st = 0; st < kUT / 16; ++st) {
#pragma unroll
              for (int db = 0; db < kDV / 128; ++db) {
                // V^T: dims 128db.. (two 64-dim blocks, BLK apart), tokens 16st..
                const uint64_t ad = dv0 + kvo + ((uint32_t)(2 * db * BLK + st * 2048) >> 4);
                const uint64_t bd = dp0 + kvo + (uint32_t)(st * 2);
                mma_f16_if(leader, tmem + kTmemO + 64 * db, ad, bd, kIdescPV,
                           !(np == u0 && st == 0));
              }
            }
            if (leader) mma_commit(&kv_free[b]);
            __syncwarp();
            ++np;
            did = true;
          }
        }
        if (!did && ns < ue && ns - np < kNKV) {  // ---- S(ns) = Q K^T
          const int b = (int)(ns & 1);
          if (__all_sync(0xffffffffu, mbar_test(&kv_ready[b], (uint32_t)((ns >> 1) & 1)))) {
            tc_fence_after();
            const uint32_t kvo = (uint32_t)(b * KV_BYTES) >> 4;
#pragma unroll
            for (int st = 0; st < kDK / 16; ++st) {
              const uint32_t off = (uint32_t)((st >> 2) * BLK + (st & 3) * 32) >> 4;
              if (st < kQTmemSlices)  // A (Q) from tensor memory
                mma_f16_ts_if(leader, tmem + kTmemS + 64 * b, tmem + kTmemQ + 8 * st,
                              dk0 + kvo + off, kIdescS, st > 0);
              else
                mma_f16_if(leader, tmem + kTmemS + 64 * b, dq0 + off, dk0 + kvo + off, kIdescS,
                           st > 0);
            }
            if (leader) {
              mma_commit(&s_full[b]);
              if (ns == ue - 1) mma_commit(q_free);  // every S of this piece is issued
            }
            __syncwarp();
            ++ns;
            did = true;
          }
        }
        if (did) {
          idle = 0;
        } else if ((++idle & 63u) == 1u) {  // the clock is read only now and then
          if (idle == 1u) t_idle = global_ns();
          if (*abort_flag) {
            go = false;
          } else if (global_ns() - t_idle > kWaitLimitNs) {
            *abort_flag = 1;
            if (lane == 0 &&
                atomicCAS(reinterpret_cast<int*>(ctl + KV_CTL_ERROR), 0, KV_ERR_TIMEOUT) == 0)
              ctl[KV_CTL_WAIT_INFO] = wait_info(warp, 0, np < ns ? 48 : 40);
            go = false;
          }
          go = __all_sync(0xffffffffu, go);
          if (!go) break;
        }
      }
      u = ue;
      ++piece;
      x = piece_end;
      if (x == seg_end) seg_next(s, pfx, B, NRB);
    }
    // let every tensor-core operation issued here finish (bounded) before
    // tensor memory is freed: a commit tracks all earlier ones
    if (leader) {
      mma_commit(drain);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(drain, 0) && global_ns() - t0 < 100000000ull) {
      }
    }
    __syncwarp();
  } else if (warp < kSoftmaxWarps) {
    // ============================ softmax (warps 0-3) ============================
    // Row r = 16 q4 + (lane & 15) of the block; lanes < 16 hold its tokens
    // 0..31 of a unit, lanes >= 16 its tokens 32..63.  Logits are in log2
    // units.  The page scale enters P as a bias log2(scale) on the exponent,
    // and the reference max M tracks max(logit + bias) lazily (the output is
    // rescaled only when it grows by more than 2^8), so P <= 2^8 and small
    // scales do not push P into f16's subnormal range; the row sum l takes
    // the bias back out.
    const int q4 = warp;
    const int r = 16 * q4 + (lane & 15), h = lane >> 4;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const float ssl = a.sm_scale_log2;
    Seg s = start;
    long long x = x_begin, u = 0;
    bool go = true;
    while (x < x_end) {
      const long long seg_end = s.start + s.np, piece_end = min(seg_end, x_end);
      const int L = a.seq_lens[s.r];
      // row rb*64 + r of the request's (t, hq) rows: draft token t = row / Hq
      const int tq = (s.rb * kRB + r) / a.Hq;
      const int lim = L - a.T + min(tq, a.T - 1);  // last visible position (inclusive)
      // this row's query scale 2^e (the converters staged Q times 2^e): its
      // scores take 2^-e; the two threads of the row (lanes l, l ^ 16) each
      // read half of it
      const float qsc = ssl * pow2f(-q_row_exp_pair(
          a.q + ((long long)s.r * a.T * a.Hq + (long long)s.rb * kRB + r) * kDK, h, 16));
      float M = -INFINITY, l = 0.0f;
      bool bad = false;  // the piece met a page it must not read
      const long long u0 = u;
      // every softmax warp runs every unit (and every named barrier), even
      // after a wait gave up, so the barrier sequence never diverges
      for (long long xu = x; xu < piece_end; ++xu, ++u) {
        const int b = (int)(u & 1);
        go = go && mbar_wait(&s_full[b], (uint32_t)((u >> 1) & 1), abort_flag, ctl,
                             wait_info(warp, 0, 52 + b));
        go = go && mbar_wait(&kv_ready[b], (uint32_t)((u >> 1) & 1), abort_flag, ctl,
                             wait_info(warp, 0, 44 + b));
        go = __all_sync(0xffffffffu, go);  // tensor-memory loads are warp-collective
        float v[32];
        if (go) {
          tc_fence_after();
          tmem_ld16x2(tmem + kTmemS + 64 * b + lane_off, v);
        }
        const UnitMeta m = kv_meta[b];
        bad = bad || (go && m.unit == (int)u && m.n_valid < 0);
        if (go && m.unit != (int)u) {
          if (lane == 0) set_error(ctl, KV_ERR_INTERNAL);
          *abort_flag = 1;
          go = false;
        }
        go = __all_sync(0xffffffffu, go);
        float alpha = 1.0f;
        if (go) {
          const float sc = m.scale * qsc, bias = __log2f(m.scale);
          // tokens i <= thr of this thread's 32 are visible
          const int thr = min(m.n_valid - 1, lim - m.pos0) - 32 * h;
          float mx = -INFINITY;
          if (thr >= 31) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v[i] *= sc;
              mx = fmaxf(mx, v[i]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v[i] = (i <= thr) ? v[i] * sc : -INFINITY;
              mx = fmaxf(mx, v[i]);
            }
          }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mb = mx + bias;
          if (mb > M + 8.0f) {
            alpha = (M == -INFINITY) ? 0.0f : ex2(M - mb);
            l *= alpha;
            M = mb;
          }
          const float c = (M == -INFINITY) ? -INFINITY : bias - M;
          float sum = 0.0f;
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float p0 = ex2(v[i] + c), p1 = ex2(v[i + 1] + c);
            sum += p0 + p1;
            pk[i >> 1] = pack_f16(p0, p1);
          }
          l += sum * ex2(-bias);
          // P row r, tokens 32h..32h+31 = chunks 4h..4h+3 of a 128B-swizzled row
          uint8_t* prow = kv_s + b * KV_BYTES + OFF_P_IN_KV;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            *reinterpret_cast<uint4*>(prow + swz(r, 4 * h + c4)) =
                make_uint4(pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
          if (alpha != 1.0f) flag_s[b] = (int)u;  // unit number: never stale
        }
        if (h == 0) alpha_s[b * kRB + r] = alpha;
        fence_async_smem();
        named_bar_sync(2, kSoftmaxWarps * 32);
        if (flag_s[b] == (int)u && u > u0) {
          // O^T columns are query rows: column n *= alpha[n], after PV(u-1)
          const long long pu = u - 1;
          go = go && mbar_wait(&kv_free[pu & 1], (uint32_t)((pu >> 1) & 1), abort_flag, ctl,
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
                for (int i = 0; i < 32; ++i) o[i] *= alpha_s[b * kRB + 32 * half + i];
                tmem_st32(ta, o);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_ready[b]);
      }
      // ---- epilogue: partial (o, m, l) of this piece
      if (u > u0) {
        const long long last = u - 1;
        go = go && mbar_wait(&kv_free[last & 1], (uint32_t)((last >> 1) & 1), abort_flag, ctl,
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
      const float l_row = l + __shfl_xor_sync(0xffffffffu, l, 16);
      if (h == 0 && go) {
        a.ws.ml_part[(slot * kRB + r) * 2 + 0] = M;
        a.ws.ml_part[(slot * kRB + r) * 2 + 1] = bad ? -1.0f : l_row;
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
  const cudaError_t e = launch_pdl(latent_split_kernel, dim3(a.grid), dim3(kThreads), SMEM, s, a);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace kvfp8
