// api.cu -- the C ABI declared in include/kvfp8.h: argument validation,
// launch configuration and workspace carve-up.  All compute is in the
// kernels of append.cu, verify.cu, release.cu, decode_gqa.cu and
// decode_latent.cu; kv_decode_step chains them on one stream.
#include <math.h>

#include <new>

#include "internal.h"

using namespace kvfp8;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

namespace kvfp8 {

kv_status decode_config(const kv_pool* pool, int B, int Hq, int T, DecodeConfig* cfg) {
  const kv_pool_desc& d = pool->d;
  if (B < 0 || Hq <= 0 || T <= 0) return KV_ERR_INVALID_ARG;
  if (d.layout == KV_LAYOUT_GQA) {
    if (Hq % d.num_kv_heads != 0) return KV_ERR_INVALID_ARG;
    const int G = Hq / d.num_kv_heads;
    // query rows per kv head, in blocks of 8 or 16 (one consumer warp each)
    const long long R = (long long)T * G;
    if (d.head_dim_k != 128 || d.head_dim_v != 128 || d.page_size != 16 || R > 64)
      return KV_ERR_UNSUPPORTED;
    // more than 8 rows: consumer warps of 16 rows (kinds 3: e4m3, 4: bf16)
    cfg->kind = d.dtype == KV_DTYPE_E4M3 ? (R > 8 ? 3 : 0) : (R > 8 ? 4 : 1);
    const bool bf16 = cfg->kind == 1 || cfg->kind == 4, wide = cfg->kind >= 3;
    // heads per unit: the largest power of two <= 8 (<= 4 for bf16, whose
    // tiles are twice as large) dividing Hkv, with heads x row blocks dividing
    // the consumer warp count; 16-row blocks may be padded with whole unused
    // blocks until such a split exists; ring depth from the ring size
    int rbw = wide ? (int)((R + 15) / 16) : (int)((R + 7) / 8);  // row blocks, one warp each
    int hs = 0;
    for (; rbw <= (wide ? 4 : 1); ++rbw) {
      hs = bf16 ? 4 : 8;
      while (hs > 0 &&
             (d.num_kv_heads % hs != 0 || gqa_consumer_warps(cfg->kind) % (hs * rbw) != 0))
        hs >>= 1;
      if (hs > 0) break;
    }
    if (hs == 0) return KV_ERR_UNSUPPORTED;  // no split of the consumers fits
    const int rb = wide ? 2 * rbw : rbw;  // row blocks of 8 in the partial layout
    cfg->Hs = hs;
    const int stage_bytes = 2 * hs * d.page_size * d.head_dim_k * (bf16 ? 2 : 1);
    cfg->stages = gqa_ring_bytes(cfg->kind) / stage_bytes;
    if (cfg->stages > gqa_max_stages()) cfg->stages = gqa_max_stages();
    // A consumer warp serves every (consumers/Hs)-th unit; the ring depth must
    // be a multiple of that stride so each warp sees every phase of the stages
    // it uses (parity waits cannot tell phase n from phase n-2).
    const int wph = gqa_consumer_warps(cfg->kind) / (hs * rbw);
    cfg->stages -= cfg->stages % wph;
    if (cfg->stages < 2 || cfg->stages < wph) return KV_ERR_UNSUPPORTED;
    const int sms = sm_count();
    const int per_sm = sms > 0 ? gqa_split_ctas_per_sm(cfg->kind) : 0;
    if (sms <= 0 || per_sm <= 0) return KV_ERR_CUDA;
    cfg->grid = sms * per_sm;
    cfg->R8 = 8 * rb;
    cfg->HG = d.num_kv_heads / hs;
    cfg->unit_tokens = d.page_size;
    // the split kernel's CTAs plan a batch that fits their shared-memory
    // prefix cache themselves: no separate plan launch
    cfg->self_plan = (gqa_kind_self_plans(cfg->kind) && B <= gqa_self_plan_max_batch()) ? 1 : 0;
    return KV_OK;
  }
  // latent layout: query rows (T tokens x Hq heads) in blocks of 64; the
  // row count stays far inside int range (2^20 rows)
  const int rb = latent_row_block();
  if ((long long)T * Hq > (1ll << 20)) return KV_ERR_UNSUPPORTED;
  if (d.head_dim_k != 576 || d.head_dim_v != 512 || d.page_size != 64 || (T * Hq) % rb != 0 ||
      d.dtype != KV_DTYPE_E4M3)
    return KV_ERR_UNSUPPORTED;
  const int sms = sm_count();
  const int per_sm = sms > 0 ? latent_split_ctas_per_sm() : 0;
  if (sms <= 0 || per_sm <= 0) return KV_ERR_CUDA;
  cfg->kind = 2;
  cfg->self_plan = 0;
  cfg->grid = sms * per_sm;
  cfg->R8 = rb;
  cfg->Hs = 1;
  cfg->HG = T * Hq / rb;
  cfg->stages = 0;
  cfg->unit_tokens = latent_unit_tokens();
  return KV_OK;
}

size_t decode_ws_layout(const kv_pool_desc& d, int B, int Hkv, const DecodeConfig& cfg,
                        void* base, DecodeWs* ws) {
  // one partial slot per (CTA, segment) piece; segments are (request, head
  // group) or (request, row block); each slot holds Hs heads x R8 rows
  (void)Hkv;
  const long long slots = (long long)B * cfg.HG + cfg.grid;
  size_t off = 0;
  const size_t o_pfx = off;
  off = align256(off + sizeof(int32_t) * (size_t)(B + 1));
  const size_t o_skip = off;
  off = align256(off + (size_t)B);
  const size_t o_ml = off;
  off = align256(off + sizeof(float) * 2 * (size_t)slots * cfg.Hs * cfg.R8);
  const size_t o_o = off;
  off = align256(off + sizeof(float) * (size_t)slots * cfg.Hs * cfg.R8 * d.head_dim_v);
  if (ws) {
    uint8_t* b = static_cast<uint8_t*>(base);
    ws->pfx = reinterpret_cast<int32_t*>(b + o_pfx);
    ws->rq_skip = b + o_skip;
    ws->ml_part = reinterpret_cast<float*>(b + o_ml);
    ws->o_part = reinterpret_cast<float*>(b + o_o);
    ws->bytes = off;
  }
  return off;
}

}  // namespace kvfp8

namespace {

kv_status decode_prepare(kv_pool* pool, int32_t B, int32_t Hq, int32_t T, const void* q,
                         const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                         const uint8_t* abort_mask, float sm_scale, void* out, void* workspace,
                         size_t workspace_bytes, bool need_inputs, bool need_out,
                         DecodeArgs* a, int* kind) {
  if (!pool) return KV_ERR_INVALID_ARG;
  const kv_pool_desc& d = pool->d;
  if (B < 0 || Hq <= 0 || T <= 0) return KV_ERR_INVALID_ARG;
  if (B > 0) {
    if (need_inputs && (!q || !page_table || !seq_lens || max_pages <= 0 || !aligned16(q) ||
                        !isfinite(sm_scale)))
      return KV_ERR_INVALID_ARG;
    if (need_out && !out) return KV_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return KV_ERR_INVALID_ARG;
  }
  DecodeConfig cfg;
  const kv_status st = decode_config(pool, B, Hq, T, &cfg);
  if (st != KV_OK) return st;
  const int Hkv = d.num_kv_heads;
  DecodeArgs& x = *a;
  x.d = d;
  x.B = B;
  x.Hq = Hq;
  x.T = T;
  x.G = Hq / Hkv;
  x.R = (d.layout == KV_LAYOUT_GQA) ? T * x.G : T * Hq;
  x.q = static_cast<const uint16_t*>(q);
  x.page_table = page_table;
  x.max_pages = max_pages;
  x.seq_lens = seq_lens;
  x.abort_mask = abort_mask;
  x.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  x.out = static_cast<uint16_t*>(out);
  x.grid = cfg.grid;
  x.R8 = cfg.R8;
  x.Hs = cfg.Hs;
  x.HG = cfg.HG;
  x.stages = cfg.stages;
  x.unit_tokens = cfg.unit_tokens;
  x.self_plan = cfg.self_plan;
  x.exp_tags = nullptr;
  x.abort_out = nullptr;
  const size_t need = decode_ws_layout(d, B, Hkv, cfg, workspace, &x.ws);
  if (B > 0 && workspace_bytes < need) return KV_ERR_INVALID_ARG;
  *kind = cfg.kind;
  return KV_OK;
}

}  // namespace

extern "C" {

kv_status kv_pool_create(const kv_pool_desc* desc, kv_pool** out) {
  if (!desc || !out) return KV_ERR_INVALID_ARG;
  *out = nullptr;
  const kv_pool_desc& d = *desc;
  if (d.num_pages <= 0 || d.page_size <= 0 || d.page_size > 1024 || d.num_kv_heads <= 0 ||
      d.head_dim_k <= 0 || d.head_dim_v <= 0 || d.head_dim_k % 16 != 0 ||
      d.head_dim_v % 16 != 0 || d.head_dim_k > 1024 || d.head_dim_v > 1024)
    return KV_ERR_INVALID_ARG;
  if (d.dtype != KV_DTYPE_E4M3 && d.dtype != KV_DTYPE_BF16) return KV_ERR_INVALID_ARG;
  if (d.layout != KV_LAYOUT_GQA && d.layout != KV_LAYOUT_LATENT) return KV_ERR_INVALID_ARG;
  if (d.scale_mode != KV_SCALE_FROZEN && d.scale_mode != KV_SCALE_REQUANTIZE)
    return KV_ERR_INVALID_ARG;
  if (!d.k_cache || !d.tags || !d.free_list || !d.ctl) return KV_ERR_INVALID_ARG;
  if (!aligned16(d.k_cache) || !aligned16(d.tags) || !aligned16(d.free_list) ||
      !aligned16(d.ctl))
    return KV_ERR_INVALID_ARG;
  if (d.layout == KV_LAYOUT_GQA) {
    if (!d.v_cache || !aligned16(d.v_cache)) return KV_ERR_INVALID_ARG;
    if (d.dtype == KV_DTYPE_E4M3 && (!d.k_scale || !d.v_scale)) return KV_ERR_INVALID_ARG;
    // the dim-major V tile of one page must fit the append kernel's staging
    if ((long long)d.head_dim_v * d.page_size * (d.dtype == KV_DTYPE_E4M3 ? 1 : 2) > 160 * 1024)
      return KV_ERR_UNSUPPORTED;
  } else {
    // a bf16 latent pool holds rows for appends and handoffs (attention over
    // it is not supported)
    if (d.num_kv_heads != 1 || d.head_dim_v > d.head_dim_k ||
        (d.dtype == KV_DTYPE_E4M3 && !d.k_scale))
      return KV_ERR_INVALID_ARG;
  }
  kv_pool* p = new (std::nothrow) kv_pool;
  if (!p) return KV_ERR_INVALID_ARG;
  p->d = d;
  p->last_launches = 0;
  *out = p;
  return KV_OK;
}

kv_status kv_pool_destroy(kv_pool* pool) {
  if (!pool) return KV_ERR_INVALID_ARG;
  delete pool;
  return KV_OK;
}

kv_status kv_append_quantize(kv_pool* pool, void* stream, int32_t B, const void* k_new,
                             const void* v_new, const int32_t* new_indptr,
                             int32_t max_new_per_req, int32_t* page_table, uint32_t* exp_tags,
                             int32_t max_pages_per_req, int32_t* seq_lens) {
  if (!pool) return KV_ERR_INVALID_ARG;
  pool->last_launches = 0;
  const kv_pool_desc& d = pool->d;
  if (B < 0 || max_new_per_req < 0 || max_pages_per_req <= 0) return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!new_indptr || !page_table || !exp_tags || !seq_lens) return KV_ERR_INVALID_ARG;
  if (max_new_per_req > 0) {
    if (!k_new || !aligned16(k_new)) return KV_ERR_INVALID_ARG;
    if (d.layout == KV_LAYOUT_GQA && (!v_new || !aligned16(v_new))) return KV_ERR_INVALID_ARG;
  }
  AppendArgs a;
  a.d = d;
  a.B = B;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.new_indptr = new_indptr;
  a.max_new = max_new_per_req;
  a.page_table = page_table;
  a.exp_tags = exp_tags;
  a.max_pages = max_pages_per_req;
  a.seq_lens = seq_lens;
  a.step_mask = nullptr;
  a.fuse_plan = false;
  a.from_pool = false;
  int n = 0;
  const cudaError_t e = launch_append(a, static_cast<cudaStream_t>(stream), &n);
  pool->last_launches = n;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kv_status kv_append_from_pool(kv_pool* pool, void* stream, int32_t B, const kv_pool* src,
                              const int32_t* src_page_table, int32_t src_max_pages_per_req,
                              const int32_t* src_seq_lens, int32_t* page_table,
                              uint32_t* exp_tags, int32_t max_pages_per_req, int32_t* seq_lens) {
  if (!pool) return KV_ERR_INVALID_ARG;
  pool->last_launches = 0;
  if (!src || B < 0 || max_pages_per_req <= 0 || src_max_pages_per_req <= 0)
    return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!src_page_table || !src_seq_lens || !page_table || !exp_tags || !seq_lens)
    return KV_ERR_INVALID_ARG;
  const kv_pool_desc& d = pool->d;
  const kv_pool_desc& sd = src->d;
  if (sd.dtype != KV_DTYPE_BF16 || sd.layout != d.layout || sd.num_kv_heads != d.num_kv_heads ||
      sd.head_dim_k != d.head_dim_k || sd.head_dim_v != d.head_dim_v ||
      sd.page_size != d.page_size)
    return KV_ERR_INVALID_ARG;
  if (!append_handoff_supported(d, B, src_max_pages_per_req)) return KV_ERR_UNSUPPORTED;
  AppendArgs a;
  a.d = d;
  a.B = B;
  a.k_new = nullptr;
  a.v_new = nullptr;
  a.new_indptr = nullptr;
  a.max_new = INT32_MAX;  // bounded by the page tables instead
  a.page_table = page_table;
  a.exp_tags = exp_tags;
  a.max_pages = max_pages_per_req;
  a.seq_lens = seq_lens;
  a.step_mask = nullptr;
  a.fuse_plan = false;
  a.from_pool = true;
  a.src = sd;
  a.src_page_table = src_page_table;
  a.src_max_pages = src_max_pages_per_req;
  a.src_lens = src_seq_lens;
  int n = 0;
  const cudaError_t e = launch_append(a, static_cast<cudaStream_t>(stream), &n);
  pool->last_launches = n;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kv_status kv_verify_tags(kv_pool* pool, void* stream, int32_t B, const int32_t* page_table,
                         const uint32_t* exp_tags, int32_t max_pages_per_req,
                         const int32_t* seq_lens, uint8_t* abort_mask) {
  if (!pool) return KV_ERR_INVALID_ARG;
  pool->last_launches = 0;
  if (B < 0 || max_pages_per_req <= 0) return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!page_table || !exp_tags || !seq_lens || !abort_mask) return KV_ERR_INVALID_ARG;
  VerifyArgs a;
  a.num_pages = pool->d.num_pages;
  a.page_size = pool->d.page_size;
  a.B = B;
  a.max_pages = max_pages_per_req;
  a.tags = pool->d.tags;
  a.page_table = page_table;
  a.exp_tags = exp_tags;
  a.seq_lens = seq_lens;
  a.abort_mask = abort_mask;
  int n = 0;
  const cudaError_t e = launch_verify(a, static_cast<cudaStream_t>(stream), &n);
  pool->last_launches = n;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

size_t kv_release_workspace_size(int32_t B) { return B < 0 ? 0 : release_ws_bytes(B); }

kv_status kv_release_pages(kv_pool* pool, void* stream, int32_t B, int32_t* page_table,
                           uint32_t* exp_tags, int32_t max_pages_per_req, int32_t* seq_lens,
                           const uint8_t* release_mask, void* workspace,
                           size_t workspace_bytes) {
  if (!pool) return KV_ERR_INVALID_ARG;
  pool->last_launches = 0;
  if (B < 0 || max_pages_per_req <= 0) return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!page_table || !exp_tags || !seq_lens || !workspace) return KV_ERR_INVALID_ARG;
  if (!aligned16(workspace) || workspace_bytes < release_ws_bytes(B)) return KV_ERR_INVALID_ARG;
  ReleaseArgs a;
  a.d = pool->d;
  a.B = B;
  a.max_pages = max_pages_per_req;
  a.page_table = page_table;
  a.exp_tags = exp_tags;
  a.seq_lens = seq_lens;
  a.mask = release_mask;
  a.mask_bits = 0xFF;
  a.offsets = static_cast<long long*>(workspace);
  int n = 0;
  const cudaError_t e = launch_release(a, static_cast<cudaStream_t>(stream), &n);
  pool->last_launches = n;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

size_t paged_decode_workspace_size(const kv_pool* pool, int32_t B, int32_t num_q_heads,
                                   int32_t q_tokens) {
  if (!pool || B < 0) return 0;
  DecodeConfig cfg;
  if (decode_config(pool, B, num_q_heads, q_tokens, &cfg) != KV_OK) return 0;
  return decode_ws_layout(pool->d, B, pool->d.num_kv_heads, cfg, nullptr, nullptr);
}

kv_status paged_decode_attn_split(kv_pool* pool, void* stream, int32_t B, int32_t num_q_heads,
                                  int32_t q_tokens, const void* q, const int32_t* page_table,
                                  int32_t max_pages_per_req, const int32_t* seq_lens,
                                  const uint8_t* abort_mask, float sm_scale, void* workspace,
                                  size_t workspace_bytes) {
  if (!pool) return KV_ERR_INVALID_ARG;
  pool->last_launches = 0;
  DecodeArgs a;
  int kind = 0;
  const kv_status st =
      decode_prepare(pool, B, num_q_heads, q_tokens, q, page_table, max_pages_per_req, seq_lens,
                     abort_mask, sm_scale, nullptr, workspace, workspace_bytes, true, false, &a,
                     &kind);
  if (st != KV_OK || B == 0) return st;
  int n = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = a.self_plan ? cudaSuccess : launch_decode_plan(a, s, &n);
  if (e == cudaSuccess) e = launch_decode_split(a, kind, s, &n);
  pool->last_launches = n;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kv_status paged_decode_attn_combine(kv_pool* pool, void* stream, int32_t B, int32_t num_q_heads,
                                    int32_t q_tokens, const uint8_t* abort_mask, void* out,
                                    void* workspace, size_t workspace_bytes) {
  if (!pool) return KV_ERR_INVALID_ARG;
  pool->last_launches = 0;
  DecodeArgs a;
  int kind = 0;
  const kv_status st =
      decode_prepare(pool, B, num_q_heads, q_tokens, nullptr, nullptr, 1, nullptr, abort_mask,
                     1.0f, out, workspace, workspace_bytes, false, true, &a, &kind);
  if (st != KV_OK || B == 0) return st;
  int n = 0;
  const cudaError_t e = launch_decode_combine(a, static_cast<cudaStream_t>(stream), &n);
  pool->last_launches = n;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kv_status paged_decode_attn(kv_pool* pool, void* stream, int32_t B, int32_t num_q_heads,
                            int32_t q_tokens, const void* q, const int32_t* page_table,
                            int32_t max_pages_per_req, const int32_t* seq_lens,
                            const uint8_t* abort_mask, float sm_scale, void* out,
                            void* workspace, size_t workspace_bytes) {
  if (!pool) return KV_ERR_INVALID_ARG;
  pool->last_launches = 0;
  if (B > 0 && !out) return KV_ERR_INVALID_ARG;
  // one argument set (and one validation) for the plan, the split and the combine
  DecodeArgs a;
  int kind = 0;
  const kv_status st =
      decode_prepare(pool, B, num_q_heads, q_tokens, q, page_table, max_pages_per_req, seq_lens,
                     abort_mask, sm_scale, out, workspace, workspace_bytes, true, true, &a, &kind);
  if (st != KV_OK || B == 0) return st;
  int n = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = a.self_plan ? cudaSuccess : launch_decode_plan(a, s, &n);
  if (e == cudaSuccess) e = launch_decode_split(a, kind, s, &n);
  if (e == cudaSuccess) e = launch_decode_combine(a, s, &n);
  pool->last_launches = n;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kv_status paged_decode_attn_checked(kv_pool* pool, void* stream, int32_t B, int32_t num_q_heads,
                                    int32_t q_tokens, const void* q, const int32_t* page_table,
                                    const uint32_t* exp_tags, int32_t max_pages_per_req,
                                    const int32_t* seq_lens, float sm_scale, void* out,
                                    uint8_t* abort_mask, void* workspace,
                                    size_t workspace_bytes) {
  if (!pool) return KV_ERR_INVALID_ARG;
  pool->last_launches = 0;
  if (B > 0 && (!out || !exp_tags || !abort_mask)) return KV_ERR_INVALID_ARG;
  DecodeArgs a;
  int kind = 0;
  const kv_status st =
      decode_prepare(pool, B, num_q_heads, q_tokens, q, page_table, max_pages_per_req, seq_lens,
                     nullptr, sm_scale, out, workspace, workspace_bytes, true, true, &a, &kind);
  if (st != KV_OK || B == 0) return st;
  a.exp_tags = exp_tags;
  a.abort_out = abort_mask;
  int n = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = a.self_plan ? cudaSuccess : launch_decode_plan(a, s, &n);
  if (e == cudaSuccess) e = launch_decode_split(a, kind, s, &n);
  if (e == cudaSuccess) e = launch_decode_combine(a, s, &n);
  pool->last_launches = n;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

size_t kv_decode_step_workspace_size(const kv_pool* pool, int32_t B, int32_t num_q_heads,
                                     int32_t q_tokens) {
  if (!pool || B < 0) return 0;
  DecodeConfig cfg;
  if (decode_config(pool, B, num_q_heads, q_tokens, &cfg) != KV_OK) return 0;
  const size_t dec = decode_ws_layout(pool->d, B, pool->d.num_kv_heads, cfg, nullptr, nullptr);
  return align256(dec) + release_ws_bytes(B);
}

kv_status kv_decode_step(kv_pool* pool, void* stream, int32_t B, int32_t num_q_heads,
                         int32_t q_tokens, const uint8_t* leave_mask, const void* k_new,
                         const void* v_new, const int32_t* new_indptr, int32_t max_new_per_req,
                         int32_t* page_table, uint32_t* exp_tags, int32_t max_pages_per_req,
                         int32_t* seq_lens, const void* q, float sm_scale, void* out,
                         uint8_t* abort_mask, int32_t flags, void* workspace,
                         size_t workspace_bytes) {
  if (!pool) return KV_ERR_INVALID_ARG;
  pool->last_launches = 0;
  const kv_pool_desc& d = pool->d;
  if (B < 0 || (flags & ~KV_STEP_REMOVE_ABORTED) != 0) return KV_ERR_INVALID_ARG;
  if (max_new_per_req < 0 || max_pages_per_req <= 0) return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!new_indptr || !page_table || !exp_tags || !seq_lens || !abort_mask)
    return KV_ERR_INVALID_ARG;
  if (max_new_per_req > 0) {
    if (!k_new || !aligned16(k_new)) return KV_ERR_INVALID_ARG;
    if (d.layout == KV_LAYOUT_GQA && (!v_new || !aligned16(v_new))) return KV_ERR_INVALID_ARG;
  }
  // attention arguments and the workspace, before anything is launched
  DecodeArgs da;
  int kind = 0;
  kv_status st = decode_prepare(pool, B, num_q_heads, q_tokens, q, page_table, max_pages_per_req,
                                seq_lens, abort_mask, sm_scale, out, workspace, workspace_bytes,
                                true, true, &da, &kind);
  if (st != KV_OK) return st;
  const size_t need = kv_decode_step_workspace_size(pool, B, num_q_heads, q_tokens);
  if (need == 0 || workspace_bytes < need) return KV_ERR_INVALID_ARG;
  const size_t dec = need - release_ws_bytes(B);
  long long* rel_ws = reinterpret_cast<long long*>(static_cast<uint8_t*>(workspace) + dec);

  ReleaseArgs ra;
  ra.d = d;
  ra.B = B;
  ra.max_pages = max_pages_per_req;
  ra.page_table = page_table;
  ra.exp_tags = exp_tags;
  ra.seq_lens = seq_lens;
  ra.offsets = rel_ws;
  VerifyArgs va;
  va.num_pages = d.num_pages;
  va.page_size = d.page_size;
  va.B = B;
  va.max_pages = max_pages_per_req;
  va.tags = d.tags;
  va.page_table = page_table;
  va.exp_tags = exp_tags;
  va.seq_lens = seq_lens;
  va.abort_mask = abort_mask;
  AppendArgs aa;
  aa.d = d;
  aa.B = B;
  aa.k_new = static_cast<const uint16_t*>(k_new);
  aa.v_new = static_cast<const uint16_t*>(v_new);
  aa.new_indptr = new_indptr;
  aa.max_new = max_new_per_req;
  aa.page_table = page_table;
  aa.exp_tags = exp_tags;
  aa.max_pages = max_pages_per_req;
  aa.seq_lens = seq_lens;
  aa.step_mask = abort_mask;
  aa.from_pool = false;
  aa.fuse_plan = true;  // the append's plan kernel also writes the attention plan
  da.self_plan = 0;     // ... so the split kernel reads it
  aa.plan = da;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int n = 0;
  cudaError_t e = cudaSuccess;
  if (leave_mask != nullptr) {
    ra.mask = leave_mask;
    ra.mask_bits = 0xFF;
    e = launch_release(ra, s, &n);
  }
  if (e == cudaSuccess) e = launch_verify(va, s, &n);
  if (e == cudaSuccess) e = launch_append(aa, s, &n);
  if (e == cudaSuccess) e = launch_decode_split(da, kind, s, &n);
  if (e == cudaSuccess) e = launch_decode_combine(da, s, &n);
  if (e == cudaSuccess && (flags & KV_STEP_REMOVE_ABORTED) != 0) {
    ra.mask = abort_mask;
    ra.mask_bits = KV_ABORT_TAG;
    e = launch_release(ra, s, &n);
  }
  pool->last_launches = n;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

const char* kv_status_string(kv_status s) {
  switch (s) {
    case KV_OK: return "KV_OK";
    case KV_ERR_INVALID_ARG: return "KV_ERR_INVALID_ARG";
    case KV_ERR_UNSUPPORTED: return "KV_ERR_UNSUPPORTED";
    case KV_ERR_CUDA: return "KV_ERR_CUDA";
    case KV_ERR_OUT_OF_PAGES: return "KV_ERR_OUT_OF_PAGES";
    case KV_ERR_BAD_PAGE_ID: return "KV_ERR_BAD_PAGE_ID";
    case KV_ERR_TIMEOUT: return "KV_ERR_TIMEOUT";
    case KV_ERR_INTERNAL: return "KV_ERR_INTERNAL";
    case KV_ERR_TAG_MISMATCH: return "KV_ERR_TAG_MISMATCH";
  }
  return "KV_ERR_UNKNOWN";
}

int32_t kv_last_launch_count(const kv_pool* pool) { return pool ? pool->last_launches : 0; }

}  // extern "C"

namespace kvfp8 {

cudaError_t launch_decode_split(const DecodeArgs& a, int kind, cudaStream_t s, int* launches) {
  if (kind == 2) return launch_latent_split(a, s, launches);
  return launch_gqa_split(a, kind, s, launches);
}

}  // namespace kvfp8
