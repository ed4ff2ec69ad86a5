// internal.h -- host-side declarations shared by the C-ABI layer (api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvfp8.h"

struct kv_pool {
  kv_pool_desc d;
  int32_t last_launches;
};

namespace kvfp8 {

// ---- verify -------------------------------------------------------------
struct VerifyArgs {
  int32_t num_pages, page_size, B, max_pages;
  const uint32_t* tags;
  const int32_t* page_table;
  const uint32_t* exp_tags;
  const int32_t* seq_lens;
  uint8_t* abort_mask;
};
cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s, int* launches);

// ---- release ------------------------------------------------------------
struct ReleaseArgs {
  kv_pool_desc d;
  int32_t B, max_pages;
  int32_t* page_table;
  uint32_t* exp_tags;
  int32_t* seq_lens;
  const uint8_t* mask;   // NULL: every request
  uint8_t mask_bits;     // with a mask: release r iff mask[r] & mask_bits
  long long* offsets;    // workspace: [B+1] released-page prefix, then [1] base, [1] ok
};
size_t release_ws_bytes(int B);
cudaError_t launch_release(const ReleaseArgs& a, cudaStream_t s, int* launches);

// ---- decode -------------------------------------------------------------
// Workspace carve-up (all offsets 256-byte aligned).
struct DecodeWs {
  int32_t* pfx;       // [B+1] exclusive prefix of pages per request (0 if skipped)
  uint8_t* rq_skip;   // [B] 1: request gets no output (aborted / invalid length)
  // [slots][Hs][R8][2]  running max (log2 domain) and sum; a sum of -1 marks a
  // piece that met a page it must not read (id out of range, or, with the
  // fused tag check, a stale tag): its request gets no output
  float* ml_part;
  float* o_part;      // [slots][Hs][R8][Dv] unnormalised partial outputs
  size_t bytes;
};

struct DecodeArgs {
  kv_pool_desc d;
  int32_t B, Hq, T, G, R;  // R = T*G query rows per kv head (latent: T*Hq)
  const uint16_t* q;       // bf16 bits [B][T][Hq][Dk]
  const int32_t* page_table;
  int32_t max_pages;
  const int32_t* seq_lens;
  const uint8_t* abort_mask;
  float sm_scale_log2;  // sm_scale * log2(e)
  uint16_t* out;        // bf16 bits [B][T][Hq][Dv]
  int32_t grid;         // CTAs of the split kernel
  int32_t R8;           // rows per (partial slot, head) (R rounded up)
  int32_t Hs;           // kv heads per unit of work (a head group)
  int32_t HG;           // segments per request: head groups (GQA) or 64-row blocks (latent)
  int32_t stages;       // ring stages of the split kernel
  int32_t unit_tokens;  // tokens per unit of work (a page)
  // the split kernel builds the batch plan itself (B + 1 <= its shared-memory
  // prefix cache) instead of reading the plan kernel's; its CTA 0 writes the
  // plan to the workspace for the combine
  int32_t self_plan;
  // fused tag check (NULL: none): the split reads a page only after its tag
  // matched exp_tags[r][j]; the combine writes abort_out[r] (1: a stale tag,
  // an out-of-range page id or an invalid length; 0 otherwise)
  const uint32_t* exp_tags;
  uint8_t* abort_out;
  DecodeWs ws;
};

// ---- append -------------------------------------------------------------
struct AppendArgs {
  kv_pool_desc d;
  int32_t B;
  const uint16_t* k_new;  // bf16 bits
  const uint16_t* v_new;
  const int32_t* new_indptr;
  int32_t max_new;
  int32_t* page_table;
  uint32_t* exp_tags;
  int32_t max_pages;
  int32_t* seq_lens;
  // NULL, or [B] (the step driver's abort mask): a request with a nonzero
  // entry appends no rows; the plan then sets KV_ABORT_UNSERVED on every
  // request at or after its stop index.
  uint8_t* step_mask;
  // with fuse_plan the plan kernel also writes the attention plan of `plan`
  // (the one-call step: the lengths and abort bits it leaves are final)
  bool fuse_plan;
  DecodeArgs plan;
  // pool-to-pool handoff: request r's rows are the first src_lens[r] rows of
  // request r in the bf16 pool `src`, read through src_page_table (then
  // k_new, v_new and new_indptr are unused and every request appends into an
  // empty destination, so that destination page j takes source page j)
  bool from_pool;
  kv_pool_desc src;
  const int32_t* src_page_table;
  int32_t src_max_pages;
  const int32_t* src_lens;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s, int* launches);
// whether a pool-to-pool handoff of B requests into a pool of this shape fits
// the bulk append kernels
bool append_handoff_supported(const kv_pool_desc& d, int B, int src_max_pages);

// Kernel configuration chosen for a pool (shape checks + grid).
struct DecodeConfig {
  int kind;         // 0 = GQA e4m3, 1 = GQA bf16, 2 = latent e4m3, 3 / 4 = GQA e4m3 / bf16 > 8 rows
  int self_plan;    // the split kernel plans the batch itself (no plan launch)
  int grid;         // split-kernel CTAs
  int R8;           // partial rows per (slot, head)
  int Hs;           // kv heads per unit of work
  int HG;           // segments per request
  int stages;       // ring stages
  int unit_tokens;  // tokens per unit of work
};

// Ring bytes and stage limit of the GQA split kernel (for the host-side
// choice of heads per unit and ring depth).
int gqa_ring_bytes(int kind);
int gqa_max_stages();
int gqa_consumer_warps(int kind);
int gqa_self_plan_max_batch();
bool gqa_kind_self_plans(int kind);

kv_status decode_config(const kv_pool* pool, int B, int Hq, int T, DecodeConfig* cfg);
size_t decode_ws_layout(const kv_pool_desc& d, int B, int Hkv, const DecodeConfig& cfg,
                        void* base, DecodeWs* ws);

cudaError_t launch_decode_plan(const DecodeArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_decode_split(const DecodeArgs& a, int kind, cudaStream_t s, int* launches);
cudaError_t launch_gqa_split(const DecodeArgs& a, int kind, cudaStream_t s, int* launches);
cudaError_t launch_latent_split(const DecodeArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t s, int* launches);

// Occupancy-derived CTAs per SM for the split kernels (cached per device).
int gqa_split_ctas_per_sm(int kind);
int latent_split_ctas_per_sm();
int latent_unit_tokens();
int latent_row_block();

}  // namespace kvfp8
