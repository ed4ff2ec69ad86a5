/*
 * kvfp8.h -- C ABI of the GB300 (sm_103a) paged FP8 KV cache decode library.
 *
 * The operations come from the Cloudflare post "Smaller, faster, safer:
 * running Kimi and GLM at scale" ("SFS" below):
 *   - section "Quantizing the KV cache": the decode KV cache is held as FP8
 *     e4m3 instead of BF16 (half the bytes, twice the resident context), and
 *     the FP8 attention kernel converts values as it reads them; BF16 stays
 *     available as the baseline cache format;
 *   - section "Protecting a shared KV cache": every physical page carries a
 *     tag that changes whenever the page is reallocated; the server records
 *     which pages and tags each request expects; before decode reads the
 *     cache the mappings are checked as a separate batched pass, and a request
 *     with any mismatch is aborted instead of returning data from the wrong
 *     page; the default deployment uses a no-op tracker.
 * The post gives no API, scale rule or kernel design.  The readings used
 * here: one fp32 scale per (page, kv-head) (per page for the latent layout),
 * scale = amax/448 over the rows a call writes into a fresh page, frozen at
 * that first write; e4m3 by round-to-nearest-even with saturation to +-448;
 * tag += 1 (mod 2^32) on every allocation; split-K decode with a separate
 * combine step.
 *
 * Conventions for every entry point:
 *   - All buffer arguments are DEVICE pointers owned by the caller (for
 *     example torch tensors); the library never allocates, frees or keeps
 *     them beyond the call.  The pool handle is host memory owned by the
 *     library (kv_pool_create / kv_pool_destroy) and holds no device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; no entry point synchronises
 *     the host with the device.
 *   - Argument errors are found on the host and returned synchronously
 *     (nothing is enqueued).  Errors the device finds (out of pages, a bad
 *     page id, a wait that timed out) are written into the pool's error word
 *     ctl[KV_CTL_ERROR] with first-error-wins semantics; the caller reads it
 *     when it chooses.  No kernel traps, asserts or spins without a bound.
 *   - Every page id read from a page table or free list is range-checked
 *     before use.
 *   - Integers are int32 unless stated; sizes are in elements unless stated.
 */
#ifndef KVFP8_H
#define KVFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = 1,   /* bad argument (host) or a request that does not fit its page table (device) */
  KV_ERR_UNSUPPORTED = 2,   /* valid but not implemented shape / dtype combination */
  KV_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute query) */
  KV_ERR_OUT_OF_PAGES = 4,  /* device: free list exhausted during an append */
  KV_ERR_BAD_PAGE_ID = 5,   /* device: a page id outside [0, num_pages) was met */
  KV_ERR_TIMEOUT = 6,       /* device: a bounded wait inside a kernel gave up */
  KV_ERR_INTERNAL = 7,      /* device: an internal consistency check failed (a library bug) */
  KV_ERR_TAG_MISMATCH = 8   /* device: append met a partly filled page whose tag changed */
} kv_status;

typedef enum { KV_DTYPE_E4M3 = 0, KV_DTYPE_BF16 = 1 } kv_dtype;

typedef enum {
  /* separate K and V; K rows token-major, V dim-major inside a page;
   * one fp32 scale per (page, kv-head) for K and one for V (e4m3) */
  KV_LAYOUT_GQA = 0,
  /* MLA-style latent cache: one row of head_dim_k values per token, the
   * first head_dim_v of which are V; one KV head; one fp32 scale per page
   * (e4m3).  A bf16 latent pool can be appended to and be the source of
   * kv_append_from_pool; attention needs an e4m3 latent pool. */
  KV_LAYOUT_LATENT = 1
} kv_layout;

/* How an append treats a partly filled e4m3 block (page, kv head, K|V; a
 * whole page for the latent layout) whose new rows need a larger scale. */
typedef enum {
  /* the scale stays as its first write set it; larger rows saturate at
   * +-448 * scale (the default) */
  KV_SCALE_FROZEN = 0,
  /* the block takes scale = amax/448 of the new rows and its codes already
   * written are re-encoded: code' = e4m3(fp32(decode(code) * old) / new),
   * rounding those values a second time */
  KV_SCALE_REQUANTIZE = 1
} kv_scale_mode;

/* kv_decode_step: abort-mask bits it writes, and its flags. */
enum {
  KV_ABORT_TAG = 1,          /* failed the page-tag check (stale or out-of-range mapping,
                                or a length its page table cannot hold) */
  KV_ABORT_UNSERVED = 2,     /* the step's append stopped at or before this request */
  KV_STEP_REMOVE_ABORTED = 1 /* flag: release the pages of KV_ABORT_TAG requests */
};

/* Slots of the pool's int32 control block (device memory, KV_CTL_WORDS
 * ints, caller-owned; zero it when creating a pool). */
enum {
  KV_CTL_FREE_HEAD = 0,    /* next unused position of free_list */
  KV_CTL_ERROR = 1,        /* first device-side error (kv_status), 0 = none */
  KV_CTL_APPEND_STOP = 2,  /* last append: first request not served (B if all were) */
  KV_CTL_WAIT_INFO = 3,    /* first timed-out wait: (cta << 12) | (warp << 7) | (barrier << 6) | stage;
                              barrier 0 = data-ready, 1 = slot-free; 0 = none */
  KV_CTL_WORDS = 4
};

/*
 * Pool descriptor.  Every pointer is caller-owned device memory.
 *
 * GQA layout (element = 1 byte for e4m3, 2 bytes for bf16):
 *   k_cache  [num_pages][num_kv_heads][page_size][head_dim_k]   token-major
 *   v_cache  [num_pages][num_kv_heads][head_dim_v][page_size]   dim-major
 *   k_scale, v_scale [num_pages][num_kv_heads] fp32 (e4m3 only; NULL for bf16)
 * LATENT layout (e4m3 only, num_kv_heads == 1):
 *   k_cache  [num_pages][page_size][head_dim_k]; v_cache NULL (V = first
 *   head_dim_v dims of each row); k_scale [num_pages]; v_scale NULL.
 * Shared:
 *   tags      [num_pages] uint32 -- physical page tags (SFS "Protecting a
 *             shared KV cache"); the library adds 1 on every allocation.
 *   free_list [num_pages] int32 -- page ids handed out in order from
 *             ctl[KV_CTL_FREE_HEAD]; entries must be distinct.
 *   ctl       [KV_CTL_WORDS] int32 control block (see above).
 * All base pointers must be 16-byte aligned.
 */
typedef struct {
  int32_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim_k;
  int32_t head_dim_v;
  int32_t dtype;   /* kv_dtype */
  int32_t layout;  /* kv_layout */
  void* k_cache;
  void* v_cache;
  float* k_scale;
  float* v_scale;
  uint32_t* tags;
  int32_t* free_list;
  int32_t* ctl;
  int32_t scale_mode;  /* kv_scale_mode (e4m3 pools; ignored for bf16) */
} kv_pool_desc;

typedef struct kv_pool kv_pool; /* opaque host handle */

/* Validate a descriptor and create a host handle that keeps a copy of it.
 * No device work and no CUDA call.  Returns KV_ERR_INVALID_ARG for a bad
 * descriptor, KV_ERR_UNSUPPORTED for a shape the kernels do not cover. */
kv_status kv_pool_create(const kv_pool_desc* desc, kv_pool** out);

/* Free the host handle (never the caller's device buffers). */
kv_status kv_pool_destroy(kv_pool* pool);

/*
 * Append new K/V rows and quantise them on write (SFS "Quantizing the KV
 * cache"); allocate pages and stamp tags (SFS "Protecting a shared KV cache").
 *
 *   B              number of requests.
 *   k_new          bf16 [total_new][num_kv_heads][head_dim_k]   (device)
 *   v_new          bf16 [total_new][num_kv_heads][head_dim_v]   (device;
 *                  NULL for LATENT, whose rows are k_new [total_new][head_dim_k])
 *   new_indptr     int32 [B+1] (device): request r appends rows
 *                  new_indptr[r] .. new_indptr[r+1]-1, in order.
 *   max_new_per_req host upper bound on any request's row count in this call
 *                  (sizes the launch; a request above it is rejected on the
 *                  device with KV_ERR_INVALID_ARG).
 *   page_table     int32 [B][max_pages_per_req] (device, in/out)
 *   exp_tags       uint32 [B][max_pages_per_req] (device, in/out): the tag each
 *                  mapped page is expected to carry.
 *   seq_lens       int32 [B] (device, in/out): tokens already cached.
 *
 * Requests are served in index order.  For request r with L tokens and n new
 * rows, logical pages ceil(L/P) .. ceil((L+n)/P)-1 are popped from the free
 * list, each popped page's tag is incremented, and page_table / exp_tags /
 * seq_lens are updated.  e4m3: every (fresh page, kv-head) gets
 * scale = amax/448 (IEEE fp32; 1.0 if that is 0) from the rows this call
 * writes into it, separately for K and V; a partly filled page keeps its
 * scale; each element becomes e4m3_rne_satfinite(x / scale).  bf16: the bits
 * are copied.  Before rows go into a request's partly filled last page (n > 0
 * and L not a multiple of P) that mapping is checked like a read: the page
 * id must be in range and its tag must still be the expected one, so a page
 * reallocated since is never written.  The first request that cannot be
 * served (free list exhausted: KV_ERR_OUT_OF_PAGES; bad free-list entry or
 * out-of-range partly filled page: KV_ERR_BAD_PAGE_ID; partly filled page
 * with a changed tag: KV_ERR_TAG_MISMATCH; too many rows for max_new_per_req
 * or for its page table, or a new length past 2^31 - 1: KV_ERR_INVALID_ARG) and every later request are left
 * untouched; its index goes to ctl[KV_CTL_APPEND_STOP] and the code to
 * ctl[KV_CTL_ERROR].  Two kernel launches.
 */
kv_status kv_append_quantize(kv_pool* pool, void* stream, int32_t B,
                             const void* k_new, const void* v_new,
                             const int32_t* new_indptr, int32_t max_new_per_req,
                             int32_t* page_table, uint32_t* exp_tags,
                             int32_t max_pages_per_req, int32_t* seq_lens);

/*
 * Prefill-to-decode handoff without a gather copy (SFS "Quantizing the KV
 * cache": prefill keeps a BF16 cache, decode reads an FP8 one).  For each
 * request r in index order, the first src_seq_lens[r] rows of request r in
 * the bf16 pool `src` -- read through src_page_table (int32
 * [B][src_max_pages_per_req], device) -- are appended to request r of
 * `pool` exactly as kv_append_quantize would append the same rows given as
 * k_new / v_new (page pops, tag stamps, per-(page, kv head) scales, codes;
 * bf16 destinations copy the bits).
 *   src          a pool with dtype KV_DTYPE_BF16 and the same layout, kv heads,
 *                head dims and page size as `pool` (else KV_ERR_INVALID_ARG);
 *                read only.
 *   src_seq_lens int32 [B] (device): rows to hand off per request (0: none).
 *   page_table, exp_tags, max_pages_per_req, seq_lens: `pool`'s, as for
 *                kv_append_quantize.
 * A request with rows to hand off must be empty in `pool` (seq_lens 0) and
 * its rows must fit src_page_table; otherwise it and every later request are
 * left untouched (KV_ERR_INVALID_ARG in ctl, stop index in
 * ctl[KV_CTL_APPEND_STOP]), like the other stops of kv_append_quantize.  A
 * source page id outside `src` sets KV_ERR_BAD_PAGE_ID and the rows of that
 * page are not written.  Shapes outside the bulk append kernels' limits
 * (GQA: page_size * head_dim <= 2048; latent: page_size <= 64) and batches
 * of more than 16,384 requests return KV_ERR_UNSUPPORTED.  Two kernel
 * launches; nothing is allocated.
 */
kv_status kv_append_from_pool(kv_pool* pool, void* stream, int32_t B, const kv_pool* src,
                              const int32_t* src_page_table, int32_t src_max_pages_per_req,
                              const int32_t* src_seq_lens, int32_t* page_table,
                              uint32_t* exp_tags, int32_t max_pages_per_req, int32_t* seq_lens);

/*
 * Batched page-tag integrity check (SFS "Protecting a shared KV cache"; run
 * as its own pass before attention, not fused into it).
 *
 *   abort_mask  uint8 [B] (device, out): 1 iff some j < ceil(seq_lens[r]/P)
 *               has page_table[r][j] outside [0, num_pages) or
 *               tags[page_table[r][j]] != exp_tags[r][j]; also 1 for a
 *               negative length or one that needs more than
 *               max_pages_per_req pages; else 0.
 * One kernel launch; reads only page tables, expected tags and the tag array.
 */
kv_status kv_verify_tags(kv_pool* pool, void* stream, int32_t B,
                         const int32_t* page_table, const uint32_t* exp_tags,
                         int32_t max_pages_per_req, const int32_t* seq_lens,
                         uint8_t* abort_mask);

/* Bytes of device workspace kv_release_pages needs for B requests (the
 * per-request offsets of the released pages). */
size_t kv_release_workspace_size(int32_t B);

/*
 * Return the pages of finished requests to the pool (SFS "Protecting a
 * shared KV cache": a page's tag changes whenever it is reallocated, so once
 * a released page is handed out again every mapping still recorded for it
 * fails the tag check).  No counterpart in the pages beyond that lifecycle;
 * the free list is used as a stack.
 *
 *   page_table, exp_tags  [B][max_pages_per_req] (device, in/out)
 *   seq_lens              int32 [B] (device, in/out)
 *   release_mask          uint8 [B] (device): release request r iff nonzero;
 *                         NULL releases every request.
 *   workspace             device, >= kv_release_workspace_size(B) bytes,
 *                         16-byte aligned, caller-owned scratch.
 *
 * Request r owns its first ceil(seq_lens[r]/P) page-table entries.  With T
 * the total over the released requests, the free head moves down by T and
 * the released pages, in (request, page) order, are written to
 * free_list[head ...], so the next appends pop them in that order and bump
 * their tags.  Their page-table entries become -1, their expected tags 0 and
 * their seq_lens 0.  Page ids are returned as recorded; an id outside
 * [0, num_pages) is refused later, when an append pops it.  Nothing changes,
 * and ctl[KV_CTL_ERROR] gets KV_ERR_INVALID_ARG, when a released request has
 * a negative length or one needing more than max_pages_per_req pages, or T
 * exceeds the free head (more pages than the pool has handed out).  Tags are
 * not touched.  Two kernel launches.
 */
kv_status kv_release_pages(kv_pool* pool, void* stream, int32_t B, int32_t* page_table,
                           uint32_t* exp_tags, int32_t max_pages_per_req, int32_t* seq_lens,
                           const uint8_t* release_mask, void* workspace,
                           size_t workspace_bytes);

/* Bytes of device workspace paged_decode_attn needs for this batch shape on
 * the current device (0 for invalid arguments or when no device is
 * visible).  Workspace holds the split-K partials and the batch plan. */
size_t paged_decode_workspace_size(const kv_pool* pool, int32_t B,
                                   int32_t num_q_heads, int32_t q_tokens);

/*
 * Paged decode attention (SFS "Quantizing the KV cache": the FP8 kernel
 * dequantises while reading; BF16 is the baseline cache).
 *
 *   q           bf16 [B][q_tokens][num_q_heads][head_dim_k] (device)
 *   page_table  int32 [B][max_pages_per_req], seq_lens int32 [B] (device);
 *               seq_lens count every cached token, including the q_tokens
 *               newest ones whose K/V were appended for this step.
 *   abort_mask  uint8 [B] from kv_verify_tags, or NULL (the no-op tracker).
 *               Aborted requests read no page and their output rows are
 *               left untouched (SFS: an aborted request returns no data).
 *   sm_scale    softmax scale applied to q.k (fp32).
 *   out         bf16 [B][q_tokens][num_q_heads][head_dim_v] (device)
 *   workspace   device scratch of at least paged_decode_workspace_size bytes,
 *               256-byte aligned; contents need not be initialised.
 *
 * Query token i of request r and query head h (kv head h / (Hq/Hkv); the
 * latent layout has one kv head) attends to positions 0 .. L_r - q_tokens + i;
 * a row with no visible position is written as zeros.  A request whose pages
 * include an id outside [0, num_pages) is not written and sets
 * KV_ERR_BAD_PAGE_ID.  Split-K: pages are spread evenly over a persistent grid
 * sized to the device, partials (fp32 o, running max, sum) go to the
 * workspace, and a combine kernel merges them.  Output is bf16 (RNE).
 * e4m3 pools multiply in f16 (every e4m3 code is exact in f16): each query
 * row is scaled by an exact power of two that puts its largest magnitude in
 * [2^15, 2^16) before it is narrowed to f16, and the row's scores take the
 * inverse factor, so any finite bf16 query is accepted; bf16 pools keep the
 * query in bf16.
 * Supported: GQA with head_dim 128, page_size 16 and up to 64 query rows per
 * kv head, q_tokens * (Hq/Hkv) <= 64 (e4m3 and bf16); LATENT
 * with head_dim_k 576, head_dim_v 512, page_size 64, e4m3.  Other shapes
 * return KV_ERR_UNSUPPORTED.
 */
kv_status paged_decode_attn(kv_pool* pool, void* stream, int32_t B,
                            int32_t num_q_heads, int32_t q_tokens,
                            const void* q, const int32_t* page_table,
                            int32_t max_pages_per_req, const int32_t* seq_lens,
                            const uint8_t* abort_mask, float sm_scale,
                            void* out, void* workspace, size_t workspace_bytes);

/*
 * paged_decode_attn with the page-tag check fused into the page reads (SFS
 * "Protecting a shared KV cache": each request's expected (page, tag) list
 * is compared with the physical tags before decode reads the cache, and a
 * request that fails is aborted and returns no data).  Instead of a separate
 * kv_verify_tags pass, the thread that fetches a page compares tags[p] with
 * exp_tags[r][j] (uint32 [B][max_pages_per_req], device) first and fetches
 * only a page that matches; the combine step then writes abort_mask
 * (uint8 [B], device, out): 1 for a request that met a stale tag or a page id
 * outside [0, num_pages) or whose length is invalid (as kv_verify_tags
 * decides it), else 0.  An aborted request's output rows are left untouched.
 * Unlike the separate pass, the pages of an aborted request whose tags do
 * match may still be read (their data never reaches an output); a page whose
 * tag does not match is never read.  Other arguments, results and errors are
 * those of paged_decode_attn (a page id out of range also sets
 * KV_ERR_BAD_PAGE_ID); the same workspace size applies.
 */
kv_status paged_decode_attn_checked(kv_pool* pool, void* stream, int32_t B,
                                    int32_t num_q_heads, int32_t q_tokens,
                                    const void* q, const int32_t* page_table,
                                    const uint32_t* exp_tags, int32_t max_pages_per_req,
                                    const int32_t* seq_lens, float sm_scale, void* out,
                                    uint8_t* abort_mask, void* workspace,
                                    size_t workspace_bytes);

/* The two phases of paged_decode_attn, for callers that schedule or time
 * them separately.  _split plans the batch (inside the split kernel for
 * batches of up to 1023 requests on GQA pools, else in a plan launch) and
 * writes the partials; _combine merges them into `out` (one launch).
 * Calling _split then _combine with the same arguments and workspace is
 * exactly paged_decode_attn. */
kv_status paged_decode_attn_split(kv_pool* pool, void* stream, int32_t B,
                                  int32_t num_q_heads, int32_t q_tokens,
                                  const void* q, const int32_t* page_table,
                                  int32_t max_pages_per_req,
                                  const int32_t* seq_lens,
                                  const uint8_t* abort_mask, float sm_scale,
                                  void* workspace, size_t workspace_bytes);
kv_status paged_decode_attn_combine(kv_pool* pool, void* stream, int32_t B,
                                    int32_t num_q_heads, int32_t q_tokens,
                                    const uint8_t* abort_mask, void* out,
                                    void* workspace, size_t workspace_bytes);

/*
 * paged_decode_attn without a caller-provided workspace.  No counterpart in
 * the post: this entry point exists for callers that cannot allocate device
 * memory -- a serving runtime (or a plug-in inside one) that owns all of the
 * GPU's memory and hands out no scratch buffers, and so can neither call
 * cudaMalloc nor pass `workspace`.  Arguments and results are exactly those of
 * paged_decode_attn; the caller still provides q, page tables, lengths and
 * `out`.
 *   - Scratch comes from one fixed 32 MiB device array compiled into the
 *     library (held by every GPU that loads the library until the process
 *     exits).  A batch whose workspace (paged_decode_workspace_size) exceeds
 *     32 MiB is rejected with KV_ERR_UNSUPPORTED before anything is enqueued.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 *   - A call made outside stream capture looks up the array's device
 *     address (cudaGetSymbolAddress) with the current device, so the address
 *     stays right after a device reset.  A call made while its stream is
 *     being captured reuses the address that the last uncaptured call on the
 *     same device found; make the first call on a device before any stream
 *     capture on it (the first lookup may load the library's device code).
 *   - All calls share the one array and nothing in it needs clearing between
 *     calls (each call rewrites what it reads), but calls that overlap on the
 *     GPU (concurrent streams) race on it: serialise them.
 */
kv_status paged_decode_attn_noalloc(kv_pool* pool, void* stream, int32_t B,
                                    int32_t num_q_heads, int32_t q_tokens, const void* q,
                                    const int32_t* page_table, int32_t max_pages_per_req,
                                    const int32_t* seq_lens, const uint8_t* abort_mask,
                                    float sm_scale, void* out);

/* Human-readable name of a status code (static string). */
const char* kv_status_string(kv_status status);

/* Number of kernel launches the last call on this pool enqueued (for
 * launch accounting by benchmarks). */
int32_t kv_last_launch_count(const kv_pool* pool);

/* Bytes of device workspace kv_decode_step needs (0 for invalid arguments
 * or when no device is visible). */
size_t kv_decode_step_workspace_size(const kv_pool* pool, int32_t B,
                                     int32_t num_q_heads, int32_t q_tokens);

/*
 * One continuous-batching decode step over B request slots, in one call
 * with no host synchronisation (SFS "Protecting a shared KV cache": the
 * page-tag check stays on for every step while requests join and leave, and
 * a request whose pages were reallocated is aborted and returns no data).
 * A slot whose seq_lens entry is 0 is empty.  The call runs, on `stream`:
 *
 *   1. leave_mask (uint8 [B], device, or NULL): requests with a nonzero
 *      entry release their pages, as kv_release_pages does;
 *   2. the tag check of kv_verify_tags over the mappings that exist now,
 *      writing abort_mask (uint8 [B], device, out): KV_ABORT_TAG or 0;
 *   3. the append of kv_append_quantize (k_new, v_new, new_indptr,
 *      max_new_per_req: a joining request's prompt rows, a decoding one's
 *      new rows), in which a request with KV_ABORT_TAG appends nothing (its
 *      rows are skipped; the request is still checked for a negative length
 *      or rows beyond its page table); every request at or after the index
 *      at which the append stopped gets KV_ABORT_UNSERVED;
 *   4. paged_decode_attn over q, for every request whose abort_mask is 0;
 *      the others' output rows are left untouched;
 *   5. with flags & KV_STEP_REMOVE_ABORTED, requests with KV_ABORT_TAG
 *      release their pages (seq_lens 0: the slot is empty again).
 *      KV_ABORT_UNSERVED requests keep their state.
 *
 * The check runs before the append: every mapping the append adds is a page
 * it has just popped and stamped, and rows go into a partly filled page only
 * after that page passed the check, so attention reads only checked pages
 * and a stale request costs no other request its step.  Arguments are those
 * of the calls above (same meaning, layout and ownership); workspace is
 * device scratch of at least kv_decode_step_workspace_size bytes, 256-byte
 * aligned.  Every argument is checked before anything is launched
 * (KV_ERR_INVALID_ARG / KV_ERR_UNSUPPORTED, nothing launched); device-found
 * errors go to ctl[KV_CTL_ERROR], first error wins.  Five kernel launches
 * (the append's plan kernel also writes the attention plan), plus two for
 * each release phase that runs.
 */
kv_status kv_decode_step(kv_pool* pool, void* stream, int32_t B, int32_t num_q_heads,
                         int32_t q_tokens, const uint8_t* leave_mask, const void* k_new,
                         const void* v_new, const int32_t* new_indptr,
                         int32_t max_new_per_req, int32_t* page_table, uint32_t* exp_tags,
                         int32_t max_pages_per_req, int32_t* seq_lens, const void* q,
                         float sm_scale, void* out, uint8_t* abort_mask, int32_t flags,
                         void* workspace, size_t workspace_bytes);

#ifdef __cplusplus
}
#endif

#endif /* KVFP8_H */
