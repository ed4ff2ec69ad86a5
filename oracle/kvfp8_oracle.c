/*
 * kvfp8_oracle.c -- CPU oracle for the paged FP8 KV cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded
 * statement of what the path computes.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg load it.  It shares no code, header,
 * table or helper with the CUDA library in paged_fp8_kv_append_gb300/csrc,
 * and the library never calls it.
 *
 * Sources.  "SFS" below is the Cloudflare post "Smaller, faster, safer:
 * running Kimi and GLM at scale":
 *   - section "Quantizing the KV cache": the cache is stored as FP8 e4m3
 *     instead of BF16 (half the bytes), and the FP8 attention kernel converts
 *     the values as it reads them;
 *   - section "Protecting a shared KV cache": each physical page carries a tag
 *     that changes whenever the page is reallocated; the server records which
 *     pages and tags each request expects; before decode reads the cache the
 *     mappings are checked, and a mismatch aborts the affected request.
 * The e4m3 format itself is the OCP "8-bit Floating Point Specification
 * (OFP8)", revision 1.0, E4M3 column: exponent bias 7, no infinities, one NaN
 * mantissa pattern (S.1111.111), largest finite 448.
 *
 * The pages give no algorithm for scales, rounding or tag updates.  The
 * readings used here (one fp32 scale per (page, kv-head) = amax/448, scale
 * frozen at the page's first write, tag += 1 on every allocation, ...) are
 * listed with their reasons in the repository's design notes and restated
 * next to each function.
 *
 * Layouts (the same byte layouts the library documents for its caller-owned
 * device buffers):
 *   GQA   k_cache[page][kv_head][slot][d]      (token-major inside a page)
 *         v_cache[page][kv_head][d][slot]      (dim-major inside a page)
 *         k_scale[page][kv_head], v_scale[page][kv_head]  fp32
 *   LATENT cache[page][slot][dk], scale[page]; V is the first dv dims of a row.
 *   Element size is 1 byte (e4m3) or 2 bytes (bf16, stored bit-for-bit).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math (no FMA
 * contraction, IEEE fp32 division, no flush-to-zero).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* status codes (same numeric meaning as the library's, restated here) */
#define OR_OK 0
#define OR_ERR_INVALID_ARG 1
#define OR_ERR_OUT_OF_PAGES 4
#define OR_ERR_BAD_PAGE_ID 5
#define OR_ERR_TAG_MISMATCH 8

/* ------------------------------------------------------------------------ */
/* OFP8 E4M3 codec                                                           */
/* ------------------------------------------------------------------------ */

/* Value of an e4m3 code: s = bit 7, E = bits 6..3, M = bits 2..0.
 * E = 15 and M = 7 is NaN.  E = 0 is subnormal: M * 2^-9.  Otherwise
 * (1 + M/8) * 2^(E-7).  (OFP8 rev 1.0, E4M3.) */
double or_e4m3_decode(uint32_t code) {
  code &= 0xFFu;
  int s = (int)(code >> 7);
  int E = (int)((code >> 3) & 15u);
  int M = (int)(code & 7u);
  double mag;
  if (E == 15 && M == 7) return NAN;
  if (E == 0)
    mag = ldexp((double)M, -9);
  else
    mag = ldexp(1.0 + (double)M / 8.0, E - 7);
  return s ? -mag : mag;
}

/* Round a non-negative double to the nearest integer, ties to even.  Used
 * only on values that are exact in double. */
static double rne_nonneg(double x) {
  double f = floor(x);
  double d = x - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* fp32 -> e4m3, round to nearest even with saturation to +-448 (the
 * "satfinite" behaviour).  NaN maps to the NaN code with the input's sign.
 * Every step is exact in double: |v| * 2^9 and the mantissa fraction of a
 * float are exact. */
uint32_t or_e4m3_encode(float v) {
  uint32_t sign = signbit(v) ? 0x80u : 0u;
  double a;
  if (isnan(v)) return sign | 0x7Fu;
  a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7Eu; /* saturate (also covers +-inf) */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: step 2^-9.  r == 8 is the smallest normal, whose
     * code is also 8 (E=1, M=0). */
    double r = rne_nonneg(a * 512.0);
    return sign | (uint32_t)r;
  } else {
    int e;
    double f = frexp(a, &e);     /* a = f * 2^e, f in [0.5, 1) */
    int ex = e - 1;              /* a = (2f) * 2^ex, 2f in [1, 2) */
    double m = rne_nonneg((2.0 * f - 1.0) * 8.0);
    if (m == 8.0) { /* mantissa carried into the exponent */
      m = 0.0;
      ex += 1;
    }
    /* a < 448 keeps the result at or below 0x7E (E = 15, M = 6) */
    return sign | ((uint32_t)(ex + 7) << 3) | (uint32_t)m;
  }
}

/* Encode a contiguous range of fp32 bit patterns [first, first + count).
 * Lets a test sweep the whole fp32 space without one foreign call per value. */
void or_e4m3_encode_bits_range(uint32_t first, uint32_t count, uint8_t* out) {
  uint32_t i;
  for (i = 0; i < count; ++i) {
    uint32_t bits = first + i;
    float v;
    memcpy(&v, &bits, 4);
    out[i] = (uint8_t)or_e4m3_encode(v);
  }
}

void or_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = (uint8_t)or_e4m3_encode(x[i]);
}

/* bf16 bit pattern -> fp32 (exact: bf16 is the top half of an fp32). */
static float bf16_to_f32(uint16_t b) {
  uint32_t bits = (uint32_t)b << 16;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}

/* Scale of a freshly written (page, kv-head) block: amax / 448 in IEEE fp32,
 * so that the largest magnitude lands on the largest e4m3 value.  amax == 0
 * (or an amax so small that the quotient underflows to 0) gives 1.0, so that
 * every code is +-0 and nothing divides by zero. */
float or_scale_from_amax(float amax) {
  float s = amax / 448.0f;
  return (s > 0.0f) ? s : 1.0f;
}

/* One element quantised with a given scale: e4m3(x / scale), fp32 division. */
uint32_t or_quantize(float x, float scale) {
  float q = x / scale;
  return or_e4m3_encode(q);
}

/* ------------------------------------------------------------------------ */
/* Page allocation and tag stamping                                          */
/* ------------------------------------------------------------------------ */

static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

/*
 * Bookkeeping of one append call, in request order (SFS, "Protecting a
 * shared KV cache": every physical page has a tag that changes whenever the
 * page is reallocated; the server records the pages and tags each request
 * expects).
 *
 * For request r with L = seq_lens[r] tokens and n = indptr[r+1]-indptr[r]
 * new rows, the new logical pages ceil(L/P) .. ceil((L+n)/P)-1 are popped in
 * order from free_list[free_head ...].  Each popped page p gets
 * tags[p] += 1 (mod 2^32); page_table[r][j] = p; exp_tags[r][j] = tags[p].
 *
 * Before a request's rows go into its partly filled last page (n > 0 and
 * L not a multiple of P), that page's recorded mapping is checked like a
 * read: page_table[r][L/P] must be a page id in [0, num_pages) whose tag is
 * still exp_tags[r][L/P]; a page reallocated since (its tag changed) is not
 * written.
 *
 * The call stops at the first request that cannot be served, and leaves
 * that request and every later one untouched:
 *   - n < 0, L < 0, n > max_new or L + n > max_pages * P  -> INVALID_ARG
 *   - the partly filled page's id is out of range         -> BAD_PAGE_ID
 *   - the partly filled page's tag differs                -> TAG_MISMATCH
 *   - not enough entries left in the free list             -> OUT_OF_PAGES
 *   - a popped entry is not a page id in [0, num_pages)    -> BAD_PAGE_ID
 * *stop_req receives the index of that request (B if every request was
 * served).  fresh[p] (optional, num_pages bytes) is set to 1 for every page
 * popped by this call.  Returns the status of the stopping request or OK.
 */
int or_alloc(int num_pages, int page_size, uint32_t* tags,
             const int32_t* free_list, int32_t* free_head, int B,
             const int32_t* new_indptr, int max_new, int32_t* page_table,
             uint32_t* exp_tags, int max_pages, int32_t* seq_lens,
             int32_t* stop_req, uint8_t* fresh) {
  int r;
  int64_t P = page_size;
  *stop_req = B;
  for (r = 0; r < B; ++r) {
    int64_t L = seq_lens[r];
    int64_t n = (int64_t)new_indptr[r + 1] - new_indptr[r];
    int64_t first, need, j;
    /* the new length must fit its page table and stay an int32 length */
    if (n < 0 || L < 0 || n > max_new || L + n > (int64_t)max_pages * P ||
        L + n > INT32_MAX) {
      *stop_req = r;
      return OR_ERR_INVALID_ARG;
    }
    if (n > 0 && L % P != 0) {
      int64_t jl = L / P;
      int32_t p = page_table[(int64_t)r * max_pages + jl];
      if (p < 0 || p >= num_pages) {
        *stop_req = r;
        return OR_ERR_BAD_PAGE_ID;
      }
      if (tags[p] != exp_tags[(int64_t)r * max_pages + jl]) {
        *stop_req = r;
        return OR_ERR_TAG_MISMATCH;
      }
    }
    first = ceil_div64(L, P);
    need = ceil_div64(L + n, P) - first;
    if ((int64_t)*free_head + need > num_pages) {
      *stop_req = r;
      return OR_ERR_OUT_OF_PAGES;
    }
    for (j = 0; j < need; ++j) {
      int32_t p = free_list[*free_head + j];
      if (p < 0 || p >= num_pages) {
        *stop_req = r;
        return OR_ERR_BAD_PAGE_ID;
      }
    }
    for (j = 0; j < need; ++j) {
      int32_t p = free_list[*free_head + j];
      tags[p] += 1u;
      page_table[(int64_t)r * max_pages + first + j] = p;
      exp_tags[(int64_t)r * max_pages + first + j] = tags[p];
      if (fresh) fresh[p] = 1;
    }
    *free_head += (int32_t)need;
    seq_lens[r] = (int32_t)(L + n);
  }
  return OR_OK;
}

/*
 * Release: the pages of finished requests go back to the pool (SFS,
 * "Protecting a shared KV cache": a page's tag changes whenever it is
 * reallocated, so once a released page is handed out again every mapping
 * still recorded for it is stale).
 *
 * Requests r < B with mask[r] != 0 (every request when mask is NULL) are
 * released, in request order.  Request r owns its first n_r = ceil(L_r / P)
 * page-table entries, L_r = seq_lens[r].  Nothing changes when
 *   - a released request has L_r < 0 or n_r > max_pages     -> INVALID_ARG
 *   - the total T = sum of n_r exceeds *free_head (more pages
 *     than the free list has handed out)                      -> INVALID_ARG.
 * Otherwise *free_head -= T and the pages, in (request, page) order, are
 * written to free_list[*free_head ...], so the next allocations pop them in
 * that order (the free list is used as a stack).  Their page-table entries
 * become -1, their expected tags 0, and seq_lens[r] = 0.  Page ids are
 * returned as recorded: an id outside [0, num_pages) is refused when an
 * append pops it.  Tags are not touched here; each page's tag changes when
 * it is popped again.
 */
int or_release(int page_size, int32_t* free_list, int32_t* free_head, int B,
               int32_t* page_table, uint32_t* exp_tags, int max_pages,
               int32_t* seq_lens, const uint8_t* mask) {
  int64_t P = page_size, total = 0, k = 0, j;
  int r;
  for (r = 0; r < B; ++r) {
    int64_t L = seq_lens[r], n;
    if (mask && !mask[r]) continue;
    if (L < 0) return OR_ERR_INVALID_ARG;
    n = ceil_div64(L, P);
    if (n > max_pages) return OR_ERR_INVALID_ARG;
    total += n;
  }
  if (total > *free_head) return OR_ERR_INVALID_ARG;
  *free_head -= (int32_t)total;
  for (r = 0; r < B; ++r) {
    int64_t n;
    if (mask && !mask[r]) continue;
    n = ceil_div64(seq_lens[r], P);
    for (j = 0; j < n; ++j) {
      free_list[*free_head + k++] = page_table[(int64_t)r * max_pages + j];
      page_table[(int64_t)r * max_pages + j] = -1;
      exp_tags[(int64_t)r * max_pages + j] = 0;
    }
    seq_lens[r] = 0;
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Append with quantise-on-write                                             */
/* ------------------------------------------------------------------------ */

/*
 * scale_mode 1 (re-quantise; the default mode 0 keeps a block's scale frozen
 * at its first write, and later rows saturate at +-448 * scale).  When the
 * rows an append writes into a partly filled (page, kv head, K|V) block need
 * a larger scale, s_new = or_scale_from_amax(amax of those rows) > s_old,
 * the block takes s_new and each code c already in it is re-encoded:
 * v = fp32(decode(c) * s_old), c' = encode(v / s_new) (fp32 division, e4m3
 * RNE with saturation), so those values are rounded a second time.  This
 * re-encodes n codes at codes[i * stride].
 */
static void requant_codes(uint8_t* codes, int64_t n, int64_t stride, float s_old,
                          float s_new) {
  int64_t i;
  for (i = 0; i < n; ++i) {
    float v = (float)or_e4m3_decode(codes[i * stride]) * s_old;
    codes[i * stride] = (uint8_t)or_quantize(v, s_new);
  }
}

/* byte offset of element (p, h, slot, d) in the GQA K cache / V cache */
static int64_t k_off(int64_t p, int64_t h, int64_t slot, int64_t d, int64_t H,
                     int64_t P, int64_t D) {
  return ((p * H + h) * P + slot) * D + d;
}
static int64_t v_off(int64_t p, int64_t h, int64_t slot, int64_t d, int64_t H,
                     int64_t P, int64_t D) {
  return ((p * H + h) * D + d) * P + slot;
}

/*
 * Append new K/V rows of a GQA pool (SFS, "Quantizing the KV cache": the
 * cache is held as FP8 e4m3, half the bytes of BF16).
 *
 *   k_new[row][kv_head][Dk], v_new[row][kv_head][Dv]  bf16 bit patterns;
 *   request r owns rows new_indptr[r] .. new_indptr[r+1]-1, in order.
 *
 * dtype 0 (e4m3): for every page popped in this call and every kv head, the
 * K scale is scale(amax) over the |k| of all rows this call writes into that
 * (page, head); the same, separately, for V.  A page that already held rows
 * (the request's partly filled last page) keeps the scale it was given when
 * it was first written: later rows are quantised with it and saturate at
 * +-448 * scale.  Each element is stored as e4m3(x / scale).
 * dtype 1 (bf16): the bf16 bits are stored unchanged; scales are not used.
 * Bookkeeping is or_alloc's; rows of requests at or after the stopping
 * request are not written.  Rows are written after all of the call's pops:
 * a partly filled page that those pops handed to a later request (its tag
 * changed in this call) is not written through the earlier, now stale,
 * mapping (SFS, "Protecting a shared KV cache": a reallocated page is not
 * used through a mapping recorded before).  Returns or_alloc's status.
 */
int or_append_gqa(int num_pages, int page_size, int num_kv_heads, int Dk,
                  int Dv, int dtype, uint8_t* k_cache, uint8_t* v_cache,
                  float* k_scale, float* v_scale, uint32_t* tags,
                  const int32_t* free_list, int32_t* free_head, int B,
                  const uint16_t* k_new, const uint16_t* v_new,
                  const int32_t* new_indptr, int max_new, int32_t* page_table,
                  uint32_t* exp_tags, int max_pages, int32_t* seq_lens,
                  int32_t* stop_req, int scale_mode) {
  int64_t P = page_size, H = num_kv_heads;
  int32_t* old_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
  uint8_t* fresh = (uint8_t*)calloc((size_t)num_pages, 1);
  int status, r;
  memcpy(old_len, seq_lens, sizeof(int32_t) * (size_t)B);
  status = or_alloc(num_pages, page_size, tags, free_list, free_head, B,
                    new_indptr, max_new, page_table, exp_tags, max_pages,
                    seq_lens, stop_req, fresh);
  for (r = 0; r < *stop_req; ++r) {
    int64_t L0 = old_len[r];
    int64_t row0 = new_indptr[r];
    int64_t n = (int64_t)new_indptr[r + 1] - row0;
    int64_t jp;
    if (n == 0) continue;
    /* every logical page this call touches: floor(L0/P) .. floor((L0+n-1)/P) */
    for (jp = L0 / P; jp <= (L0 + n - 1) / P; ++jp) {
      int64_t p = page_table[(int64_t)r * max_pages + jp];
      int64_t pos_lo = (jp * P > L0) ? jp * P : L0;
      int64_t pos_hi = ((jp + 1) * P < L0 + n) ? (jp + 1) * P : L0 + n;
      int64_t h, pos, d;
      if (jp * P < L0 && fresh[p]) continue; /* partly filled, re-allocated now */
      for (h = 0; h < H; ++h) {
        float ks = 1.0f, vs = 1.0f;
        if (dtype == 0) {
          if (fresh[p]) {
            float ka = 0.0f, va = 0.0f;
            for (pos = pos_lo; pos < pos_hi; ++pos) {
              int64_t row = row0 + (pos - L0);
              for (d = 0; d < Dk; ++d) {
                float x = fabsf(bf16_to_f32(k_new[(row * H + h) * Dk + d]));
                if (x > ka) ka = x;
              }
              for (d = 0; d < Dv; ++d) {
                float x = fabsf(bf16_to_f32(v_new[(row * H + h) * Dv + d]));
                if (x > va) va = x;
              }
            }
            k_scale[p * H + h] = or_scale_from_amax(ka);
            v_scale[p * H + h] = or_scale_from_amax(va);
          } else if (scale_mode == 1) {
            int64_t n_old = pos_lo - jp * P;  /* slots already written */
            float ka = 0.0f, va = 0.0f, kn, vn;
            for (pos = pos_lo; pos < pos_hi; ++pos) {
              int64_t row = row0 + (pos - L0);
              for (d = 0; d < Dk; ++d) {
                float x = fabsf(bf16_to_f32(k_new[(row * H + h) * Dk + d]));
                if (x > ka) ka = x;
              }
              for (d = 0; d < Dv; ++d) {
                float x = fabsf(bf16_to_f32(v_new[(row * H + h) * Dv + d]));
                if (x > va) va = x;
              }
            }
            kn = or_scale_from_amax(ka);
            vn = or_scale_from_amax(va);
            if (kn > k_scale[p * H + h]) {  /* K rows: Dk codes per slot */
              requant_codes(k_cache + k_off(p, h, 0, 0, H, P, Dk), n_old * Dk, 1,
                            k_scale[p * H + h], kn);
              k_scale[p * H + h] = kn;
            }
            if (vn > v_scale[p * H + h]) {  /* V: per dim, its slots are contiguous */
              for (d = 0; d < Dv; ++d)
                requant_codes(v_cache + v_off(p, h, 0, d, H, P, Dv), n_old, 1,
                              v_scale[p * H + h], vn);
              v_scale[p * H + h] = vn;
            }
          }
          ks = k_scale[p * H + h];
          vs = v_scale[p * H + h];
        }
        for (pos = pos_lo; pos < pos_hi; ++pos) {
          int64_t row = row0 + (pos - L0);
          int64_t slot = pos - jp * P;
          for (d = 0; d < Dk; ++d) {
            uint16_t b = k_new[(row * H + h) * Dk + d];
            int64_t o = k_off(p, h, slot, d, H, P, Dk);
            if (dtype == 0)
              k_cache[o] = (uint8_t)or_quantize(bf16_to_f32(b), ks);
            else
              memcpy(k_cache + 2 * o, &b, 2);
          }
          for (d = 0; d < Dv; ++d) {
            uint16_t b = v_new[(row * H + h) * Dv + d];
            int64_t o = v_off(p, h, slot, d, H, P, Dv);
            if (dtype == 0)
              v_cache[o] = (uint8_t)or_quantize(bf16_to_f32(b), vs);
            else
              memcpy(v_cache + 2 * o, &b, 2);
          }
        }
      }
    }
  }
  free(old_len);
  free(fresh);
  return status;
}

/*
 * Append to a latent (MLA-style) pool: one row of Dk dims per token; the
 * first Dv dims of the row double as V.  One fp32 scale per page, from the
 * amax over all Dk dims of every row this call writes into a fresh page;
 * frozen afterwards, as in or_append_gqa, which also states the rule for a
 * partly filled page re-allocated by the same call.  dtype 0 (e4m3): codes
 * as above.  dtype 1 (bf16, the prefill pool a handoff reads from): the
 * rows' bf16 bits are stored unchanged (cache holds 2-byte elements) and no
 * scale is used, as for the BF16 cache of or_append_gqa.
 */
int or_append_latent(int num_pages, int page_size, int Dk, int dtype, uint8_t* cache,
                     float* scale, uint32_t* tags, const int32_t* free_list,
                     int32_t* free_head, int B, const uint16_t* kv_new,
                     const int32_t* new_indptr, int max_new,
                     int32_t* page_table, uint32_t* exp_tags, int max_pages,
                     int32_t* seq_lens, int32_t* stop_req, int scale_mode) {
  int64_t P = page_size;
  int32_t* old_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
  uint8_t* fresh = (uint8_t*)calloc((size_t)num_pages, 1);
  int status, r;
  memcpy(old_len, seq_lens, sizeof(int32_t) * (size_t)B);
  status = or_alloc(num_pages, page_size, tags, free_list, free_head, B,
                    new_indptr, max_new, page_table, exp_tags, max_pages,
                    seq_lens, stop_req, fresh);
  for (r = 0; r < *stop_req; ++r) {
    int64_t L0 = old_len[r];
    int64_t row0 = new_indptr[r];
    int64_t n = (int64_t)new_indptr[r + 1] - row0;
    int64_t jp;
    if (n == 0) continue;
    for (jp = L0 / P; jp <= (L0 + n - 1) / P; ++jp) {
      int64_t p = page_table[(int64_t)r * max_pages + jp];
      int64_t pos_lo = (jp * P > L0) ? jp * P : L0;
      int64_t pos_hi = ((jp + 1) * P < L0 + n) ? (jp + 1) * P : L0 + n;
      int64_t pos, d;
      float s;
      if (jp * P < L0 && fresh[p]) continue; /* partly filled, re-allocated now */
      if (dtype == 1) {
        for (pos = pos_lo; pos < pos_hi; ++pos) {
          int64_t row = row0 + (pos - L0);
          int64_t slot = pos - jp * P;
          memcpy(cache + 2 * ((p * P + slot) * Dk), kv_new + row * Dk, 2 * (size_t)Dk);
        }
        continue;
      }
      if (fresh[p]) {
        float a = 0.0f;
        for (pos = pos_lo; pos < pos_hi; ++pos) {
          int64_t row = row0 + (pos - L0);
          for (d = 0; d < Dk; ++d) {
            float x = fabsf(bf16_to_f32(kv_new[row * Dk + d]));
            if (x > a) a = x;
          }
        }
        scale[p] = or_scale_from_amax(a);
      } else if (scale_mode == 1) {
        float a = 0.0f;
        for (pos = pos_lo; pos < pos_hi; ++pos) {
          int64_t row = row0 + (pos - L0);
          for (d = 0; d < Dk; ++d) {
            float x = fabsf(bf16_to_f32(kv_new[row * Dk + d]));
            if (x > a) a = x;
          }
        }
        if (or_scale_from_amax(a) > scale[p]) {  /* the rows already written */
          requant_codes(cache + p * P * Dk, (pos_lo - jp * P) * Dk, 1, scale[p],
                        or_scale_from_amax(a));
          scale[p] = or_scale_from_amax(a);
        }
      }
      s = scale[p];
      for (pos = pos_lo; pos < pos_hi; ++pos) {
        int64_t row = row0 + (pos - L0);
        int64_t slot = pos - jp * P;
        for (d = 0; d < Dk; ++d)
          cache[(p * P + slot) * Dk + d] =
              (uint8_t)or_quantize(bf16_to_f32(kv_new[row * Dk + d]), s);
      }
    }
  }
  free(old_len);
  free(fresh);
  return status;
}

/* ------------------------------------------------------------------------ */
/* Tag verification                                                          */
/* ------------------------------------------------------------------------ */

/*
 * SFS, "Protecting a shared KV cache": before decode reads the cache, each
 * request's recorded (page, tag) mappings are checked against the physical
 * tags, and a request with any mismatch is aborted.
 *
 * abort_mask[r] = 1 iff, for some j < ceil(L_r / P), page_table[r][j] is not
 * a page id in [0, num_pages) or tags[page_table[r][j]] != exp_tags[r][j].
 * A length that is negative or needs more than max_pages pages also aborts
 * (the mapping cannot be checked).  Otherwise 0.
 */
void or_verify(int num_pages, int page_size, const uint32_t* tags, int B,
               const int32_t* page_table, const uint32_t* exp_tags,
               int max_pages, const int32_t* seq_lens, uint8_t* abort_mask) {
  int r;
  for (r = 0; r < B; ++r) {
    int64_t L = seq_lens[r];
    int64_t n, j;
    uint8_t bad = 0;
    if (L < 0) {
      abort_mask[r] = 1;
      continue;
    }
    n = ceil_div64(L, page_size);
    if (n > max_pages) {
      abort_mask[r] = 1;
      continue;
    }
    for (j = 0; j < n; ++j) {
      int32_t p = page_table[(int64_t)r * max_pages + j];
      if (p < 0 || p >= num_pages) {
        bad = 1;
        break;
      }
      if (tags[p] != exp_tags[(int64_t)r * max_pages + j]) {
        bad = 1;
        break;
      }
    }
    abort_mask[r] = bad;
  }
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                 */
/* ------------------------------------------------------------------------ */

/* Dequantised cache element, exactly as the definition states it: the e4m3
 * value times its scale, rounded to fp32 (or the bf16 value), then widened. */
static double deq_e4m3(uint8_t code, float scale) {
  float v = (float)or_e4m3_decode(code) * scale; /* one fp32 rounding */
  return (double)v;
}
static double deq_bf16(const uint8_t* base, int64_t elem) {
  uint16_t b;
  memcpy(&b, base + 2 * elem, 2);
  return (double)bf16_to_f32(b);
}

/* Check the page ids a request needs; 1 if all are in range. */
static int pages_in_range(int num_pages, const int32_t* pt_row, int64_t n) {
  int64_t j;
  for (j = 0; j < n; ++j)
    if (pt_row[j] < 0 || pt_row[j] >= num_pages) return 0;
  return 1;
}

/*
 * Decode attention over a paged GQA cache, in fp64.  SFS, "Quantizing the KV
 * cache": the attention reads the FP8 cache and converts values as it reads
 * them; the BF16 cache is the baseline format.
 *
 * For request r (skipped when abort_mask[r] != 0: SFS "Protecting a shared KV
 * cache" -- an aborted request returns no data), query token i in [0, T) and
 * query head h, with kv head g = h / (Hq / Hkv):
 *   visible positions t = 0 .. L_r - T + i          (causal among the T
 *                                                    newest positions)
 *   k_t, v_t = dequantised cache rows of (page_table[r][t / P], g, t % P)
 *   s_t = (sum_d q_d k_{t,d}) * sm_scale            (sm_scale: the fp32
 *                                                    value, widened)
 *   w_t = exp(s_t - max s) / sum exp(s - max s)
 *   out[r][i][h][d] = sum_t w_t v_{t,d}
 * No visible position gives an all-zero row.  A request whose pages are not
 * all valid ids is not written either (written[r] = 0), as for an abort.
 * q is bf16 [B][T][Hq][Dk]; out is fp64 [B][T][Hq][Dv].
 */
void or_attn_gqa(int num_pages, int page_size, int num_kv_heads, int Dk,
                 int Dv, int dtype, const uint8_t* k_cache,
                 const uint8_t* v_cache, const float* k_scale,
                 const float* v_scale, int B, int Hq, int T,
                 const int32_t* page_table, int max_pages,
                 const int32_t* seq_lens, const uint8_t* abort_mask,
                 const uint16_t* q, float sm_scale, double* out,
                 uint8_t* written) {
  int64_t P = page_size, H = num_kv_heads;
  int64_t G = Hq / num_kv_heads;
  int r;
  for (r = 0; r < B; ++r) {
    int64_t L = seq_lens[r];
    const int32_t* pt = page_table + (int64_t)r * max_pages;
    int64_t i, h;
    written[r] = 0;
    if (abort_mask && abort_mask[r]) continue;
    if (L < 0 || ceil_div64(L, P) > max_pages) continue;
    if (!pages_in_range(num_pages, pt, ceil_div64(L, P))) continue;
    written[r] = 1;
    for (i = 0; i < T; ++i) {
      int64_t last = L - T + i; /* inclusive */
      for (h = 0; h < Hq; ++h) {
        int64_t g = h / G;
        const uint16_t* qr = q + ((((int64_t)r * T + i) * Hq) + h) * Dk;
        double* o = out + ((((int64_t)r * T + i) * Hq) + h) * Dv;
        double mx = -INFINITY, den = 0.0;
        double* s;
        int64_t t, d;
        for (d = 0; d < Dv; ++d) o[d] = 0.0;
        if (last < 0) continue;
        s = (double*)malloc(sizeof(double) * (size_t)(last + 1));
        for (t = 0; t <= last; ++t) {
          int64_t p = pt[t / P], slot = t % P;
          double acc = 0.0;
          for (d = 0; d < Dk; ++d) {
            int64_t e = k_off(p, g, slot, d, H, P, Dk);
            double kv = (dtype == 0) ? deq_e4m3(k_cache[e], k_scale[p * H + g])
                                     : deq_bf16(k_cache, e);
            acc += (double)bf16_to_f32(qr[d]) * kv;
          }
          s[t] = acc * (double)sm_scale;
          if (s[t] > mx) mx = s[t];
        }
        for (t = 0; t <= last; ++t) {
          int64_t p = pt[t / P], slot = t % P;
          double w = exp(s[t] - mx);
          den += w;
          for (d = 0; d < Dv; ++d) {
            int64_t e = v_off(p, g, slot, d, H, P, Dv);
            double vv = (dtype == 0) ? deq_e4m3(v_cache[e], v_scale[p * H + g])
                                     : deq_bf16(v_cache, e);
            o[d] += w * vv;
          }
        }
        for (d = 0; d < Dv; ++d) o[d] /= den;
        free(s);
      }
    }
  }
}

/*
 * Decode attention over a latent (MLA-style) pool, fp64: every query head
 * reads the same single cache row per token; scores use all Dk dims, values
 * the first Dv dims of the same dequantised row.  T query tokens per request
 * with the same causal rule as or_attn_gqa (the speculative-verify shape:
 * draft tokens scored in one pass).  q is bf16 [B][T][Hq][Dk]; out fp64
 * [B][T][Hq][Dv].  e4m3 cache with one scale per page.
 */
void or_attn_latent(int num_pages, int page_size, int Dk, int Dv,
                    const uint8_t* cache, const float* scale, int B, int Hq,
                    int T, const int32_t* page_table, int max_pages,
                    const int32_t* seq_lens, const uint8_t* abort_mask,
                    const uint16_t* q, float sm_scale, double* out,
                    uint8_t* written) {
  int64_t P = page_size;
  int r;
  for (r = 0; r < B; ++r) {
    int64_t L = seq_lens[r];
    const int32_t* pt = page_table + (int64_t)r * max_pages;
    int64_t i, h, t, d;
    double* kv = NULL; /* dequantised rows of this request, [L][Dk] */
    written[r] = 0;
    if (abort_mask && abort_mask[r]) continue;
    if (L < 0 || ceil_div64(L, P) > max_pages) continue;
    if (!pages_in_range(num_pages, pt, ceil_div64(L, P))) continue;
    written[r] = 1;
    kv = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * (size_t)Dk);
    for (t = 0; t < L; ++t) {
      int64_t p = pt[t / P], slot = t % P;
      for (d = 0; d < Dk; ++d)
        kv[t * Dk + d] = deq_e4m3(cache[(p * P + slot) * Dk + d], scale[p]);
    }
    for (i = 0; i < T; ++i) {
      int64_t last = L - T + i;
      for (h = 0; h < Hq; ++h) {
        const uint16_t* qr = q + ((((int64_t)r * T + i) * Hq) + h) * Dk;
        double* o = out + ((((int64_t)r * T + i) * Hq) + h) * Dv;
        double mx = -INFINITY, den = 0.0;
        double* s;
        for (d = 0; d < Dv; ++d) o[d] = 0.0;
        if (last < 0) continue;
        s = (double*)malloc(sizeof(double) * (size_t)(last + 1));
        for (t = 0; t <= last; ++t) {
          double acc = 0.0;
          for (d = 0; d < Dk; ++d)
            acc += (double)bf16_to_f32(qr[d]) * kv[t * Dk + d];
          s[t] = acc * (double)sm_scale;
          if (s[t] > mx) mx = s[t];
        }
        for (t = 0; t <= last; ++t) {
          double w = exp(s[t] - mx);
          den += w;
          for (d = 0; d < Dv; ++d) o[d] += w * kv[t * Dk + d];
        }
        for (d = 0; d < Dv; ++d) o[d] /= den;
        free(s);
      }
    }
    free(kv);
  }
}
