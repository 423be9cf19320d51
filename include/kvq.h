/*
 * kvq.h -- C ABI of the GB300 (sm_103a) low-bit KV-cache library.
 *
 * Write side: asymmetric min-max quantization of the KV cache
 *   - KIVI keys per channel over groups of G tokens and values per token over
 *     groups of Gv channels, 2-bit codes with fp16 (scale, zero)
 *     (KIVI, zenmind.me summary, section 3.3 and section 4 steps 2-3;
 *      the affine formula of Kitty, Observation 1);
 *   - Kitty pages: top-K channel precision boost (Eq. 2 score), 4-bit boosted
 *     key channels stored as two dense 2-bit planes plus a boost index, 2-bit
 *     per-token value pages (Kitty summary, "The Channel-Wise Precision Boost
 *     Mechanism", "Page-Centric Memory Layout and Dense-Sparse Decomposition");
 *   - WitCert INT8 with subtractive Philox4x32-10 dither and per-256-token,
 *     per-channel fp16 scales amax/126.5 (WitCert, arxiv 2607.28699, sec. 6),
 *     and its token-granular form for a slot-paged pool: one fp16 scale per
 *     token and group of Gc channels, dither keyed by the slot (WitCert, the
 *     SGLang storage subsection of sec. 6.2).
 * Read side: split-KV flash-decoding attention that dequantizes codes in
 * registers, concatenates the fp16 residual / sink / buffer segments, and
 * merges the splits by log-sum-exp (WitCert sec. 6.2.2 two-stage structure;
 * KIVI Eq. 3; Kitty "Lightweight Attention Execution Pipeline").
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *     aligned (KVQ_ERR_MISALIGNED otherwise).  The library allocates no
 *     memory, never synchronizes the host, and enqueues its kernels on the
 *     given stream (0 = legacy default stream).  Calls are graph-capturable.
 *   - Argument errors are detected on the host before anything is launched;
 *     nothing is launched when a call returns an error.  Launch failures
 *     return KVQ_ERR_CUDA.  No device code traps or asserts; a bounded wait
 *     that expires inside a kernel records KVQ_DEVICE_ERR_* in a device flag
 *     that kvq_get_device_error() reads.
 *   - fp16 = IEEE binary16 stored as uint16; "fp16x2 (s, z)" = a pair of
 *     fp16 values, scale first.
 *   - head_dim must be 128 (KVQ_ERR_UNSUPPORTED otherwise).
 *
 * Byte layouts (D = 128):
 *   KIVI key group (G tokens, G % 32 == 0): G*D/4 bytes made of G/32 tiles of
 *     1024 bytes.  Within a tile write token t = q + 8p (q = t%8) and
 *     channel c = 16k + cc, cc = 2r + e + 8h (r = (cc%8)/2, e = cc%2,
 *     h = cc/8).  The 2-bit code sits in bits 2p of the byte at
 *       (t/32)*1024 + (k/4)*512 + (4q + r)*16 + (k%4)*4 + (e + 2h)
 *     so a byte holds tokens q, q+8, q+16, q+24 of one channel, and lane
 *     4q + r of a warp finds all of its tokens {q + 8p} x channels
 *     {16k + 2r + {0,1,8,9}} in the 16-byte chunks lane and lane + 32.
 *     Parameters: 256 fp16 per group, the 128 scales then the 128 zeros,
 *     channel c at index ((k/2)*4 + r)*8 + (k%2)*4 + e + 2h of each half.
 *     At 4 bits (KIVI-4) a tile is 2048 bytes, two planes of 1024: token
 *     q + 8p goes to plane p/2, at bits 4*(p%2) of the byte that the 2-bit
 *     layout above gives inside the plane (t%8 in place of t).
 *   KIVI value codes, token-major: D*b/8 bytes per token for b-bit codes,
 *     channel c in bits b*(c % (8/b)) of byte c/(8/b).  Parameters: fp16x2
 *     (s, z) [D/Gv] per token.
 *   KIVI value tiles: a config whose query heads decode on the grouped-query
 *     tensor-core kernel (2 <= n_q_heads / n_kv_heads <= 4, or an even ratio
 *     up to 8; at 4-bit widths with Gv = 32) stores its value codes in
 *     32-token tiles instead (the tile of token t is tile t/32 of its (batch
 *     row, kv head) or page record), in the order of the A operands of the
 *     tensor-core value products.  2 bits, tiles of 1024 bytes: with
 *     t % 32 = 16kv + 4i + r and c = 32g + 4q + p, the code sits in bits 2p
 *     of byte (t/32)*1024 + kv*512 + (4q + r)*16 + 4g + i (a byte holds four
 *     channels of one token; lane 4q + r finds byte 8g + q of the tokens r,
 *     r+4, r+8, r+12 of each 16-token half, g = 0..3, in one 16-byte chunk).
 *     4 bits, tiles of 2048 bytes: with t % 32 = 16kv + 8w + 4s + r and
 *     c % 64 = 16m + 8h + q, the code sits in nibble c/64 of byte
 *     (t/32)*2048 + kv*1024 + (4q + r)*32 + (2m + w)*4 + 2h + s (a byte holds
 *     channels c % 64 and c % 64 + 64 of one token).
 *   Kitty key page (G = 128 tokens, K boosted channels), one record of
 *     kvq_kitty_key_page_bytes() bytes: low plane (D*G/4 bytes, code & 3 of
 *     every channel), high plane (Kp*G/4 bytes, Kp = K rounded up to a
 *     multiple of 4; row r = r-th boosted channel in ascending channel order,
 *     code >> 2; rows K..Kp-1 zero), idx uint8 [D] (r, or K+1 for channels
 *     that are not boosted), s fp16 [D], z fp16 [D].  Both planes are in
 *     the fragment order of the KIVI key tiles: the low plane is the KIVI
 *     2-bit key layout above over the page's 128 tokens (token t, channel c
 *     at bits 2p of byte (t/32)*1024 + (k/4)*512 + (4q + r)*16 + (k%4)*4 +
 *     (e + 2h)); the high plane gives each 32-token tile t/32 a block of
 *     Kp*8 bytes, row r = 16kh + 4rb + b of token t = q + 8p (mod 32) at
 *     bits 2p of byte (t/32)*Kp*8 + kh*128 + 32*rb + 4q + b, so one 4-byte
 *     word holds four rows at four tokens.
 *   Kitty value page: codes [G][D/4] token-major as above, s fp16 [G],
 *     z fp16 [G].
 *   INT8 cache: codes int8 [tokens][D]; scale fp16 [blocks][D].
 *   Token-granular INT8 slot pool: codes int8 [n_slots][Hkv][D]; scale fp16
 *     [n_slots][Hkv][D/Gc] (136 bytes per token, kv head and side at Gc = 32).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent config */
    KVQ_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim != 128, bits not 2 or 4, ...) */
    KVQ_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned */
    KVQ_ERR_CUDA = 4,          /* a CUDA runtime call or a launch failed */
    KVQ_ERR_WORKSPACE = 5      /* workspace smaller than kv_decode_attn_plan() asked for */
} kvq_status;

/* device error flags (bitmask) written by kernels instead of trapping */
#define KVQ_DEVICE_ERR_WAIT_TIMEOUT 1u
#define KVQ_DEVICE_ERR_CAPACITY 2u      /* kv_append_* on a row already at max_seq_len: nothing written */
#define KVQ_DEVICE_ERR_POOL 4u          /* slot pool exhausted (or overfilled by a release): nothing written */

typedef enum {
    KVQ_VARIANT_KIVI = 0,
    KVQ_VARIANT_KITTY = 1,
    KVQ_VARIANT_INT8 = 2,
    KVQ_VARIANT_INT8_TOKEN = 3,
    KVQ_VARIANT_KIVI_PAGED = 4
} kvq_variant;

/* Free-slot (or free-page) pool: a stack of free ids.  slots int32
 * [capacity] and top int32 [1] are device memory owned by the caller; the
 * ids below *top are free. */
typedef struct {
    int32_t capacity;
    int32_t *slots;
    int32_t *top;
} kvq_slot_pool;

typedef struct {
    int32_t head_dim;     /* D; 128 */
    int32_t n_q_heads;    /* Hq */
    int32_t n_kv_heads;   /* Hkv; Hq % Hkv == 0 */
    int32_t bits_k;       /* KIVI key bits: 2 or 4 */
    int32_t bits_v;       /* KIVI value bits: 2 or 4; Kitty value bits: 2 */
    int32_t group_k;      /* G: tokens per KIVI key group (32, 64, 128) or Kitty page (128) */
    int32_t group_v;      /* Gv: channels per KIVI value group (32, 64 or 128) */
    int32_t residual;     /* R: KIVI fp16 residual (R % G == 0), Kitty value local window */
    int32_t sink;         /* S: Kitty fp16 sink tokens */
    int32_t boost_k;      /* K: Kitty boosted key channels, 0..head_dim */
    int32_t int8_block;   /* INT8 dither block length in tokens: 256 */
    float sm_scale;       /* softmax scale; 0 means 1/sqrt(head_dim) */
    int32_t int8_group;   /* Gc: channels per token-granular INT8 scale (32, 64 or 128) */
} kvq_config;

/* --------------------------------------------------------------------- */
/* Write side                                                              */
/* --------------------------------------------------------------------- */

/* a1: quantize n_groups KIVI key groups at b = cfg->bits_k bits (2 or 4).
 *   k       fp16 [n_groups][G][D], token-major (as the K projection emits it)
 *   codes   uint8 [n_groups][G*D*b/8]  (tile layout above)
 *   sz      fp16 [n_groups][2*D]       (scales then zeros, order above)
 * Per channel over the group's G tokens, with Q = 2^b - 1: z = fp16
 * round-down(min), s = fp16 round-up(fp32 (max - z) / Q), raised by one fp16
 * step while z + Q s < max; code = clamp(rint((x - z) / s), 0, Q) in fp32
 * with the stored fp16 s, z; s = 0 (all codes 0) when max == min.
 * (KIVI section 3.3 key split, section 4 KIVI-2 / KIVI-4; Kitty Observation 1
 * formula.)
 * n_groups == 0 launches nothing and returns KVQ_OK. */
KVQ_API kvq_status kv_quant_key(const kvq_config *cfg, const void *k, int64_t n_groups,
                        void *codes, void *sz, cudaStream_t stream);

/* a2: quantize n_tokens KIVI values, per token over groups of Gv channels,
 * at b = cfg->bits_v bits (2 or 4).
 *   v       fp16 [n_tokens][D]
 *   codes   token-major uint8 [n_tokens][D*b/8], or, for a config stored in
 *           value tiles, ceil(n_tokens/32) tiles of 32*D*b/8 bytes (token 0
 *           of the call starts a tile; bytes of the last tile's tokens past
 *           n_tokens are left unchanged)
 *   sz      fp16x2 [n_tokens][D/Gv]
 * Same rounding rules as kv_quant_key.  (KIVI section 3.3 value split.) */
KVQ_API kvq_status kv_quant_value(const kvq_config *cfg, const void *v, int64_t n_tokens,
                          void *codes, void *sz, cudaStream_t stream);

/* a5: quantize n_pages Kitty key pages (G = cfg->group_k = 128 tokens).
 *   k          fp16 [n_pages][G][D]
 *   score_mode 0: Eq. 2 score sum_t |x| (exact integer sum in units of 2^-24);
 *              1: population variance over the page from sequential fp32
 *                 sums in token order (sum x^2 / G - (sum x / G)^2)
 *   pages      [n_pages] records of kvq_kitty_key_page_bytes(cfg) bytes
 * The K = cfg->boost_k channels with the largest score (ties to the lower
 * channel) get 4-bit codes, the rest 2-bit; each channel has its own (s, z)
 * with the rounding rules of kv_quant_key and 2^b - 1 = 15 or 3.
 * (Kitty Eq. 2, "Selecting the Top-K Channels", "The Decomposition".) */
KVQ_API kvq_status kv_quant_key_kitty(const kvq_config *cfg, const void *k, int64_t n_pages,
                              int32_t score_mode, void *pages, cudaStream_t stream);

/* a6: quantize n_pages Kitty value pages: per token over all D channels,
 * 2-bit.  v fp16 [n_pages][G][D]; pages [n_pages] records of
 * kvq_kitty_value_page_bytes(cfg) bytes.  (Kitty "Value Cache Quantization".) */
KVQ_API kvq_status kv_quant_value_kitty(const kvq_config *cfg, const void *v, int64_t n_pages,
                                void *pages, cudaStream_t stream);

/* a8: INT8 subtractive-dither quantization of n_blocks blocks of
 * T = cfg->int8_block (256) tokens.
 *   x        fp16 [n_blocks][T][D]
 *   req_id, kv_head, tok0   int32 [n_blocks] (device): request id, kv head
 *            and absolute position of the block's first token
 *   layer    layer index (0 .. 2^15-1), kv_sel 0 for keys, 1 for values
 *   seed     64-bit Philox key
 *   codes    int8 [n_blocks][T][D];  scale fp16 [n_blocks][D]
 * s_c = fp16 round-to-nearest(fp32 amax_c / 126.5); xi = Philox4x32-10 word
 * (c % 4) of counter (token, c / 4, layer << 17 | kv_sel << 16 | kv_head,
 * request) under key (seed lo, seed hi), xi = (word >> 8) * 2^-24 - 1/2;
 * code = clamp(rint(x / s + xi), -127, 127) in fp32 with the stored fp16 s;
 * s = 0 gives code 0.  (WitCert sec. 6.1 write kernel.) */
KVQ_API kvq_status kv_quant_int8_dither(const kvq_config *cfg, const void *x, int64_t n_blocks,
                                const int32_t *req_id, const int32_t *kv_head, const int32_t *tok0,
                                int32_t layer, int32_t kv_sel, uint64_t seed,
                                void *codes, void *scale, cudaStream_t stream);

/* Record sizes of the Kitty pages for this config (0 on invalid config). */
KVQ_API size_t kvq_kitty_key_page_bytes(const kvq_config *cfg);
KVQ_API size_t kvq_kitty_value_page_bytes(const kvq_config *cfg);

/* --------------------------------------------------------------------- */
/* Read side: caches at attention time                                     */
/* --------------------------------------------------------------------- */
/* seq_len[b] = L_b = tokens in the cache of batch row b INCLUDING the
 * current token (its k, v are inserted before attention; quantization of a
 * full group happens after attention, the Kitty step order).  The dense
 * caches are [batch][n_kv_heads][capacity][...] with the capacity derived
 * from max_seq_len, and 1 <= seq_len[b] <= max_seq_len; the paged caches
 * and the token-granular slot pool state their own layouts below (a slot-pool
 * request may be empty, seq_len[b] = 0). */

/* KIVI: the key residual holds r_K = ((L-1) mod R) + 1 tokens and the first
 * L - r_K keys are quantized in whole groups; the value residual holds
 * min(L, R) tokens and the first L - min(L, R) values are quantized.
 * Residual token t is stored at slot t % R.  (KIVI section 3.3, Eq. 3.) */
typedef struct {
    int32_t batch;
    int32_t max_seq_len;     /* token capacity CAP = max_seq_len rounded up to a multiple of 128 */
    const int32_t *seq_len;  /* [B] */
    const void *k_codes;     /* uint8  [B][Hkv][CAP/G][G*D*bits_k/8] */
    const void *k_sz;        /* fp16 [B][Hkv][CAP/G][2*D]: scales, then zeros (layout above) */
    const void *v_codes;     /* uint8  [B][Hkv][CAP][D*bits_v/8] */
    const void *v_sz;        /* fp16x2 [B][Hkv][CAP][D/Gv] */
    const void *k_res;       /* fp16   [B][Hkv][R][D] */
    const void *v_res;       /* fp16   [B][Hkv][R][D] */
} kvq_kivi_cache;

/* Streaming append of one token per (batch row, kv head) to a KIVI cache,
 * for a decode loop that calls it before kv_decode_attn at every step.
 *   k_new, v_new  fp16 [batch][n_kv_heads][D]: the new token's key and value
 *   c             the cache (written: codes, (s, z), residual rings, seq_len)
 * With L = seq_len[b] tokens cached it first completes the quantization that
 * follows the attention of the step with L tokens (KIVI section 3.3 with the
 * Kitty step order insert -> attend -> quantize): when L is a positive
 * multiple of R the R keys of the full key residual become R/G quantized
 * groups, and when L >= R value token L - R, which leaves the fp16 window,
 * is quantized; then it writes the new token to ring slot L % R and sets
 * seq_len[b] = L + 1.  The quantizers are those of kv_quant_key and
 * kv_quant_value, so a cache grown token by token holds the same bytes as one
 * filled at once.  Two kernels on `stream`, graph-capturable.  A row with
 * seq_len[b] >= max_seq_len is left unchanged and KVQ_DEVICE_ERR_CAPACITY is
 * recorded (kvq_get_device_error).  Beyond the pages' hot path: this is the
 * streaming write side of their decode loop, on the dense cache layout above. */
KVQ_API kvq_status kv_append_kivi(const kvq_config *cfg, const kvq_kivi_cache *c, const void *k_new,
                                  const void *v_new, cudaStream_t stream);

/* Paged KIVI cache: the quantized part of every request lives in pages of
 * 128 tokens taken from a shared pool (a page table per request, a free-page
 * stack: kvq_slot_pool with page ids), the fp16 residual stays per (batch
 * row, kv head).  A page record holds one kv head's 128 tokens in the order a
 * decode stage uses them:
 *   key codes   128*D*bits_k/8 bytes  (128/G key groups in the tile layout)
 *   key (s, z)  2048 bytes            (128/G blocks of 256 fp16, order above)
 *   value codes 128*D*bits_v/8 bytes  (token-major)
 *   value (s,z) 2048 bytes            (fp16x2 [128][D/Gv])
 * so a decode stage is one contiguous copy of kvq_kivi_page_bytes(cfg)
 * bytes.  Token t of request b is in logical page t/128, physical page
 * page_table[b][t/128], record pages + (page * Hkv + kv_head) * page_bytes.
 * (Page management as in Kitty's "Page-Centric Memory Layout and
 * Dense-Sparse Decomposition": fixed-size pages in a pool addressed through
 * a page table, PagedAttention style; applied here to the KIVI segments.) */
typedef struct {
    int32_t batch;
    int32_t max_seq_len;       /* page_table row stride = ceil(max_seq_len / 128) */
    const int32_t *seq_len;    /* [B] */
    const int32_t *page_table; /* int32 [B][ceil(max_seq_len/128)] */
    int32_t n_pages;           /* pages in the pool */
    const void *pages;         /* [n_pages][Hkv][kvq_kivi_page_bytes(cfg)] */
    const void *k_res;         /* fp16 [B][Hkv][R][D] */
    const void *v_res;         /* fp16 [B][Hkv][R][D] */
} kvq_kivi_paged_cache;

/* Bytes of one paged KIVI page record for cfg (0 for an invalid cfg). */
KVQ_API size_t kvq_kivi_page_bytes(const kvq_config *cfg);

/* a1 / a2 into pages: quantize n_groups key groups (fp16 [n_groups][G][D]
 * of kv head kv_head) that are groups group0 .. group0 + n_groups - 1 of
 * request `row`, or n_tokens value tokens (fp16 [n_tokens][D]) that are its
 * tokens tok0 .., into the pages page_table[row] names.  Same arithmetic as
 * kv_quant_key / kv_quant_value. */
KVQ_API kvq_status kv_quant_key_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const void *k,
                                      int64_t n_groups, int32_t group0, int32_t row, int32_t kv_head,
                                      cudaStream_t stream);
KVQ_API kvq_status kv_quant_value_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const void *v,
                                        int64_t n_tokens, int32_t tok0, int32_t row, int32_t kv_head,
                                        cudaStream_t stream);

/* Streaming append to a paged KIVI cache, as kv_append_kivi: a row with
 * L = seq_len[b] a multiple of 128 first takes a page from the pool for
 * logical page L/128 (rows in order of b take pages from the top of the free
 * stack, deterministic under graph replay); then the pending flush and value
 * quantization write into the row's pages, token L goes to ring slot L % R,
 * and seq_len[b] = L + 1.  A row that needs a page when the pool has too few
 * is left unchanged and KVQ_DEVICE_ERR_POOL is recorded; a full row records
 * KVQ_DEVICE_ERR_CAPACITY.  Three kernels on `stream`, graph-capturable. */
KVQ_API kvq_status kv_append_kivi_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c,
                                        const kvq_slot_pool *pool, const void *k_new, const void *v_new,
                                        cudaStream_t stream);

/* Return the pages of request `row` (logical pages 0 .. ceil(seq_len/128)-1)
 * to the pool and set seq_len[row] = 0; overfilling the pool records
 * KVQ_DEVICE_ERR_POOL and changes nothing. */
KVQ_API kvq_status kv_release_kivi_paged(const kvq_kivi_paged_cache *c, int32_t row, const kvq_slot_pool *pool,
                                         cudaStream_t stream);

/* Kitty: sink tokens [0, min(L,S)) fp16; key pages, then a key Q-buffer of
 * n_kb = ((L-S-1) mod G) + 1 tokens (slot (t-S) % G); value pages, a value
 * Q-buffer of n_vb = ((E-1) mod G) + 1 tokens with E = L-S-R > 0 (slot
 * (t-S) % G), then a local window of the last min(L-S, R) tokens (slot
 * t % R).  (Kitty "Stage 1: Inserting New KV Vectors", "Stage 3".) */
typedef struct {
    int32_t batch;
    int32_t max_seq_len;
    const int32_t *seq_len;  /* [B] */
    const void *k_pages;     /* [B][Hkv][P][key page record], P = ceil(max(max_seq_len-S,0)/G) */
    const void *v_pages;     /* [B][Hkv][P][value page record] */
    const void *k_sink;      /* fp16 [B][Hkv][S][D] */
    const void *v_sink;      /* fp16 [B][Hkv][S][D] */
    const void *k_qbuf;      /* fp16 [B][Hkv][G][D] */
    const void *v_qbuf;      /* fp16 [B][Hkv][G][D] */
    const void *v_local;     /* fp16 [B][Hkv][R][D] */
    /* Paged form (page_table non-null): key and value page records come from
     * shared pools k_pages [n_pages][Hkv][key page record] and v_pages
     * [n_pages][Hkv][value page record]; logical page j of request b (tokens
     * S + G j .. S + G j + G - 1, keys and values) is physical page
     * page_table[b][j], int32 [B][P].  NULL: the per-request arrays above. */
    const int32_t *page_table;
    int32_t n_pages;
} kvq_kitty_cache;

/* Streaming append of one token per (batch row, kv head) to a Kitty cache,
 * called before kv_decode_attn_kitty at every step.
 *   k_new, v_new  fp16 [batch][n_kv_heads][D]
 *   score_mode    as kv_quant_key_kitty
 * With L = seq_len[b] cached it completes the quantization that follows the
 * attention of the step with L tokens: a full key Q-buffer ((L-S) a positive
 * multiple of G) becomes key page (L-S)/G - 1, a full value Q-buffer (E = L-S-R
 * a positive multiple of G) becomes value page E/G - 1, and token L-R leaves
 * the local window for value Q-buffer slot (L-R-S) % G; then token L goes to
 * the sink (L < S) or to key Q-buffer slot (L-S) % G and local slot L % R,
 * and seq_len[b] = L + 1 (Kitty "Stage 1: Inserting New KV Vectors",
 * "Stage 3").  The page quantizers are those of kv_quant_key_kitty and
 * kv_quant_value_kitty.  Two kernels on `stream`, graph-capturable; a row
 * with seq_len[b] >= max_seq_len is left unchanged and
 * KVQ_DEVICE_ERR_CAPACITY is recorded. */
KVQ_API kvq_status kv_append_kitty(const kvq_config *cfg, const kvq_kitty_cache *c, const void *k_new,
                                   const void *v_new, int score_mode, cudaStream_t stream);

/* a5 / a6 into a paged Kitty cache: n_pages key (value) pages, fp16
 * [n_pages][G][D] of kv head kv_head, that are logical pages page0 .. of
 * request `row`, quantized into the pool pages page_table[row] names.  Same
 * arithmetic as kv_quant_key_kitty / kv_quant_value_kitty. */
KVQ_API kvq_status kv_quant_key_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const void *k,
                                            int64_t n_pages, int32_t page0, int32_t row, int32_t kv_head,
                                            int32_t score_mode, cudaStream_t stream);
KVQ_API kvq_status kv_quant_value_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const void *v,
                                              int64_t n_pages, int32_t page0, int32_t row, int32_t kv_head,
                                              cudaStream_t stream);

/* Streaming append to a paged Kitty cache, as kv_append_kitty: a row whose
 * L = seq_len[b] is S + G j first takes pool page j for its next tokens
 * (rows in order of b, from the top of the free stack; deterministic under
 * graph replay).  A row that needs a page when too few are free is left
 * unchanged and KVQ_DEVICE_ERR_POOL is recorded.  Three kernels. */
KVQ_API kvq_status kv_append_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const kvq_slot_pool *pool,
                                         const void *k_new, const void *v_new, int32_t score_mode,
                                         cudaStream_t stream);

/* Return the pages of request `row` (logical pages 0 .. ceil(max(seq_len-S, 0)/G) - 1)
 * of a paged Kitty cache to the pool and set seq_len[row] = 0. */
KVQ_API kvq_status kv_release_kitty(const kvq_config *cfg, const kvq_kitty_cache *c, int32_t row,
                                    const kvq_slot_pool *pool, cudaStream_t stream);

/* INT8 dither: the first L - n_tail tokens are quantized in blocks of T,
 * n_tail = ((L-1) mod T) + 1 tokens of the active block stay fp16 (slot
 * t % T).  Dither is regenerated from (req_id[b], layer, kv head, token,
 * channel).  (WitCert sec. 6.1 read kernel; "active block" tail.) */
typedef struct {
    int32_t batch;
    int32_t max_seq_len;
    const int32_t *seq_len;  /* [B] */
    const int32_t *req_id;   /* [B] */
    int32_t layer;
    uint64_t seed;
    const void *k_codes;     /* int8 [B][Hkv][max_seq_len][D] */
    const void *v_codes;     /* int8 [B][Hkv][max_seq_len][D] */
    const void *k_scale;     /* fp16 [B][Hkv][ceil(max_seq_len/T)][D] */
    const void *v_scale;     /* fp16 [B][Hkv][ceil(max_seq_len/T)][D] */
    const void *k_tail;      /* fp16 [B][Hkv][T][D] */
    const void *v_tail;      /* fp16 [B][Hkv][T][D] */
} kvq_int8_cache;

/* Streaming append of one token per (batch row, kv head) to an INT8 cache,
 * called before kv_decode_attn_int8 at every step.
 *   k_new, v_new  fp16 [batch][n_kv_heads][D]
 * With L = seq_len[b] cached: when L is a positive multiple of T the fp16
 * tail becomes INT8 block (L-T)/T of keys and values with the same scales,
 * codes and Philox dither streams as kv_quant_int8_dither (WitCert section
 * 6.1, active-block tail); then the new token goes to tail slot L % T and
 * seq_len[b] = L + 1.  Two kernels on `stream`, graph-capturable.  A row
 * with seq_len[b] >= max_seq_len is left unchanged and
 * KVQ_DEVICE_ERR_CAPACITY is recorded. */
KVQ_API kvq_status kv_append_int8(const kvq_config *cfg, const kvq_int8_cache *c, const void *k_new,
                                  const void *v_new, cudaStream_t stream);

/* --------------------------------------------------------------------- */
/* Token-granular INT8 over a slot pool                                     */
/* --------------------------------------------------------------------- */
/* The form WitCert gives for an engine whose KV pool is paged at token-slot
 * granularity (the SGLang storage subsection of sec. 6.2): a token's slot is
 * any free slot of the pool, a request's tokens need not be contiguous, and
 * a token is quantized when it is written, with
 *   s = fp16_RN(amax / 126.5) per token and group of Gc channels,
 *   code = clamp(rint(x/s + xi), -127, 127) with the stored s (0 if s == 0),
 *   x^ = s (code - xi),
 * and xi = (w >> 8) 2^-24 - 1/2 from Philox4x32-10 keyed by (layer, kv head,
 * slot, channel): counter (slot, channel/4, layer << 17 | kv_sel << 16 |
 * kv_head, 0), key (seed low, seed high), word channel % 4; kv_sel 0 = K,
 * 1 = V.  The dither follows the slot, so moving a request never changes
 * what a written slot decodes to. */
typedef struct {
    int32_t batch;
    int32_t max_seq_len;      /* row stride of slot_table */
    const int32_t *seq_len;   /* [B] tokens per request (0 allowed) */
    const int32_t *slot_table; /* int32 [B][max_seq_len]: slot of token t of request b */
    int32_t n_slots;
    int32_t layer;            /* 0 .. 2^15 - 1 */
    uint64_t seed;
    const void *k_codes;      /* int8 [n_slots][Hkv][D] */
    const void *v_codes;      /* int8 [n_slots][Hkv][D] */
    const void *k_scale;      /* fp16 [n_slots][Hkv][D/Gc] */
    const void *v_scale;      /* fp16 [n_slots][Hkv][D/Gc] */
} kvq_int8_token_cache;

/* Quantize n tokens (all kv heads) into their slots.
 *   x      fp16 [n][Hkv][D]
 *   slots  int32 [n] device array of distinct slots in [0, n_slots)
 *   kv_sel 0 for keys (writes k_codes / k_scale of c), 1 for values
 * Slots outside [0, n_slots) are skipped. */
KVQ_API kvq_status kv_quant_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c, const void *x,
                                       int64_t n, const int32_t *slots, int32_t kv_sel, cudaStream_t stream);

/* Fill the pool with every slot 0 .. capacity-1 (pops then return 0, 1, 2, ...). */
KVQ_API kvq_status kv_slot_pool_init(const kvq_slot_pool *pool, cudaStream_t stream);

/* Streaming append of one token per request: k_new, v_new fp16 [B][Hkv][D].
 * Every row b with seq_len[b] < max_seq_len takes one slot from the pool
 * (rows in order of b take the slots from the top of the stack down, so the
 * assignment is deterministic and a replayed graph writes the same slots),
 * records it in slot_table[b][seq_len[b]], quantizes the token into it and
 * sets seq_len[b] += 1.  Rows already at max_seq_len record
 * KVQ_DEVICE_ERR_CAPACITY and are left unchanged; if the pool holds fewer
 * free slots than rows that need one, KVQ_DEVICE_ERR_POOL is recorded and
 * no row is changed.  Two kernels on `stream`, graph-capturable. */
KVQ_API kvq_status kv_append_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c,
                                        const kvq_slot_pool *pool, const void *k_new, const void *v_new,
                                        cudaStream_t stream);

/* Return the slots of request `row` (slot_table[row][0 .. seq_len[row])) to
 * the pool and set seq_len[row] = 0.  A release that would overfill the pool
 * records KVQ_DEVICE_ERR_POOL and changes nothing.  Slots shared between
 * requests are not reference-counted: release each slot once. */
KVQ_API kvq_status kv_release_int8_token(const kvq_int8_token_cache *c, int32_t row, const kvq_slot_pool *pool,
                                         cudaStream_t stream);

/* Split-KV plan: number of splits per (batch row, query head) and the
 * workspace bytes the decode calls need for this config, variant, batch and
 * max_seq_len.  Deterministic: the decode calls recompute the same plan. */
KVQ_API kvq_status kv_decode_attn_plan(const kvq_config *cfg, int32_t variant, int32_t batch,
                               int32_t max_seq_len, int32_t *n_splits, size_t *workspace_bytes);

/* a3 + a4: out fp16 [B][Hq][D] = softmax(sm_scale q K^T) V over every cached
 * token, q fp16 [B][Hq][D]; query head h reads kv head h / (Hq / Hkv).
 * Stage 1 writes per-split (o_s = acc / l, lse_s) into the workspace
 * (fp32, caller-owned, at least the planned size); stage 2 merges
 * o = sum_s exp(lse_s - LSE) o_s with LSE = log sum_s exp(lse_s). */
KVQ_API kvq_status kv_decode_attn(const kvq_config *cfg, const kvq_kivi_cache *cache, const void *q,
                          void *out, void *workspace, size_t workspace_bytes, cudaStream_t stream);
KVQ_API kvq_status kv_decode_attn_kitty(const kvq_config *cfg, const kvq_kitty_cache *cache, const void *q,
                                void *out, void *workspace, size_t workspace_bytes, cudaStream_t stream);
KVQ_API kvq_status kv_decode_attn_int8(const kvq_config *cfg, const kvq_int8_cache *cache, const void *q,
                               void *out, void *workspace, size_t workspace_bytes, cudaStream_t stream);
/* Paged KIVI: the quantized tiles are read page by page through the page
 * table (one copy per 128-token stage). */
KVQ_API kvq_status kv_decode_attn_kivi_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *cache,
                                             const void *q, void *out, void *workspace, size_t workspace_bytes,
                                             cudaStream_t stream);
/* Token-granular INT8: every token t < seq_len[b] is read from slot
 * slot_table[b][t] and dequantized with its slot's dither; a row with
 * seq_len[b] == 0 gets out = 0. */
KVQ_API kvq_status kv_decode_attn_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *cache,
                                             const void *q, void *out, void *workspace, size_t workspace_bytes,
                                             cudaStream_t stream);

/* Allocation-free kv_decode_attn (no counterpart on the pages: an addition
 * for callers that cannot provide a workspace, such as engines whose own
 * pool owns all device memory or deployments that allow no device
 * allocation after start-up).  Same computation and kernels as
 * kv_decode_attn, with the split workspace in a fixed device array of
 * KVQ_NOALLOC_SCRATCH_BYTES compiled into the library; it holds that memory
 * on every GPU that loads the library until the process exits.
 *   - Returns KVQ_ERR_WORKSPACE, launching nothing, when the planned
 *     workspace (kv_decode_attn_plan) exceeds KVQ_NOALLOC_SCRATCH_BYTES.
 *   - The first call on each device looks the array's device address up
 *     (cudaGetSymbolAddress); make that first call before any stream
 *     capture on that device.  The address is kept per device and context:
 *     after a device reset the next call looks it up again (so, again,
 *     outside a capture).
 *   - Every call uses the same array: calls whose kernels can overlap on the
 *     GPU (other streams, other host threads) race and must be serialized
 *     by the caller.  No part of the array needs clearing between calls.
 * It calls no cudaMalloc or cudaFree. */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)
KVQ_API kvq_status kv_decode_attn_noalloc(const kvq_config *cfg, const kvq_kivi_cache *cache, const void *q,
                                          void *out, cudaStream_t stream);

/* The two stages separately (kv_decode_attn* = stage1 then merge). */
KVQ_API kvq_status kv_decode_attn_stage1(const kvq_config *cfg, int32_t variant, const void *cache,
                                 const void *q, void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream);
KVQ_API kvq_status kv_decode_attn_merge(const kvq_config *cfg, int32_t variant, int32_t batch,
                                int32_t max_seq_len, const void *workspace, size_t workspace_bytes,
                                void *out, cudaStream_t stream);

/* --------------------------------------------------------------------- */
/* Diagnostics                                                             */
/* --------------------------------------------------------------------- */

/* The library's Philox4x32-10 on the GPU: out[i][0..3] = Philox4x32-10 of
 * counter ctr[i][0..3] under key (key[i][0], key[i][1]); uint32 device
 * arrays.  (Salmon et al., SC'11.) */
KVQ_API kvq_status kvq_philox4x32_10(const uint32_t *ctr, const uint32_t *key, int64_t n,
                             uint32_t *out, cudaStream_t stream);

/* Reads and clears the device error bitmask of the current device
 * (synchronous; not for use inside a stream capture). */
KVQ_API kvq_status kvq_get_device_error(uint32_t *flags);

KVQ_API const char *kvq_status_string(kvq_status s);
KVQ_API const char *kvq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
