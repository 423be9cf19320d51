// extern "C" entry points of libkvq: host-side argument validation, the
// split-KV plan, and dispatch to the kernels.  Nothing here allocates device
// memory or synchronizes the host (except kvq_get_device_error, documented
// as synchronous).
#include <math.h>
#include <string.h>

#include <initializer_list>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

// Device error bitmask: kernels atomically OR KVQ_DEVICE_ERR_* into it
// instead of trapping.  Its device address is passed to every kernel that
// can wait.
__device__ unsigned g_device_error;

static const int kMaxDevices = 64;

int num_sms() {
    static int cached[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 152;
    }
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 152;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

unsigned *device_error_ptr() {
    static unsigned *cached[kMaxDevices] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!cached[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        cached[dev] = static_cast<unsigned *>(p);
    }
    return cached[dev];
}

float sm_scale_of(const kvq_config *cfg) {
    return cfg->sm_scale > 0.f ? cfg->sm_scale : 1.0f / sqrtf((float)cfg->head_dim);
}

// Splits: chunks of a multiple of 128 tokens (the stage), sized so that the
// persistent decode grid (4 CTAs per SM; 3 for grouped-query KIVI, 2 for
// INT8) gets about 6 (per-head units) or 8 (kv-head units) units per CTA,
// within [128, 4096] tokens and at most 256 + 1 splits per row (the last split of
// a row holds the tokens outside the quantized tiles, e.g. the fp16 residual;
// the token-granular INT8 cache has none and leaves that split empty).
kvq_status plan_decode(const kvq_config *cfg, int variant, int batch, int max_seq_len, DecodePlan *p) {
    const int64_t rows = (int64_t)batch * cfg->n_q_heads;
    // the INT8 kernel (2 CTAs per SM) and the grouped-query KIVI (3) and Kitty (4) kernels handle all
    // query heads of a kv head in one unit; the per-head kernels run 4 CTAs per SM
    const bool int8 = variant == KVQ_VARIANT_INT8 || variant == KVQ_VARIANT_INT8_TOKEN;
    const bool kivi = variant == KVQ_VARIANT_KIVI || variant == KVQ_VARIANT_KIVI_PAGED;
    const bool kv_units = int8 || (kivi && kivi_gqa_supported(cfg)) ||
                          (variant == KVQ_VARIANT_KITTY && kitty_gqa_supported(cfg));
    const int vsub = kivi && kivi_gqa_supported(cfg)                               ? kivi_gqa_units_per_kv_head(cfg)
                     : variant == KVQ_VARIANT_KITTY && kitty_gqa_supported(cfg) ? kitty_gqa_units_per_kv_head(cfg)
                                                                                : 1;
    const int64_t unit_rows = kv_units ? (int64_t)batch * cfg->n_kv_heads * vsub : rows;
    const int ctas = int8 ? 2 : (kivi && kivi_gqa_supported(cfg)) ? 3 : 4;
    // units per CTA aimed at: fewer, longer units amortize the per-unit merge, more units balance the
    // static round-robin; measured on the MHA decode layer (B32, 32 heads, L4096) 6 beat 8 by 3.5 % and
    // 5 lost 19 %, on the grouped-query layer (B64, 32q/8kv, L32768) 8 beat 6 and 10.  A dynamic
    // schedule (a ticket counter in the workspace, largest units first) measured 2-11 % slower on
    // both layers: the SM's issue slots pass to its other CTAs as one drains, so the static imbalance
    // costs less than the tickets' round trips and the spills they added
    const int64_t per_cta = kv_units ? 8 : 6;
    const int64_t target_units = per_cta * num_sms() * ctas;
    int64_t chunk = (unit_rows * max_seq_len + target_units - 1) / target_units;
    chunk = (chunk + 127) / 128 * 128;
    if (chunk < 128) chunk = 128;
    if (chunk > 4096) chunk = 4096;
    const int64_t min_chunk = (((int64_t)max_seq_len + 255) / 256 + 127) / 128 * 128;
    if (chunk < min_chunk) chunk = min_chunk;
    // quantized-tile splits, plus one split per row for the tokens outside the tiles
    const int splits = (int)(((int64_t)max_seq_len + chunk - 1) / chunk) + 1;
    p->splits = splits;
    p->chunk = (int)chunk;
    p->off_o = 256;
    p->off_lse = p->off_o + (size_t)rows * p->splits * KVQ_D * sizeof(float);
    p->ws_bytes = (p->off_lse + (size_t)rows * p->splits * sizeof(float) + 255) / 256 * 256;
    return KVQ_OK;
}

}  // namespace kvq

using namespace kvq;

// ---------------------------------------------------------------------------
// validation helpers
// ---------------------------------------------------------------------------
static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static kvq_status check_common(const kvq_config *cfg) {
    if (!cfg) return KVQ_ERR_INVALID_ARG;
    if (cfg->n_q_heads < 1 || cfg->n_kv_heads < 1 || cfg->n_q_heads % cfg->n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
    if (cfg->sm_scale < 0.f || !(cfg->sm_scale == cfg->sm_scale)) return KVQ_ERR_INVALID_ARG;
    if (cfg->head_dim != KVQ_D) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

static kvq_status check_kivi(const kvq_config *cfg) {
    kvq_status s = check_common(cfg);
    if (s) return s;
    if (cfg->group_k <= 0 || cfg->group_v <= 0 || cfg->residual <= 0) return KVQ_ERR_INVALID_ARG;
    if ((cfg->bits_k != 2 && cfg->bits_k != 4) || (cfg->bits_v != 2 && cfg->bits_v != 4)) return KVQ_ERR_UNSUPPORTED;
    if (cfg->group_k != 32 && cfg->group_k != 64 && cfg->group_k != 128) return KVQ_ERR_UNSUPPORTED;
    if (cfg->group_v != 32 && cfg->group_v != 64 && cfg->group_v != 128) return KVQ_ERR_UNSUPPORTED;
    if (cfg->residual % cfg->group_k != 0) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

static kvq_status check_kitty(const kvq_config *cfg) {
    kvq_status s = check_common(cfg);
    if (s) return s;
    if (cfg->group_k <= 0 || cfg->residual <= 0 || cfg->sink < 0 || cfg->boost_k < 0 || cfg->boost_k > cfg->head_dim)
        return KVQ_ERR_INVALID_ARG;
    if (cfg->group_k != 128 || cfg->bits_v != 2) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

static kvq_status check_int8(const kvq_config *cfg) {
    kvq_status s = check_common(cfg);
    if (s) return s;
    if (cfg->int8_block <= 0) return KVQ_ERR_INVALID_ARG;
    if (cfg->int8_block % 128 != 0) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

static kvq_status check_int8_token(const kvq_config *cfg) {
    kvq_status s = check_common(cfg);
    if (s) return s;
    if (cfg->int8_group <= 0) return KVQ_ERR_INVALID_ARG;
    if (cfg->int8_group != 32 && cfg->int8_group != 64 && cfg->int8_group != 128) return KVQ_ERR_UNSUPPORTED;
    if (cfg->n_q_heads / cfg->n_kv_heads > 8) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

static kvq_status ptrs_ok(std::initializer_list<const void *> ps) {
    for (const void *p : ps) {
        if (!p) return KVQ_ERR_INVALID_ARG;
        if (!aligned16(p)) return KVQ_ERR_MISALIGNED;
    }
    return KVQ_OK;
}

static kvq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

static kvq_status check_pool(const kvq_slot_pool *pool) {
    if (!pool || pool->capacity < 1) return KVQ_ERR_INVALID_ARG;
    return ptrs_ok({pool->slots, pool->top});
}

static kvq_status check_kivi_paged_cache(const kvq_kivi_paged_cache *c) {
    if (!c || c->batch < 1 || c->max_seq_len < 1 || c->n_pages < 1) return KVQ_ERR_INVALID_ARG;
    return ptrs_ok({c->seq_len, c->page_table, c->pages, c->k_res, c->v_res});
}

// ---------------------------------------------------------------------------
// write side
// ---------------------------------------------------------------------------
extern "C" kvq_status kv_quant_key(const kvq_config *cfg, const void *k, int64_t n_groups, void *codes, void *sz,
                                   cudaStream_t stream) {
    kvq_status s = check_kivi(cfg);
    if (s) return s;
    if (n_groups < 0) return KVQ_ERR_INVALID_ARG;
    if (n_groups == 0) return KVQ_OK;
    if ((s = ptrs_ok({k, codes, sz}))) return s;
    return cuda_status(launch_quant_key_kivi(cfg, k, n_groups, codes, sz, stream));
}

extern "C" kvq_status kv_quant_value(const kvq_config *cfg, const void *v, int64_t n_tokens, void *codes, void *sz,
                                     cudaStream_t stream) {
    kvq_status s = check_kivi(cfg);
    if (s) return s;
    if (n_tokens < 0) return KVQ_ERR_INVALID_ARG;
    if (n_tokens == 0) return KVQ_OK;
    if ((s = ptrs_ok({v, codes, sz}))) return s;
    return cuda_status(launch_quant_value_kivi(cfg, v, n_tokens, codes, sz, stream));
}

extern "C" kvq_status kv_append_kivi(const kvq_config *cfg, const kvq_kivi_cache *c, const void *k_new,
                                     const void *v_new, cudaStream_t stream) {
    kvq_status s = check_kivi(cfg);
    if (s) return s;
    if (!c || c->batch < 1 || c->max_seq_len < 1) return KVQ_ERR_INVALID_ARG;
    if ((s = ptrs_ok({k_new, v_new, c->seq_len, c->k_codes, c->k_sz, c->v_codes, c->v_sz, c->k_res, c->v_res})))
        return s;
    return cuda_status(launch_append_kivi(cfg, c, k_new, v_new, stream));
}

extern "C" size_t kvq_kivi_page_bytes(const kvq_config *cfg) {
    if (check_kivi(cfg)) return 0;
    return (size_t)kivi_page_bytes(cfg->bits_k, cfg->bits_v);
}

static kvq_status check_kivi_paged_write(const kvq_config *cfg, const kvq_kivi_paged_cache *c, int64_t n,
                                         int64_t first, int64_t unit, int32_t row, int32_t kv_head) {
    kvq_status s = check_kivi(cfg);
    if (s) return s;
    if (!c || c->batch < 1 || c->max_seq_len < 1 || c->n_pages < 1) return KVQ_ERR_INVALID_ARG;
    if (n < 0 || first < 0 || row < 0 || row >= c->batch || kv_head < 0 || kv_head >= cfg->n_kv_heads)
        return KVQ_ERR_INVALID_ARG;
    const int64_t row_tokens = ((int64_t)c->max_seq_len + 127) / 128 * 128;
    if ((first + n) * unit > row_tokens) return KVQ_ERR_INVALID_ARG;
    return ptrs_ok({c->page_table, c->pages});
}

extern "C" kvq_status kv_quant_key_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const void *k,
                                         int64_t n_groups, int32_t group0, int32_t row, int32_t kv_head,
                                         cudaStream_t stream) {
    kvq_status s = check_kivi_paged_write(cfg, c, n_groups, group0, cfg ? cfg->group_k : 1, row, kv_head);
    if (s) return s;
    if (n_groups == 0) return KVQ_OK;
    if ((s = ptrs_ok({k}))) return s;
    return cuda_status(launch_quant_key_paged(cfg, c, k, n_groups, group0, row, kv_head, stream));
}

extern "C" kvq_status kv_quant_value_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const void *v,
                                           int64_t n_tokens, int32_t tok0, int32_t row, int32_t kv_head,
                                           cudaStream_t stream) {
    kvq_status s = check_kivi_paged_write(cfg, c, n_tokens, tok0, 1, row, kv_head);
    if (s) return s;
    if (n_tokens == 0) return KVQ_OK;
    if ((s = ptrs_ok({v}))) return s;
    return cuda_status(launch_quant_value_paged(cfg, c, v, n_tokens, tok0, row, kv_head, stream));
}

extern "C" kvq_status kv_append_kivi_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c,
                                           const kvq_slot_pool *pool, const void *k_new, const void *v_new,
                                           cudaStream_t stream) {
    kvq_status s = check_kivi(cfg);
    if (s) return s;
    if ((s = check_kivi_paged_cache(c))) return s;
    if ((s = check_pool(pool))) return s;
    if ((s = ptrs_ok({k_new, v_new}))) return s;
    return cuda_status(launch_append_kivi_paged(cfg, c, pool, k_new, v_new, stream));
}

extern "C" kvq_status kv_release_kivi_paged(const kvq_kivi_paged_cache *c, int32_t row, const kvq_slot_pool *pool,
                                            cudaStream_t stream) {
    kvq_status s = check_kivi_paged_cache(c);
    if (s) return s;
    if (row < 0 || row >= c->batch) return KVQ_ERR_INVALID_ARG;
    if ((s = check_pool(pool))) return s;
    const int stride = (int)(((int64_t)c->max_seq_len + 127) / 128);
    return cuda_status(launch_release_ids(const_cast<int32_t *>(c->seq_len), c->page_table, row, c->max_seq_len, 128,
                                          stride, 0, pool, stream));
}

extern "C" kvq_status kv_append_int8(const kvq_config *cfg, const kvq_int8_cache *c, const void *k_new,
                                     const void *v_new, cudaStream_t stream) {
    kvq_status s = check_int8(cfg);
    if (s) return s;
    if (!c || c->batch < 1 || c->max_seq_len < 1) return KVQ_ERR_INVALID_ARG;
    if (c->layer < 0 || c->layer >= (1 << 15)) return KVQ_ERR_INVALID_ARG;
    if ((s = ptrs_ok({k_new, v_new, c->seq_len, c->req_id, c->k_codes, c->v_codes, c->k_scale, c->v_scale, c->k_tail,
                      c->v_tail})))
        return s;
    return cuda_status(launch_append_int8(cfg, c, k_new, v_new, stream));
}

static int kitty_page_cap(const kvq_config *cfg, const kvq_kitty_cache *c) {
    const int pc = (int)(((c->max_seq_len - cfg->sink > 0 ? c->max_seq_len - cfg->sink : 0) + 127) / 128);
    return pc < 1 ? 1 : pc;
}

static kvq_status check_kitty_cache(const kvq_config *cfg, const kvq_kitty_cache *c, bool paged) {
    if (!c || c->batch < 1 || c->max_seq_len < 1) return KVQ_ERR_INVALID_ARG;
    if (paged != (c->page_table != nullptr)) return KVQ_ERR_INVALID_ARG;
    if (paged && c->n_pages < 1) return KVQ_ERR_INVALID_ARG;
    kvq_status s = ptrs_ok({c->seq_len, c->k_pages, c->v_pages, c->k_qbuf, c->v_qbuf, c->v_local});
    if (s) return s;
    if (paged && (s = ptrs_ok({c->page_table}))) return s;
    if (cfg->sink > 0 && (s = ptrs_ok({c->k_sink, c->v_sink}))) return s;
    return KVQ_OK;
}

extern "C" kvq_status kv_quant_key_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const void *k,
                                               int64_t n_pages, int32_t page0, int32_t row, int32_t kv_head,
                                               int32_t score_mode, cudaStream_t stream) {
    kvq_status s = check_kitty(cfg);
    if (s) return s;
    if (score_mode != 0 && score_mode != 1) return KVQ_ERR_INVALID_ARG;
    if (!c || !c->page_table || c->batch < 1 || c->max_seq_len < 1 || c->n_pages < 1) return KVQ_ERR_INVALID_ARG;
    if (n_pages < 0 || page0 < 0 || row < 0 || row >= c->batch || kv_head < 0 || kv_head >= cfg->n_kv_heads ||
        page0 + n_pages > kitty_page_cap(cfg, c))
        return KVQ_ERR_INVALID_ARG;
    if (n_pages == 0) return KVQ_OK;
    if ((s = ptrs_ok({k, c->k_pages, c->page_table}))) return s;
    return cuda_status(launch_quant_key_kitty_paged(cfg, c, k, n_pages, page0, row, kv_head, score_mode, stream));
}

extern "C" kvq_status kv_quant_value_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const void *v,
                                                 int64_t n_pages, int32_t page0, int32_t row, int32_t kv_head,
                                                 cudaStream_t stream) {
    kvq_status s = check_kitty(cfg);
    if (s) return s;
    if (!c || !c->page_table || c->batch < 1 || c->max_seq_len < 1 || c->n_pages < 1) return KVQ_ERR_INVALID_ARG;
    if (n_pages < 0 || page0 < 0 || row < 0 || row >= c->batch || kv_head < 0 || kv_head >= cfg->n_kv_heads ||
        page0 + n_pages > kitty_page_cap(cfg, c))
        return KVQ_ERR_INVALID_ARG;
    if (n_pages == 0) return KVQ_OK;
    if ((s = ptrs_ok({v, c->v_pages, c->page_table}))) return s;
    return cuda_status(launch_quant_value_kitty_paged(cfg, c, v, n_pages, page0, row, kv_head, stream));
}

extern "C" kvq_status kv_append_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const kvq_slot_pool *pool,
                                            const void *k_new, const void *v_new, int32_t score_mode,
                                            cudaStream_t stream) {
    kvq_status s = check_kitty(cfg);
    if (s) return s;
    if (score_mode != 0 && score_mode != 1) return KVQ_ERR_INVALID_ARG;
    if ((s = check_kitty_cache(cfg, c, true))) return s;
    if ((s = check_pool(pool))) return s;
    if ((s = ptrs_ok({k_new, v_new}))) return s;
    return cuda_status(launch_append_kitty_paged(cfg, c, pool, k_new, v_new, score_mode, stream));
}

extern "C" kvq_status kv_release_kitty(const kvq_config *cfg, const kvq_kitty_cache *c, int32_t row,
                                       const kvq_slot_pool *pool, cudaStream_t stream) {
    kvq_status s = check_kitty(cfg);
    if (s) return s;
    if ((s = check_kitty_cache(cfg, c, true))) return s;
    if (row < 0 || row >= c->batch) return KVQ_ERR_INVALID_ARG;
    if ((s = check_pool(pool))) return s;
    return cuda_status(launch_release_ids(const_cast<int32_t *>(c->seq_len), c->page_table, row, c->max_seq_len, 128,
                                          kitty_page_cap(cfg, c), cfg->sink, pool, stream));
}

extern "C" kvq_status kv_append_kitty(const kvq_config *cfg, const kvq_kitty_cache *c, const void *k_new,
                                      const void *v_new, int score_mode, cudaStream_t stream) {
    kvq_status s = check_kitty(cfg);
    if (s) return s;
    if (score_mode != 0 && score_mode != 1) return KVQ_ERR_INVALID_ARG;
    if (!c || c->batch < 1 || c->max_seq_len < 1) return KVQ_ERR_INVALID_ARG;
    if (c->page_table) return KVQ_ERR_INVALID_ARG;          // a paged cache appends through kv_append_kitty_paged
    if ((s = ptrs_ok({k_new, v_new, c->seq_len, c->k_pages, c->v_pages, c->k_qbuf, c->v_qbuf, c->v_local}))) return s;
    if (cfg->sink > 0 && (s = ptrs_ok({c->k_sink, c->v_sink}))) return s;
    return cuda_status(launch_append_kitty(cfg, c, k_new, v_new, score_mode, stream));
}

static kvq_status check_int8_token_cache(const kvq_int8_token_cache *c) {
    if (!c || c->batch < 1 || c->max_seq_len < 1 || c->n_slots < 1) return KVQ_ERR_INVALID_ARG;
    if (c->layer < 0 || c->layer >= (1 << 15)) return KVQ_ERR_INVALID_ARG;
    if ((int64_t)c->batch * c->max_seq_len > INT32_MAX) return KVQ_ERR_UNSUPPORTED;
    return ptrs_ok({c->seq_len, c->slot_table, c->k_codes, c->v_codes, c->k_scale, c->v_scale});
}


extern "C" kvq_status kv_quant_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c, const void *x,
                                          int64_t n, const int32_t *slots, int32_t kv_sel, cudaStream_t stream) {
    kvq_status s = check_int8_token(cfg);
    if (s) return s;
    if (n < 0 || (kv_sel != 0 && kv_sel != 1)) return KVQ_ERR_INVALID_ARG;
    if ((s = check_int8_token_cache(c))) return s;
    if (n == 0) return KVQ_OK;
    if ((s = ptrs_ok({x, slots}))) return s;
    return cuda_status(launch_quant_int8_token(cfg, c, x, n, slots, kv_sel, stream));
}

extern "C" kvq_status kv_slot_pool_init(const kvq_slot_pool *pool, cudaStream_t stream) {
    kvq_status s = check_pool(pool);
    if (s) return s;
    return cuda_status(launch_slot_pool_init(pool, stream));
}

extern "C" kvq_status kv_append_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c,
                                           const kvq_slot_pool *pool, const void *k_new, const void *v_new,
                                           cudaStream_t stream) {
    kvq_status s = check_int8_token(cfg);
    if (s) return s;
    if ((s = check_int8_token_cache(c))) return s;
    if ((s = check_pool(pool))) return s;
    if ((s = ptrs_ok({k_new, v_new}))) return s;
    return cuda_status(launch_append_int8_token(cfg, c, pool, k_new, v_new, stream));
}

extern "C" kvq_status kv_release_int8_token(const kvq_int8_token_cache *c, int32_t row, const kvq_slot_pool *pool,
                                            cudaStream_t stream) {
    kvq_status s = check_int8_token_cache(c);
    if (s) return s;
    if (row < 0 || row >= c->batch) return KVQ_ERR_INVALID_ARG;
    if ((s = check_pool(pool))) return s;
    return cuda_status(launch_release_int8_token(c, row, pool, stream));
}

extern "C" size_t kvq_kitty_key_page_bytes(const kvq_config *cfg) {
    if (check_kitty(cfg)) return 0;
    return (size_t)kitty_key_page_bytes(cfg->boost_k);   // group_k = 128 (check_kitty)
}

extern "C" size_t kvq_kitty_value_page_bytes(const kvq_config *cfg) {
    if (check_kitty(cfg)) return 0;
    return (size_t)cfg->group_k * KVQ_D / 4 + 4 * (size_t)cfg->group_k;
}

extern "C" kvq_status kv_quant_key_kitty(const kvq_config *cfg, const void *k, int64_t n_pages, int32_t score_mode,
                                         void *pages, cudaStream_t stream) {
    kvq_status s = check_kitty(cfg);
    if (s) return s;
    if (n_pages < 0 || (score_mode != 0 && score_mode != 1)) return KVQ_ERR_INVALID_ARG;
    if (n_pages == 0) return KVQ_OK;
    if ((s = ptrs_ok({k, pages}))) return s;
    return cuda_status(launch_quant_key_kitty(cfg, k, n_pages, score_mode, pages, stream));
}

extern "C" kvq_status kv_quant_value_kitty(const kvq_config *cfg, const void *v, int64_t n_pages, void *pages,
                                           cudaStream_t stream) {
    kvq_status s = check_kitty(cfg);
    if (s) return s;
    if (n_pages < 0) return KVQ_ERR_INVALID_ARG;
    if (n_pages == 0) return KVQ_OK;
    if ((s = ptrs_ok({v, pages}))) return s;
    return cuda_status(launch_quant_value_kitty(cfg, v, n_pages, pages, stream));
}

extern "C" kvq_status kv_quant_int8_dither(const kvq_config *cfg, const void *x, int64_t n_blocks,
                                           const int32_t *req_id, const int32_t *kv_head, const int32_t *tok0,
                                           int32_t layer, int32_t kv_sel, uint64_t seed, void *codes, void *scale,
                                           cudaStream_t stream) {
    kvq_status s = check_int8(cfg);
    if (s) return s;
    if (n_blocks < 0 || layer < 0 || layer >= (1 << 15) || (kv_sel != 0 && kv_sel != 1)) return KVQ_ERR_INVALID_ARG;
    if (n_blocks == 0) return KVQ_OK;
    if ((s = ptrs_ok({x, codes, scale}))) return s;
    if (!req_id || !kv_head || !tok0) return KVQ_ERR_INVALID_ARG;
    return cuda_status(launch_quant_int8(cfg, x, n_blocks, req_id, kv_head, tok0, layer, kv_sel, seed, codes, scale,
                                         stream));
}

// ---------------------------------------------------------------------------
// read side
// ---------------------------------------------------------------------------
extern "C" kvq_status kv_decode_attn_plan(const kvq_config *cfg, int32_t variant, int32_t batch, int32_t max_seq_len,
                                          int32_t *n_splits, size_t *workspace_bytes) {
    kvq_status s = variant == KVQ_VARIANT_KIVI    ? check_kivi(cfg)
                   : variant == KVQ_VARIANT_KITTY ? check_kitty(cfg)
                   : variant == KVQ_VARIANT_INT8  ? check_int8(cfg)
                   : variant == KVQ_VARIANT_INT8_TOKEN ? check_int8_token(cfg)
                   : variant == KVQ_VARIANT_KIVI_PAGED ? check_kivi(cfg)
                                                  : KVQ_ERR_INVALID_ARG;
    if (s) return s;
    if (batch < 1 || max_seq_len < 1) return KVQ_ERR_INVALID_ARG;
    DecodePlan p;
    plan_decode(cfg, variant, batch, max_seq_len, &p);
    if (n_splits) *n_splits = p.splits;
    if (workspace_bytes) *workspace_bytes = p.ws_bytes;
    return KVQ_OK;
}

static kvq_status check_ws(const kvq_config *cfg, int variant, int batch, int max_seq_len, const void *ws,
                           size_t ws_bytes, DecodePlan *p) {
    if (batch < 1 || max_seq_len < 1) return KVQ_ERR_INVALID_ARG;
    plan_decode(cfg, variant, batch, max_seq_len, p);
    if (!ws) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(ws)) return KVQ_ERR_MISALIGNED;
    if (ws_bytes < p->ws_bytes) return KVQ_ERR_WORKSPACE;
    return KVQ_OK;
}

static kvq_status stage1_kivi(const kvq_config *cfg, const kvq_kivi_cache *c, const void *q, void *ws, size_t wsb,
                              cudaStream_t st, DecodePlan *p) {
    kvq_status s = check_kivi(cfg);
    if (s) return s;
    if (!c) return KVQ_ERR_INVALID_ARG;
    if ((s = check_ws(cfg, KVQ_VARIANT_KIVI, c->batch, c->max_seq_len, ws, wsb, p))) return s;
    if ((s = ptrs_ok({q, c->seq_len, c->k_codes, c->k_sz, c->v_codes, c->v_sz, c->k_res, c->v_res}))) return s;
    if (kivi_gqa_supported(cfg)) return cuda_status(launch_decode_kivi_gqa(cfg, kivi_src(c), q, *p, ws, st));
    return cuda_status(launch_decode_kivi(cfg, kivi_src(c), q, *p, ws, st));
}


static kvq_status stage1_kivi_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const void *q, void *ws,
                                    size_t wsb, cudaStream_t st, DecodePlan *p) {
    kvq_status s = check_kivi(cfg);
    if (s) return s;
    if ((s = check_kivi_paged_cache(c))) return s;
    if ((s = check_ws(cfg, KVQ_VARIANT_KIVI_PAGED, c->batch, c->max_seq_len, ws, wsb, p))) return s;
    if ((s = ptrs_ok({q}))) return s;
    if (kivi_gqa_supported(cfg)) return cuda_status(launch_decode_kivi_gqa(cfg, kivi_src(c), q, *p, ws, st));
    return cuda_status(launch_decode_kivi(cfg, kivi_src(c), q, *p, ws, st));
}

static kvq_status stage1_kitty(const kvq_config *cfg, const kvq_kitty_cache *c, const void *q, void *ws, size_t wsb,
                               cudaStream_t st, DecodePlan *p) {
    kvq_status s = check_kitty(cfg);
    if (s) return s;
    if (!c) return KVQ_ERR_INVALID_ARG;
    if (cfg->boost_k > 92) return KVQ_ERR_UNSUPPORTED;   // key record must fit the decode stage slot
    if ((s = check_ws(cfg, KVQ_VARIANT_KITTY, c->batch, c->max_seq_len, ws, wsb, p))) return s;
    if ((s = check_kitty_cache(cfg, c, c->page_table != nullptr))) return s;
    if ((s = ptrs_ok({q}))) return s;
    if (kitty_gqa_supported(cfg)) return cuda_status(launch_decode_kitty_gqa(cfg, c, q, *p, ws, st));
    return cuda_status(launch_decode_kitty(cfg, c, q, *p, ws, st));
}

static kvq_status stage1_int8(const kvq_config *cfg, const kvq_int8_cache *c, const void *q, void *ws, size_t wsb,
                              cudaStream_t st, DecodePlan *p) {
    kvq_status s = check_int8(cfg);
    if (s) return s;
    if (!c) return KVQ_ERR_INVALID_ARG;
    if (c->layer < 0 || c->layer >= (1 << 15)) return KVQ_ERR_INVALID_ARG;
    if ((s = check_ws(cfg, KVQ_VARIANT_INT8, c->batch, c->max_seq_len, ws, wsb, p))) return s;
    if ((s = ptrs_ok({q, c->seq_len, c->req_id, c->k_codes, c->v_codes, c->k_scale, c->v_scale, c->k_tail,
                      c->v_tail})))
        return s;
    return cuda_status(launch_decode_int8(cfg, c, q, *p, ws, st));
}

static kvq_status stage1_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c, const void *q, void *ws,
                                    size_t wsb, cudaStream_t st, DecodePlan *p) {
    kvq_status s = check_int8_token(cfg);
    if (s) return s;
    if ((s = check_int8_token_cache(c))) return s;
    if ((s = check_ws(cfg, KVQ_VARIANT_INT8_TOKEN, c->batch, c->max_seq_len, ws, wsb, p))) return s;
    if ((s = ptrs_ok({q}))) return s;
    return cuda_status(launch_decode_int8_token(cfg, c, q, *p, ws, st));
}

extern "C" kvq_status kv_decode_attn_stage1(const kvq_config *cfg, int32_t variant, const void *cache, const void *q,
                                            void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    DecodePlan p;
    switch (variant) {
        case KVQ_VARIANT_KIVI:
            return stage1_kivi(cfg, static_cast<const kvq_kivi_cache *>(cache), q, workspace, workspace_bytes, stream, &p);
        case KVQ_VARIANT_KITTY:
            return stage1_kitty(cfg, static_cast<const kvq_kitty_cache *>(cache), q, workspace, workspace_bytes, stream,
                                &p);
        case KVQ_VARIANT_INT8:
            return stage1_int8(cfg, static_cast<const kvq_int8_cache *>(cache), q, workspace, workspace_bytes, stream, &p);
        case KVQ_VARIANT_INT8_TOKEN:
            return stage1_int8_token(cfg, static_cast<const kvq_int8_token_cache *>(cache), q, workspace,
                                     workspace_bytes, stream, &p);
        case KVQ_VARIANT_KIVI_PAGED:
            return stage1_kivi_paged(cfg, static_cast<const kvq_kivi_paged_cache *>(cache), q, workspace,
                                     workspace_bytes, stream, &p);
        default:
            return KVQ_ERR_INVALID_ARG;
    }
}

extern "C" kvq_status kv_decode_attn_merge(const kvq_config *cfg, int32_t variant, int32_t batch, int32_t max_seq_len,
                                           const void *workspace, size_t workspace_bytes, void *out,
                                           cudaStream_t stream) {
    kvq_status s = variant == KVQ_VARIANT_KIVI    ? check_kivi(cfg)
                   : variant == KVQ_VARIANT_KITTY ? check_kitty(cfg)
                   : variant == KVQ_VARIANT_INT8  ? check_int8(cfg)
                   : variant == KVQ_VARIANT_INT8_TOKEN ? check_int8_token(cfg)
                   : variant == KVQ_VARIANT_KIVI_PAGED ? check_kivi(cfg)
                                                  : KVQ_ERR_INVALID_ARG;
    if (s) return s;
    DecodePlan p;
    if ((s = check_ws(cfg, variant, batch, max_seq_len, workspace, workspace_bytes, &p))) return s;
    if ((s = ptrs_ok({out}))) return s;
    return cuda_status(launch_merge(cfg, batch, p, workspace, out, stream));
}

extern "C" kvq_status kv_decode_attn(const kvq_config *cfg, const kvq_kivi_cache *cache, const void *q, void *out,
                                     void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!out) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(out)) return KVQ_ERR_MISALIGNED;
    DecodePlan p;
    kvq_status s = stage1_kivi(cfg, cache, q, workspace, workspace_bytes, stream, &p);
    if (s) return s;
    return cuda_status(launch_merge(cfg, cache->batch, p, workspace, out, stream));
}

extern "C" kvq_status kv_decode_attn_kitty(const kvq_config *cfg, const kvq_kitty_cache *cache, const void *q,
                                           void *out, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!out) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(out)) return KVQ_ERR_MISALIGNED;
    DecodePlan p;
    kvq_status s = stage1_kitty(cfg, cache, q, workspace, workspace_bytes, stream, &p);
    if (s) return s;
    return cuda_status(launch_merge(cfg, cache->batch, p, workspace, out, stream));
}

extern "C" kvq_status kv_decode_attn_int8(const kvq_config *cfg, const kvq_int8_cache *cache, const void *q,
                                          void *out, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!out) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(out)) return KVQ_ERR_MISALIGNED;
    DecodePlan p;
    kvq_status s = stage1_int8(cfg, cache, q, workspace, workspace_bytes, stream, &p);
    if (s) return s;
    return cuda_status(launch_merge(cfg, cache->batch, p, workspace, out, stream));
}

extern "C" kvq_status kv_decode_attn_kivi_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *cache,
                                                const void *q, void *out, void *workspace, size_t workspace_bytes,
                                                cudaStream_t stream) {
    if (!out) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(out)) return KVQ_ERR_MISALIGNED;
    DecodePlan p;
    kvq_status s = stage1_kivi_paged(cfg, cache, q, workspace, workspace_bytes, stream, &p);
    if (s) return s;
    return cuda_status(launch_merge(cfg, cache->batch, p, workspace, out, stream));
}

extern "C" kvq_status kv_decode_attn_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *cache,
                                                const void *q, void *out, void *workspace, size_t workspace_bytes,
                                                cudaStream_t stream) {
    if (!out) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(out)) return KVQ_ERR_MISALIGNED;
    DecodePlan p;
    kvq_status s = stage1_int8_token(cfg, cache, q, workspace, workspace_bytes, stream, &p);
    if (s) return s;
    return cuda_status(launch_merge(cfg, cache->batch, p, workspace, out, stream));
}

// ---------------------------------------------------------------------------
// diagnostics
// ---------------------------------------------------------------------------
extern "C" kvq_status kvq_philox4x32_10(const uint32_t *ctr, const uint32_t *key, int64_t n, uint32_t *out,
                                        cudaStream_t stream) {
    if (n < 0) return KVQ_ERR_INVALID_ARG;
    if (n == 0) return KVQ_OK;
    kvq_status s = ptrs_ok({ctr, key, out});
    if (s) return s;
    return cuda_status(launch_philox(ctr, key, n, out, stream));
}

#ifdef KVQ_FAULT_INJECT
namespace kvq {
TestInject g_test_inject;
}
// Test builds only: arm (skip_stage >= 0) or disarm (-1) the KIVI decode
// wait injection; spin_limit 0 restores the product limit.
extern "C" KVQ_API void kvq_test_inject_wait(int skip_stage, unsigned spin_limit) {
    kvq::g_test_inject.skip_stage = skip_stage;
    kvq::g_test_inject.spin_limit = spin_limit;
}
#endif

extern "C" kvq_status kvq_get_device_error(uint32_t *flags) {
    if (!flags) return KVQ_ERR_INVALID_ARG;
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return KVQ_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return KVQ_ERR_CUDA;
    *flags = v;
    return KVQ_OK;
}

extern "C" const char *kvq_status_string(kvq_status s) {
    switch (s) {
        case KVQ_OK: return "ok";
        case KVQ_ERR_INVALID_ARG: return "invalid argument";
        case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
        case KVQ_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case KVQ_ERR_CUDA: return "CUDA error";
        case KVQ_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

extern "C" const char *kvq_version(void) { return "kvq 0.1 (sm_103a)"; }
