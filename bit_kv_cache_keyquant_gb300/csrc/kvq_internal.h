// Host-side declarations shared by the kvq translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

struct DecodePlan {
    int splits;        // splits per (batch row, query head)
    int chunk;         // tokens per split (multiple of 128)
    size_t ws_bytes;   // workspace bytes
    size_t off_o;      // byte offset of o_s  fp32 [B][Hq][splits][D]
    size_t off_lse;    // byte offset of lse_s fp32 [B][Hq][splits]
};

int num_sms();
unsigned *device_error_ptr();   // device address of the error bitmask (current device)

float sm_scale_of(const kvq_config *cfg);
kvq_status plan_decode(const kvq_config *cfg, int variant, int batch, int max_seq_len, DecodePlan *p);

// launchers (return a CUDA error code; arguments already validated)
cudaError_t launch_quant_key_kivi(const kvq_config *cfg, const void *k, int64_t n_groups, void *codes,
                                  void *sz, cudaStream_t st);
cudaError_t launch_quant_value_kivi(const kvq_config *cfg, const void *v, int64_t n_tokens, void *codes,
                                    void *sz, cudaStream_t st);
cudaError_t launch_quant_key_kitty(const kvq_config *cfg, const void *k, int64_t n_pages, int score_mode,
                                   void *pages, cudaStream_t st);
cudaError_t launch_quant_value_kitty(const kvq_config *cfg, const void *v, int64_t n_pages, void *pages,
                                     cudaStream_t st);
cudaError_t launch_quant_int8(const kvq_config *cfg, const void *x, int64_t n_blocks, const int32_t *req,
                              const int32_t *head, const int32_t *tok0, int layer, int kv_sel, uint64_t seed,
                              void *codes, void *scale, cudaStream_t st);

cudaError_t launch_append_kivi(const kvq_config *cfg, const kvq_kivi_cache *c, const void *k_new, const void *v_new,
                               cudaStream_t st);
cudaError_t launch_append_int8(const kvq_config *cfg, const kvq_int8_cache *c, const void *k_new, const void *v_new,
                               cudaStream_t st);
cudaError_t launch_append_kitty(const kvq_config *cfg, const kvq_kitty_cache *c, const void *k_new, const void *v_new,
                                int score_mode, cudaStream_t st);
cudaError_t launch_decode_kivi(const kvq_config *cfg, const kvq_kivi_cache *c, const void *q,
                               const DecodePlan &p, void *ws, cudaStream_t st);
// grouped-query KIVI decode on the tensor cores (2 <= n_q_heads / n_kv_heads <= 4)
bool kivi_gqa_supported(const kvq_config *cfg);
cudaError_t launch_decode_kivi_gqa(const kvq_config *cfg, const kvq_kivi_cache *c, const void *q,
                                   const DecodePlan &p, void *ws, cudaStream_t st);
// grouped-query Kitty decode on the tensor cores (2 <= n_q_heads / n_kv_heads <= 4)
bool kitty_gqa_supported(const kvq_config *cfg);
cudaError_t launch_decode_kitty_gqa(const kvq_config *cfg, const kvq_kitty_cache *c, const void *q,
                                    const DecodePlan &p, void *ws, cudaStream_t st);
cudaError_t launch_decode_kitty(const kvq_config *cfg, const kvq_kitty_cache *c, const void *q,
                                const DecodePlan &p, void *ws, cudaStream_t st);
cudaError_t launch_decode_int8(const kvq_config *cfg, const kvq_int8_cache *c, const void *q,
                               const DecodePlan &p, void *ws, cudaStream_t st);
cudaError_t launch_decode_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c, const void *q,
                                     const DecodePlan &p, void *ws, cudaStream_t st);
cudaError_t launch_quant_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c, const void *x, int64_t n,
                                    const int32_t *slots, int kv_sel, cudaStream_t st);
cudaError_t launch_slot_pool_init(const kvq_slot_pool *pool, cudaStream_t st);
cudaError_t launch_append_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c, const kvq_slot_pool *pool,
                                     const void *k_new, const void *v_new, cudaStream_t st);
cudaError_t launch_release_int8_token(const kvq_int8_token_cache *c, int row, const kvq_slot_pool *pool,
                                      cudaStream_t st);
cudaError_t launch_merge(const kvq_config *cfg, int batch, const DecodePlan &p, const void *ws, void *out,
                         cudaStream_t st);

cudaError_t launch_philox(const uint32_t *ctr, const uint32_t *key, int64_t n, uint32_t *out, cudaStream_t st);

}  // namespace kvq
