// Host-side declarations shared by the kvq translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/kvq.h"

namespace kvq {

struct DecodePlan {
    int splits;        // splits per (batch row, query head)
    int chunk;         // tokens per split (multiple of 128)
    size_t ws_bytes;   // workspace bytes
    size_t off_o;      // byte offset of o_s  fp32 [B][Hq][splits][D]
    size_t off_lse;    // byte offset of lse_s fp32 [B][Hq][splits]
};

// A dense or a paged KIVI cache as the decode kernels read it: dense caches
// set the four code / parameter arrays, paged caches the page table and pool.
struct KiviSrc {
    int batch = 0, max_seq_len = 0;
    const int32_t *seq_len = nullptr;
    const void *k_codes = nullptr, *k_sz = nullptr, *v_codes = nullptr, *v_sz = nullptr;
    const int32_t *page_table = nullptr;
    const void *pages = nullptr;
    int n_pages = 0;
    const void *k_res = nullptr, *v_res = nullptr;
};

inline KiviSrc kivi_src(const kvq_kivi_cache *c) {
    KiviSrc s;
    s.batch = c->batch;
    s.max_seq_len = c->max_seq_len;
    s.seq_len = c->seq_len;
    s.k_codes = c->k_codes;
    s.k_sz = c->k_sz;
    s.v_codes = c->v_codes;
    s.v_sz = c->v_sz;
    s.k_res = c->k_res;
    s.v_res = c->v_res;
    return s;
}

inline KiviSrc kivi_src(const kvq_kivi_paged_cache *c) {
    KiviSrc s;
    s.batch = c->batch;
    s.max_seq_len = c->max_seq_len;
    s.seq_len = c->seq_len;
    s.page_table = c->page_table;
    s.pages = c->pages;
    s.n_pages = c->n_pages;
    s.k_res = c->k_res;
    s.v_res = c->v_res;
    return s;
}

// Byte offset of channel quad c4 (channels 4 c4 .. 4 c4 + 3, c4 = 8g + q) of token t in 2-bit KIVI value
// codes stored in value tiles (kivi_value_tiles), of one (batch row, kv head) or page record: 32-token tiles
// of 1024 bytes in the fragment order of the grouped-query kernel's tensor-core value products.  With t % 32 = 16 kv + 4 i + r the byte is
// tile * 1024 + kv * 512 + (4q + r) * 16 + 4g + i, so lane 4q + r of a warp finds byte c4 of the tokens
// r, r + 4, r + 8, r + 12 of a 16-token half (for g = 0..3) in one 16-byte chunk.
__host__ __device__ constexpr int64_t kivi_value_byte(int64_t t, int c4) {
    return (t >> 5) * 1024 + ((t >> 4) & 1) * 512 + (4 * (c4 & 7) + (int)(t & 3)) * 16 + 4 * (c4 >> 3) + (int)((t >> 2) & 3);
}

// Byte offset of channel c of token t in 4-bit KIVI value tiles (32-token tiles of 2048 bytes); the code is
// nibble c / 64 of the byte, which holds channels c % 64 and c % 64 + 64 of one token.  With
// t % 32 = 16 kv + 8 w + 4 s + r and c % 64 = 16 m + 8 h + q the byte is
// tile * 2048 + kv * 1024 + (4q + r) * 32 + (2m + w) * 4 + 2h + s: lane 4q + r finds in its 32 bytes of a
// 16-token half the A words of m-tiles m (low nibbles) and m + 4 (high nibbles), two words each.
__host__ __device__ constexpr int64_t kivi_value_byte4(int64_t t, int c) {
    return (t >> 5) * 2048 + ((t >> 4) & 1) * 1024 + (4 * (c & 7) + (int)(t & 3)) * 32 +
           (2 * ((c & 63) >> 4) + (int)((t >> 3) & 1)) * 4 + 2 * ((c >> 3) & 1) + (int)((t >> 2) & 1);
}

// Rows of a Kitty key page's high plane: the K boosted channels rounded up to
// a multiple of 4 (each 4-byte word of the plane holds a group of four rows).
__host__ __device__ constexpr int kitty_high_rows(int K) { return (K + 3) & ~3; }

// bytes of one Kitty key page record of 128 tokens (D = 128): low plane, high plane, idx [D], s [D], z [D]
__host__ __device__ constexpr int64_t kitty_key_page_bytes(int K) {
    return 128LL * 128 / 4 + (int64_t)kitty_high_rows(K) * 128 / 4 + 128 + 4 * 128;
}

// bytes of one paged KIVI page record: key codes, key (s, z), value codes, value (s, z) of 128 tokens
inline int64_t kivi_page_bytes(int bits_k, int bits_v) {
    return 16LL * 128 * bits_k + 2048 + 16LL * 128 * bits_v + 2048;   // D = 128
}

// Opts a kernel into `smem` bytes of dynamic shared memory, once per device:
// `done` is that kernel's own bitmask of devices already set up.  Host
// threads that make a first launch together may both set the attribute (it
// is idempotent); none can skip it.
template <typename Kern>
inline cudaError_t smem_opt_in(Kern *kernel, size_t smem, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

#ifdef KVQ_FAULT_INJECT
// Test builds only (never the product library): the KIVI decode producer of
// CTA 0 leaves its stage skip_stage unfilled, and the KIVI decode waits give
// up after spin_limit tries when it is nonzero, so that a test can watch the
// bounded waits expire.  Set through kvq_test_inject_wait.
struct TestInject {
    int skip_stage = -1;
    unsigned spin_limit = 0;
};
extern TestInject g_test_inject;
#endif

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
cudaError_t launch_decode_kivi(const kvq_config *cfg, const KiviSrc &c, const void *q,
                               const DecodePlan &p, void *ws, cudaStream_t st);
// grouped-query KIVI decode on the tensor cores (2 <= n_q_heads / n_kv_heads <= 4)
bool kivi_gqa_supported(const kvq_config *cfg);
// KIVI value codes of a config that decodes on the grouped-query kernel are stored in its value tiles
// (kivi_value_byte at 2 bits, kivi_value_byte4 at 4 bits); every other KIVI value cache is token-major
bool kivi_value_tiles(const kvq_config *cfg);
int kivi_gqa_units_per_kv_head(const kvq_config *cfg);   // 1, or 2 for 4 < g <= 8
cudaError_t launch_decode_kivi_gqa(const kvq_config *cfg, const KiviSrc &c, const void *q,
                                   const DecodePlan &p, void *ws, cudaStream_t st);
// grouped-query Kitty decode on the tensor cores (2 <= n_q_heads / n_kv_heads <= 4)
bool kitty_gqa_supported(const kvq_config *cfg);
int kitty_gqa_units_per_kv_head(const kvq_config *cfg);
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
// paged KIVI write side
cudaError_t launch_quant_key_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const void *k, int64_t n,
                                   int group0, int row, int kvh, cudaStream_t st);
cudaError_t launch_quant_value_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const void *v, int64_t n,
                                     int tok0, int row, int kvh, cudaStream_t st);
cudaError_t launch_append_kivi_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const kvq_slot_pool *pool,
                                     const void *k_new, const void *v_new, cudaStream_t st);
// free-id stack (token slots: unit 1; pages: unit 128, after `base` sink tokens for Kitty): rows with
// seq_len >= base and (seq_len - base) % unit == 0 take an id for table[b][(seq_len - base) / unit];
// release pushes table[row][0 .. ceil(max(seq_len - base, 0) / unit)) back
cudaError_t launch_alloc_ids(const int32_t *seq_len, int32_t *table, int batch, int cap, int unit, int stride,
                             int base, const kvq_slot_pool *pool, cudaStream_t st);
cudaError_t launch_release_ids(int32_t *seq_len, const int32_t *table, int row, int cap, int unit, int stride,
                               int base, const kvq_slot_pool *pool, cudaStream_t st);
cudaError_t launch_quant_key_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const void *k, int64_t n,
                                         int page0, int row, int kvh, int score_mode, cudaStream_t st);
cudaError_t launch_quant_value_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const void *v, int64_t n,
                                           int page0, int row, int kvh, cudaStream_t st);
cudaError_t launch_append_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const kvq_slot_pool *pool,
                                      const void *k_new, const void *v_new, int score_mode, cudaStream_t st);
cudaError_t launch_merge(const kvq_config *cfg, int batch, const DecodePlan &p, const void *ws, void *out,
                         cudaStream_t st);

cudaError_t launch_philox(const uint32_t *ctr, const uint32_t *key, int64_t n, uint32_t *out, cudaStream_t st);

}  // namespace kvq
