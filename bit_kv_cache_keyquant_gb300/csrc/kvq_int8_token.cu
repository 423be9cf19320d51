// Token-granular INT8 over a slot pool, write side (WitCert, the SGLang
// storage subsection of sec. 6.2): the engine's KV pool is paged at token
// slots, so every token is quantized on its own when it is written, with one
// fp16 scale amax/126.5 per group of Gc channels and the Philox4x32-10
// dither keyed by (layer, kv head, slot, channel).
//
//   quant_int8_token_kernel   one warp per (token, kv head); lane l owns
//                             channels 4l..4l+3, so one Philox call gives
//                             its four dithers and the group amax is a
//                             shuffle over Gc/4 lanes.
//   slot_pool_init_kernel     free stack = every slot.
//   slot_alloc_kernel         one CTA: the rows that append this step take
//                             slots from the top of the free stack in row
//                             order (a block-wide scan), so the assignment
//                             and therefore the dither are the same on every
//                             replay of a captured graph.
//   append_int8_token_kernel  one CTA per row: quantize the row's new K and V
//                             into its new slot, then seq_len += 1.
//   slot_release_kernel       one CTA: push a request's slots back.
#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_quant.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

// One token of one kv head: lane holds channels 4*lane..4*lane+3 of src.
// Returns the lane's four codes packed little-endian and the scale of its
// channel group (all lanes of a group agree).
template <int LG>
__device__ __forceinline__ void int8t_token_quant(const uint16_t *__restrict__ src, int lane, uint32_t slot,
                                                  uint32_t c2, uint32_t k0, uint32_t k1, uint32_t &word,
                                                  uint16_t &s) {
    const uint2 u = *reinterpret_cast<const uint2 *>(src + 4 * lane);
    const float xs[4] = {h2f(lo16(u.x)), h2f(hi16(u.x)), h2f(lo16(u.y)), h2f(hi16(u.y))};
    float a = fmaxf(fmaxf(fabsf(xs[0]), fabsf(xs[1])), fmaxf(fabsf(xs[2]), fabsf(xs[3])));
#pragma unroll
    for (int o = 1; o < LG; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    s = f2h_rn(__fdiv_rn(a, 126.5f));
    const float sf = h2f(s), rf = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
    const uint4 r = philox4x32_10(make_uint4(slot, (uint32_t)lane, c2, 0u), k0, k1);
    const uint32_t wr[4] = {r.x, r.y, r.z, r.w};
    word = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int code = 0;
        if (sf != 0.0f) code = dither_code(xs[i], sf, rf, dither_from_word(wr[i]));
        word |= ((uint32_t)(code & 0xFF)) << (8 * i);
    }
}

template <int LG>
__device__ __forceinline__ void int8t_store(int8_t *__restrict__ codes, uint16_t *__restrict__ scale, int64_t rec,
                                            int lane, uint32_t word, uint16_t s) {
    constexpr int NSC = KVQ_D / (4 * LG);   // scales per record
    reinterpret_cast<uint32_t *>(codes + rec * KVQ_D)[lane] = word;
    if (lane % LG == 0) scale[rec * NSC + lane / LG] = s;
}

template <int LG>
__global__ void __launch_bounds__(256) quant_int8_token_kernel(const uint16_t *__restrict__ x, int64_t n, int Hkv,
                                                               const int32_t *__restrict__ slots, int n_slots,
                                                               uint32_t c2base, uint32_t k0, uint32_t k1,
                                                               int8_t *__restrict__ codes,
                                                               uint16_t *__restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < n * Hkv; w += nw) {
        const int64_t i = w / Hkv;
        const int h = (int)(w - i * Hkv);
        const int32_t slot = slots[i];
        if (slot < 0 || slot >= n_slots) continue;
        uint32_t word;
        uint16_t s;
        int8t_token_quant<LG>(x + w * KVQ_D, lane, (uint32_t)slot, c2base | (uint32_t)h, k0, k1, word, s);
        int8t_store<LG>(codes, scale, (int64_t)slot * Hkv + h, lane, word, s);
    }
}

__global__ void slot_pool_init_kernel(int32_t *__restrict__ free_slots, int32_t *__restrict__ top, int capacity) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < capacity; i += gridDim.x * blockDim.x)
        free_slots[i] = capacity - 1 - i;
    if (blockIdx.x == 0 && threadIdx.x == 0) *top = capacity;
}

// Exclusive scan of one flag per thread over a block of 1024 threads.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wt = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
        int wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += t;
        }
        warp_tot[lane] = wi - wt;   // exclusive prefix of warp totals
        if (lane == 31) warp_tot[32] = wi;
    }
    __syncthreads();
    const int r = warp_tot[warp] + incl - v;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

// Rows b with base <= L = seq_len[b] < cap and (L - base) % unit == 0 take one
// id each (token slots: unit 1; pages of 128 tokens: unit 128; Kitty pages
// start after the base = S sink tokens) for table[b][(L - base) / unit].
__global__ void __launch_bounds__(1024) slot_alloc_kernel(const int32_t *__restrict__ seq_len,
                                                          int32_t *__restrict__ table, int B, int cap, int unit,
                                                          int stride, int base,
                                                          const int32_t *__restrict__ free_slots,
                                                          int32_t *__restrict__ top, int capacity,
                                                          unsigned *err) {
    __shared__ int warp_tot[33];
    __shared__ int s_need;
    if (threadIdx.x == 0) s_need = 0;
    __syncthreads();
    int cnt = 0;
    bool full = false;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int L = seq_len[b];
        if (L >= 0 && L < cap) cnt += (L >= base && (L - base) % unit == 0) ? 1 : 0;
        else full = true;
    }
    if (full) atomicOr(err, KVQ_DEVICE_ERR_CAPACITY);
    atomicAdd(&s_need, cnt);
    __syncthreads();
    const int need = s_need;
    const int t0 = *top;
    const bool fail = need > t0 || t0 > capacity;
    if (fail && threadIdx.x == 0) atomicOr(err, KVQ_DEVICE_ERR_POOL);
    int done = 0;
    for (int c0 = 0; c0 < B; c0 += blockDim.x) {
        const int b = c0 + threadIdx.x;
        const int L = b < B ? seq_len[b] : -1;
        const int f = (L >= base && L < cap && (L - base) % unit == 0) ? 1 : 0;
        int tot;
        const int r = block_excl_scan(f, warp_tot, tot) + done;
        if (f) table[(int64_t)b * stride + (L - base) / unit] = fail ? -1 : free_slots[t0 - 1 - r];
        done += tot;
    }
    __syncthreads();
    if (threadIdx.x == 0 && !fail) *top = t0 - need;
}

struct AppendT {
    int32_t *seq_len;
    const int32_t *table;
    const uint16_t *k_new, *v_new;
    int8_t *k_codes, *v_codes;
    uint16_t *k_scale, *v_scale;
    int Hkv, cap, n_slots;
    uint32_t ctr2_layer, k0, k1;
};

template <int LG>
__global__ void __launch_bounds__(256) append_int8_token_kernel(AppendT P) {
    const int b = blockIdx.x;
    const int L = P.seq_len[b];
    if (L < 0 || L >= P.cap) return;
    const int32_t slot = P.table[(int64_t)b * P.cap + L];
    if (slot < 0 || slot >= P.n_slots) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < 2 * P.Hkv; j += (int)(blockDim.x >> 5)) {
        const int sel = j >= P.Hkv ? 1 : 0;
        const int h = j - sel * P.Hkv;
        const uint16_t *src = (sel ? P.v_new : P.k_new) + ((int64_t)b * P.Hkv + h) * KVQ_D;
        uint32_t word;
        uint16_t s;
        int8t_token_quant<LG>(src, lane, (uint32_t)slot, P.ctr2_layer | ((uint32_t)sel << 16) | (uint32_t)h, P.k0,
                              P.k1, word, s);
        int8t_store<LG>(sel ? P.v_codes : P.k_codes, sel ? P.v_scale : P.k_scale, (int64_t)slot * P.Hkv + h, lane,
                        word, s);
    }
    __syncthreads();
    if (threadIdx.x == 0) P.seq_len[b] = L + 1;
}

// Push the ids of request `row` (table[row][0 .. ceil(max(seq_len[row] - base, 0) / unit))) back.
__global__ void __launch_bounds__(1024) slot_release_kernel(int32_t *__restrict__ seq_len,
                                                            const int32_t *__restrict__ table, int row, int cap,
                                                            int unit, int stride, int base,
                                                            int32_t *__restrict__ free_slots,
                                                            int32_t *__restrict__ top, int capacity, unsigned *err) {
    const int L = seq_len[row];
    const int n = L >= 0 && L <= cap ? (max(L - base, 0) + unit - 1) / unit : -1;
    const int t0 = *top;
    if (n < 0 || t0 < 0 || t0 + n > capacity) {
        if (threadIdx.x == 0) atomicOr(err, KVQ_DEVICE_ERR_POOL);
        return;
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x) free_slots[t0 + i] = table[(int64_t)row * stride + i];
    __syncthreads();
    if (threadIdx.x == 0) {
        *top = t0 + n;
        seq_len[row] = 0;
    }
}

template <typename F>
cudaError_t by_group(int Gc, F f) {
    switch (Gc) {
        case 32: return f(std::integral_constant<int, 8>());
        case 64: return f(std::integral_constant<int, 16>());
        case 128: return f(std::integral_constant<int, 32>());
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_quant_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c, const void *x, int64_t n,
                                    const int32_t *slots, int kv_sel, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int Hkv = cfg->n_kv_heads;
    int64_t grid = (n * Hkv + 7) / 8;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (grid > cap) grid = cap;
    const uint32_t c2base = ((uint32_t)c->layer << 17) | ((uint32_t)(kv_sel & 1) << 16);
    const uint32_t k0 = (uint32_t)(c->seed & 0xFFFFFFFFu), k1 = (uint32_t)(c->seed >> 32);
    int8_t *codes = static_cast<int8_t *>(const_cast<void *>(kv_sel ? c->v_codes : c->k_codes));
    uint16_t *scale = static_cast<uint16_t *>(const_cast<void *>(kv_sel ? c->v_scale : c->k_scale));
    const uint16_t *xs = static_cast<const uint16_t *>(x);
    cudaError_t e = by_group(cfg->int8_group, [&](auto lg) {
        quant_int8_token_kernel<decltype(lg)::value><<<(unsigned)grid, 256, 0, st>>>(
            xs, n, Hkv, slots, c->n_slots, c2base, k0, k1, codes, scale);
        return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_slot_pool_init(const kvq_slot_pool *pool, cudaStream_t st) {
    int grid = (pool->capacity + 255) / 256;
    if (grid > num_sms() * 8) grid = num_sms() * 8;
    if (grid < 1) grid = 1;
    slot_pool_init_kernel<<<grid, 256, 0, st>>>(pool->slots, pool->top, pool->capacity);
    return cudaGetLastError();
}

cudaError_t launch_append_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c, const kvq_slot_pool *pool,
                                     const void *k_new, const void *v_new, cudaStream_t st) {
    unsigned *err = device_error_ptr();
    if (!err) return cudaErrorInvalidDevicePointer;
    int32_t *table = const_cast<int32_t *>(c->slot_table);
    int32_t *seq_len = const_cast<int32_t *>(c->seq_len);
    cudaError_t e = launch_alloc_ids(seq_len, table, c->batch, c->max_seq_len, 1, c->max_seq_len, 0, pool, st);
    if (e != cudaSuccess) return e;
    AppendT P;
    P.seq_len = seq_len;
    P.table = table;
    P.k_new = static_cast<const uint16_t *>(k_new);
    P.v_new = static_cast<const uint16_t *>(v_new);
    P.k_codes = static_cast<int8_t *>(const_cast<void *>(c->k_codes));
    P.v_codes = static_cast<int8_t *>(const_cast<void *>(c->v_codes));
    P.k_scale = static_cast<uint16_t *>(const_cast<void *>(c->k_scale));
    P.v_scale = static_cast<uint16_t *>(const_cast<void *>(c->v_scale));
    P.Hkv = cfg->n_kv_heads;
    P.cap = c->max_seq_len;
    P.n_slots = c->n_slots;
    P.ctr2_layer = (uint32_t)c->layer << 17;
    P.k0 = (uint32_t)(c->seed & 0xFFFFFFFFu);
    P.k1 = (uint32_t)(c->seed >> 32);
    e = by_group(cfg->int8_group, [&](auto lg) {
        append_int8_token_kernel<decltype(lg)::value><<<(unsigned)c->batch, 256, 0, st>>>(P);
        return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_release_int8_token(const kvq_int8_token_cache *c, int row, const kvq_slot_pool *pool,
                                      cudaStream_t st) {
    return launch_release_ids(const_cast<int32_t *>(c->seq_len), c->slot_table, row, c->max_seq_len, 1,
                              c->max_seq_len, 0, pool, st);
}

cudaError_t launch_alloc_ids(const int32_t *seq_len, int32_t *table, int batch, int cap, int unit, int stride,
                             int base, const kvq_slot_pool *pool, cudaStream_t st) {
    unsigned *err = device_error_ptr();
    if (!err) return cudaErrorInvalidDevicePointer;
    slot_alloc_kernel<<<1, 1024, 0, st>>>(seq_len, table, batch, cap, unit, stride, base, pool->slots, pool->top,
                                          pool->capacity, err);
    return cudaGetLastError();
}

cudaError_t launch_release_ids(int32_t *seq_len, const int32_t *table, int row, int cap, int unit, int stride,
                               int base, const kvq_slot_pool *pool, cudaStream_t st) {
    unsigned *err = device_error_ptr();
    if (!err) return cudaErrorInvalidDevicePointer;
    slot_release_kernel<<<1, 1024, 0, st>>>(seq_len, table, row, cap, unit, stride, base, pool->slots, pool->top,
                                            pool->capacity, err);
    return cudaGetLastError();
}

}  // namespace kvq
