// a4: split-KV merge.  Stage 1 leaves, per (batch row, query head, split),
// o_s = acc_s / l_s and lse_s = m_s + log2 l_s (base-2 softmax domain);
//   LSE = log2 sum_s 2^(lse_s),  o = sum_s 2^(lse_s - LSE) o_s  -> fp16.
// (WitCert sec. 6.2.2: stage 2 merges the per-split results with LSE weights.)
// The merge is launched as a programmatic dependent of stage 1 on the same
// stream: its CTAs may be scheduled while stage 1 drains and wait in
// griddepcontrol.wait until stage 1 has completed and its writes are visible.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

// One warp per (batch row, query head); lane i holds channels 4i..4i+3.  The
// split weights 2^(lse_s - LSE) are computed one split per lane and
// broadcast by shuffles; the o_s rows are read eight at a time with every
// load of a batch in flight together, so a row costs a few memory latencies
// instead of one per split.  An empty split (lse_s = -inf) has weight 0 and
// its o_s is not used.
constexpr int MERGE_ROWS = 4;             // rows (warps) per CTA
constexpr int MERGE_BATCH = 8;            // o_s rows in flight per lane

__global__ void __launch_bounds__(32 * MERGE_ROWS) merge_kernel(const float *__restrict__ o,
                                                                const float *__restrict__ lse, int splits,
                                                                int64_t rows, uint16_t *__restrict__ out) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * MERGE_ROWS + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float *ls = lse + row * splits;
    float M = -INFINITY;
    for (int s = lane; s < splits; s += 32) M = fmaxf(M, ls[s]);
    M = warp_max(M);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (M > -INFINITY) {
        const float4 *orow = reinterpret_cast<const float4 *>(o + row * splits * KVQ_D) + lane;
        for (int s0 = 0; s0 < splits; s0 += 32) {
            const float l = s0 + lane < splits ? ls[s0 + lane] : -INFINITY;
            const float w = l > -INFINITY ? exp2f(l - M) : 0.f;
            den += w;
            const int n = min(32, splits - s0);
            for (int j0 = 0; j0 < n; j0 += MERGE_BATCH) {
                float4 v[MERGE_BATCH];
#pragma unroll
                for (int k = 0; k < MERGE_BATCH; ++k)
                    v[k] = j0 + k < n ? orow[(int64_t)(s0 + j0 + k) * (KVQ_D / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < MERGE_BATCH; ++k) {
                    const float wk = __shfl_sync(0xFFFFFFFFu, w, (j0 + k) & 31);
                    if (j0 + k < n && wk > 0.f) {
                        acc.x = fmaf(wk, v[k].x, acc.x);
                        acc.y = fmaf(wk, v[k].y, acc.y);
                        acc.z = fmaf(wk, v[k].z, acc.z);
                        acc.w = fmaf(wk, v[k].w, acc.w);
                    }
                }
            }
        }
        den = warp_sum(den);
    }
    if (den > 0.f) {
        acc.x /= den;
        acc.y /= den;
        acc.z /= den;
        acc.w /= den;
    }
    const uint32_t h01 = (uint32_t)f2h_rn(acc.x) | ((uint32_t)f2h_rn(acc.y) << 16);
    const uint32_t h23 = (uint32_t)f2h_rn(acc.z) | ((uint32_t)f2h_rn(acc.w) << 16);
    *reinterpret_cast<uint2 *>(out + row * KVQ_D + 4 * lane) = make_uint2(h01, h23);
}

cudaError_t launch_merge(const kvq_config *cfg, int batch, const DecodePlan &p, const void *ws, void *out,
                         cudaStream_t st) {
    const uint8_t *w = static_cast<const uint8_t *>(ws);
    const int64_t rows = (int64_t)batch * cfg->n_q_heads;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((rows + MERGE_ROWS - 1) / MERGE_ROWS));
    lc.blockDim = dim3(32 * MERGE_ROWS);
    lc.dynamicSmemBytes = 0;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, merge_kernel, reinterpret_cast<const float *>(w + p.off_o),
                              reinterpret_cast<const float *>(w + p.off_lse), p.splits, rows,
                              static_cast<uint16_t *>(out));
}

}  // namespace kvq
