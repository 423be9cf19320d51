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

__global__ void __launch_bounds__(128) merge_kernel(const float *__restrict__ o, const float *__restrict__ lse,
                                                    int splits, uint16_t *__restrict__ out) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t row = blockIdx.x;
    const int c = threadIdx.x;
    const float *ls = lse + row * splits;
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, ls[s]);
    float acc = 0.f, den = 0.f;
    if (M > -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float l = ls[s];
            if (l == -INFINITY) continue;
            const float w = exp2f(l - M);
            den += w;
            acc += w * o[(row * splits + s) * KVQ_D + c];
        }
    }
    out[row * KVQ_D + c] = f2h_rn(den > 0.f ? acc / den : 0.f);
}

cudaError_t launch_merge(const kvq_config *cfg, int batch, const DecodePlan &p, const void *ws, void *out,
                         cudaStream_t st) {
    const uint8_t *w = static_cast<const uint8_t *>(ws);
    const int64_t rows = (int64_t)batch * cfg->n_q_heads;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)rows);
    lc.blockDim = dim3(128);
    lc.dynamicSmemBytes = 0;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, merge_kernel, reinterpret_cast<const float *>(w + p.off_o),
                              reinterpret_cast<const float *>(w + p.off_lse), p.splits, static_cast<uint16_t *>(out));
}

}  // namespace kvq
