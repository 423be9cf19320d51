// Allocation-free variant of the KIVI decode call.
//
// Some callers cannot hand the library a workspace buffer: engines whose own
// pool owns all device memory and forbids allocations it did not plan, or
// deployments that allow no device allocation after start-up.  For them,
// kv_decode_attn_noalloc runs the same two kernels as kv_decode_attn (split
// stage 1, then the LSE merge) with the split workspace placed in a fixed
// array compiled into this library instead of a caller buffer.
//
// The array (KVQ_NOALLOC_SCRATCH_BYTES) lives in device memory of every GPU
// on which the library is loaded, until the process exits.  All calls share
// it: two calls whose kernels overlap on the GPU (different streams, or
// different host threads) race on it and give wrong results; serialize them.
// Nothing in it needs to start at zero: stage 1 writes every (o, lse) entry
// of the splits before the merge reads them, so the contents a previous call
// left behind are never read.
#include <mutex>

#include "kvq_internal.h"

namespace kvq {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
struct ScratchEntry {
    void *ctx;    // the context the address belongs to
    void *ptr;
};
ScratchEntry g_scratch[kMaxDev] = {};

// The calling thread's current CUDA context (null if none, or if the driver
// does not hand out cuCtxGetCurrent), reached through the runtime's driver
// entry-point query so that the library needs no link to the driver library.
void *current_context() {
    typedef int (*ctx_get_t)(void **);
    static ctx_get_t fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (ctx_get_t) nullptr;
        return reinterpret_cast<ctx_get_t>(p);
    }();
    void *ctx = nullptr;
    if (!fn || fn(&ctx) != 0) return nullptr;
    return ctx;
}

// Device address of the scratch array in the current device's context
// (host code cannot use the array's name as a device pointer).  Looked up
// once per device and context: after a device reset the context, and with it
// the array's address, changes, and the next call looks it up again.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchEntry &ent = g_scratch[dev];
    void *ctx = current_context();
    if (!ent.ptr || !ctx || ent.ctx != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        ent.ptr = p;
        ent.ctx = current_context();     // the lookup makes the device's primary context current
    }
    *out = ent.ptr;
    return cudaSuccess;
}
}  // namespace

}  // namespace kvq

extern "C" kvq_status kv_decode_attn_noalloc(const kvq_config *cfg, const kvq_kivi_cache *cache, const void *q,
                                             void *out, cudaStream_t stream) {
    if (!cfg || !cache) return KVQ_ERR_INVALID_ARG;
    int32_t splits = 0;
    size_t need = 0;
    kvq_status s = kv_decode_attn_plan(cfg, KVQ_VARIANT_KIVI, cache->batch, cache->max_seq_len, &splits, &need);
    if (s != KVQ_OK) return s;
    if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;   // too large for the fixed scratch
    void *scratch = nullptr;
    if (kvq::scratch_address(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
    return kv_decode_attn(cfg, cache, q, out, scratch, (size_t)KVQ_NOALLOC_SCRATCH_BYTES, stream);
}
