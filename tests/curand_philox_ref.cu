// Test-only: cuRAND's Philox4x32-10 (device API) evaluated at a raw
// (counter, key), used as an independent known-answer source for the
// library's and the oracle's Philox.  curand_init(seed, subsequence, offset)
// starts at counter (offset/4 low, offset/4 high, subsequence low,
// subsequence high) with key (seed low, seed high).
#include <curand_kernel.h>

__global__ void curand_ref_kernel(const unsigned *ctr, const unsigned *key, int n, unsigned *out) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    unsigned long long seed = (unsigned long long)key[2 * i] | ((unsigned long long)key[2 * i + 1] << 32);
    unsigned long long sub = (unsigned long long)ctr[4 * i + 2] | ((unsigned long long)ctr[4 * i + 3] << 32);
    unsigned long long off = ((unsigned long long)ctr[4 * i] | ((unsigned long long)ctr[4 * i + 1] << 32)) * 4ull;
    curandStatePhilox4_32_10_t st;
    curand_init(seed, sub, off, &st);
    uint4 r = curand4(&st);
    out[4 * i] = r.x; out[4 * i + 1] = r.y; out[4 * i + 2] = r.z; out[4 * i + 3] = r.w;
}

extern "C" int curand_philox_ref(const unsigned *ctr, const unsigned *key, int n, unsigned *out) {
    curand_ref_kernel<<<(n + 127) / 128, 128>>>(ctr, key, n, out);
    return (int)cudaGetLastError();
}
