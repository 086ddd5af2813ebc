// Test-only helper: Philox4x32-10 words from cuRAND's device API, to check
// the oracle's generator against a library routine.  curand_init(seed,
// subsequence, offset) starts the counter at (offset/4 in words 0-1,
// subsequence in words 2-3) under key (seed low, seed high); curand4 returns
// the four words of the current counter and advances it.
#include <curand_kernel.h>

__global__ void curand_blocks(unsigned long long seed, const unsigned long long* subseq,
                              const unsigned long long* offset, uint4* out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    curandStatePhilox4_32_10_t st;
    curand_init(seed, subseq[i], offset[i], &st);
    out[i] = curand4(&st);
}

extern "C" int curand_philox_blocks(unsigned long long seed, const unsigned long long* subseq,
                                    const unsigned long long* offset, unsigned* out, int n) {
    curand_blocks<<<(n + 127) / 128, 128>>>(seed, subseq, offset, reinterpret_cast<uint4*>(out), n);
    if (cudaGetLastError() != cudaSuccess) return -1;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -1;
}
