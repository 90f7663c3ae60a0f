// Measurement helper: the sustained rate of the search's inner integer operation on this GPU.
#include <cuda_runtime.h>

#include "mce_probe.h"

namespace {

// acc + popc(a & (b ^ acc)): one 3-input logic op (the AND of the search, here fed with a
// loop-carried operand so that no iteration can be folded or hoisted), one popcount, one add --
// the same three integer instructions the search spends on each 32-bit word it scores.
__device__ __forceinline__ unsigned and_popc_add(unsigned acc, unsigned a, unsigned b)
{
    return acc + __popc(a & (b ^ acc));
}

__global__ void __launch_bounds__(256) word_rate_kernel(const unsigned *in, unsigned *out,
                                                        int iters)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    unsigned a[8], b[8], acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        a[k] = in[(t + k) & 1023];
        b[k] = in[(t * 7 + k * 13) & 1023];
        acc[k] = 0;
    }
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = and_popc_add(acc[k], a[k], b[k]);
    }
    unsigned r = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) r += acc[k];
    if (r == 0xdeadbeefu) out[t] = r;   // practically never: keeps the work observable
}

}  // namespace

extern "C" int mce_probe_word_rate(int iters, int reps, double *words_per_s, float *ms)
{
    if (iters < 1 || reps < 1 || !words_per_s) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 9;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 9;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, word_rate_kernel, 256, 0) !=
        cudaSuccess || per_sm < 1)
        return 9;
    const int blocks = per_sm * sms, threads = 256;
    unsigned *in = nullptr, *out = nullptr;
    if (cudaMalloc(&in, 1024 * sizeof(unsigned)) != cudaSuccess) return 9;
    if (cudaMalloc(&out, (size_t)blocks * threads * sizeof(unsigned)) != cudaSuccess) {
        cudaFree(in);
        return 9;
    }
    unsigned host[1024];
    for (int i = 0; i < 1024; ++i) host[i] = 0x9E3779B9u * (unsigned)(i + 1);
    cudaMemcpy(in, host, sizeof(host), cudaMemcpyHostToDevice);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    word_rate_kernel<<<blocks, threads>>>(in, out, iters / 8 + 1);   // warm-up
    float best = 1e30f;
    for (int r = 0; r < reps; ++r) {
        cudaEventRecord(e0);
        word_rate_kernel<<<blocks, threads>>>(in, out, iters);
        cudaEventRecord(e1);
        cudaEventSynchronize(e1);
        float t = 0.f;
        cudaEventElapsedTime(&t, e0, e1);
        if (t < best) best = t;
    }
    const cudaError_t err = cudaGetLastError();
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(in);
    cudaFree(out);
    if (err != cudaSuccess) return 9;
    *words_per_s = (double)blocks * threads * 8.0 * (double)iters / (best * 1e-3);
    if (ms) *ms = best;
    return 0;
}
