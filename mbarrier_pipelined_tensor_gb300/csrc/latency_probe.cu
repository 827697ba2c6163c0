// Dependent-chain latency probe ("hardware-hazards-b200" note, section
// "Fixed-latency RAW under-stalls"): a chain a = a * 1 + 1 of `chain`
// fused multiply-adds, each reading the previous one's result, timed with
// clock64 by one thread. The result must be exactly seed + chain; the cycles
// per link bound the FMA's read-after-write latency from above (the loop
// around the unrolled block and the clock reads add a little). Written with
// inline fma.rn so the compiler cannot fold the chain; nothing here reads
// or edits compiled code.
#include <cstdint>

#include "common.cuh"

namespace tp {

struct ProbeOut {
    double result;
    long long cycles;
};

// One slot per kind; written by the probe, read back by the host.
static __device__ ProbeOut g_probe_out[2];

__global__ void fma_f32_chain_kernel(float seed, int blocks)
{
    float a = seed;
    const float one = 1.0f;
    const long long t0 = clock64();
    for (int b = 0; b < blocks; ++b) {
#pragma unroll
        for (int i = 0; i < 64; ++i) asm volatile("fma.rn.f32 %0, %0, %1, %1;" : "+f"(a) : "f"(one));
    }
    const long long t1 = clock64();
    g_probe_out[0].result = a;
    g_probe_out[0].cycles = t1 - t0;
}

__global__ void fma_f64_chain_kernel(double seed, int blocks)
{
    double a = seed;
    const double one = 1.0;
    const long long t0 = clock64();
    for (int b = 0; b < blocks; ++b) {
#pragma unroll
        for (int i = 0; i < 64; ++i) asm volatile("fma.rn.f64 %0, %0, %1, %1;" : "+d"(a) : "d"(one));
    }
    const long long t1 = clock64();
    g_probe_out[1].result = a;
    g_probe_out[1].cycles = t1 - t0;
}

// Runs the chain of 64 * blocks links and reads the result back
// (synchronizes `st`).
cudaError_t run_fma_probe(int kind, double seed, int blocks, cudaStream_t st, double* result, long long* cycles)
{
    if (kind == 0)
        fma_f32_chain_kernel<<<1, 1, 0, st>>>(static_cast<float>(seed), blocks);
    else
        fma_f64_chain_kernel<<<1, 1, 0, st>>>(seed, blocks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    ProbeOut h[2];
    e = cudaMemcpyFromSymbol(h, g_probe_out, sizeof(h));
    if (e != cudaSuccess) return e;
    *result = h[kind].result;
    *cycles = h[kind].cycles;
    return cudaSuccess;
}

}  // namespace tp
