// synth.cu -- device implementation of the seeded synthetic-tensor stream.
//
// Element i of a stream with seed s is SplitMix64 output i for initial state
// s (Steele, Lea & Flood, "Fast Splittable Pseudorandom Number Generators",
// OOPSLA 2014): z = s + (i + 1) * 0x9E3779B97F4A7C15, then the SplitMix64
// output mix.  The four 16-bit fields of z are summed and centred (an
// Irwin-Hall sum, mean 131070), converted to fp32 exactly and multiplied by
// `scale` once in fp32 (round to nearest), then rounded to bf16 (nearest
// even) for bf16 tensors.  Integer steps and one correctly rounded multiply
// make the values identical to any other implementation of the definition.
#include "common.cuh"

namespace moe {

namespace {

__global__ void synth_kernel(void* dst, int dtype, uint64_t n, uint64_t start, uint64_t seed, float scale) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        uint64_t z = seed + (start + i + 1) * 0x9E3779B97F4A7C15ull;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z = z ^ (z >> 31);
        const int sum = (int)(z & 0xFFFF) + (int)((z >> 16) & 0xFFFF) + (int)((z >> 32) & 0xFFFF) +
                        (int)(z >> 48) - 131070;
        const float v = __fmul_rn((float)sum, scale);
        if (dtype == MOE_DTYPE_BF16)
            static_cast<__nv_bfloat16*>(dst)[i] = __float2bfloat16_rn(v);
        else
            static_cast<float*>(dst)[i] = v;
    }
}

}  // namespace

cudaError_t launch_synth(void* dst, int dtype, uint64_t n, uint64_t start, uint64_t seed, float scale,
                         cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    uint64_t blocks = (n + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    synth_kernel<<<(unsigned)blocks, 256, 0, s>>>(dst, dtype, n, start, seed, scale);
    return cudaGetLastError();
}

}  // namespace moe
