// pack.cu -- moe_pack_int4: quantises a bf16 expert matrix to the packed
// INT4 image that the mixed-precision expert kernel reads (DynaExq page,
// section 3.2: an expert's low-precision version, 4-bit symmetric codes with
// a scale per group; section 2.4: a version is made off the request path
// and then published).  Done on the device, so an expert can be demoted
// without a round trip through host memory.
//
// One warp per (row, 128-column group): lane l holds columns 4l..4l+3.
//   s = bf16(fp32(max|w| / 7))   quotient in double, then nearest-even to
//                                fp32 and to bf16
//   q = clamp(rint(w / s), -7, 7) in double, ties to even; q = 0 if s = 0
// Two lanes' codes share one 32-bit word of the image (see moe.h for the
// nibble order).
#include "common.cuh"

namespace moe {

namespace {

constexpr int kPackWarps = 8;

__global__ void __launch_bounds__(kPackWarps * 32)
pack_int4_kernel(const __nv_bfloat16* __restrict__ w, int rows, int cols, int rb, uint8_t* __restrict__ out) {
    const int ng = cols / 128;
    const long long item = (long long)blockIdx.x * kPackWarps + (threadIdx.x >> 5);
    if (item >= (long long)rows * ng) return;   // the whole warp leaves together
    const int lane = threadIdx.x & 31;
    const int r = (int)(item / ng), g = (int)(item - (long long)r * ng);
    const uint2 raw = *reinterpret_cast<const uint2*>(w + (size_t)r * cols + (size_t)g * 128 + 4 * lane);
    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float v[4] = {__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1)};
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const __nv_bfloat16 s = __float2bfloat16_rn(__double2float_rn((double)m / 7.0));
    const double sd = (double)__bfloat162float(s);
    // column 4l + j of the group: offset o = 4 (l % 2) + j within its word
    const int base = (lane & 1) ? 8 : 0;
    const int bits[4] = {base, base + 16, base + 4, base + 20};
    uint32_t part = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        double q = sd > 0.0 ? rint((double)v[j] / sd) : 0.0;
        q = fmin(7.0, fmax(-7.0, q));
        part |= (uint32_t)((int)q + 8) << bits[j];
    }
    const uint32_t word = part | __shfl_xor_sync(0xffffffffu, part, 1);
    const int rbi = r / rb, rr = r - rbi * rb;
    uint8_t* chunk = out + ((size_t)rbi * ng + g) * (size_t)(rb * 64 + rb * 2);
    if (!(lane & 1)) *reinterpret_cast<uint32_t*>(chunk + rr * 64 + (lane >> 1) * 4) = word;
    if (lane == 0) *reinterpret_cast<__nv_bfloat16*>(chunk + rb * 64 + rr * 2) = s;
}

}  // namespace

cudaError_t launch_pack_int4(const void* w, int rows, int cols, int rb, void* out, cudaStream_t s) {
    const long long items = (long long)rows * (cols / 128);
    const long long blocks = (items + kPackWarps - 1) / kPackWarps;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    pack_int4_kernel<<<(unsigned)blocks, kPackWarps * 32, 0, s>>>(static_cast<const __nv_bfloat16*>(w), rows, cols,
                                                                  rb, static_cast<uint8_t*>(out));
    return cudaGetLastError();
}

}  // namespace moe
