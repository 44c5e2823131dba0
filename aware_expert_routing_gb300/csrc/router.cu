// router.cu -- router scores logits[i][e] = x_i . w_router[e] + bias[e].
//
// Page "Opportunistic Expert Activation (OEA)", section 2 (Q1/Q2): every
// token scores all N experts; those scores drive top-k and OEA.
//
// bf16 path.  One CTA computes a 16-expert x 32-token tile over a slice of
// the hidden dimension with warp-level tensor-core MMAs; the KS CTAs that
// share a tile form a thread-block cluster; each rank adds one slice of the
// tile over all ranks' partial tiles through distributed shared memory, in
// rank order, so the result is deterministic and no global atomics or
// second launch are needed.
//
// Operand loads.  Both operands come straight from global memory with
// 16-byte loads.  Within a 64-column block, lane (g = lane/4, t = lane%4)
// loads columns [16t, 16t+16) of its rows; the K index of the MMA is a
// permutation of those 64 columns (k-step s, k-slot pair 2t / 2t+8 map to
// columns 16t+4s / 16t+4s+2), applied identically to both operands, so the
// dot products are unchanged and every load is a full 128-byte row segment.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kRouterWarps = 4;

__device__ __forceinline__ uint4 ldg16(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__global__ void __launch_bounds__(kRouterWarps * 32)
router_bf16_kernel(RouterArgs a) {
    __shared__ float red[kRouterWarps][4 * 128];
    __shared__ float part[4 * 128];

    grid_dependency_wait();      // hidden states come from the preceding kernel
    grid_launch_dependents();    // the routing kernel may start its prologue
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int e0 = blockIdx.x * 16;
    const int ks = blockIdx.y;
    const int tok0 = blockIdx.z * 32;
    const int ntv = min(4, (a.B - tok0 + 7) / 8);   // n-tiles holding real tokens
    const int kbtot = a.d / 64;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(a.w);

    float acc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;

    const int r0 = e0 + g, r1 = e0 + g + 8;
    int q = 0;
    for (int kb = ks; kb < kbtot; kb += a.ks, ++q) {
        if ((q & (kRouterWarps - 1)) != warp) continue;
        const int col = kb * 64 + 16 * t;
        uint4 wa0 = make_uint4(0, 0, 0, 0), wa1 = wa0, wb0 = wa0, wb1 = wa0;
        if (r0 < a.N) { wa0 = ldg16(w + (size_t)r0 * a.d + col); wa1 = ldg16(w + (size_t)r0 * a.d + col + 8); }
        if (r1 < a.N) { wb0 = ldg16(w + (size_t)r1 * a.d + col); wb1 = ldg16(w + (size_t)r1 * a.d + col + 8); }
        const uint32_t A0[8] = {wa0.x, wa0.y, wa0.z, wa0.w, wa1.x, wa1.y, wa1.z, wa1.w};
        const uint32_t A1[8] = {wb0.x, wb0.y, wb0.z, wb0.w, wb1.x, wb1.y, wb1.z, wb1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j >= ntv) break;
            const int tok = tok0 + 8 * j + g;
            uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
            if (tok < a.B) { xa = ldg16(x + (size_t)tok * a.d + col); xb = ldg16(x + (size_t)tok * a.d + col + 8); }
            const uint32_t X[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_16816(acc[j], A0[2 * s], A1[2 * s], A0[2 * s + 1], A1[2 * s + 1], X[2 * s], X[2 * s + 1]);
        }
    }

    // Sum the warps of this CTA in warp order (fragment-linear layout).
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) red[warp][j * 128 + lane * 4 + q2] = acc[j][q2];
    __syncthreads();
    for (int l = threadIdx.x; l < 512; l += blockDim.x) {
        float s = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kRouterWarps; ++w2) s += red[w2][l];
        part[l] = s;
    }
    cluster_sync();
    {   // each cluster rank adds up and stores its slice of the tile
        const int rank = (int)cluster_ctarank();
        const int per = (512 + a.ks - 1) / a.ks;
        const int lend = min(512, (rank + 1) * per);
        for (int l = rank * per + (int)threadIdx.x; l < lend; l += blockDim.x) {
            float v[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) v[r] = r < a.ks ? ld_dsmem_f32(&part[l], r) : 0.f;
            float s = 0.f;
#pragma unroll
            for (int r = 0; r < 8; ++r) s += v[r];   // rank order
            const int j = l >> 7, ln = (l >> 2) & 31, q2 = l & 3;
            const int row = (ln >> 2) + 8 * (q2 >> 1);
            const int tok = tok0 + 8 * j + 2 * (ln & 3) + (q2 & 1);
            const int e = e0 + row;
            if (tok < a.B && e < a.N) {
                if (a.bias) s += a.bias[e];
                a.logits[(size_t)tok * a.N + e] = s;
            }
        }
    }
    cluster_sync();   // keep every CTA's shared memory alive until all ranks have read it
}

// fp32 path: one thread per score, plain FMA over the hidden dimension.
__global__ void router_f32_kernel(RouterArgs a) {
    extern __shared__ float xs[];
    grid_dependency_wait();
    const int i = blockIdx.y;
    const float* x = static_cast<const float*>(a.x) + (size_t)i * a.d;
    for (int c = threadIdx.x; c < a.d; c += blockDim.x) xs[c] = x[c];
    __syncthreads();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= a.N) return;
    const float* w = static_cast<const float*>(a.w) + (size_t)e * a.d;
    float acc = 0.f;
    for (int c = 0; c < a.d; ++c) acc = fmaf(xs[c], w[c], acc);
    if (a.bias) acc += a.bias[e];
    a.logits[(size_t)i * a.N + e] = acc;
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a_in, int dtype, cudaStream_t s) {
    RouterArgs a = a_in;
    if (a.B == 0) return cudaSuccess;
    if (dtype == MOE_DTYPE_F32) {
        dim3 grid((a.N + 127) / 128, a.B);
        size_t smem = sizeof(float) * a.d;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(router_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        router_f32_kernel<<<grid, 128, smem, s>>>(a);
        return cudaGetLastError();
    }
    const int kbtot = a.d / 64;
    a.ks = kbtot < 8 ? kbtot : 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.N + 15) / 16, a.ks, (a.B + 31) / 32);
    cfg.blockDim = dim3(kRouterWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = a.ks;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, router_bf16_kernel, a);
}

}  // namespace moe
