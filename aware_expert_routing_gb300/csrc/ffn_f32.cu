// ffn_f32.cu -- expert FFN + combine with fp32 weights and activations.
//
// Same computation as the bf16 kernel (page "Opportunistic Expert
// Activation (OEA)", section 2: the experts chosen by routing, SwiGLU form
// y = W_down (silu(W_gate x) * (W_up x)), combine out_i = sum_j w_ij y_ij),
// kept in fp32 throughout on CUDA cores.  It serves fp32 models, whose
// expert weights are read once per activated expert like the bf16 path,
// but without tensor cores: three plain kernels (h, y, combine).
#include "common.cuh"

namespace moe {

namespace {

// h[pos][f] = silu(W_gate[e][f] . x_tok) * (W_up[e][f] . x_tok)
// grid: (N active slots, ceil(F/128)); one thread per f, all tokens of e.
__global__ void ffn_f32_h_kernel(FfnArgs A) {
    extern __shared__ float xs[];
    const int a = blockIdx.x;
    if (a >= *A.T) return;
    const int e = A.active[a];
    const int cnt = A.counts[e], off = A.offsets[e];
    const int f = blockIdx.y * blockDim.x + threadIdx.x;
    const float* wg = static_cast<const float*>(A.w_gate) + (size_t)e * A.F * A.d;
    const float* wu = static_cast<const float*>(A.w_up) + (size_t)e * A.F * A.d;
    float* hb = static_cast<float*>(A.hbuf);
    for (int n = 0; n < cnt; ++n) {
        const int tok = A.perm[off + n] / A.kslots;
        const float* x = static_cast<const float*>(A.x) + (size_t)tok * A.d;
        __syncthreads();
        for (int c = threadIdx.x; c < A.d; c += blockDim.x) xs[c] = x[c];
        __syncthreads();
        if (f < A.F) {
            float g = 0.f, u = 0.f;
            for (int c = 0; c < A.d; ++c) {
                g = fmaf(wg[(size_t)f * A.d + c], xs[c], g);
                u = fmaf(wu[(size_t)f * A.d + c], xs[c], u);
            }
            hb[(size_t)(off + n) * A.F + f] = g / (1.f + expf(-g)) * u;
        }
    }
}

// y[pos][j] = W_down[e][j] . h[pos]; grid: (N active slots, ceil(d/128)).
__global__ void ffn_f32_y_kernel(FfnArgs A) {
    extern __shared__ float hs[];
    const int a = blockIdx.x;
    if (a >= *A.T) return;
    const int e = A.active[a];
    const int cnt = A.counts[e], off = A.offsets[e];
    const int j = blockIdx.y * blockDim.x + threadIdx.x;
    const float* wd = static_cast<const float*>(A.w_down) + (size_t)e * A.d * A.F;
    const float* hb = static_cast<const float*>(A.hbuf);
    for (int n = 0; n < cnt; ++n) {
        __syncthreads();
        for (int f = threadIdx.x; f < A.F; f += blockDim.x) hs[f] = hb[(size_t)(off + n) * A.F + f];
        __syncthreads();
        if (j < A.d) {
            float y = 0.f;
            for (int f = 0; f < A.F; ++f) y = fmaf(wd[(size_t)j * A.F + f], hs[f], y);
            A.ybuf[(size_t)(off + n) * A.d + j] = y;
        }
    }
}

// out[i][j] = sum over slots (in slot order) of w[i][slot] * y[pos(i, slot)][j]
__global__ void combine_f32_kernel(FfnArgs A) {
    const int i = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= A.d) return;
    float acc = 0.f;
    for (int sl = 0; sl < A.kslots; ++sl) {
        const int pos = A.pos_of[i * A.kslots + sl];
        if (pos >= 0) acc = fmaf(A.w[i * A.kslots + sl], A.ybuf[(size_t)pos * A.d + j], acc);
    }
    static_cast<float*>(A.out)[(size_t)i * A.d + j] = acc;
}

}  // namespace

cudaError_t launch_ffn_f32(const FfnArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    const size_t smem_h = sizeof(float) * a.d, smem_y = sizeof(float) * a.F;
    cudaError_t e;
    if (smem_h > 48 * 1024 &&
        (e = cudaFuncSetAttribute(ffn_f32_h_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_h)) != cudaSuccess)
        return e;
    if (smem_y > 48 * 1024 &&
        (e = cudaFuncSetAttribute(ffn_f32_y_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_y)) != cudaSuccess)
        return e;
    ffn_f32_h_kernel<<<dim3(a.N, (a.F + 127) / 128), 128, smem_h, s>>>(a);
    ffn_f32_y_kernel<<<dim3(a.N, (a.d + 127) / 128), 128, smem_y, s>>>(a);
    combine_f32_kernel<<<dim3((a.d + 127) / 128, a.B), 128, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
