// ffn_bf16.cu -- grouped SwiGLU expert FFN + weighted combine, bf16 weights.
//
// Page "Opportunistic Expert Activation (OEA)": at decode the MoE layer is
// memory bound and its latency is set by fetching every activated expert's
// weights from HBM (section 2 Q1, section 4 check 4).  This kernel streams
// each activated expert's gate, up and down matrices from HBM exactly once
// and does the arithmetic of all the tokens routed to it while the tile is
// on chip.  Expert form (Qwen3): y = W_down (silu(W_gate x) * (W_up x));
// combine: out_i = sum_j w_ij y_{e_ij}(x_i) (kept scores, section 2 Q2).
//
// Structure (one persistent CTA per SM):
//   * Work is a list of tiles.  Phase-A tile (expert a, 16 rows of d_ff,
//     token chunk c) computes h = silu(W_gate x) * (W_up x) for those rows
//     and up to 32 tokens and writes h (bf16) to the workspace.  Phase-B
//     tile (expert a, 32 rows of d, chunk c) computes y = W_down h.  Each
//     CTA takes an equal, contiguous share of the phase-A tiles and then of
//     the phase-B tiles, so every CTA streams the same number of bytes.
//   * Warp 4 is the producer: one lane issues TMA tile loads (128-byte
//     swizzle, L2 evict-first) into a 12-stage shared-memory ring guarded by
//     mbarriers.  A stage is 16 KB: 256 K-columns of two 16-row tiles (gate
//     and up) or of one 32-row tile (down).  The weight stream does not wait
//     for any other CTA, so it continues across the phase boundary.
//   * Warps 0-3 are consumers: warp w owns the w-th 64-column block of every
//     stage and runs warp-level bf16 tensor-core MMAs with the weights as
//     the M side and the tokens as the N side (8 tokens per MMA column
//     tile), accumulating in fp32.  Tokens' hidden states (phase A) or h
//     rows (phase B) are loaded straight from global/L2 with 16-byte loads;
//     the K index inside each 64-column block is permuted identically for
//     both operands so that every lane reads 32 contiguous bytes.
//   * At the end of a tile the four warps' partial sums are added in warp
//     order through shared memory.  Phase A then applies SwiGLU and bumps a
//     per-expert counter; a phase-B tile first waits (bounded) until all
//     phase-A tiles of its expert are counted.  Phase B bumps a counter per
//     32-row output block; the CTA whose tile completes a block performs the
//     weighted combine of that block for all tokens, in slot order.
//   * The last CTA to finish resets the counters for the next launch.
// Every result is computed in a fixed order, so runs are bit-reproducible.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kCW = 4;                  // consumer warps
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kStageBytes = 16384;
constexpr int kStages = 12;
constexpr int kChunk = 32;              // tokens per tile pass
constexpr long long kWaitCycles = 4000000000LL;   // about two seconds

struct Smem {
    float red[kCW][1024];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int chunk_off[MOE_MAX_EXPERTS + 1];
    int abort_flag;
    int combine_flag;
    int last_flag;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + sizeof(Smem);

struct Tile {
    int a, e, rb, c, off, ntok;
};

__device__ __forceinline__ Tile decode_tile(long long t, int rbn, const int* chunk_off, int Tn,
                                            const FfnArgs& A) {
    int lo = 0, hi = Tn - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)chunk_off[mid] * rbn <= t) lo = mid; else hi = mid - 1;
    }
    Tile T;
    T.a = lo;
    T.e = A.active[lo];
    const int cnt = A.counts[T.e];
    T.off = A.offsets[T.e];
    const int nch = chunk_off[lo + 1] - chunk_off[lo];
    const long long r = t - (long long)chunk_off[lo] * rbn;
    T.rb = (int)(r / nch);
    T.c = (int)(r % nch);
    T.ntok = min(kChunk, cnt - kChunk * T.c);
    return T;
}

// Bounded mbarrier wait; once the CTA has given up, every later wait
// returns at once so that the control flow (and every barrier) still
// completes.
__device__ __forceinline__ void wait_bar(uint64_t* bar, uint32_t parity, Smem& S, uint32_t* flags) {
    if (mbar_try_wait(bar, parity)) return;
    const long long t0 = clock64();
    while (!*(volatile int*)&S.abort_flag) {
        if (mbar_try_wait(bar, parity)) return;
        if (clock64() - t0 > kWaitCycles) {
            *(volatile int*)&S.abort_flag = 1;
            raise_flag(flags, kFlagTimeout);
            return;
        }
    }
}

__device__ __forceinline__ uint4 lds16(const unsigned char* p) {
    return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ void unpack8(uint32_t (&r)[8], uint4 a, uint4 b) {
    r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
    r[4] = b.x; r[5] = b.y; r[6] = b.z; r[7] = b.w;
}

// One 16-row x 64-column weight block of a stage (128-byte swizzled rows):
// the A fragments of rows g and g+8 for the four k-steps.
__device__ __forceinline__ void load_a_block(const unsigned char* blk, int g, int t4,
                                             uint32_t (&r0)[8], uint32_t (&r1)[8]) {
    const int c0 = ((2 * t4) ^ g) << 4, c1 = ((2 * t4 + 1) ^ g) << 4;
    unpack8(r0, lds16(blk + g * 128 + c0), lds16(blk + g * 128 + c1));
    unpack8(r1, lds16(blk + (g + 8) * 128 + c0), lds16(blk + (g + 8) * 128 + c1));
}

__device__ __forceinline__ void mma_block(float (&acc)[4], const uint32_t (&r0)[8], const uint32_t (&r1)[8],
                                          const uint32_t (&xb)[8]) {
#pragma unroll
    for (int s = 0; s < 4; ++s)
        mma_bf16_16816(acc, r0[2 * s], r1[2 * s], r0[2 * s + 1], r1[2 * s + 1], xb[2 * s], xb[2 * s + 1]);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }

__global__ void __launch_bounds__(kThreads, 1)
ffn_bf16_kernel(const FfnArgs A, const __grid_constant__ CUtensorMap tm_gate,
                const __grid_constant__ CUtensorMap tm_up, const __grid_constant__ CUtensorMap tm_down) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem& S = *reinterpret_cast<Smem*>(ring + (size_t)kStages * kStageBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = A.d, F = A.F;
    uint32_t* flags = &A.hdr->flags;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], kCW);
        }
        fence_barrier_init();
        S.abort_flag = 0;
    }
    int Tn = *A.T;
    if (Tn < 0 || Tn > A.N) {
        if (threadIdx.x == 0 && blockIdx.x == 0) raise_flag(flags, kFlagBadIndex);
        Tn = 0;
    }
    if (warp == 0) {   // chunk offsets of the active experts
        int run = 0;
        if (lane == 0) S.chunk_off[0] = 0;
        for (int a0 = 0; a0 < Tn; a0 += 32) {
            const int a = a0 + lane;
            const int nch = a < Tn ? (A.counts[A.active[a]] + kChunk - 1) / kChunk : 0;
            int inc = nch;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += u;
            }
            if (a < Tn) S.chunk_off[a + 1] = run + inc;
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
    }
    if (warp == kCW && lane == 0) {
        prefetch_tensormap(&tm_gate);
        prefetch_tensormap(&tm_up);
        prefetch_tensormap(&tm_down);
    }
    __syncthreads();

    const int Ctot = S.chunk_off[Tn];
    const int rbA = F / 16, rbB = d / 32;
    const long long TA = (long long)Ctot * rbA, TB = (long long)Ctot * rbB;
    const long long G = gridDim.x, b = blockIdx.x;
    const long long a_beg = TA * b / G, a_end = TA * (b + 1) / G;
    const long long b_beg = TB * b / G, b_end = TB * (b + 1) / G;
    const int SA = (d + 255) / 256, SB = (F + 255) / 256;

    if (warp == kCW) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            uint32_t it = 0;
            for (long long t = a_beg; t < a_end; ++t) {
                const Tile T = decode_tile(t, rbA, S.chunk_off, Tn, A);
                const int row = T.e * F + 16 * T.rb;
                for (int s = 0; s < SA; ++s, ++it) {
                    const int slot = it % kStages;
                    if (it >= kStages) wait_bar(&S.empty[slot], ((it / kStages) - 1) & 1, S, flags);
                    const int kq = min(4, (d - 256 * s) / 64);
                    mbar_arrive_expect_tx(&S.full[slot], kq * 2 * 2048);
                    unsigned char* dst = ring + (size_t)slot * kStageBytes;
                    for (int q = 0; q < kq; ++q) {
                        tma_load_2d(dst + q * 2048, &tm_gate, 256 * s + 64 * q, row, &S.full[slot], pol);
                        tma_load_2d(dst + 8192 + q * 2048, &tm_up, 256 * s + 64 * q, row, &S.full[slot], pol);
                    }
                }
            }
            for (long long t = b_beg; t < b_end; ++t) {
                const Tile T = decode_tile(t, rbB, S.chunk_off, Tn, A);
                const int row = T.e * d + 32 * T.rb;
                for (int s = 0; s < SB; ++s, ++it) {
                    const int slot = it % kStages;
                    if (it >= kStages) wait_bar(&S.empty[slot], ((it / kStages) - 1) & 1, S, flags);
                    const int kq = min(4, (F - 256 * s) / 64);
                    mbar_arrive_expect_tx(&S.full[slot], kq * 4096);
                    unsigned char* dst = ring + (size_t)slot * kStageBytes;
                    for (int q = 0; q < kq; ++q)
                        tma_load_2d(dst + q * 4096, &tm_down, 256 * s + 64 * q, row, &S.full[slot], pol);
                }
            }
            // Every issued stage is consumed before the consumers reach the
            // final barrier, so no copy is in flight when the CTA exits.
        }
        __syncwarp();
    } else {
        // ------------------------------ consumers -----------------------------
        const int w = warp, g = lane >> 2, t4 = lane & 3, tid = threadIdx.x;
        const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(A.x);
        __nv_bfloat16* hb = static_cast<__nv_bfloat16*>(A.hbuf);
        uint32_t it = 0;

        // ---- phase A: h = silu(W_gate x) * (W_up x) ----
        for (long long t = a_beg; t < a_end; ++t) {
            const Tile T = decode_tile(t, rbA, S.chunk_off, Tn, A);
            const int NT = (T.ntok + 7) >> 3;
            const __nv_bfloat16* xr[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int nn = 8 * j + g;
                xr[j] = nullptr;
                if (nn < T.ntok) {
                    const int tok = A.perm[T.off + kChunk * T.c + nn] / A.kslots;
                    xr[j] = xg + (size_t)tok * d;
                }
            }
            float acc[2][4][4];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[m][j][q] = 0.f;

            for (int s = 0; s < SA; ++s, ++it) {
                const int slot = it % kStages;
                const int kq = min(4, (d - 256 * s) / 64);
                const bool has = w < kq;
                uint32_t X[4][8];
                const int col = 256 * s + 64 * w + 16 * t4;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                    if (has && j < NT && xr[j]) {
                        lo = __ldg(reinterpret_cast<const uint4*>(xr[j] + col));
                        hi = __ldg(reinterpret_cast<const uint4*>(xr[j] + col + 8));
                    }
                    unpack8(X[j], lo, hi);
                }
                wait_bar(&S.full[slot], (it / kStages) & 1, S, flags);
                if (has) {
                    const unsigned char* st = ring + (size_t)slot * kStageBytes;
                    uint32_t g0[8], g1[8], u0[8], u1[8];
                    load_a_block(st + w * 2048, g, t4, g0, g1);
                    load_a_block(st + 8192 + w * 2048, g, t4, u0, u1);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j < NT) {
                            mma_block(acc[0][j], g0, g1, X[j]);
                            mma_block(acc[1][j], u0, u1, X[j]);
                        }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }
            // reduce the four warps, SwiGLU, store h
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) S.red[w][(m * 4 + j) * 128 + lane * 4 + q] = acc[m][j][q];
            named_barrier(1, kCW * 32);
            for (int l = tid; l < 512; l += kCW * 32) {
                const int j = l >> 7, ln = (l >> 2) & 31, q = l & 3;
                const int nn = 8 * j + 2 * (ln & 3) + (q & 1);
                if (nn < T.ntok) {
                    float gs = 0.f, us = 0.f;
#pragma unroll
                    for (int ww = 0; ww < kCW; ++ww) {
                        gs += S.red[ww][j * 128 + ln * 4 + q];
                        us += S.red[ww][(4 + j) * 128 + ln * 4 + q];
                    }
                    const int row = (ln >> 2) + 8 * (q >> 1);
                    const size_t pos = (size_t)T.off + kChunk * T.c + nn;
                    hb[pos * F + 16 * T.rb + row] = __float2bfloat16_rn(silu_f(gs) * us);
                }
            }
            __threadfence();
            named_barrier(1, kCW * 32);
            if (tid == 0) atomicAdd(&A.hdone[T.a], 1u);
        }

        // ---- phase B: y = W_down h, combine when an output block is complete ----
        int ready_a = -1;
        for (long long t = b_beg; t < b_end; ++t) {
            const Tile T = decode_tile(t, rbB, S.chunk_off, Tn, A);
            const int NT = (T.ntok + 7) >> 3;
            if (T.a != ready_a) {
                if (tid == 0) {
                    const uint32_t need = (uint32_t)rbA * (S.chunk_off[T.a + 1] - S.chunk_off[T.a]);
                    const long long t0 = clock64();
                    while (ld_acquire_gpu(&A.hdone[T.a]) < need) {
                        if (*(volatile int*)&S.abort_flag) break;
                        if (clock64() - t0 > kWaitCycles) {
                            *(volatile int*)&S.abort_flag = 1;
                            raise_flag(flags, kFlagTimeout);
                            break;
                        }
                        __nanosleep(64);
                    }
                }
                named_barrier(1, kCW * 32);
                ready_a = T.a;
            }
            const __nv_bfloat16* hr[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int nn = 8 * j + g;
                hr[j] = nn < T.ntok ? hb + ((size_t)T.off + kChunk * T.c + nn) * F : nullptr;
            }
            float acc[2][4][4];
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[m][j][q] = 0.f;

            for (int s = 0; s < SB; ++s, ++it) {
                const int slot = it % kStages;
                const int kq = min(4, (F - 256 * s) / 64);
                const bool has = w < kq;
                uint32_t X[4][8];
                const int col = 256 * s + 64 * w + 16 * t4;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                    if (has && j < NT && hr[j]) {
                        lo = __ldcg(reinterpret_cast<const uint4*>(hr[j] + col));
                        hi = __ldcg(reinterpret_cast<const uint4*>(hr[j] + col + 8));
                    }
                    unpack8(X[j], lo, hi);
                }
                wait_bar(&S.full[slot], (it / kStages) & 1, S, flags);
                if (has) {
                    const unsigned char* st = ring + (size_t)slot * kStageBytes + w * 4096;
                    uint32_t a0[8], a1[8], b0[8], b1[8];
                    load_a_block(st, g, t4, a0, a1);
                    load_a_block(st + 2048, g, t4, b0, b1);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j < NT) {
                            mma_block(acc[0][j], a0, a1, X[j]);
                            mma_block(acc[1][j], b0, b1, X[j]);
                        }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) S.red[w][(m * 4 + j) * 128 + lane * 4 + q] = acc[m][j][q];
            named_barrier(1, kCW * 32);
            for (int l = tid; l < 1024; l += kCW * 32) {
                const int m = l >> 9, j = (l >> 7) & 3, ln = (l >> 2) & 31, q = l & 3;
                const int nn = 8 * j + 2 * (ln & 3) + (q & 1);
                if (nn < T.ntok) {
                    float ys = 0.f;
#pragma unroll
                    for (int ww = 0; ww < kCW; ++ww) ys += S.red[ww][l];
                    const int row = 16 * m + (ln >> 2) + 8 * (q >> 1);
                    const size_t pos = (size_t)T.off + kChunk * T.c + nn;
                    A.ybuf[pos * d + 32 * T.rb + row] = ys;
                }
            }
            __threadfence();
            named_barrier(1, kCW * 32);
            if (tid == 0) {
                const uint32_t old = atomicAdd(&A.ydone[T.rb], 1u);
                S.combine_flag = (old + 1 == (uint32_t)Ctot);
                __threadfence();
            }
            named_barrier(1, kCW * 32);
            if (S.combine_flag) {
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(A.out);
                const int c0 = 32 * T.rb;
                for (int l = tid; l < A.B * 32; l += kCW * 32) {
                    const int i = l >> 5, jr = l & 31;
                    float acc2 = 0.f;
                    for (int sl = 0; sl < A.kslots; ++sl) {
                        const int pos = A.pos_of[i * A.kslots + sl];
                        if (pos >= 0) acc2 += A.w[i * A.kslots + sl] * __ldcg(A.ybuf + (size_t)pos * d + c0 + jr);
                    }
                    out[(size_t)i * d + c0 + jr] = __float2bfloat16_rn(acc2);
                }
            }
            named_barrier(1, kCW * 32);
        }

        if (Ctot == 0 && blockIdx.x == 0) {   // nothing routed: the output is zero
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(A.out);
            for (long long l = tid; l < (long long)A.B * d; l += kCW * 32) out[l] = __float2bfloat16_rn(0.f);
        }
    }

    // ---- the last CTA resets the counters for the next launch ----
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(&A.hdr->ctas_done, 1u);
        S.last_flag = (old + 1 == gridDim.x);
    }
    __syncthreads();
    if (S.last_flag) {
        __threadfence();
        for (int i = threadIdx.x; i < A.N; i += kThreads) A.hdone[i] = 0;
        for (int i = threadIdx.x; i < d / 32; i += kThreads) A.ydone[i] = 0;
        if (threadIdx.x == 0) A.hdr->ctas_done = 0;
    }
}

}  // namespace

cudaError_t launch_ffn_bf16(const FfnArgs& a, const CUtensorMap* maps, int num_sms, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(ffn_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    ffn_bf16_kernel<<<num_sms, kThreads, kSmemBytes, s>>>(a, maps[0], maps[1], maps[2]);
    return cudaGetLastError();
}

size_t ffn_bf16_smem_bytes() { return kSmemBytes; }

}  // namespace moe
