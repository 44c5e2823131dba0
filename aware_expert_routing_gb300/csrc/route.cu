// route.cu -- per-token expert selection (plain top-k or OEA) and grouping of
// the (token, slot) pairs by expert, in one CTA.
//
// Page "Opportunistic Expert Activation (OEA)":
//   section 2 Q2  phase 1: n_i = min(k0, t_i), t_i the adaptive top-p count;
//                 baseline S_i^base = the token's top-n_i; S_base = union;
//                 phase 2: add experts of the token's own ranked list that
//                 are in S_base; kept scores renormalised.
//   section 3     the phase-2 gate "e_ij in S_base".
//   sections 4-5  maxP (rank depth of phase 2) and k^max (experts per token).
//   section 4     per-expert loads cnt_e, T = number of experts with cnt_e > 0.
//   section 7     padding tokens select nothing.
// Ranking: larger score first, equal scores by the lower expert id.
//
// One warp handles one token at a time; lane l holds the scores of experts
// l, l+32, l+64, ... in registers.  The k-th best expert is found by k rounds
// of a warp-wide (score, id) arg-max.  The batch union S_base is an N-bit
// mask in shared memory built with __ballot_sync + atomicOr.  Grouping by
// expert uses per-token N-bit masks: one warp per expert counts its tokens
// with ballots, a block scan gives the offsets, and a second ballot pass
// writes each pair's position (tokens ascending within an expert).
#include <float.h>
#include <limits.h>

#include "common.cuh"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int NPL>
__device__ __forceinline__ void load_scores(const float* row, int N, int lane, float (&v)[NPL],
                                            bool& nonfinite) {
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
        const int e = lane + 32 * j;
        float x = e < N ? row[e] : -INFINITY;
        if (e < N && !isfinite(x)) {
            nonfinite = true;
            x = -INFINITY;
        }
        v[j] = x;
    }
}

// Warp-wide arg-max over the scores whose bit in `excl` is clear.
// Returns -inf / INT_MAX when no candidate is left.
template <int NPL>
__device__ __forceinline__ void warp_argmax(const float (&v)[NPL], uint32_t excl, int lane,
                                            float& bv, int& bid) {
    float best = -INFINITY;
    int id = INT_MAX;
#pragma unroll
    for (int j = 0; j < NPL; ++j)
        if (!((excl >> j) & 1u) && v[j] > best) {   // ascending j = ascending id
            best = v[j];
            id = lane + 32 * j;
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ob = __shfl_xor_sync(kFull, best, off);
        const int oi = __shfl_xor_sync(kFull, id, off);
        if (ob > best || (ob == best && oi < id)) {
            best = ob;
            id = oi;
        }
    }
    bv = best;
    bid = id;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, off));
    return x;
}

struct RouteSmem {
    uint32_t* sbase;    // [32]      S_base bit mask
    int* snb;           // [B]       n_i
    int* sidx;          // [B][kslots]
    uint32_t* tokmask;  // [B][NW]   experts kept by each token
    int* scnt;          // [N]
    int* soff;          // [N]
    int* sact;          // [N]
    int* scan;          // [64]
};

// Writes the routing of token i: lane r < cnt holds slot r (myid, myval);
// `kept` holds the lane's bits of the token's expert mask.
template <int NPL>
__device__ __forceinline__ void finish_token(const RouteArgs& a, RouteSmem& sm, int i, int lane, int cnt,
                                             int myid, float myval, uint32_t kept, int NW) {
    const float l0 = __shfl_sync(kFull, myval, 0);
    const float ex = lane < cnt ? expf(myval - l0) : 0.f;
    const float z = warp_sum(ex);
    if (lane < a.kslots) {
        const size_t q = (size_t)i * a.kslots + lane;
        const bool used = lane < cnt;
        a.idx[q] = used ? myid : -1;
        a.w[q] = used ? ex / z : 0.f;
        sm.sidx[q] = used ? myid : -1;
        if (!used) a.pos_of[q] = -1;
    }
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
        const uint32_t word = __ballot_sync(kFull, (kept >> j) & 1u);
        if (lane == 0 && j < NW) sm.tokmask[(size_t)i * NW + j] = word;
    }
}

template <int NPL>
__global__ void route_kernel(RouteArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int nthreads = blockDim.x;
    const int nwarps = nthreads >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = a.N, B = a.B;
    const int NW = (N + 31) >> 5;

    RouteSmem sm;
    unsigned char* p = smem_raw;
    sm.sbase = reinterpret_cast<uint32_t*>(p); p += 32 * 4;
    sm.scan = reinterpret_cast<int*>(p); p += 64 * 4;
    sm.snb = reinterpret_cast<int*>(p); p += MOE_MAX_TOKENS * 4;
    sm.scnt = reinterpret_cast<int*>(p); p += MOE_MAX_EXPERTS * 4;
    sm.soff = reinterpret_cast<int*>(p); p += MOE_MAX_EXPERTS * 4;
    sm.sact = reinterpret_cast<int*>(p); p += MOE_MAX_EXPERTS * 4;
    sm.sidx = reinterpret_cast<int*>(p); p += (size_t)B * a.kslots * 4;
    sm.tokmask = reinterpret_cast<uint32_t*>(p);

    if (threadIdx.x < 32) sm.sbase[threadIdx.x] = 0;
    __syncthreads();

    bool nonfinite = false;
    const bool oea = a.mode == MOE_MODE_OEA;

    // ---- plain top-k, or OEA phase 1 (baseline and union) ------------------
    for (int i = warp; i < B; i += nwarps) {
        float v[NPL];
        load_scores<NPL>(a.logits + (size_t)i * N, N, lane, v, nonfinite);
        if (i >= a.B_valid) {           // padding token: selects nothing
            if (lane == 0) {
                sm.snb[i] = 0;
                if (a.n_base) a.n_base[i] = 0;
            }
            if (!oea) finish_token<NPL>(a, sm, i, lane, 0, -1, 0.f, 0u, NW);
            continue;
        }
        uint32_t taken = 0;
        int myid = -1;
        float myval = -INFINITY;
        int n = 0;
        if (!oea) {
            for (int r = 0; r < a.k; ++r) {
                float bv; int bid;
                warp_argmax<NPL>(v, taken, lane, bv, bid);
                if (bv == -INFINITY) break;
                if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
                if (lane == r) { myid = bid; myval = bv; }
                n = r + 1;
            }
            if (lane == 0 && a.n_base) a.n_base[i] = n;
            finish_token<NPL>(a, sm, i, lane, n, myid, myval, taken, NW);
            continue;
        }
        // Phase 1: softmax over all N scores, prefix in rank order, fp32.
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < NPL; ++j) m = fmaxf(m, v[j]);
        m = warp_max(m);
        float zl = 0.f;
#pragma unroll
        for (int j = 0; j < NPL; ++j)
            if (lane + 32 * j < N && v[j] != -INFINITY) zl += expf(v[j] - m);
        const float Z = warp_sum(zl);
        float prefix = 0.f;
        for (int r = 0; r < a.k0; ++r) {
            float bv; int bid;
            warp_argmax<NPL>(v, taken, lane, bv, bid);
            if (bv == -INFINITY) break;
            if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
            n = r + 1;
            if (a.p < 1.f) {
                prefix += expf(bv - m) / Z;
                if (prefix >= a.p) break;
            }
        }
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
            const uint32_t word = __ballot_sync(kFull, (taken >> j) & 1u);
            if (lane == 0 && word) atomicOr(&sm.sbase[j], word);
        }
        if (lane == 0) {
            sm.snb[i] = n;
            if (a.n_base) a.n_base[i] = n;
        }
    }
    __syncthreads();

    // ---- OEA phase 2: piggyback inside S_base -------------------------------
    if (oea) {
        uint32_t notin = 0;
#pragma unroll
        for (int j = 0; j < NPL; ++j)
            if (!((sm.sbase[j] >> lane) & 1u)) notin |= 1u << j;
        for (int i = warp; i < a.B_valid; i += nwarps) {
            float v[NPL];
            bool dummy = false;
            load_scores<NPL>(a.logits + (size_t)i * N, N, lane, v, dummy);
            uint32_t taken = 0, kept = 0;
            int cnt = 0, myid = -1;
            float myval = -INFINITY;
            if (a.maxP >= N) {
                // the in-union experts in rank order; the first n_i are the baseline
                for (int r = 0; r < a.kmax; ++r) {
                    float bv; int bid;
                    warp_argmax<NPL>(v, taken | notin, lane, bv, bid);
                    if (bv == -INFINITY) break;
                    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
                    if (lane == r) { myid = bid; myval = bv; }
                    cnt = r + 1;
                }
                kept = taken;
            } else {
                // walk the ranked list to depth max(maxP, n_i)
                const int nb = sm.snb[i];
                const int depth = a.maxP > nb ? a.maxP : nb;
                for (int r = 0; r < depth && cnt < a.kmax; ++r) {
                    float bv; int bid;
                    warp_argmax<NPL>(v, taken, lane, bv, bid);
                    if (bv == -INFINITY) break;
                    const bool mine = (bid & 31) == lane;
                    if (mine) taken |= 1u << (bid >> 5);
                    const bool in_union = (sm.sbase[bid >> 5] >> (bid & 31)) & 1u;
                    if (r < nb || in_union) {
                        if (mine) kept |= 1u << (bid >> 5);
                        if (lane == cnt) { myid = bid; myval = bv; }
                        ++cnt;
                    }
                }
            }
            finish_token<NPL>(a, sm, i, lane, cnt, myid, myval, kept, NW);
        }
        for (int i = a.B_valid + warp; i < B; i += nwarps)
            finish_token<NPL>(a, sm, i, lane, 0, -1, 0.f, 0u, NW);
    }
    if (__any_sync(kFull, nonfinite) && lane == 0) raise_flag(a.flags, kFlagNonFinite);
    __syncthreads();

    // ---- per-expert counts ---------------------------------------------------
    for (int e = warp; e < N; e += nwarps) {
        int c = 0;
        for (int i0 = 0; i0 < B; i0 += 32) {
            const int i = i0 + lane;
            const uint32_t bit = i < B ? (sm.tokmask[(size_t)i * NW + (e >> 5)] >> (e & 31)) & 1u : 0u;
            c += __popc(__ballot_sync(kFull, bit));
        }
        if (lane == 0) sm.scnt[e] = c;
    }
    __syncthreads();

    // ---- block exclusive scan of counts and of (count > 0) -------------------
    {
        const int per = (N + nthreads - 1) / nthreads;
        const int e0 = threadIdx.x * per;
        int s1 = 0, s2 = 0;
        for (int q = 0; q < per; ++q) {
            const int e = e0 + q;
            if (e < N) { s1 += sm.scnt[e]; s2 += sm.scnt[e] > 0; }
        }
        int i1 = s1, i2 = s2;   // warp inclusive scans
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u1 = __shfl_up_sync(kFull, i1, off), u2 = __shfl_up_sync(kFull, i2, off);
            if (lane >= off) { i1 += u1; i2 += u2; }
        }
        if (lane == 31) { sm.scan[warp] = i1; sm.scan[32 + warp] = i2; }
        __syncthreads();
        if (warp == 0) {
            int t1 = lane < nwarps ? sm.scan[lane] : 0, t2 = lane < nwarps ? sm.scan[32 + lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u1 = __shfl_up_sync(kFull, t1, off), u2 = __shfl_up_sync(kFull, t2, off);
                if (lane >= off) { t1 += u1; t2 += u2; }
            }
            __syncwarp();
            if (lane < nwarps) { sm.scan[lane] = t1; sm.scan[32 + lane] = t2; }
        }
        __syncthreads();
        int ex1 = (warp ? sm.scan[warp - 1] : 0) + i1 - s1;
        int ex2 = (warp ? sm.scan[32 + warp - 1] : 0) + i2 - s2;
        for (int q = 0; q < per; ++q) {
            const int e = e0 + q;
            if (e < N) {
                const int c = sm.scnt[e];
                sm.soff[e] = ex1;
                a.counts[e] = c;
                a.offsets[e] = ex1;
                if (c > 0) a.active[ex2] = e;
                ex1 += c;
                ex2 += c > 0;
            }
        }
        const int total = sm.scan[nwarps - 1], T = sm.scan[32 + nwarps - 1];
        if (threadIdx.x == 0) {
            a.offsets[N] = total;
            *a.T = T;
        }
        for (int q = T + threadIdx.x; q < N; q += nthreads) a.active[q] = -1;
    }
    __syncthreads();

    // ---- positions: pairs grouped by expert, tokens ascending -----------------
    for (int e = warp; e < N; e += nwarps) {
        if (sm.scnt[e] == 0) continue;
        int run = 0;
        const int off = sm.soff[e];
        for (int i0 = 0; i0 < B; i0 += 32) {
            const int i = i0 + lane;
            const uint32_t bit = i < B ? (sm.tokmask[(size_t)i * NW + (e >> 5)] >> (e & 31)) & 1u : 0u;
            const uint32_t bal = __ballot_sync(kFull, bit);
            if (bit) {
                const int pos = off + run + __popc(bal & lanemask_lt());
                int slot = -1;
                for (int j = 0; j < a.kslots; ++j)
                    if (sm.sidx[(size_t)i * a.kslots + j] == e) slot = j;
                if (slot < 0) {
                    raise_flag(a.flags, kFlagBadIndex);
                } else {
                    a.perm[pos] = i * a.kslots + slot;
                    a.pos_of[(size_t)i * a.kslots + slot] = pos;
                }
            }
            run += __popc(bal);
        }
    }
}

template <int NPL>
cudaError_t launch_route_t(const RouteArgs& a, cudaStream_t s) {
    const int threads = NPL <= 8 ? 1024 : 512;
    const size_t smem = 32 * 4 + 64 * 4 + MOE_MAX_TOKENS * 4 + 3 * MOE_MAX_EXPERTS * 4 +
                        (size_t)a.B * a.kslots * 4 + (size_t)a.B * ((a.N + 31) / 32) * 4;
    cudaError_t e = cudaFuncSetAttribute(route_kernel<NPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    route_kernel<NPL><<<1, threads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, cudaStream_t s) {
    const int nw = (a.N + 31) / 32;
    if (nw <= 1) return launch_route_t<1>(a, s);
    if (nw <= 2) return launch_route_t<2>(a, s);
    if (nw <= 4) return launch_route_t<4>(a, s);
    if (nw <= 8) return launch_route_t<8>(a, s);
    if (nw <= 16) return launch_route_t<16>(a, s);
    return launch_route_t<32>(a, s);
}

}  // namespace moe
