// route.cu -- per-token expert selection (plain top-k or OEA) and grouping of
// the (token, slot) pairs by expert, in one thread-block cluster.
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
// Each token's kept-slot count also seeds one counter per 128 rows of d,
// which the expert kernel counts down as the token's y slices are written.
// Ranking: larger score first, equal scores by the lower expert id.
//
// CTA r of the cluster (one CTA per 32 tokens, up to 8) handles tokens
// 32r..32r+31, one warp per token (two with 512 threads).  Lane l holds
// experts l, l+32, ... as order-preserving 32-bit keys of their fp32 scores
// (the map is a bijection, so a key gives back its exact score).  The
// next-ranked expert is one warp max-reduction of the keys and one
// min-reduction of the ids that hold the maximum.  Each CTA builds the union
// of its tokens' baselines as an N-bit mask in shared memory (__ballot_sync +
// atomicOr); after a cluster barrier every CTA ORs the masks of all CTAs
// (distributed shared memory) into S_base.  Grouping by expert: every kept
// (token, expert) sets bit (token mod 32) of the CTA's word [expert]; after a
// second cluster barrier every CTA reads all CTAs' words, and its warps, 32
// experts each, turn them into per-expert counts, offsets and the pairs of
// earlier CTAs, which give each pair's position directly (tokens ascending
// within an expert).  CTA 0 writes the per-expert arrays.
//
// With OEA and up to 64 tokens (one or two CTAs), S_base is published to
// the workspace as soon as phase 1 (and the cluster's union) is done, each
// word with the routing call's epoch: the expert kernel, already resident,
// starts on the activated experts' weights while phase 2 and the grouping
// run.
//
// For bf16 batches of up to 32 tokens with N <= 128, route_fused_kernel
// also computes the router scores (page section 2 Q1/Q2: every token scores
// all N experts), in one cluster of N/16 CTAs, and runs the same selection
// and grouping on them from shared memory, so a layer needs no separate
// router kernel.
#include <limits.h>

#include "common.cuh"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxCtas = MOE_MAX_TOKENS / 32;   // cluster size for the largest batch
static_assert(kMaxCtas <= 8, "a portable cluster holds at most 8 CTAs");

// Order-preserving key of a finite fp32 score (-0 and +0 map to one key);
// 0 is below every score and marks "not selectable".
__device__ __forceinline__ uint32_t score_key(float f) {
    const uint32_t b = __float_as_uint(f + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int NPL>
__device__ __forceinline__ void load_keys(const float* row, int N, int lane, uint32_t (&kv)[NPL], bool& nonfinite) {
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
        const int e = lane + 32 * j;
        uint32_t k = 0;
        if (e < N) {
            const float x = row[e];
            if (isfinite(x)) k = score_key(x); else nonfinite = true;
        }
        kv[j] = k;
    }
}

// Best remaining expert: largest key among entries whose bit in `excl` is
// clear, lowest expert id among equal keys.  Returns key 0 when none is left.
template <int NPL>
__device__ __forceinline__ uint32_t warp_best(const uint32_t (&kv)[NPL], uint32_t excl, int lane, int& id) {
    uint32_t lk = 0;
    int lid = INT_MAX;
#pragma unroll
    for (int j = 0; j < NPL; ++j)
        if (!((excl >> j) & 1u) && kv[j] > lk) {   // ascending j = ascending id
            lk = kv[j];
            lid = lane + 32 * j;
        }
    const uint32_t m = __reduce_max_sync(kFull, lk);
    id = (int)__reduce_min_sync(kFull, lk == m ? (uint32_t)lid : 0xffffffffu);
    return m;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    return x;
}

__device__ __forceinline__ uint32_t ld_dsmem_u32(const uint32_t* local, uint32_t rank) {
    uint32_t raddr, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(raddr) : "memory");
    return v;
}

struct RouteSmem {
    uint32_t* sbase;   // [32]          union of this CTA's tokens' baselines
    uint32_t* sball;   // [32]          S_base: union over the cluster
    uint32_t* btot;    // [32]          packed totals of 32-expert blocks
    int* snb;          // [32]          n_i of this CTA's tokens
    int* soff;         // [N]           first pair of expert e
    int* pre;          // [N]           pairs of expert e of earlier CTAs' tokens
    uint32_t* bits;    // [N]           bit il set if this CTA's token il keeps expert e
    int* sidx;         // [32][kslots]  kept experts of this CTA's tokens
};

// Writes the routing of token i (this CTA's token il): lane r < cnt holds
// slot r (myid, myval).
__device__ __forceinline__ void finish_token(const RouteArgs& a, RouteSmem& sm, int i, int il, int lane, int cnt,
                                             int myid, float myval) {
    const float l0 = __shfl_sync(kFull, myval, 0);
    const float ex = lane < cnt ? expf(myval - l0) : 0.f;
    const float z = warp_sum(ex);
    if (lane == 0) a.nused[i] = cnt;
    for (int r = lane; r < a.rbd; r += 32) a.ycnt[(size_t)i * a.rbd + r] = (uint32_t)cnt;
    if (lane < a.kslots) {
        const size_t q = (size_t)i * a.kslots + lane;
        const bool used = lane < cnt;
        a.idx[q] = used ? myid : -1;
        a.w[q] = used ? ex / z : 0.f;
        sm.sidx[il * a.kslots + lane] = used ? myid : -1;
        if (used) atomicOr(&sm.bits[myid], 1u << il);
        else a.pos_of[q] = -1;
    }
}

// Publishes the OEA union S_base: lane j stores word j (bit b: expert
// 32j + b) together with the call's epoch in one 64-bit store, so a reader
// that sees the epoch sees the word.  The activated set is S_base as soon
// as phase 1 is done: phase 2 only adds tokens to experts inside it, and
// every expert in it keeps the token whose baseline put it there.  The
// expert kernel, launched early, starts on those experts' weights from it
// while phase 2 and the grouping run.  CTA 0's last warp.
__device__ __forceinline__ void publish_union(const RouteArgs& a, uint32_t word, int lane) {
    st_relaxed_gpu_u64(&a.uwords[lane], ((uint64_t)a.epoch << 32) | (lane < (a.N + 31) / 32 ? word : 0u));
}

// Zeroes the shared union and per-expert token words of route_body's layout
// and, in CTA 0, the counter set that the expert call after the previous
// routing call used (it has completed: the caller has waited for the
// preceding kernel); the expert call after the next routing call uses it.
// The last warp, which publishes S_base, takes no part in the clearing.
// The caller synchronises the CTA before route_body reads them.
__device__ __forceinline__ void route_prepare(const RouteArgs& a, unsigned char* smem_raw, const uint32_t rank) {
    const int nthreads = blockDim.x;
    const int warp = threadIdx.x >> 5, nwarps = nthreads >> 5;
    uint32_t* sbase = reinterpret_cast<uint32_t*>(smem_raw);
    uint32_t* bits = reinterpret_cast<uint32_t*>(smem_raw + 4 * 32 * 4 + 2 * (size_t)a.N * 4);
    if (threadIdx.x < 32) sbase[threadIdx.x] = 0;
    for (int q = threadIdx.x; q < a.N; q += nthreads) bits[q] = 0;
    if (rank == 0 && a.clr_hdone && warp < nwarps - 1) {
        for (int q = threadIdx.x; q < kHdoneSet; q += nthreads - 32) a.clr_hdone[q] = 0u;
        if (threadIdx.x == 0) {
            *a.clr_next = 0u;
            *a.clr_gathered = 0u;
        }
    }
}

// The routing of tokens [32 rank, 32 rank + 32) by one CTA of `ncta` in a
// cluster, from the scores at `logits` (global or shared memory).  Prepared:
// the caller has run route_prepare and synchronised the CTA after its
// dependency wait.
template <int NPL, bool kPrepared>
__device__ __forceinline__ void route_body(const RouteArgs& a, const float* logits, unsigned char* smem_raw,
                                           const uint32_t rank, const uint32_t ncta) {
    const int nthreads = blockDim.x;
    const int nwarps = nthreads >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = a.N, B = a.B;
    const int tb = 32 * (int)rank;                   // this CTA's tokens: [tb, te)
    const int te = min(B, tb + 32);
    const int bv = min(te, max(tb, a.B_valid));      // valid tokens of this CTA: [tb, bv)

    RouteSmem sm;
    unsigned char* p = smem_raw;
    sm.sbase = reinterpret_cast<uint32_t*>(p); p += 32 * 4;
    sm.sball = reinterpret_cast<uint32_t*>(p); p += 32 * 4;
    sm.btot = reinterpret_cast<uint32_t*>(p); p += 32 * 4;
    sm.snb = reinterpret_cast<int*>(p); p += 32 * 4;
    sm.soff = reinterpret_cast<int*>(p); p += (size_t)N * 4;
    sm.pre = reinterpret_cast<int*>(p); p += (size_t)N * 4;
    sm.bits = reinterpret_cast<uint32_t*>(p); p += (size_t)N * 4;
    sm.sidx = reinterpret_cast<int*>(p);

    if (!kPrepared) {
        grid_launch_dependents();    // the expert kernel may start its prologue
        grid_dependency_wait();      // scores come from the router kernel
        route_prepare(a, smem_raw, rank);
        __syncthreads();
    }

    bool nonfinite = false;
    const bool oea = a.mode == MOE_MODE_OEA;
    const bool keep_keys = te - tb <= nwarps;   // one token per warp: keys and picks stay in registers
    uint32_t kv[NPL];
    // Phase-1 picks of this warp's token (used by phase 2 when keep_keys).
    uint32_t taken1 = 0;
    int n1 = 0, myid1 = -1;
    float myval1 = 0.f;

    // ---- plain top-k, or OEA phase 1 (baseline and union) ------------------
    for (int i = tb + warp; i < te; i += nwarps) {
        const int il = i - tb;
        load_keys<NPL>(logits + (size_t)i * N, N, lane, kv, nonfinite);
        if (i >= a.B_valid) {           // padding token: selects nothing
            if (lane == 0) {
                sm.snb[il] = 0;
                if (a.n_base && !oea) a.n_base[i] = 0;   // OEA: after S_base is published
            }
            if (!oea) finish_token(a, sm, i, il, lane, 0, -1, 0.f);
            continue;
        }
        uint32_t taken = 0;
        int myid = -1, n = 0;
        float myval = 0.f;
        if (!oea) {
            for (int r = 0; r < a.k; ++r) {
                int id;
                const uint32_t m = warp_best<NPL>(kv, taken, lane, id);
                if (m == 0) break;
                if ((id & 31) == lane) taken |= 1u << (id >> 5);
                if (lane == r) { myid = id; myval = key_score(m); }
                n = r + 1;
            }
            if (lane == 0 && a.n_base) a.n_base[i] = n;
            finish_token(a, sm, i, il, lane, n, myid, myval);
            continue;
        }
        // Phase 1: top-n_i in rank order; with top-p on, the softmax over all
        // N scores (fp32) gives the prefix mass that stops the selection.
        const bool top_p = a.p < 1.f;
        float m = 0.f, Z = 1.f;
        if (top_p) {
            int id0;
            m = key_score(warp_best<NPL>(kv, 0u, lane, id0));
            float zl = 0.f;
#pragma unroll
            for (int j = 0; j < NPL; ++j)
                if (kv[j]) zl += expf(key_score(kv[j]) - m);
            Z = warp_sum(zl);
        }
        float prefix = 0.f;
        for (int r = 0; r < a.k0; ++r) {
            int id;
            const uint32_t bk = warp_best<NPL>(kv, taken, lane, id);
            if (bk == 0) break;
            if ((id & 31) == lane) taken |= 1u << (id >> 5);
            if (lane == r) { myid = id; myval = key_score(bk); }
            n = r + 1;
            if (top_p) {
                prefix += expf(key_score(bk) - m) / Z;
                if (prefix >= a.p) break;
            }
        }
#pragma unroll
        for (int j = 0; j < NPL; ++j) {
            const uint32_t word = __ballot_sync(kFull, (taken >> j) & 1u);
            if (lane == 0 && word) atomicOr(&sm.sbase[j], word);
        }
        if (lane == 0) sm.snb[il] = n;   // n_base is written after S_base is published
        taken1 = taken; n1 = n; myid1 = myid; myval1 = myval;
    }

    // ---- OEA phase 2: piggyback inside S_base -------------------------------
    // The baseline (the token's top-n_i) lies inside S_base and heads both the
    // in-union list and the walked list, so with the phase-1 picks still in
    // registers the selection resumes at rank n_i.
    if (oea) {
        const uint32_t* sb = sm.sbase;   // S_base
        if (ncta > 1) {
            cluster_sync();   // every CTA's union is complete
            if (threadIdx.x < 32) {
                uint32_t w = 0;
                for (uint32_t r = 0; r < ncta; ++r)
                    w |= r == rank ? sm.sbase[threadIdx.x] : ld_dsmem_u32(&sm.sbase[threadIdx.x], r);
                sm.sball[threadIdx.x] = w;
            }
            sb = sm.sball;
        }
        __syncthreads();
        // S_base (over the cluster), from CTA 0's last warp.  Each word holds
        // the routing call's epoch in the same 64-bit store, and the expert
        // kernel reads everything else of this kernel's only after its
        // completion, so the stores are relaxed: no fence, which would wait
        // for this CTA's earlier stores (1.8 us measured).
        if (rank == 0 && a.uwords && warp == nwarps - 1) publish_union(a, sb[lane], lane);
        if (a.n_base)
            for (int i = tb + (int)threadIdx.x; i < te; i += nthreads) a.n_base[i] = sm.snb[i - tb];
        uint32_t notin = 0;
#pragma unroll
        for (int j = 0; j < NPL; ++j)
            if (!((sb[j] >> lane) & 1u)) notin |= 1u << j;
        for (int i = tb + warp; i < bv; i += nwarps) {
            const int il = i - tb;
            uint32_t taken = 0;
            int cnt = 0, myid = -1, r0 = 0;
            float myval = 0.f;
            if (keep_keys) {
                taken = taken1; cnt = n1; r0 = n1; myid = myid1; myval = myval1;
            } else {
                bool dummy = false;
                load_keys<NPL>(logits + (size_t)i * N, N, lane, kv, dummy);
            }
            if (a.maxP >= N) {
                // the in-union experts in rank order; the first n_i are the baseline
                for (int r = r0; r < a.kmax; ++r) {
                    int id;
                    const uint32_t m = warp_best<NPL>(kv, taken | notin, lane, id);
                    if (m == 0) break;
                    if ((id & 31) == lane) taken |= 1u << (id >> 5);
                    if (lane == r) { myid = id; myval = key_score(m); }
                    cnt = r + 1;
                }
            } else {
                // walk the ranked list to depth max(maxP, n_i)
                const int nb = sm.snb[il];
                const int depth = a.maxP > nb ? a.maxP : nb;
                for (int r = r0; r < depth && cnt < a.kmax; ++r) {
                    int id;
                    const uint32_t m = warp_best<NPL>(kv, taken, lane, id);
                    if (m == 0) break;
                    if ((id & 31) == lane) taken |= 1u << (id >> 5);
                    const bool in_union = (sb[id >> 5] >> (id & 31)) & 1u;
                    if (r < nb || in_union) {
                        if (lane == cnt) { myid = id; myval = key_score(m); }
                        ++cnt;
                    }
                }
            }
            finish_token(a, sm, i, il, lane, cnt, myid, myval);
        }
        for (int i = bv + warp; i < te; i += nwarps) finish_token(a, sm, i, i - tb, lane, 0, -1, 0.f);
    }
    if (__any_sync(kFull, nonfinite) && lane == 0) raise_flag(a.flags, kFlagNonFinite);
    if (ncta > 1) cluster_sync(); else __syncthreads();   // every CTA's (token, expert) words are complete

    // ---- counts, offsets, active list and per-expert info ---------------------
    // Warp w scans expert blocks w, w + nwarps, ... (32 experts each): per
    // expert the pairs of every CTA (its words, read across the cluster) and
    // of the CTAs before this one, then one packed inclusive scan of
    // (count | active << 26) across the block; the block totals meet in
    // shared memory and each warp adds the totals of the blocks before its
    // own.  A block's count is at most B * kslots < 2^26 and its active count
    // at most 32, so the packed sum never carries across fields.
    constexpr int kBlkPerWarp = NPL <= 16 ? 1 : 2;   // 32 (or 16) warps cover N / 32 blocks
    const int nblk = (N + 31) >> 5;
    int cnt_r[kBlkPerWarp];
    uint32_t inc_r[kBlkPerWarp];
    uint32_t m0_r[kBlkPerWarp], m1_r[kBlkPerWarp];   // tokens 0-31 and 32-63 of expert e (batches of up to 64)
#pragma unroll
    for (int u = 0; u < kBlkPerWarp; ++u) {
        const int b = warp + u * nwarps;
        cnt_r[u] = 0;
        inc_r[u] = 0;
        m0_r[u] = m1_r[u] = 0u;
        if (b < nblk) {
            const int e = (b << 5) + lane;
            int c = 0;
            if (e < N) {
                uint32_t w[kMaxCtas];
#pragma unroll
                for (int r = 0; r < kMaxCtas; ++r)
                    w[r] = r < (int)ncta ? (r == (int)rank ? sm.bits[e] : ld_dsmem_u32(&sm.bits[e], r)) : 0u;
#pragma unroll
                for (int r = 0; r < kMaxCtas; ++r) {
                    if (r == (int)rank) sm.pre[e] = c;
                    c += __popc(w[r]);
                }
                m0_r[u] = w[0];
                m1_r[u] = kMaxCtas > 1 ? w[1] : 0u;
            }
            uint32_t v = (uint32_t)c | ((uint32_t)(c > 0) << 26);
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t t = __shfl_up_sync(kFull, v, off);
                if (lane >= off) v += t;
            }
            cnt_r[u] = c;
            inc_r[u] = v;
            if (lane == 31) sm.btot[b] = v;
        }
    }
    __syncthreads();
    {
        // totals of all blocks (for T and offsets[N]) and of the blocks before each of ours
        const uint32_t tv = lane < nblk ? sm.btot[lane] : 0u;
        const int tc = (int)(tv & ((1u << 26) - 1)), ta = (int)(tv >> 26);
        const bool writer = rank == 0;
#pragma unroll
        for (int u = 0; u < kBlkPerWarp; ++u) {
            const int b = warp + u * nwarps;
            if (b >= nblk) break;
            const int e = (b << 5) + lane;
            const int base1 = __reduce_add_sync(kFull, lane < b ? tc : 0);
            const int base2 = __reduce_add_sync(kFull, lane < b ? ta : 0);
            const int c = cnt_r[u], act = c > 0;
            const int ex1 = base1 + (int)(inc_r[u] & ((1u << 26) - 1)) - c;
            const int ex2 = base2 + (int)(inc_r[u] >> 26) - act;
            if (e < N) {
                sm.soff[e] = ex1;
                if (writer) {
                    a.counts[e] = c;
                    a.offsets[e] = ex1;
                    if (act) {
                        a.active[ex2] = e;
                        a.exinfo[ex2] = (uint32_t)e | ((uint32_t)c << 10) | ((uint32_t)ex1 << 19);
                        // the expert's tokens (batches of up to 64: the first two CTAs' words)
                        a.exinfo[N + ex2] = B <= 64 ? m0_r[u] : 0u;
                        a.exinfo[2 * N + ex2] = B <= 64 ? m1_r[u] : 0u;
                    }
                }
            }
        }
        const int total = __reduce_add_sync(kFull, tc);
        const int T = __reduce_add_sync(kFull, ta);
        if (writer) {
            if (threadIdx.x == 0) {
                a.offsets[N] = total;
                *a.T = T;
            }
            for (int q = T + threadIdx.x; q < N; q += nthreads) {
                a.active[q] = -1;
                a.exinfo[q] = 0;
                a.exinfo[N + q] = 0;
                a.exinfo[2 * N + q] = 0;
            }
        }
    }
    __syncthreads();

    // ---- positions: pairs grouped by expert, tokens ascending -----------------
    for (int q = threadIdx.x; q < (te - tb) * a.kslots; q += nthreads) {
        const int e = sm.sidx[q];
        if (e < 0) continue;
        const int il = q / a.kslots;
        const int pos = sm.soff[e] + sm.pre[e] + __popc(sm.bits[e] & ((1u << il) - 1u));
        const int qg = tb * a.kslots + q;
        a.perm[pos] = qg;
        a.pos_of[qg] = pos;
    }
    if (ncta > 1) cluster_sync();   // no CTA leaves while another may still read its words
}

template <int NPL>
__global__ void route_kernel(RouteArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    route_body<NPL, false>(a, a.logits, smem_raw, cluster_ctarank(), gridDim.x);   // the whole grid is one cluster
}

// ---- scores and routing in one cluster (bf16, up to 32 tokens, N <= 128) ----
// CTA r of the cluster scores experts [16r, 16r + 16) for all tokens over
// the whole hidden dimension: its 32 warps take the 64-column blocks w,
// w + 32, ... with warp-level bf16 MMAs (the operand loads and the K-index
// permutation of the separate router kernel), then sum their partial tiles
// in warp order.  Each CTA stores its scores straight into CTA 0's score
// array (distributed shared memory; one cluster barrier completes it), and
// CTA 0 runs the routing above on the scores in its own shared memory, so
// the scores never make a round trip through global memory between two
// kernels (they are still written there, as the routing's logits output).
// Each warp loads its first block of router weights before the dependency
// wait: the weights do not come from the preceding kernel.
constexpr int kFusedWarps = 32;

// Opt-in dynamic shared memory per block of the current device.
size_t smem_cap() {
    static int cap[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 48 * 1024;
    if (!cap[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 48 * 1024;
        cap[dev] = v;
    }
    return (size_t)cap[dev];
}

__device__ __forceinline__ uint4 ldg16(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__host__ __device__ constexpr size_t route_smem_bytes(int N, int kslots) {
    return 4 * 32 * 4 + 3 * (size_t)N * 4 + 32 * (size_t)kslots * 4;
}

// Shared memory of the fused kernel: the routing's, the scores [32][N]
// (complete in CTA 0) and the warps' partial tiles [32][512].
__host__ __device__ constexpr size_t fused_smem_bytes(int N, int kslots) {
    return ((route_smem_bytes(N, kslots) + 15) & ~size_t(15)) + 32 * (size_t)N * 4 +
           (size_t)kFusedWarps * 512 * 4;
}

template <int NPL>
__global__ void __launch_bounds__(kFusedWarps * 32, 1) route_fused_kernel(RouterArgs r, RouteArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const size_t rsm = (route_smem_bytes(a.N, a.kslots) + 15) & ~size_t(15);
    float* lg = reinterpret_cast<float*>(smem_raw + rsm);             // [32][N] scores (CTA 0)
    float* red = lg + 32 * a.N;                                        // [32 warps][512] partial tiles
    const uint32_t rank = cluster_ctarank();   // the whole grid is one cluster
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int e0 = 16 * (int)rank;
    const int ntv = min(4, (r.B + 7) / 8);   // 8-token n-tiles holding real tokens
    const int kbtot = r.d / 64;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(r.x);
    const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(r.w);
    const int r0 = e0 + g, r1 = e0 + g + 8;
    // The router weights do not come from the preceding kernel: the warp's
    // first K block is loaded before the dependency wait.
    auto load_w = [&](int kb, uint4& wa0, uint4& wa1, uint4& wb0, uint4& wb1) {
        const int col = kb * 64 + 16 * t;
        wa0 = make_uint4(0, 0, 0, 0), wa1 = wa0, wb0 = wa0, wb1 = wa0;
        if (kb >= kbtot) return;
        if (r0 < r.N) { wa0 = ldg16(w + (size_t)r0 * r.d + col); wa1 = ldg16(w + (size_t)r0 * r.d + col + 8); }
        if (r1 < r.N) { wb0 = ldg16(w + (size_t)r1 * r.d + col); wb1 = ldg16(w + (size_t)r1 * r.d + col + 8); }
    };
    uint4 pa0, pa1, pb0, pb1;
    load_w(warp, pa0, pa1, pb0, pb1);
    grid_launch_dependents();    // the expert kernel may start its prologue
    grid_dependency_wait();      // hidden states come from the preceding kernel
    // CTA 0's routing state, set up while the token rows load; the cluster
    // barrier after the scores orders it before the routing reads it
    if (rank == 0) route_prepare(a, smem_raw, 0u);

    float acc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;
    for (int kb = warp; kb < kbtot; kb += kFusedWarps) {
        const int col = kb * 64 + 16 * t;
        uint4 wa0 = pa0, wa1 = pa1, wb0 = pb0, wb1 = pb1;
        if (kb != warp) load_w(kb, wa0, wa1, wb0, wb1);
        const uint32_t A0[8] = {wa0.x, wa0.y, wa0.z, wa0.w, wa1.x, wa1.y, wa1.z, wa1.w};
        const uint32_t A1[8] = {wb0.x, wb0.y, wb0.z, wb0.w, wb1.x, wb1.y, wb1.z, wb1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j >= ntv) break;
            const int tok = 8 * j + g;
            uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
            if (tok < r.B) { xa = ldg16(x + (size_t)tok * r.d + col); xb = ldg16(x + (size_t)tok * r.d + col + 8); }
            const uint32_t X[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16_16816(acc[j], A0[2 * s], A1[2 * s], A0[2 * s + 1], A1[2 * s + 1], X[2 * s], X[2 * s + 1]);
        }
    }
    // the warps' partial tiles (fragment-linear), summed in warp order; each
    // score goes straight into CTA 0's score array (distributed shared
    // memory), so one cluster barrier completes the [B][N] scores there
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) red[warp * 512 + j * 128 + lane * 4 + q2] = acc[j][q2];
    __syncthreads();
    if (threadIdx.x < 512) {
        const int l = threadIdx.x;
        float sum = 0.f;
        for (int w2 = 0; w2 < kFusedWarps; ++w2) sum += red[w2 * 512 + l];
        const int j = l >> 7, ln = (l >> 2) & 31, q2 = l & 3;
        const int row = (ln >> 2) + 8 * (q2 >> 1);
        const int tok = 8 * j + 2 * (ln & 3) + (q2 & 1);
        const int e = e0 + row;
        if (tok < r.B && e < r.N) {
            if (r.bias) sum += r.bias[e];
            r.logits[(size_t)tok * r.N + e] = sum;
            float* dst = &lg[tok * r.N + e];
            if (rank == 0) *dst = sum; else st_dsmem_f32(dst, 0u, sum);
        }
    }
    const bool clustered = gridDim.x > 1;   // one CTA (N <= 16) is launched without a cluster
    if (clustered) cluster_sync(); else __syncthreads();   // CTA 0 holds every score
    if (rank != 0) return;
    // the routing reads every argument from the kernel's parameters and the
    // scores from shared memory
    route_body<NPL, true>(a, lg, smem_raw, 0u, 1u);
}

template <int NPL>
cudaError_t launch_route_fused_t(const RouterArgs& r, const RouteArgs& a, cudaStream_t s) {
    const int ncta = (a.N + 15) / 16;
    const size_t smem = fused_smem_bytes(a.N, a.kslots);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(route_fused_kernel<NPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_cap());
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncta);
    cfg.blockDim = dim3(kFusedWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = ncta;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ncta > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, route_fused_kernel<NPL>, r, a);
}

template <int NPL>
cudaError_t launch_route_t(const RouteArgs& a, cudaStream_t s) {
    const int threads = NPL <= 8 ? 1024 : 512;
    const int ncta = a.B > 0 ? (a.B + 31) / 32 : 1;
    const size_t smem = 4 * 32 * 4 + 3 * (size_t)a.N * 4 + 32 * (size_t)a.kslots * 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ncta);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // batches of up to 32 tokens: one CTA, launched without a cluster
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = ncta;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ncta > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, route_kernel<NPL>, a);
}

}  // namespace

bool route_fused_supported(int dtype, int B, int N, int kslots) {
    return dtype == MOE_DTYPE_BF16 && B > 0 && B <= 32 && N <= 128 && fused_smem_bytes(N, kslots) <= smem_cap();
}

cudaError_t launch_route_fused(const RouterArgs& r, const RouteArgs& a, cudaStream_t s) {
    const int nw = (a.N + 31) / 32;
    if (nw <= 1) return launch_route_fused_t<1>(r, a, s);
    if (nw <= 2) return launch_route_fused_t<2>(r, a, s);
    return launch_route_fused_t<4>(r, a, s);
}

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
