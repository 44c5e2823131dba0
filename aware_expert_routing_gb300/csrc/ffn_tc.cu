// ffn_tc.cu -- grouped SwiGLU expert FFN + weighted combine on the
// 5th-generation tensor cores (tcgen05), bf16 weights.
//
// Page "Opportunistic Expert Activation (OEA)": at decode the MoE layer is
// memory bound and its latency is set by fetching every activated expert's
// weights from HBM (section 2 Q1, section 4 check 4).  This kernel streams
// each activated expert's gate, up and down matrices from HBM once and does
// the arithmetic of all the tokens routed to it while the tile is on chip.
// Expert form (Qwen3): y = W_down (silu(W_gate x) * (W_up x)); combine:
// out_i = sum_j w_ij y_{e_ij}(x_i) (kept scores, section 2 Q2).
//
// Structure (one persistent CTA per SM, 15 warps):
//   * Work is a list of tiles.  Phase-A tile (expert a, 64 rows of d_ff,
//     token chunk c): the 64 W_gate rows and the 64 W_up rows of the same
//     d_ff indices, interleaved 8 rows at a time (rows 16g..16g+7 = gate
//     rows 8g..8g+7, rows 16g+8..16g+15 = the up rows), form the 128-row A
//     operand of a tcgen05 MMA with M = 128; the chunk's token rows are the
//     N operand (N = the chunk's tokens rounded up to 16; a chunk holds the
//     whole batch of up to 16 tokens, else up to nmax = the largest expert's
//     token count rounded up to 16, at most 128, so most experts' weights
//     are streamed once); K = d.  Phase-B tile (expert a, 128 rows of d,
//     chunk c): W_down rows times the chunk's h rows, K = d_ff.  The list
//     holds every phase-A tile, then every phase-B tile, each in active-
//     expert order; CTA b starts with tile b and claims each next tile (two
//     ahead) from one grid-wide counter, so all CTAs finish within about
//     one tile of each other.
//   * Warp 4 claims the tiles, posts them to a 16-entry shared-memory queue
//     and streams the weights: one TMA operation per 16 KB stage (128 rows x
//     64 columns, 128-byte swizzle; the gate/up interleave comes from one 5D
//     tensor map over both matrices).  Warp 5 streams the 16 token rows of
//     each stage (16-row boxes): the whole batch of up to 16 tokens straight
//     from the hidden states, or rows of the expert-grouped copy of the
//     hidden states, or (phase B) rows of h once every phase-A tile of the
//     chunk has written them (a per-chunk counter).  Ring: 180 KB of stages
//     of 16 KB + nmax x 128 bytes (10 stages at nmax = 16, 5 at 128).
//   * Warp 6, lane 0, issues the MMAs: four K=16 steps per stage straight
//     from the swizzled shared memory (no register staging), fp32
//     accumulators in tensor memory, four accumulator buffers (16 columns
//     each for batches of up to 16 tokens, else 128).
//     tcgen05.commit frees each stage when its MMAs have completed and marks
//     a tile's accumulator full.
//   * INT4 experts (DynaExq page, section 3.2): warp 4 bulk-copies the
//     packed chunks of a stage into a 4-slot raw ring; warps 7-14 decode
//     them (exact integer codes, times the row's group scale, rounded once
//     to bf16) into the stage's 128-byte-swizzled A operand, fence it for
//     the tensor core's async proxy and arrive on the stage's barrier in
//     place of warp 4.
//   * Warps 0-3 (tensor-memory lanes 32w..32w+31, one D row per thread)
//     read a finished accumulator with tcgen05.ld and free it; phase A:
//     the lane holding gate row r takes the matching up row from the lane
//     8 above (shuffle), applies SwiGLU and stores h (bf16) for the tile's
//     tokens; phase B: stores y (fp32).  After a phase-A tile the four warps
//     meet at a shared-memory barrier and one thread releases the chunk's
//     counter.
//   * All phase-A tiles precede all phase-B tiles in the list and wait on
//     nothing later, so every wait ends.  After its last tile every CTA
//     arrives at one grid-wide counter; once all have, each CTA combines a
//     slice of the output (float4, slot order).  The last CTA resets the
//     counters for the next launch.
// Every wait is bounded; a wait that gives up raises MOE_FLAG_WAIT_TIMEOUT
// and the CTA runs to its end without waiting again.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kEpiWarps = 4;             // warps 0-3: epilogue
constexpr int kWarpW = 4;                // weight producer
constexpr int kWarpO = 5;                // operand producer
constexpr int kWarpM = 6;                // MMA issuer, owner of the tensor memory
constexpr int kWarpC = 7;                // warps 7-14: INT4 converters
constexpr int kConvWarps = 8;
constexpr int kThreads = (kWarpC + kConvWarps) * 32;
constexpr int kM = 128;                  // weight rows per tile (MMA M)
constexpr int kNMax = 128;               // most token columns per tile (MMA N)
constexpr int kWBytes = kM * 128;        // 128 rows x 64 bf16
constexpr int kRingBytes = 10 * (kWBytes + 16 * 128);   // 10 stages with 16 token rows
constexpr int kMaxStages = 10;
constexpr int kRaw = 4;                  // packed INT4 chunks in flight
constexpr int kQ4A = 64 * 32 + 64 * 2;   // INT4 chunk of W_gate / W_up: 64 rows x 64 columns + scales
constexpr int kQ4B = 128 * 32 + 128 * 2; // INT4 chunk of W_down: 128 rows x 64 columns + scales
constexpr int kRawBytes = 2 * kQ4A;      // a phase-A stage needs a W_gate and a W_up chunk
static_assert(kRawBytes == kQ4B, "one raw slot fits either stage");
constexpr int kQ = 16;                   // tile queue entries
constexpr int kAcc = 4;                  // accumulator buffers
constexpr uint32_t kTmemCols = kAcc * kNMax;   // fp32 columns (batches over 16 tokens)
constexpr uint32_t kTmemColsSmall = kAcc * 16;  // batches of up to 16 tokens
constexpr uint32_t kBarEpi = 1;          // named barrier of the four epilogue warps
constexpr long long kWaitCycles = 4000000000LL;   // about two seconds
static_assert(kTmemCols <= 512, "tensor memory has 512 columns");

struct Smem {
    uint64_t full[kMaxStages];           // both producers (+ transaction bytes)
    uint64_t empty[kMaxStages];          // tcgen05.commit after the stage's MMAs
    uint64_t acc_full[kAcc];             // tcgen05.commit after a tile's last MMA
    uint64_t acc_empty[kAcc];            // the four epilogue warps
    uint64_t tq_full[kQ];                // tile queue entry posted by the weight warp
    uint64_t tq_empty[kQ];               // entry released by the four epilogue warps
    uint64_t mma_done;                   // every MMA issued has completed
    uint64_t h_written;                  // the four epilogue warps stored a phase-A tile's h rows
    uint64_t raw_full[kRaw];             // packed INT4 chunks landed (bulk copies)
    uint64_t raw_empty[kRaw];            // the four converter warps have read them
    uint64_t conv_bar;                   // the four converter warps meet (bounded wait)
    uint32_t raw_info[kRaw];             // target ring slot | phase A << 8, or ~0u (no more chunks)
    int tq[kQ];                          // tile index, or -1 once the list is exhausted
    int chunk_off[MOE_MAX_EXPERTS + 1];
    uint32_t ex_info[MOE_MAX_EXPERTS];   // active index -> id | cnt << 10 | first pair << 19
    uint16_t tokmask[MOE_MAX_EXPERTS];   // active index -> tokens routed to it (batches of <= 16)
    int ex_slot[MOE_MAX_EXPERTS];        // active index -> bf16 expert (>= 0) or -1 - INT4 expert
    uint32_t tmem_base;
    int nmax;                            // tokens per chunk for this launch (multiple of 16)
    int abort_flag;
    int last_flag;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kRingBytes + (size_t)kRaw * kRawBytes + sizeof(Smem);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct Tile {
    int a, e, rb, c, off, ntok, nch;
};

// Tile t of a phase with rbn row blocks per (expert, chunk); shared memory only.
__device__ __forceinline__ Tile decode_tile(int t, int rbn, const Smem& S, int Tn, int nmax) {
    int lo = 0, hi = Tn - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (S.chunk_off[mid] * rbn <= t) lo = mid; else hi = mid - 1;
    }
    Tile T;
    T.a = lo;
    const uint32_t info = S.ex_info[lo];
    T.e = info & 1023u;
    const int cnt = (info >> 10) & 511u;
    T.off = info >> 19;
    T.nch = S.chunk_off[lo + 1] - S.chunk_off[lo];
    const int r = t - S.chunk_off[lo] * rbn;
    T.rb = r / T.nch;
    T.c = r - T.rb * T.nch;
    T.ntok = min(nmax, cnt - nmax * T.c);
    return T;
}

__device__ __forceinline__ void give_up(Smem& S, uint32_t* flags) {
    *(volatile int*)&S.abort_flag = 1;
    raise_flag(flags, kFlagTimeout);
}

// Bounded mbarrier wait; once the CTA has given up every later wait returns
// at once, so the control flow (and every barrier) still completes.
__device__ __forceinline__ void wait_bar(uint64_t* bar, uint32_t parity, Smem& S, uint32_t* flags) {
    if (mbar_try_wait(bar, parity)) return;
    const long long t0 = clock64();
    while (!*(volatile int*)&S.abort_flag) {
        if (mbar_try_wait(bar, parity)) return;
        if (clock64() - t0 > kWaitCycles) {
            give_up(S, flags);
            return;
        }
    }
}

// Bounded wait until *p >= need (acquire, GPU scope).
__device__ __forceinline__ void wait_counter(const uint32_t* p, uint32_t need, Smem& S, uint32_t* flags) {
    if (ld_acquire_gpu(p) >= need) return;
    const long long t0 = clock64();
    while (!*(volatile int*)&S.abort_flag) {
        if (ld_acquire_gpu(p) >= need) return;
        if (clock64() - t0 > kWaitCycles) {
            give_up(S, flags);
            return;
        }
        __nanosleep(32);
    }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }

// Eight INT4 codes (one packed word, column 2p in the low and 2p+1 in the
// high half of nibble pair p) -> eight bf16 weights q*s, columns in order.
// (w >> 4p) & 0x000f000f | 0x43004300 is the bf16 pair (128 + c, 128 + c')
// with c = q + 8; subtracting 136 leaves q exactly; the product with the
// group scale is rounded once to bf16.
__device__ __forceinline__ uint4 decode_q4_row8(uint32_t w, __nv_bfloat162 s2) {
    const __nv_bfloat162 off = __floats2bfloat162_rn(136.f, 136.f);
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t v;
        asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(v) : "r"(w >> (4 * p)), "r"(0x000f000fu), "r"(0x43004300u));
        const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), off);
        const __nv_bfloat162 x = __hmul2(q, s2);
        o[p] = *reinterpret_cast<const uint32_t*>(&x);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The four converter warps meet; every warp calls this the same number of
// times, and the wait is bounded.
__device__ __forceinline__ void conv_sync(Smem& S, uint32_t& nsync, uint32_t* flags, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.conv_bar);
    wait_bar(&S.conv_bar, nsync & 1, S, flags);
    ++nsync;
}

// Position in the stage ring (the stage count is set per launch): slot,
// phase parity, and whether the ring has wrapped once (a producer then
// waits for the slot to be freed).
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    bool wrapped = false;
    __device__ __forceinline__ void next(int nst) {
        if (++slot == nst) {
            slot = 0;
            phase ^= 1u;
            wrapped = true;
        }
    }
};

__global__ void __launch_bounds__(kThreads, 1)
ffn_tc_kernel(const FfnArgs A, const __grid_constant__ CUtensorMap tm_gu, const __grid_constant__ CUtensorMap tm_gate,
              const __grid_constant__ CUtensorMap tm_up, const __grid_constant__ CUtensorMap tm_down,
              const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_h,
              const __grid_constant__ CUtensorMap tm_hid) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* raw = ring + (size_t)kRingBytes;   // kRaw packed INT4 slots
    Smem& S = *reinterpret_cast<Smem*>(raw + (size_t)kRaw * kRawBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = A.d, F = A.F;
    uint32_t* flags = &A.hdr->flags;
    const uint32_t G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&S.full[i], 2);          // weight producer + operand producer
            mbar_init(&S.empty[i], 1);         // tcgen05.commit
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(&S.acc_full[i], 1);
            mbar_init(&S.acc_empty[i], kEpiWarps);
        }
        for (int i = 0; i < kQ; ++i) {
            mbar_init(&S.tq_full[i], 1);
            mbar_init(&S.tq_empty[i], kEpiWarps);
        }
        mbar_init(&S.mma_done, 1);
        mbar_init(&S.h_written, kEpiWarps);
        for (int i = 0; i < kRaw; ++i) {
            mbar_init(&S.raw_full[i], 1);
            mbar_init(&S.raw_empty[i], kConvWarps);
        }
        mbar_init(&S.conv_bar, kConvWarps);
        fence_barrier_init();
        S.abort_flag = 0;
    }
    // accumulator buffers: kAcc x nmax columns, nmax = 16 for batches of up to 16
    const uint32_t tmem_cols = A.B <= 16 ? kTmemColsSmall : kTmemCols;
    const int acc_stride = A.B <= 16 ? 16 : kNMax;
    if (warp == kWarpM) tmem_alloc(&S.tmem_base, tmem_cols);
    __syncthreads();             // barriers initialised (this overlaps the routing kernel)
    grid_dependency_wait();      // routing comes from the preceding kernel
    int Tn = *A.T;
    if (Tn < 0 || Tn > A.N) {
        if (threadIdx.x == 0 && blockIdx.x == 0) raise_flag(flags, kFlagBadIndex);
        Tn = 0;
    }
    // Batches of up to 16 tokens: the CTA's first tile is phase-A tile
    // blockIdx.x of a one-chunk-per-expert list, so the weight warp starts
    // its stages now, while warp 0 builds the per-expert records.
    int fast_stages = 0;
    if (warp == kWarpW && lane == 0 && A.B <= 16) {
        const int rbA0 = F / 64, t0 = (int)blockIdx.x;
        if (t0 < Tn * rbA0) {
            const int e = (int)(A.exinfo[t0 / rbA0] & 1023u);
            const int sl = A.slot ? A.slot[e] : e;
            if (sl >= 0 && sl < A.n_hot) {
                const uint64_t pol = l2_evict_first_policy();
                const int row0 = sl * F + 64 * (t0 % rbA0);
                fast_stages = min(d / 64, min(kMaxStages, kRingBytes / (kWBytes + 16 * 128)));
                for (int s = 0; s < fast_stages; ++s) {
                    unsigned char* dst = ring + (size_t)s * (kWBytes + 16 * 128);
                    mbar_arrive_expect_tx(&S.full[s], kWBytes);
                    if (A.gu_fused) {
                        tma_load_5d(dst, &tm_gu, 0, 0, 0, row0 / 8, s, &S.full[s], pol);
                    } else {
                        for (int g = 0; g < 8; ++g) {
                            tma_load_3d(dst + (2 * g) * 1024, &tm_gate, 0, row0 + 8 * g, s, &S.full[s], pol);
                            tma_load_3d(dst + (2 * g + 1) * 1024, &tm_up, 0, row0 + 8 * g, s, &S.full[s], pol);
                        }
                    }
                }
            }
        }
    }
    if (warp == 0) {   // per-expert records, chunk width and chunk offsets of the active experts
        int maxcnt = 0;
        for (int a = lane; a < Tn; a += 32) {
            const uint32_t info = A.exinfo[a];   // written by the routing kernel
            S.ex_info[a] = info;
            S.tokmask[a] = (uint16_t)A.exinfo[A.N + a];
            maxcnt = max(maxcnt, (int)((info >> 10) & 511u));
            const int e = info & 1023u;
            int sl = A.slot ? A.slot[e] : e;
            if (sl >= A.n_hot || -1 - sl >= A.n_cold) {   // out of range: flag it, read expert 0
                raise_flag(flags, kFlagBadIndex);
                sl = A.n_hot > 0 ? 0 : -1;
            }
            S.ex_slot[a] = sl;
        }
        maxcnt = __reduce_max_sync(0xffffffffu, maxcnt);
        // a chunk holds up to nmax tokens: the whole batch for batches of up to
        // 16, else the largest expert's tokens rounded up to 16, at most 128
        const int nmax = A.B <= 16 ? 16 : min(kNMax, max(16, (maxcnt + 15) & ~15));
        if (lane == 0) S.nmax = nmax;
        __syncwarp();
        int run = 0;
        if (lane == 0) S.chunk_off[0] = 0;
        for (int a0 = 0; a0 < Tn; a0 += 32) {
            const int a = a0 + lane;
            int nch = 0;
            if (a < Tn) nch = ((int)((S.ex_info[a] >> 10) & 511u) + nmax - 1) / nmax;
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
    if (warp == kWarpW && lane == 0) {
        prefetch_tensormap(A.gu_fused ? &tm_gu : &tm_gate);
        if (!A.gu_fused) prefetch_tensormap(&tm_up);
        prefetch_tensormap(&tm_down);
    }
    if (warp == kWarpO && lane == 0) {
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_hid);
        prefetch_tensormap(&tm_h);
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tmem = S.tmem_base;

    // Tiles: phase A (expert, 64 rows of d_ff, chunk) first, then phase B
    // (expert, 128 rows of d, chunk), both in active-expert order.
    const int rbA = F / 64, rbB = (d + kM - 1) / kM;
    const int SA = d / 64, SB = F / 64;             // stages per tile (K blocks of 64)
    const int TA = S.chunk_off[Tn] * rbA;
    const int Ttot = TA + S.chunk_off[Tn] * rbB;
    const bool small_b = A.B <= 16;                 // phase-A operand: the whole batch
    const int nmax = S.nmax;
    const int slot_bytes = kWBytes + nmax * 128;    // 16 KB of weights + nmax token rows
    const int nst = min(kMaxStages, kRingBytes / slot_bytes);

    if (warp == kWarpW) {
        // ---------------------------- weight producer ----------------------------
        if (lane == 0) {
            const uint64_t pol_once = l2_evict_first_policy();
            const uint64_t pol_keep = l2_evict_normal_policy();
            RingPos rp, rq;   // stage ring, packed INT4 ring
            const size_t q4_mat_a = (size_t)(F / 64) * (d / 64) * kQ4A;    // bytes of one INT4 W_gate / W_up
            const size_t q4_mat_b = (size_t)(d / kM) * (F / 64) * kQ4B;    // bytes of one INT4 W_down
            // claims run two tiles ahead so that the atomic's latency is hidden
            int next0 = (int)blockIdx.x;
            int next1 = next0 < Ttot ? (int)G + (int)atomicAdd(&A.hdr->next_tile, 1u) : Ttot;
            for (int s = 0; s < fast_stages; ++s) rp.next(nst);   // stages issued before the prologue
            for (int n = 0;; ++n) {
                const int q = n % kQ;
                if (n >= kQ) wait_bar(&S.tq_empty[q], ((n / kQ) - 1) & 1, S, flags);
                const int tile = next0 < Ttot ? next0 : -1;
                S.tq[q] = tile;
                mbar_arrive(&S.tq_full[q]);
                if (tile < 0) break;
                next0 = next1;
                next1 = next1 < Ttot ? (int)G + (int)atomicAdd(&A.hdr->next_tile, 1u) : Ttot;
                const bool ph_a = tile < TA;
                const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, S, Tn, nmax);
                const uint64_t pol = T.nch > 1 ? pol_keep : pol_once;   // chunked experts are re-read from L2
                const int sl = S.ex_slot[T.a];                          // bf16 expert, or -1 - INT4 expert
                const int row0 = ph_a ? sl * F + 64 * T.rb : sl * d + kM * T.rb;
                const int ns = ph_a ? SA : SB;
                for (int s = n == 0 ? fast_stages : 0; s < ns; ++s, rp.next(nst)) {
                    const int slot = rp.slot;
                    if (rp.wrapped) wait_bar(&S.empty[slot], rp.phase ^ 1u, S, flags);
                    unsigned char* dst = ring + (size_t)slot * slot_bytes;
                    if (sl < 0) {
                        // INT4 expert: the packed chunk(s) go to a raw slot; the converter
                        // warps write the bf16 stage and arrive on its barrier.
                        const int r = rq.slot;
                        if (rq.wrapped) wait_bar(&S.raw_empty[r], rq.phase ^ 1u, S, flags);
                        S.raw_info[r] = (uint32_t)slot | (ph_a ? 256u : 0u);
                        unsigned char* rdst = raw + (size_t)r * kRawBytes;
                        const int c = -1 - sl;
                        if (ph_a) {
                            const size_t off = (size_t)c * q4_mat_a + ((size_t)T.rb * (d / 64) + s) * kQ4A;
                            mbar_arrive_expect_tx(&S.raw_full[r], 2 * kQ4A);
                            bulk_load(rdst, A.q_gate + off, kQ4A, &S.raw_full[r], pol);
                            bulk_load(rdst + kQ4A, A.q_up + off, kQ4A, &S.raw_full[r], pol);
                        } else {
                            const size_t off = (size_t)c * q4_mat_b + ((size_t)T.rb * (F / 64) + s) * kQ4B;
                            mbar_arrive_expect_tx(&S.raw_full[r], kQ4B);
                            bulk_load(rdst, A.q_down + off, kQ4B, &S.raw_full[r], pol);
                        }
                        rq.next(kRaw);
                        continue;
                    }
                    mbar_arrive_expect_tx(&S.full[slot], kWBytes);
                    if (!ph_a) {
                        // 128 W_down rows (rows past the expert's d are computed and dropped)
                        tma_load_3d(dst, &tm_down, 0, row0, s, &S.full[slot], pol);
                    } else if (A.gu_fused) {
                        // 8 row groups x {8 rows of the lower matrix, 8 rows of the other}
                        tma_load_5d(dst, &tm_gu, 0, 0, 0, row0 / 8, s, &S.full[slot], pol);
                    } else {
#pragma unroll 1
                        for (int g = 0; g < 8; ++g) {
                            tma_load_3d(dst + (2 * g) * 1024, &tm_gate, 0, row0 + 8 * g, s, &S.full[slot], pol);
                            tma_load_3d(dst + (2 * g + 1) * 1024, &tm_up, 0, row0 + 8 * g, s, &S.full[slot], pol);
                        }
                    }
                }
            }
            {   // no more INT4 chunks: the converter warps stop
                const int r = rq.slot;
                if (rq.wrapped) wait_bar(&S.raw_empty[r], rq.phase ^ 1u, S, flags);
                S.raw_info[r] = ~0u;
                mbar_arrive(&S.raw_full[r]);
            }
            // Every issued stage is consumed before the MMA warp finishes,
            // so no copy is in flight when the CTA exits.
        }
        __syncwarp();
    } else if (warp == kWarpO) {
        // ---------------------------- operand producer ---------------------------
        const uint64_t pol = l2_evict_last_policy();
        RingPos rp;
        bool gathered = small_b;
        for (int n = 0;; ++n) {
            const int q = n % kQ;
            wait_bar(&S.tq_full[q], (n / kQ) & 1, S, flags);
            const int tile = S.tq[q];
            if (tile < 0) break;
            const bool ph_a = tile < TA;
            const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, S, Tn, nmax);
            if (ph_a && !gathered) {   // every CTA has copied its rows of the grouped hidden states
                for (int c = lane; c < (int)G; c += 32) wait_counter(&A.gflag[c], 1u, S, flags);
                __syncwarp();
                fence_proxy_async_global();
                gathered = true;
            }
            if (lane == 0) {
                if (!ph_a) {   // every phase-A tile of this token chunk has written its h rows
                    wait_counter(&A.hdone[S.chunk_off[T.a] + T.c], (uint32_t)rbA, S, flags);
                    fence_proxy_async_global();
                }
                const CUtensorMap* map = ph_a ? (small_b ? &tm_hid : &tm_x) : &tm_h;
                const int row = (ph_a && small_b) ? 0 : T.off + nmax * T.c;
                const int nb = (ph_a && small_b) ? 1 : (T.ntok + 15) >> 4;   // 16-row boxes = MMA N / 16
                const int ns = ph_a ? SA : SB;
                for (int s = 0; s < ns; ++s, rp.next(nst)) {
                    const int slot = rp.slot;
                    if (rp.wrapped) wait_bar(&S.empty[slot], rp.phase ^ 1u, S, flags);
                    mbar_arrive_expect_tx(&S.full[slot], nb * 2048);   // rows past the end read as zeros
                    unsigned char* dst = ring + (size_t)slot * slot_bytes + kWBytes;
                    for (int j = 0; j < nb; ++j)
                        tma_load_3d(dst + j * 2048, map, 0, row + 16 * j, s, &S.full[slot], pol);
                }
            }
            __syncwarp();
        }
    } else if (warp == kWarpM) {
        // ------------------------------ MMA issuer -------------------------------
        if (lane == 0) {
            RingPos rp;
            for (int n = 0;; ++n) {
                const int q = n % kQ;
                wait_bar(&S.tq_full[q], (n / kQ) & 1, S, flags);
                const int tile = S.tq[q];
                if (tile < 0) break;
                const bool ph_a = tile < TA;
                int ntile = 16;   // MMA N: batches of up to 16 always use 16 columns
                if (!small_b) {
                    const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, S, Tn, nmax);
                    ntile = (ph_a && small_b) ? 16 : (T.ntok + 15) & ~15;
                }
                const uint32_t idesc = umma_idesc_bf16(kM, ntile);
                const int ns = ph_a ? SA : SB;
                const int b = n % kAcc;
                if (n >= kAcc) {   // the epilogue has read this accumulator's previous tile
                    wait_bar(&S.acc_empty[b], ((n / kAcc) - 1) & 1, S, flags);
                    tmem_fence_after_sync();
                }
                const uint32_t dt = tmem + (uint32_t)(b * acc_stride);
                for (int s = 0; s < ns; ++s, rp.next(nst)) {
                    const int slot = rp.slot;
                    wait_bar(&S.full[slot], rp.phase, S, flags);
                    tmem_fence_after_sync();
                    const uint32_t a0 = smem_u32(ring + (size_t)slot * slot_bytes);
                    const uint32_t b0 = a0 + kWBytes;
#pragma unroll
                    for (int k = 0; k < 4; ++k)   // K = 16 per step: 32 bytes along the swizzled row
                        umma_bf16(dt, umma_sdesc_sw128(a0 + 32 * k), umma_sdesc_sw128(b0 + 32 * k), idesc,
                                  (s | k) ? 1u : 0u);
                    umma_commit(&S.empty[slot]);   // the stage is free once these MMAs are done
                }
                umma_commit(&S.acc_full[b]);
            }
            umma_commit(&S.mma_done);
            wait_bar(&S.mma_done, 0, S, flags);
        }
        __syncwarp();
    } else if (warp >= kWarpC) {
        // ----------------------------- INT4 converters ----------------------------
        // Each packed stage becomes the 128 x 64 bf16 A operand of one ring
        // stage, 128-byte swizzled like a TMA box: output row i, 16-byte unit u
        // (8 columns) at i*128 + ((u ^ (i & 7)) << 4).  Phase A: row i =
        // (2g + m)*8 + r is row 8g + r of W_gate (m = 0) or W_up (m = 1).
        const int ct = threadIdx.x - kWarpC * 32;   // 0..kConvWarps*32-1
        RingPos rq;
        uint32_t nsync = 0;
        for (;;) {
            if (A.n_cold == 0) break;                  // no INT4 experts in this launch
            const int r = rq.slot;
            wait_bar(&S.raw_full[r], rq.phase, S, flags);
            const uint32_t info = S.raw_info[r];
            if (info == ~0u) break;
            const int slot = (int)(info & 255u);
            const bool ph_a = (info >> 8) & 1u;
            const unsigned char* src = raw + (size_t)r * kRawBytes;
            unsigned char* dstA = ring + (size_t)slot * slot_bytes;
#pragma unroll
            for (int it = 0; it < 1024 / (kConvWarps * 32); ++it) {   // 128 rows x 8 units
                const int k = it * (kConvWarps * 32) + ct;
                const int i = k >> 3, u = k & 7;
                const unsigned char* ch = ph_a ? src + ((i >> 3) & 1) * kQ4A : src;
                const int srow = ph_a ? 8 * (i >> 4) + (i & 7) : i;
                const int rows = ph_a ? 64 : kM;
                const uint32_t w = *reinterpret_cast<const uint32_t*>(ch + srow * 32 + u * 4);
                const __nv_bfloat16 sc = *reinterpret_cast<const __nv_bfloat16*>(ch + rows * 32 + srow * 2);
                *reinterpret_cast<uint4*>(dstA + i * 128 + ((u ^ (i & 7)) << 4)) =
                    decode_q4_row8(w, __bfloat162bfloat162(sc));
            }
            fence_proxy_async_shared();   // the tensor core reads the stage through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.raw_empty[r]);   // this warp has read the packed chunk
            conv_sync(S, nsync, flags, lane);              // all four warps have written their rows
            if (ct == 0) mbar_arrive(&S.full[slot]);       // in place of the weight warp
            rq.next(kRaw);
        }
    } else {
        // ------------------------------- epilogue --------------------------------
        const int tid = threadIdx.x;   // 0..127

        // Prologue (batches over 16 tokens): this CTA's rows of the
        // expert-grouped hidden states (rows b, b+G, ...), eight 16-byte
        // loads in flight per thread.
        if (!small_b) {
            const int P = A.offsets[A.N];
            const int vpr = d / 8;   // 16-byte vectors per row
            const int nrow = P > (int)blockIdx.x ? (P - 1 - (int)blockIdx.x) / (int)G + 1 : 0;
            const int nvec = nrow * vpr;
            const uint4* xs = static_cast<const uint4*>(A.x);
            uint4* xp = static_cast<uint4*>(A.xperm);
            for (int v0 = 0; v0 < nvec; v0 += 8 * kEpiWarps * 32) {
                uint4 val[8];
                size_t dst[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = v0 + u * kEpiWarps * 32 + tid;
                    dst[u] = ~size_t(0);
                    if (v < nvec) {
                        const int r = v / vpr, c = v - r * vpr;
                        const int pr = (int)blockIdx.x + r * (int)G;
                        val[u] = __ldg(xs + (size_t)(A.perm[pr] / A.kslots) * vpr + c);
                        dst[u] = (size_t)pr * vpr + c;
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (dst[u] != ~size_t(0)) xp[dst[u]] = val[u];
            }
            named_barrier(kBarEpi, kEpiWarps * 32);
            if (tid == 0) {
                __threadfence();
                atomicExch(&A.gflag[blockIdx.x], 1u);
            }
        }

        __nv_bfloat16* hb = static_cast<__nv_bfloat16*>(A.hbuf);
        const int i = 32 * warp + lane;                    // this thread's D row (tensor-memory lane)
        const uint32_t lane_addr = (uint32_t)(32 * warp) << 16;
        uint32_t na = 0;   // phase-A tiles so far (parity of h_written)
        for (int n = 0;; ++n) {
            const int q = n % kQ;
            wait_bar(&S.tq_full[q], (n / kQ) & 1, S, flags);
            const int tile = S.tq[q];
            if (tile < 0) break;
            const bool ph_a = tile < TA;
            const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, S, Tn, nmax);
            const int b = n % kAcc;
            const int ngroups = (ph_a && small_b) ? 1 : (T.ntok + 15) >> 4;   // 16-column groups of D
            wait_bar(&S.acc_full[b], (n / kAcc) & 1, S, flags);
            tmem_fence_after_sync();
            if (ph_a) {
                // D row i = (2g + m) * 8 + r holds gate (m = 0) or up (m = 1) row
                // 8g + r of the tile, or the reverse when the map starts at W_up;
                // the partner row is 8 lanes away in the same warp.
                const int m = (i >> 3) & 1;
                const int frow = 64 * T.rb + 8 * (i >> 4) + (i & 7);
                const uint32_t tmask = small_b ? S.tokmask[T.a] : 0u;
                const bool swap = A.gu_swap && S.ex_slot[T.a] >= 0;   // INT4 stages hold the gate rows first
                for (int cg = 0; cg < ngroups; ++cg) {
                    float v[16];
                    tmem_ld16(tmem + lane_addr + (uint32_t)(b * acc_stride + 16 * cg), v);
                    if (cg == ngroups - 1) {   // the accumulator is in registers: free it
                        tmem_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&S.acc_empty[b]);
                    }
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = 16 * cg + jj;
                        const float other = __shfl_down_sync(0xffffffffu, v[jj], 8);
                        const float gs = swap ? other : v[jj];
                        const float us = swap ? v[jj] : other;
                        // column j: batch token j (small batches) or the chunk's j-th pair
                        const bool keep = small_b ? ((tmask >> j) & 1u) != 0 : j < T.ntok;
                        if (m == 0 && keep) {
                            const size_t pos = small_b ? (size_t)T.off + __popc(tmask & ((1u << j) - 1u))
                                                       : (size_t)T.off + nmax * T.c + j;
                            hb[pos * F + frow] = __float2bfloat16_rn(silu_f(gs) * us);
                        }
                    }
                }
                __syncwarp();
                // All four warps wait for the barrier's phase, so no warp can
                // arrive for the next phase-A tile before this one completes.
                if (lane == 0) mbar_arrive(&S.h_written);
                wait_bar(&S.h_written, na & 1, S, flags);
                if (tid == 0) {   // all four warps have stored: release the chunk's counter
                    __threadfence();
                    atomicAdd(&A.hdone[S.chunk_off[T.a] + T.c], 1u);
                }
                ++na;
            } else {
                const int row = kM * T.rb + i;
                for (int cg = 0; cg < ngroups; ++cg) {
                    float v[16];
                    tmem_ld16(tmem + lane_addr + (uint32_t)(b * acc_stride + 16 * cg), v);
                    if (cg == ngroups - 1) {
                        tmem_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&S.acc_empty[b]);
                    }
                    if (row < d) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = 16 * cg + jj;
                            if (j < T.ntok) A.ybuf[((size_t)T.off + nmax * T.c + j) * d + row] = v[jj];
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.tq_empty[q]);
        }
    }

    // ---- every CTA arrives after its last tile; then the combine ----
    // This thread's first output of the combine: its slots' pair positions
    // and weights (routing results) are loaded before the grid barrier.
    const int d4 = d / 4;
    const long long ctotal = (long long)A.B * d4;
    const long long co0 = ctotal * blockIdx.x / G, co1 = ctotal * (blockIdx.x + 1) / G;
    int pf_pos[8];
    float pf_w[8];
    if (co0 + (long long)threadIdx.x < co1) {
        const int i0 = (int)((co0 + threadIdx.x) / d4);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            pf_pos[u] = u < A.kslots ? A.pos_of[i0 * A.kslots + u] : -1;
            pf_w[u] = pf_pos[u] >= 0 ? A.w[i0 * A.kslots + u] : 0.f;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(&A.hdr->b_done, 1u);
        wait_counter(&A.hdr->b_done, G, S, flags);
        __threadfence();
    }
    __syncthreads();
    {
        const float4* y4 = reinterpret_cast<const float4*>(A.ybuf);
        uint2* out = static_cast<uint2*>(A.out);
        bool first = true;
        for (long long o = co0 + threadIdx.x; o < co1; o += kThreads, first = false) {
            const int i = (int)(o / d4), c4 = (int)(o - (long long)i * d4);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 0; s0 < A.kslots; s0 += 8) {
                float4 yv[8];
                float wv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int sl = s0 + u;
                    int pos;
                    if (first && s0 == 0) {
                        pos = pf_pos[u];
                        wv[u] = pf_w[u];
                    } else {
                        pos = sl < A.kslots ? A.pos_of[i * A.kslots + sl] : -1;
                        wv[u] = pos >= 0 ? A.w[i * A.kslots + sl] : 0.f;
                    }
                    yv[u] = pos >= 0 ? __ldcg(y4 + (size_t)pos * d4 + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {   // slot order
                    acc.x += wv[u] * yv[u].x;
                    acc.y += wv[u] * yv[u].y;
                    acc.z += wv[u] * yv[u].z;
                    acc.w += wv[u] * yv[u].w;
                }
            }
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            out[o] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
        }
    }

    // ---- release the tensor memory; the last CTA resets the counters ----
    tmem_fence_before_sync();
    __syncthreads();
    if (warp == kWarpM) {
        tmem_fence_after_sync();
        tmem_dealloc(tmem, tmem_cols);
    }
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(&A.hdr->ctas_done, 1u);
        S.last_flag = (old + 1 == G);
    }
    __syncthreads();
    if (S.last_flag) {
        __threadfence();
        for (int k = threadIdx.x; k < (int)G; k += kThreads) A.gflag[k] = 0;
        for (int k = threadIdx.x; k < S.chunk_off[Tn]; k += kThreads) A.hdone[k] = 0;
    }
    if (S.last_flag && threadIdx.x == 0) {
        A.hdr->next_tile = 0;
        A.hdr->b_done = 0;
        A.hdr->ctas_done = 0;
    }
}

}  // namespace

cudaError_t launch_ffn_tc(const FfnArgs& a, const CUtensorMap* maps, int num_sms, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(ffn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // One CTA per SM (the shared-memory size allows no second one, so the
    // tensor memory is never contended); programmatic dependent launch lets
    // the CTAs allocate and prefetch while the routing kernel finishes.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ffn_tc_kernel, a, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                              maps[6]);
}

}  // namespace moe
