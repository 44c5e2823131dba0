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
// Structure (one persistent CTA per SM, 16 warps):
//   * Work is a list of tiles.  Phase-A tile (expert a, 64 rows of d_ff,
//     token chunk c): the 64 W_gate rows and the 64 W_up rows of the same
//     d_ff indices, interleaved 8 rows at a time (rows 16g..16g+7 = gate
//     rows 8g..8g+7, rows 16g+8..16g+15 = the up rows), form the 128-row A
//     operand of a tcgen05 MMA with M = 128; the chunk's token rows are the
//     N operand; K = d.  Batches of up to 64 tokens: one chunk per expert
//     whose phase-A operand is the whole batch (N = the batch rounded up to
//     16; the tensor pipe is nearly idle at decode, so multiplying tokens
//     that the expert does not serve costs nothing, and the epilogue keeps
//     the expert's own by a 64-bit token mask).  Larger batches: chunks of
//     up to nmax = the largest expert's token count rounded up to 16, at
//     most 128, rows of an expert-grouped copy of the hidden states (N = the
//     chunk's tokens rounded up to 16), so most experts' weights are
//     streamed once.  Phase-B tile (expert a, 128 rows of d,
//     chunk c): W_down rows times the chunk's h rows, K = d_ff.  The list
//     holds every phase-A tile, then every phase-B tile, each in active-
//     expert order; CTA b starts with tile b and claims each next tile (one
//     ahead) from one grid-wide counter, so all CTAs finish within about
//     one tile of each other.
//   * Warp 4 claims the tiles, posts them to a 16-entry shared-memory queue
//     and streams the weights: one TMA operation per stage of KB blocks of
//     128 rows x 64 columns (128-byte swizzle; the gate/up interleave comes
//     from one 5D tensor map over both matrices, or, where the two cannot
//     share one, from 16 copies of 8-row groups, KB blocks each).  A TMA unit's rate per SM
//     grows with the bytes of each operation, so batches of up to 16 tokens
//     use KB = 4 (64 KB per operation) where d and d_ff allow it, larger
//     batches KB = 2 where both are even.  Warp 5 streams the token rows of
//     each stage: the whole batch of up to 64 tokens straight from the
//     hidden states (one box), or rows of the expert-grouped copy of the
//     hidden states (16-row boxes), or (phase B) rows of h once every phase-A tile
//     of the chunk has written them (a per-chunk counter).  The stage ring takes the shared memory
//     that the barriers and per-expert tables leave (3 stages of 72 KB at
//     KB = 4; 3 to 6 stages at KB = 2, by the chunk width).  For batches of
//     up to 64 tokens warp 4 also loads the first tile's first stages (token
//     rows, then weights) as soon as the activated experts are known: with
//     OEA routing, from the S_base that the routing kernel publishes after
//     phase 1 (the early start: the weights stream while phase 2 and the
//     grouping run; warp 0 adds the counts, first pairs and token masks
//     once the routing kernel has completed), else after it ends.
//   * Warp 6, lane 0, issues the MMAs: four K=16 steps per stage straight
//     from the swizzled shared memory (no register staging), fp32
//     accumulators in tensor memory, four accumulator buffers (the batch
//     rounded up to 16 columns each for batches of up to 64 tokens, else
//     128).
//     tcgen05.commit frees each stage when its MMAs have completed and marks
//     a tile's accumulator full.
//   * INT4 experts (DynaExq page, section 3.2; compiled into the kInt4
//     instantiation only): warp 4 bulk-copies the packed 128-column chunks
//     of a stage's K blocks into a raw ring of up to 16 slots (the stage
//     ring's unused tail holds all but one or two) and arrives on the stage
//     barrier without bytes; warps 7-14 decode each chunk together (exact
//     integer codes, times the row's group scale, rounded once to bf16)
//     into the stage's 128-byte-swizzled A operand, fence it for the tensor
//     core's async proxy, and after the stage's last block each arrives on
//     the stage's cfull barrier, which the MMA thread waits on besides the
//     stage barrier.  Batches of up to 48 tokens: an INT4 stage spans twice
//     the K blocks, its packed chunks land in its own ring slot after the
//     token rows, and the converters write the decoded A operand into one of
//     two tensor-memory buffers, from which the MMAs read it.
//   * Warps 0-3 (tensor-memory lanes 32w..32w+31, one D row per thread)
//     read a finished accumulator with tcgen05.ld and free it; phase A:
//     the lane holding gate row r takes the matching up row from the lane
//     8 above (shuffle), applies SwiGLU and stores h (bf16) for the tile's
//     tokens; phase B: stores y (fp32).  After a phase-A tile the four warps
//     meet at a shared-memory barrier and one thread releases the chunk's
//     counter.  A finished phase-B tile goes to warp 15 through a small
//     queue; it counts each of the tile's tokens down on the token's
//     counter for the tile's 128 rows of d (set to the token's kept slots
//     by the routing kernel), with release semantics, so the epilogue
//     warps never wait for their stores to drain.
//   * After its role every warp takes (token, 128 rows) combine items: it
//     waits until the item's counter is zero, sums the kept weights times
//     the y rows in slot order, writes the output rows and restores the
//     counter for the next launch.
//   * All phase-A tiles precede all phase-B tiles in the list and wait on
//     nothing later, so every wait ends.  Nothing is reset at the end: the
//     routing call that precedes the next launch zeroes the tile and chunk
//     counters of the set that launch uses.
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
constexpr int kWarpN = kWarpC + kConvWarps;   // warp 15: counts finished y slices down
constexpr int kThreads = (kWarpN + 1) * 32;
constexpr int kNQ = 8;                   // phase-B tiles handed to warp 15
static_assert(MOE_MAX_TOKENS <= 256, "a handed-over tile's tokens are kept as bytes");
constexpr int kM = 128;                  // weight rows per tile (MMA M)
constexpr int kNMax = 128;               // most token columns per tile (MMA N)
constexpr int kWBytes = kM * 128;        // one K block: 128 rows x 64 bf16
constexpr int kMaxStages = 12;
constexpr int kRawMax = 16;              // raw slots (one stage's chunks each) at most; the ring's unused tail holds more
constexpr int kQ4A = 64 * 64 + 64 * 2;   // INT4 chunk of W_gate / W_up: 64 rows x 128 columns (a scale group) + scales
constexpr int kQ4B = 128 * 64 + 128 * 2; // INT4 chunk of W_down: 128 rows x 128 columns + scales
constexpr int kRawPair = 2 * kQ4A;       // a W_gate and a W_up chunk (phase A), or a W_down chunk (phase B)
static_assert(kRawPair == kQ4B, "one raw unit fits either phase");
constexpr int kRawReserve = 2 * kRawPair;   // packed INT4 bytes kept after the stage ring
constexpr int kQ = 16;                   // tile queue entries
constexpr int kAcc = 4;                  // accumulator buffers
constexpr uint32_t kTmemCols = kAcc * kNMax;   // fp32 columns (batches over kWholeMax tokens)
constexpr int kWholeMax = 64;            // batches up to this size use the whole batch as the phase-A operand
constexpr uint32_t kTmA = 256;           // first TMEM column of the INT4 A buffers (whole batches)
constexpr uint32_t kTmAStride = 128;     // columns of one A buffer: up to 4 blocks of 64 bf16
constexpr uint32_t kBarGather = 2;       // named barrier of the warps that copy grouped rows
constexpr int kGatherThreads = (kEpiWarps + kConvWarps + 1) * 32;   // warps 0-3 and 7-15
constexpr int kGatherRows = 64;          // grouped rows per pass
static_assert(kTmemCols <= 512, "tensor memory has 512 columns");

struct Smem {
    uint64_t full[kMaxStages];           // both producers (+ transaction bytes)
    uint64_t empty[kMaxStages];          // tcgen05.commit after the stage's MMAs
    uint64_t acc_full[kAcc];             // tcgen05.commit after a tile's last MMA
    uint64_t acc_empty[kAcc];            // the four epilogue warps
    uint64_t tq_full[kQ];                // tile queue entry posted by the weight warp
    uint64_t tq_empty[kQ];               // entry released by the four epilogue warps
    uint64_t tma_empty[2];               // the MMAs have read a TMEM A buffer (INT4 stages of whole batches)
    uint64_t mma_done;                   // every MMA issued has completed
    uint64_t meta_full;                  // early start: counts, first pairs and token masks are in the tables
    uint64_t union_full;                 // early start: warp 4 has put the union's words in uw
    uint32_t uw[32];                     // early start: the routing kernel's union (bit b of word j: expert 32j + b)
    uint64_t epi_bar;                    // the four epilogue warps meet (bounded wait)
    uint64_t nt_full[kNQ];               // the four epilogue warps stored a phase-B tile's y rows
    uint64_t nt_empty[kNQ];              // warp 15 has counted them down
    int4 nt_info[kNQ];                   // first pair, pairs (-1: no more tiles), row block
    uint8_t nt_tok[kNQ][kNMax];          // the tile's tokens (batches of at most 256), looked up by the epilogue
    uint64_t raw_full[kRawMax];          // packed INT4 chunks landed (bulk copies)
    uint64_t raw_empty[kRawMax];         // the converter warps have read them
    uint64_t cfull[kMaxStages];          // each converter warp wrote its rows of a stage's blocks (INT4 stages)
    uint32_t raw_info[kRawMax];          // ring slot | phase A << 8, or ~0u
    int tq[kQ];                          // tile index, or -1 once the list is exhausted
    int fast_ops;                        // stages of the first tile whose token rows warp 4 has loaded
    int gtok[kGatherRows];               // tokens of the grouped rows this CTA copies in one pass
    uint32_t tmem_base;
    int nmax;                            // tokens per chunk for this launch (multiple of 16)
    int tn;                              // activated experts (T)
    int abort_flag;
    long long wait_cycles;               // bound of every wait (FfnArgs::wait_cycles)
};

// Per-expert tables in shared memory, after Smem, sized by N at launch.
struct Tabs {
    uint64_t* tokmask;    // [N] active index -> tokens routed to it (batches of up to kWholeMax)
    int* chunk_off;       // [N + 1] first token chunk of each active expert
    uint32_t* ex_info;    // [N] active index -> id | cnt << 10 | first pair << 19
    int* ex_slot;         // [N] active index -> bf16 expert (>= 0) or -1 - INT4 expert
};

__host__ __device__ constexpr size_t tabs_bytes(int N) {
    return (((size_t)N * 8 + (size_t)(N + 1) * 4 + (size_t)N * 4 + (size_t)N * 4) + 15) & ~size_t(15);
}

// Stage ring bytes left in `total` bytes of dynamic shared memory (whole KB).
__host__ __device__ constexpr size_t ring_bytes_for(size_t total, int N, bool int4) {
    return (total - 1024 - ((sizeof(Smem) + 15) & ~size_t(15)) - tabs_bytes(N) -
            (int4 ? (size_t)kRawReserve : 0)) & ~size_t(1023);
}

struct Tile {
    int a, e, rb, c, off, ntok, nch;
};

// Tile t of a phase with rbn row blocks per (expert, chunk); shared memory only.
__device__ __forceinline__ Tile decode_tile(int t, int rbn, const Tabs& X, int Tn, int nmax) {
    int lo = 0, hi = Tn - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (X.chunk_off[mid] * rbn <= t) lo = mid; else hi = mid - 1;
    }
    Tile T;
    T.a = lo;
    const uint32_t info = X.ex_info[lo];
    T.e = info & 1023u;
    const int cnt = (info >> 10) & 511u;
    T.off = info >> 19;
    T.nch = X.chunk_off[lo + 1] - X.chunk_off[lo];
    const int r = t - X.chunk_off[lo] * rbn;
    T.rb = r / T.nch;
    T.c = r - T.rb * T.nch;
    T.ntok = min(nmax, cnt - nmax * T.c);
    return T;
}

__device__ __forceinline__ bool aborted(Smem& S) { return *(volatile int*)&S.abort_flag != 0; }

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
        if (clock64() - t0 > S.wait_cycles) {
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
        if (clock64() - t0 > S.wait_cycles) {
            give_up(S, flags);
            return;
        }
        __nanosleep(32);
    }
}

// Bounded wait until *p == 0 (acquire, GPU scope), polling with a backoff
// of up to 128 ns so that waiting warps load the memory system little.
__device__ __forceinline__ void wait_zero(const uint32_t* p, Smem& S, uint32_t* flags) {
    if (ld_acquire_gpu(p) == 0u) return;
    const long long t0 = clock64();
    uint32_t ns = 32;
    while (!*(volatile int*)&S.abort_flag) {
        if (ld_acquire_gpu(p) == 0u) return;
        if (clock64() - t0 > S.wait_cycles) {
            give_up(S, flags);
            return;
        }
        __nanosleep(ns);
        if (ns < 128) ns <<= 1;
    }
}

// Early start (whole batches): waits (bounded) until the routing call
// that this launch follows has published its activated experts, then
// returns word `lane` of that union (bit b: expert 32 * lane + b).  Each
// lane polls its own word, which carries the epoch in its high half; the
// whole warp calls this.
__device__ __forceinline__ uint32_t early_union_word(const FfnArgs& A, int lane, Smem& S, uint32_t* flags) {
    const long long t0 = clock64();
    uint64_t v = ld_relaxed_gpu_u64(&A.uwords[lane]);
    while (!__all_sync(0xffffffffu, (uint32_t)(v >> 32) == A.epoch)) {
        if (__any_sync(0xffffffffu, *(volatile int*)&S.abort_flag != 0)) return 0u;
        if (__any_sync(0xffffffffu, clock64() - t0 > S.wait_cycles)) {
            if (lane == 0) give_up(S, flags);
            return 0u;
        }
        __nanosleep(64);
        v = ld_relaxed_gpu_u64(&A.uwords[lane]);
    }
    return (uint32_t)v;
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

// The four epilogue warps meet (bounded wait); every warp calls this the
// same number of times.
__device__ __forceinline__ void epi_meet(Smem& S, uint32_t& nm, uint32_t* flags, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.epi_bar);
    wait_bar(&S.epi_bar, nm & 1, S, flags);
    ++nm;
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

// Phase-A weights of one stage when W_gate and W_up have separate maps
// (8-row boxes, kb blocks wide): for each of the tile's 8 row groups g, the
// g-th 8 rows of W_gate then of W_up, each box landing as kb consecutive
// 1024-byte swizzle atoms (one per K block).  Atom (j, b) of row-group slot
// j = 2g + m (m = 0: W_gate, 1: W_up) and block b sits at (j kb + b) x 1024,
// so block b's 128 A rows are 8-row groups kb x 1024 apart, in the same
// interleaved row order as the 5D map's.
__device__ __forceinline__ void load_gate_up_groups(unsigned char* dst, const CUtensorMap* m_gate,
                                                    const CUtensorMap* m_up, int row0, int blk, int kb,
                                                    uint64_t* bar, uint64_t pol) {
#pragma unroll 1
    for (int g = 0; g < 8; ++g) {
        tma_load_3d(dst + (2 * g) * kb * 1024, m_gate, 0, row0 + 8 * g, blk, bar, pol);
        tma_load_3d(dst + (2 * g + 1) * kb * 1024, m_up, 0, row0 + 8 * g, blk, bar, pol);
    }
}

// One converter warp, q4t stages: decodes block kb of a stage's packed
// chunks at src (qch chunks per matrix) for A row i (a row of this warp's
// lane quarter) and stores its 64 bf16 as 32 columns of tensor memory from
// tb + 32 kb (the K pair (2j, 2j + 1) in column j, the lower K in the low
// half).  Phase A: row i = (2g + m) 8 + r is row 8g + r of W_gate (m = 0)
// or W_up (m = 1).
__device__ __forceinline__ void q4_block_to_tmem(const unsigned char* src, uint32_t tb, int i, int kb, int qch, bool ph_a) {
    const int ci = kb >> 1, half = kb & 1;   // chunk of the block, 64-column half of it
    const int srow = ph_a ? 8 * (i >> 4) + (i & 7) : i;
    const int rows = ph_a ? 64 : kM;
    // phase A: W_gate's chunk ci, or W_up's (after W_gate's qch)
    const unsigned char* ch = ph_a ? src + (((i >> 3) & 1) * qch + ci) * kQ4A : src + ci * kQ4B;
    const __nv_bfloat162 sc = __bfloat162bfloat162(*reinterpret_cast<const __nv_bfloat16*>(ch + rows * 64 + srow * 2));
#pragma unroll 1
    for (int g = 0; g < 2; ++g) {   // 32 columns of the block: 4 code words of 8
        const uint4 c = *reinterpret_cast<const uint4*>(ch + srow * 64 + half * 32 + 16 * g);
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
        uint32_t o[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint4 v = decode_q4_row8(w[u], sc);
            o[4 * u] = v.x;
            o[4 * u + 1] = v.y;
            o[4 * u + 2] = v.z;
            o[4 * u + 3] = v.w;
        }
        tmem_st16(tb + 32 * kb + 16 * g, o);
    }
}

// kInt4: launches with INT4 experts (the packed slots, the converter warps,
// INT4 stages).  Launches with bf16 experts only run the instantiation
// without that code, whose warps keep the registers and the instruction
// footprint that the bf16 stages alone need.
template <bool kInt4>
__global__ void __launch_bounds__(kThreads, 1)
ffn_tc_kernel(const FfnArgs A, const __grid_constant__ CUtensorMap tm_gu, const __grid_constant__ CUtensorMap tm_gate,
              const __grid_constant__ CUtensorMap tm_up, const __grid_constant__ CUtensorMap tm_down,
              const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_h,
              const __grid_constant__ CUtensorMap tm_hid, const __grid_constant__ CUtensorMap tm_gu4,
              const __grid_constant__ CUtensorMap tm_down4, const __grid_constant__ CUtensorMap tm_hid4,
              const __grid_constant__ CUtensorMap tm_h4, const __grid_constant__ CUtensorMap tm_gu2,
              const __grid_constant__ CUtensorMap tm_down2, const __grid_constant__ CUtensorMap tm_up4,
              const __grid_constant__ CUtensorMap tm_up2) {
    extern __shared__ unsigned char smem_raw[];
    // [stage ring][kRawReserve bytes of packed INT4 slots, with INT4 experts][Smem][tables]
    const bool has_q4 = kInt4 && A.n_cold > 0;
    const int ring_bytes = (int)ring_bytes_for((size_t)A.smem_bytes, A.N, has_q4);
    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* raw = ring + ring_bytes;
    Smem& S = *reinterpret_cast<Smem*>(raw + (has_q4 ? kRawReserve : 0));
    Tabs X;
    X.tokmask = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(&S) + ((sizeof(Smem) + 15) & ~size_t(15)));
    X.chunk_off = reinterpret_cast<int*>(X.tokmask + A.N);
    X.ex_info = reinterpret_cast<uint32_t*>(X.chunk_off + A.N + 1);
    X.ex_slot = reinterpret_cast<int*>(X.ex_info + A.N);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = A.d, F = A.F;
    uint32_t* flags = &A.hdr->flags;
    const uint32_t G = gridDim.x;
    // K blocks (64 columns) per stage, moved by one TMA operation for the
    // weights, since the TMA unit's rate per SM grows with the size of each
    // operation: A.kbs (up to 4) for batches of up to 16 tokens, A.kbl (up to
    // 2) for larger batches, whose token rows share the ring.
    const bool small_b = A.B <= 16;
    // Stages of A.kbs blocks (4 where d and d_ff allow them) for bf16 batches
    // of up to 16 tokens.  Launches with INT4 experts keep the packed slots'
    // reserve, which leaves room for only two such stages: they use A.kbl.
    const bool kbs_stages = small_b && !has_q4;
    // Batches of up to kWholeMax tokens: the phase-A operand is the whole
    // batch (nwb rows, the batch rounded up to 16; the tensor pipe is nearly
    // idle at decode, so multiplying every token costs nothing), each expert
    // is one token chunk, and h is stored for the expert's own tokens only.
    const bool whole = A.B <= kWholeMax;
    const int nwb = max(16, (A.B + 15) & ~15);
    const int KB = kbs_stages ? A.kbs : A.kbl;
    // weight maps, KB blocks wide: the 5D gate/up map (or, when W_gate and
    // W_up cannot share one, W_gate's and W_up's 8-row maps) and W_down's
    const CUtensorMap* const m_gu = KB == 1 ? &tm_gu : kbs_stages ? &tm_gu4 : &tm_gu2;
    const CUtensorMap* const m_up = KB == 1 ? &tm_up : kbs_stages ? &tm_up4 : &tm_up2;
    const CUtensorMap* const m_down = KB == 1 ? &tm_down : kbs_stages ? &tm_down4 : &tm_down2;
    // Batches of up to 48 tokens with INT4 experts: an INT4 stage spans
    // KBq = 2 KB blocks and its ring slot holds the token rows of those
    // blocks, then their packed chunks (2 KB x 128 x nwb + KB x 16.5 KB
    // bytes, within the slot's KB x (16 KB + 128 x nwb) while nwb <= 48).
    // The converter warps write the decoded A operand into one of two
    // tensor-memory buffers (columns kTmA and kTmA + kTmAStride) that the
    // MMAs read.  A ring slot's cycle is set by the token rows' TMA load,
    // which queues behind the HBM stream, so twice the K per slot doubles the
    // INT4 stages' rate, and the bf16 stages keep the whole ring.
    const bool q4t = has_q4 && whole && KB <= 2 && nwb * 128 + kRawPair <= kWBytes &&
                     (d / 64) % (2 * KB) == 0 && (F / 64) % (2 * KB) == 0;
    const int KBq = q4t ? 2 * KB : KB;   // blocks of an INT4 stage

    // The tensor maps' descriptors, fetched while the barriers are set up:
    // the first copies (which the early start issues the moment the
    // activated experts are known) then find them cached.
    if (warp == kWarpW && lane == 0) {
        prefetch_tensormap(m_gu);
        if (!A.gu_fused) prefetch_tensormap(m_up);
        prefetch_tensormap(m_down);
    }
    if (warp == kWarpO && lane == 0) {
        if (whole) {
            prefetch_tensormap(KB > 1 ? &tm_hid4 : &tm_hid);
            prefetch_tensormap(kbs_stages && KB > 1 ? &tm_h4 : &tm_h);
        } else {
            prefetch_tensormap(&tm_x);
            prefetch_tensormap(&tm_h);
        }
    }
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
        for (int i = 0; i < 2; ++i) mbar_init(&S.tma_empty[i], 1);
        mbar_init(&S.meta_full, 1);
        mbar_init(&S.union_full, 1);
        mbar_init(&S.epi_bar, kEpiWarps);
        for (int i = 0; i < kNQ; ++i) {
            mbar_init(&S.nt_full[i], kEpiWarps);
            mbar_init(&S.nt_empty[i], 1);
            S.nt_info[i] = make_int4(0, 0, 0, 0);
        }
        for (int i = 0; i < kRawMax; ++i) {
            mbar_init(&S.raw_full[i], 1);
            mbar_init(&S.raw_empty[i], kConvWarps);
        }
        for (int i = 0; i < kMaxStages; ++i) mbar_init(&S.cfull[i], kConvWarps);
        fence_barrier_init();
        S.abort_flag = 0;
        S.fast_ops = 0;
        S.wait_cycles = A.wait_cycles;
        for (int i = 0; i < 32; ++i) S.uw[i] = 0u;   // read as "no expert" if a wait gives up first
    }
    // accumulator buffers: kAcc x nwb columns for whole batches, else kAcc x kNMax
    const int acc_stride = whole ? nwb : kNMax;
    const uint32_t tmem_cols = q4t ? 512u : whole ? (kAcc * nwb <= 64 ? 64u : kAcc * nwb <= 128 ? 128u : 256u)
                                                  : kTmemCols;
    if (warp == kWarpM) tmem_alloc(&S.tmem_base, tmem_cols);
    __syncthreads();             // barriers initialised (this overlaps the routing kernel)
    // Early start (OEA routing of whole batches, whose routing
    // call publishes S_base after phase 1): the activated experts are fixed
    // before the routing kernel ends, and they are all that phase A needs (its operand
    // is the whole batch; the token masks and first pairs are read only by
    // the epilogue and phase B).  The tables start from the union, in
    // ascending expert id like the routing kernel's active list, and the
    // weights stream while the routing finishes; warp 0 then adds the counts,
    // first pairs and token masks once the routing kernel has completed.
    // Every warp that reads the routing's other outputs waits for its
    // completion first.
    const bool early = whole && A.epoch != 0u;
    int Tn = 0;
    if (!early) {
        grid_dependency_wait();      // routing comes from the preceding kernel
        Tn = *A.T;
        if (Tn < 0 || Tn > A.N) {
            if (threadIdx.x == 0 && blockIdx.x == 0) raise_flag(flags, kFlagBadIndex);
            Tn = 0;
        }
    }
    // Whole batches: the CTA's first tile is phase-A tile blockIdx.x of a
    // one-chunk-per-expert list, so the weight warp starts its stages now
    // (each stage's token rows first, then its weights), while warp 0 builds
    // the per-expert records.
    int fast_stages = 0;
    if (warp == kWarpW && whole) {
        const int rbA0 = F / 64, t0 = (int)blockIdx.x;
        int e = -1;   // expert of phase-A tile t0 (active index t0 / rbA0), if there is one
        if (early) {
            // experts N and above do not exist: their bits are dropped
            const int nb = A.N - 32 * lane;
            const uint32_t word = early_union_word(A, lane, S, flags) &
                                  (nb >= 32 ? 0xffffffffu : nb > 0 ? (1u << nb) - 1u : 0u);
            S.uw[lane] = word;   // for warp 0's tables
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.union_full);
            const int c = __popc(word);
            int inc = c;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += u;
            }
            const int a0 = t0 / rbA0;
            const bool mine = a0 >= inc - c && a0 < inc;   // active index a0 is a bit of this lane's word
            int eo = -1;
            if (mine) {
                uint32_t w = word;
                for (int k = inc - c; k < a0; ++k) w &= w - 1u;   // drop the lower set bits
                eo = 32 * lane + __ffs(w) - 1;
            }
            const uint32_t who = __ballot_sync(0xffffffffu, mine);
            e = who ? __shfl_sync(0xffffffffu, eo, __ffs(who) - 1) : -1;
        } else if (t0 < Tn * rbA0) {
            e = (int)(A.exinfo[t0 / rbA0] & 1023u);
        }
        if (lane == 0 && e >= 0) {
            const int sl = A.slot ? A.slot[e] : e;
            if (sl >= 0 && sl < A.n_hot) {
                const uint64_t pol = l2_evict_first_policy();
                const int row0 = sl * F + 64 * (t0 % rbA0);
                const int sb = KB * (kWBytes + nwb * 128);   // the slot size of this launch (nmax = nwb)
                fast_stages = min(d / 64 / KB, min(kMaxStages, ring_bytes / sb));
                const uint64_t pol_x = l2_evict_last_policy();
                for (int s = 0; s < fast_stages; ++s) {
                    unsigned char* dst = ring + (size_t)s * sb;
                    mbar_arrive_expect_tx(&S.full[s], KB * nwb * 128);   // rows past B read as zeros
                    tma_load_3d(dst + KB * kWBytes, KB > 1 ? &tm_hid4 : &tm_hid, 0, 0, s * KB, &S.full[s], pol_x);
                    mbar_arrive_expect_tx(&S.full[s], KB * kWBytes);
                    if (A.gu_fused) {
                        tma_load_5d(dst, m_gu, 0, 0, 0, row0 / 8, s * KB, &S.full[s], pol);
                    } else {
                        load_gate_up_groups(dst, m_gu, m_up, row0, s * KB, KB, &S.full[s], pol);
                    }
                }
                S.fast_ops = fast_stages;   // read by the operand warp after the barrier below
            }
        }
    }
    if (warp == 0 && early) {   // the tables from the union: one chunk per expert
        wait_bar(&S.union_full, 0, S, flags);
        const int nbits = A.N - 32 * lane;   // at most N experts, so the tables stay in bounds
        const uint32_t word = *(volatile uint32_t*)&S.uw[lane] &
                              (nbits >= 32 ? 0xffffffffu : nbits > 0 ? (1u << nbits) - 1u : 0u);
        const int c = __popc(word);
        int inc = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += u;
        }
        const int tot = __shfl_sync(0xffffffffu, inc, 31);
        uint32_t w = word;
        for (int a = inc - c; w; ++a, w &= w - 1u) {
            const int e = 32 * lane + __ffs(w) - 1;
            int sl = A.slot ? A.slot[e] : e;
            if (sl >= A.n_hot || -1 - sl >= A.n_cold) {   // out of range: flag it, read expert 0
                raise_flag(flags, kFlagBadIndex);
                sl = A.n_hot > 0 ? 0 : -1;
            }
            X.ex_info[a] = (uint32_t)e;   // the count and first pair follow with the routing's completion
            X.tokmask[a] = 0ull;
            X.ex_slot[a] = sl;
            X.chunk_off[a] = a;
        }
        if (lane == 0) {
            X.chunk_off[tot] = tot;
            S.nmax = nwb;
            S.tn = tot;
        }
    } else if (warp == 0) {   // per-expert records, chunk width and chunk offsets of the active experts
        if (lane == 0) S.tn = Tn;
        int maxcnt = 0;
        for (int a = lane; a < Tn; a += 32) {
            const uint32_t info = A.exinfo[a];   // written by the routing kernel
            X.ex_info[a] = info;
            X.tokmask[a] = (uint64_t)A.exinfo[A.N + a] | ((uint64_t)A.exinfo[2 * A.N + a] << 32);
            maxcnt = max(maxcnt, (int)((info >> 10) & 511u));
            const int e = info & 1023u;
            int sl = A.slot ? A.slot[e] : e;
            if (sl >= A.n_hot || -1 - sl >= A.n_cold) {   // out of range: flag it, read expert 0
                raise_flag(flags, kFlagBadIndex);
                sl = A.n_hot > 0 ? 0 : -1;
            }
            X.ex_slot[a] = sl;
        }
        maxcnt = __reduce_max_sync(0xffffffffu, maxcnt);
        // a chunk holds up to nmax tokens: the whole batch for whole batches,
        // else the largest expert's tokens rounded up to 16, at most 128
        const int nmax = whole ? nwb : min(kNMax, max(16, (maxcnt + 15) & ~15));
        if (lane == 0) S.nmax = nmax;
        __syncwarp();
        int run = 0;
        if (lane == 0) X.chunk_off[0] = 0;
        for (int a0 = 0; a0 < Tn; a0 += 32) {
            const int a = a0 + lane;
            int nch = 0;
            if (a < Tn) nch = ((int)((X.ex_info[a] >> 10) & 511u) + nmax - 1) / nmax;
            int inc = nch;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, inc, off);
                if (lane >= off) inc += u;
            }
            if (a < Tn) X.chunk_off[a + 1] = run + inc;
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tmem = S.tmem_base;
    Tn = S.tn;
    if (early && warp == 0) {
        // The routing kernel has completed: the counts, first pairs and token
        // masks join the union's tables (the same experts, in the same order).
        grid_dependency_wait();
        if (lane == 0 && *A.T != Tn) raise_flag(flags, kFlagBadIndex);
        for (int a = lane; a < Tn; a += 32) {
            const uint32_t info = A.exinfo[a];
            if ((info & 1023u) != X.ex_info[a]) raise_flag(flags, kFlagBadIndex);
            X.ex_info[a] = info;
            X.tokmask[a] = (uint64_t)A.exinfo[A.N + a] | ((uint64_t)A.exinfo[2 * A.N + a] << 32);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.meta_full);
    }

    // Batches over kWholeMax tokens: the expert-grouped copy of the hidden states.
    // Warps 0-3 and 7-15 copy this CTA's rows b, b+G, ... (their tokens
    // first, so that every 16-byte load depends on shared memory only), then
    // one thread counts the CTA in; the operand warp starts phase A once all
    // CTAs have.
    if (!whole && (warp < kEpiWarps || warp >= kWarpC)) {
        const int gt = warp < kEpiWarps ? (int)threadIdx.x : (int)threadIdx.x - (kWarpC - kEpiWarps) * 32;
        const int P = A.offsets[A.N];
        const int vpr = d / 8;   // 16-byte vectors per row
        const int nrow = P > (int)blockIdx.x ? (P - 1 - (int)blockIdx.x) / (int)G + 1 : 0;
        const uint4* xs = static_cast<const uint4*>(A.x);
        uint4* xp = static_cast<uint4*>(A.xperm);
        for (int r0 = 0; r0 < nrow; r0 += kGatherRows) {
            const int nr = min(kGatherRows, nrow - r0);
            if (gt < nr) S.gtok[gt] = A.perm[(int)blockIdx.x + (r0 + gt) * (int)G] / A.kslots;
            named_barrier(kBarGather, kGatherThreads);
            const int nvec = nr * vpr;
            for (int v0 = 0; v0 < nvec; v0 += 4 * kGatherThreads) {
                uint4 val[4];
                size_t dst[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int v = v0 + u * kGatherThreads + gt;
                    dst[u] = ~size_t(0);
                    if (v < nvec) {
                        const int r = v / vpr, c = v - r * vpr;
                        val[u] = __ldg(xs + (size_t)S.gtok[r] * vpr + c);
                        dst[u] = (size_t)((int)blockIdx.x + (r0 + r) * (int)G) * vpr + c;
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (dst[u] != ~size_t(0)) xp[dst[u]] = val[u];
            }
            named_barrier(kBarGather, kGatherThreads);   // every row stored; gtok is free again
        }
        if (gt == 0) {
            __threadfence();
            atomicAdd(A.gathered, 1u);
        }
    }

    // Tiles: phase A (expert, 64 rows of d_ff, chunk) first, then phase B
    // (expert, 128 rows of d, chunk), both in active-expert order.
    const int rbA = F / 64, rbB = (d + kM - 1) / kM;
    const int SA = d / 64 / KB, SB = F / 64 / KB;   // stages per tile (KB blocks of 64 columns)
    const int TA = X.chunk_off[Tn] * rbA;
    const int Ttot = TA + X.chunk_off[Tn] * rbB;
    const int nmax = S.nmax;
    // a slot: KB weight blocks of 16 KB, then KB operand blocks of nmax rows
    const int slot_bytes = KB * (kWBytes + nmax * 128);
    const int obytes = nmax * 128;                  // one operand block
    const int nst = min(kMaxStages, ring_bytes / slot_bytes);
    // Packed INT4 chunk slots: kRawReserve bytes after the ring, more in the
    // ring's tail that the whole stages leave unused (deeper raw rings keep
    // more bytes in flight for the converter warps without costing a stage).
    // A packed chunk spans 128 columns (two K blocks); a raw slot holds the
    // chunks of one stage's KB blocks (W_gate's, then W_up's, in phase A),
    // each matrix's moved by one bulk copy.  With KB = 1 a stage reads half
    // of its chunk.
    // With q4t the packed chunks sit in the stage's ring slot (after its
    // KBq operand blocks) and a raw slot is only the converters' queue entry.
    const int qch = KBq > 1 ? KBq / 2 : 1;         // packed chunks per matrix and stage
    const int rslot = qch * kRawPair;
    const int nraw_a = kRawReserve / rslot;        // slots after the ring
    const int nraw = q4t ? kRawMax : nraw_a + min(kRawMax - nraw_a, (ring_bytes - nst * slot_bytes) / rslot);
    auto raw_slot = [&](int r) -> unsigned char* {
        return r < nraw_a ? raw + (size_t)r * rslot : ring + (size_t)nst * slot_bytes + (size_t)(r - nraw_a) * rslot;
    };
    // q4t: the packed chunks of the INT4 stage in ring slot `slot`
    auto packed_in_slot = [&](int slot) -> unsigned char* {
        return ring + (size_t)slot * slot_bytes + (size_t)KBq * obytes;
    };

    if (warp == kWarpW) {
        // ---------------------------- weight producer ----------------------------
        if (lane == 0) {
            const uint64_t pol_once = l2_evict_first_policy();
            const uint64_t pol_keep = l2_evict_normal_policy();
            RingPos rp, rq;   // stage ring, packed INT4 ring
            const size_t q4_mat_a = (size_t)(F / 64) * (d / 128) * kQ4A;   // bytes of one INT4 W_gate / W_up
            const size_t q4_mat_b = (size_t)(d / kM) * (F / 128) * kQ4B;   // bytes of one INT4 W_down
            // CTA b starts with tile b; the next tile is claimed when this
            // one is posted, so the atomic's latency hides behind its stages
            int next0 = (int)blockIdx.x;
            for (int s = 0; s < fast_stages; ++s) rp.next(nst);   // stages issued before the prologue
            for (int n = 0;; ++n) {
                const int q = n % kQ;
                if (n >= kQ) wait_bar(&S.tq_empty[q], ((n / kQ) - 1) & 1, S, flags);
                const int tile = next0 < Ttot && !aborted(S) ? next0 : -1;   // no new copies once a wait gave up
                S.tq[q] = tile;
                mbar_arrive(&S.tq_full[q]);
                if (tile < 0) break;
                next0 = (int)G + (int)atomicAdd(A.next_tile, 1u);
                const bool ph_a = tile < TA;
                const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, X, Tn, nmax);
                const uint64_t pol = T.nch > 1 ? pol_keep : pol_once;   // chunked experts are re-read from L2
                const int sl = X.ex_slot[T.a];                          // bf16 expert, or -1 - INT4 expert
                const int row0 = ph_a ? sl * F + 64 * T.rb : sl * d + kM * T.rb;
                const int ns = (ph_a ? SA : SB) >> (q4t && sl < 0 ? 1 : 0);   // INT4 stages of KBq blocks
                for (int s = n == 0 ? fast_stages : 0; s < ns; ++s, rp.next(nst)) {
                    const int slot = rp.slot;
                    if (rp.wrapped) wait_bar(&S.empty[slot], rp.phase ^ 1u, S, flags);
                    if (aborted(S)) break;
                    unsigned char* dst = ring + (size_t)slot * slot_bytes;
                    if (has_q4 && sl < 0) {
                        // INT4 expert: the packed chunks of the stage's KB blocks are
                        // contiguous per matrix and go to one raw slot; the converter
                        // warps write the bf16 blocks and each arrives on the stage's
                        // cfull barrier.  This warp's arrival on full carries no bytes.
                        const int c = -1 - sl;
                        mbar_arrive(&S.full[slot]);
                        const int r = rq.slot;
                        if (rq.wrapped) wait_bar(&S.raw_empty[r], rq.phase ^ 1u, S, flags);
                        // slot, phase A, and (KB = 1) which half of the chunk the stage reads
                        S.raw_info[r] = (uint32_t)slot | (ph_a ? 256u : 0u) | ((uint32_t)((s * KB) & 1) << 9);
                        unsigned char* rdst = q4t ? packed_in_slot(slot) : raw_slot(r);
                        const int cg = s * KBq / 2;   // the stage's first 128-column group
                        if (ph_a) {
                            const size_t off = (size_t)c * q4_mat_a + ((size_t)T.rb * (d / 128) + cg) * kQ4A;
                            mbar_arrive_expect_tx(&S.raw_full[r], 2 * qch * kQ4A);
                            bulk_load(rdst, A.q_gate + off, qch * kQ4A, &S.raw_full[r], pol);
                            bulk_load(rdst + qch * kQ4A, A.q_up + off, qch * kQ4A, &S.raw_full[r], pol);
                        } else {
                            const size_t off = (size_t)c * q4_mat_b + ((size_t)T.rb * (F / 128) + cg) * kQ4B;
                            mbar_arrive_expect_tx(&S.raw_full[r], qch * kQ4B);
                            bulk_load(rdst, A.q_down + off, qch * kQ4B, &S.raw_full[r], pol);
                        }
                        rq.next(nraw);
                        continue;
                    }
                    mbar_arrive_expect_tx(&S.full[slot], KB * kWBytes);
                    if (!ph_a) {
                        // 128 W_down rows (rows past the expert's d are computed and dropped)
                        tma_load_3d(dst, m_down, 0, row0, s * KB, &S.full[slot], pol);
                    } else if (A.gu_fused) {
                        // 8 row groups x {8 rows of the lower matrix, 8 rows of the other}
                        tma_load_5d(dst, m_gu, 0, 0, 0, row0 / 8, s * KB, &S.full[slot], pol);
                    } else {
                        load_gate_up_groups(dst, m_gu, m_up, row0, s * KB, KB, &S.full[slot], pol);
                    }
                }
            }
            if (has_q4) {   // no more INT4 chunks: the converter warps stop
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
        const int fast_ops = S.fast_ops;   // stages of the first tile already loaded by warp 4
        for (int s = 0; s < fast_ops; ++s) rp.next(nst);
        bool gathered = whole;
        bool meta = !early;   // the tables hold the counts and first pairs
        for (int n = 0;; ++n) {
            const int q = n % kQ;
            wait_bar(&S.tq_full[q], (n / kQ) & 1, S, flags);
            if (aborted(S)) break;
            const int tile = S.tq[q];
            if (tile < 0) break;
            const bool ph_a = tile < TA;
            if (!ph_a && !meta) {   // phase B reads the chunk's first pair and tokens
                wait_bar(&S.meta_full, 0, S, flags);
                meta = true;
            }
            const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, X, Tn, nmax);
            if (ph_a && !gathered) {   // every CTA has copied its rows of the grouped hidden states
                if (lane == 0) {
                    wait_counter(A.gathered, G, S, flags);
                    fence_proxy_async_global();
                }
                __syncwarp();
                gathered = true;
            }
            if (lane == 0) {
                if (!ph_a) {   // every phase-A tile of this token chunk has written its h rows
                    wait_counter(&A.hdone[X.chunk_off[T.a] + T.c], (uint32_t)rbA, S, flags);
                    fence_proxy_async_global();
                }
                // Phase A of whole batches: one box of nwb rows and KB blocks,
                // which lands as KB consecutive [nwb rows][64] operand blocks.
                // Phase B of batches of up to 16 tokens: one 16-row box of KB
                // blocks.  Otherwise: one 16-row box per 16 tokens and block,
                // block kb at kb x nmax rows.
                const bool wide = ph_a && whole;
                const CUtensorMap* map = ph_a ? (whole ? (KB > 1 ? &tm_hid4 : &tm_hid) : &tm_x)
                                              : (kbs_stages && KB > 1 ? &tm_h4 : &tm_h);
                const int row = wide ? 0 : T.off + nmax * T.c;
                const int nb = wide ? nwb >> 4 : (T.ntok + 15) >> 4;   // 16-row boxes = MMA N / 16
                // an INT4 stage of a q4t launch: KBq operand blocks at the slot's start
                const bool pk = q4t && X.ex_slot[T.a] < 0;
                const int ns = (ph_a ? SA : SB) >> (pk ? 1 : 0);
                for (int s = n == 0 ? fast_ops : 0; s < ns; ++s, rp.next(nst)) {
                    const int slot = rp.slot;
                    if (rp.wrapped) wait_bar(&S.empty[slot], rp.phase ^ 1u, S, flags);
                    if (aborted(S)) break;
                    unsigned char* dst = ring + (size_t)slot * slot_bytes + (pk ? 0 : KB * kWBytes);
                    if (pk) {
                        mbar_arrive_expect_tx(&S.full[slot], nb * 2048 * KBq);
                        if (wide) {   // KBq / KB boxes of KB blocks
                            for (int h = 0; h < KBq; h += KB)
                                tma_load_3d(dst + h * obytes, map, 0, 0, s * KBq + h, &S.full[slot], pol);
                        } else {
                            for (int kb = 0; kb < KBq; ++kb)
                                for (int j = 0; j < nb; ++j)
                                    tma_load_3d(dst + kb * obytes + j * 2048, map, 0, row + 16 * j, s * KBq + kb,
                                                &S.full[slot], pol);
                        }
                        continue;
                    }
                    mbar_arrive_expect_tx(&S.full[slot], nb * 2048 * KB);   // rows past the end read as zeros
                    if (wide) {
                        tma_load_3d(dst, map, 0, 0, s * KB, &S.full[slot], pol);
                    } else if (kbs_stages) {
                        for (int j = 0; j < nb; ++j)
                            tma_load_3d(dst + j * 2048, map, 0, row + 16 * j, s * KB, &S.full[slot], pol);
                    } else {
                        for (int kb = 0; kb < KB; ++kb)
                            for (int j = 0; j < nb; ++j)
                                tma_load_3d(dst + kb * obytes + j * 2048, map, 0, row + 16 * j, s * KB + kb,
                                            &S.full[slot], pol);
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == kWarpM) {
        // ------------------------------ MMA issuer -------------------------------
        if (lane == 0) {
            RingPos rp;
            uint32_t cpar = 0;   // per ring slot: parity of its next cfull phase (INT4 stages)
            uint32_t q4n = 0;    // INT4 stages of a q4t launch so far (TMEM A buffer q4n & 1)
            bool meta = !early;  // the tables hold the counts
            for (int n = 0;; ++n) {
                const int q = n % kQ;
                wait_bar(&S.tq_full[q], (n / kQ) & 1, S, flags);
                if (aborted(S)) break;
                const int tile = S.tq[q];
                if (tile < 0) break;
                const bool ph_a = tile < TA;
                // MMA N: every token (phase A of whole batches; phase B of
                // batches of up to 16, whose chunks hold at most 16), else the
                // chunk's tokens rounded up to 16, read once the routing has
                // completed (before that an early table holds no counts)
                const bool by_count = !small_b && !(whole && ph_a);
                if (by_count && !meta) {
                    wait_bar(&S.meta_full, 0, S, flags);
                    if (aborted(S)) break;
                    meta = true;
                }
                int ntile = nwb;
                bool q4 = false;  // INT4 expert: the converter warps write the A operand
                if (by_count || has_q4) {
                    const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, X, Tn, nmax);
                    if (by_count) ntile = max(16, (T.ntok + 15) & ~15);
                    q4 = has_q4 && X.ex_slot[T.a] < 0;
                }
                const uint32_t idesc = umma_idesc_bf16(kM, ntile);
                const bool pk = q4 && q4t;   // A from tensor memory, KBq blocks per stage
                const int ns = (ph_a ? SA : SB) >> (pk ? 1 : 0);
                const int b = n % kAcc;
                if (n >= kAcc) {   // the epilogue has read this accumulator's previous tile
                    wait_bar(&S.acc_empty[b], ((n / kAcc) - 1) & 1, S, flags);
                    tmem_fence_after_sync();
                }
                const uint32_t dt = tmem + (uint32_t)(b * acc_stride);
                for (int s = 0; s < ns; ++s, rp.next(nst)) {
                    const int slot = rp.slot;
                    wait_bar(&S.full[slot], rp.phase, S, flags);
                    if (q4) {
                        wait_bar(&S.cfull[slot], (cpar >> slot) & 1u, S, flags);
                        cpar ^= 1u << slot;
                    }
                    if (aborted(S)) break;   // the stage may not have landed: issue nothing more
                    tmem_fence_after_sync();
                    const uint32_t a0 = smem_u32(ring + (size_t)slot * slot_bytes);
                    if (pk) {
                        const uint32_t ta = tmem + kTmA + (q4n & 1u) * kTmAStride;
#pragma unroll 1
                        for (int kb = 0; kb < KBq; ++kb) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)   // 8 columns of A, 32 bytes of the swizzled B row
                                umma_bf16_tmem_a(dt, ta + 32 * kb + 8 * k, umma_sdesc_sw128(a0 + kb * obytes + 32 * k),
                                                 idesc, (s | kb | k) ? 1u : 0u);
                        }
                        umma_commit(&S.empty[slot]);
                        umma_commit(&S.tma_empty[q4n & 1u]);   // the converters may refill this A buffer
                        ++q4n;
                        continue;
                    }
                    const uint32_t b0 = a0 + KB * kWBytes;
                    // bf16 phase-A stages of separate W_gate / W_up maps hold
                    // their K blocks' swizzle atoms interleaved (see
                    // load_gate_up_groups): block kb at kb x 1024, 8-row
                    // groups KB x 1024 apart
                    const bool grouped = ph_a && !q4 && !A.gu_fused;
                    const uint32_t a_blk = grouped ? 1024u : (uint32_t)kWBytes;
                    const uint32_t a_sbo = grouped ? 1024u * KB : 1024u;
#pragma unroll 1
                    for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)   // K = 16 per step: 32 bytes along the swizzled row
                            umma_bf16(dt, umma_sdesc_sw128_sbo(a0 + kb * a_blk + 32 * k, a_sbo),
                                      umma_sdesc_sw128(b0 + kb * obytes + 32 * k), idesc, (s | kb | k) ? 1u : 0u);
                    }
                    umma_commit(&S.empty[slot]);   // the stage is free once these MMAs are done
                }
                umma_commit(&S.acc_full[b]);
            }
            umma_commit(&S.mma_done);
            // Every MMA issued has completed before the tensor memory is
            // freed, also after a wait gave up (bounded, not cut short).
            for (const long long t0 = clock64(); !mbar_try_wait(&S.mma_done, 0) && clock64() - t0 < S.wait_cycles;) {
            }
        }
        __syncwarp();
    } else if (warp == kWarpN) {
        // ----------------------------- count-down warp ----------------------------
        // Each finished phase-B tile's tokens (at most kNMax, four per lane,
        // looked up by the epilogue warps while the tile's MMAs ran) count
        // down their counters for the tile's 128 rows of d: one fence (after
        // the acquire of the epilogue warps' barrier) makes their y stores
        // visible before the plain atomic subtractions -- a release.
        if (early) grid_dependency_wait();   // the pairs and counters come from the routing kernel
        for (uint32_t p = 0;; ++p) {
            const int slot = (int)(p % kNQ);
            wait_bar(&S.nt_full[slot], (p / kNQ) & 1, S, flags);
            if (*(volatile int*)&S.abort_flag) break;
            const int4 inf = S.nt_info[slot];
            if (inf.y < 0) break;
            int tk[kNMax / 32];
#pragma unroll
            for (int u = 0; u < kNMax / 32; ++u) {
                const int j = lane + 32 * u;
                tk[u] = j < inf.y ? (int)S.nt_tok[slot][j] : -1;   // written by the epilogue warps
            }
            __threadfence();
#pragma unroll
            for (int u = 0; u < kNMax / 32; ++u)
                if (tk[u] >= 0) atomicAdd(&A.ycnt[(size_t)tk[u] * rbB + inf.z], 0xffffffffu);
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.nt_empty[slot]);
        }
    } else if (warp >= kWarpC) {
        // ----------------------------- INT4 converters ----------------------------
        // Each packed stage becomes the 128 x 64 bf16 A operand of one ring
        // stage, 128-byte swizzled like a TMA box: output row i, 16-byte unit u
        // (8 columns) at i*128 + ((u ^ (i & 7)) << 4).  Phase A: row i =
        // (2g + m)*8 + r is row 8g + r of W_gate (m = 0) or W_up (m = 1).
        // A stage's KB chunks sit in one raw slot: the warps decode them in
        // one pass (KB x 4 units per lane), then fence once and arrive on the
        // slot and on the stage.
        const int ct = threadIdx.x - kWarpC * 32;   // 0..kConvWarps*32-1
        RingPos rq;
        uint32_t cq = 0;   // INT4 stages decoded so far (q4t launches)
        for (;;) {
            if (!has_q4) break;                        // no INT4 experts in this launch
            const int r = rq.slot;
            wait_bar(&S.raw_full[r], rq.phase, S, flags);
            if (*(volatile int*)&S.abort_flag) break;
            const uint32_t info = S.raw_info[r];
            if (info == ~0u) break;                    // no more chunks
            const int slot = (int)(info & 255u);
            if (slot >= nst) {   // never posted so: flag it and write nothing
                if (lane == 0) {
                    raise_flag(flags, kFlagBadIndex);
                    give_up(S, flags);
                }
                break;
            }
            const bool ph_a = (info >> 8) & 1u;
            const int half1 = (info >> 9) & 1u;          // KB = 1: the stage's half of its chunk
            const int rows = ph_a ? 64 : kM;
            if (q4t) {
                // The stage's KBq blocks go to tensor-memory A buffer cq & 1:
                // row i (this warp's lane quarter) in lane i, block kb at
                // column 32 kb, the K pair (2j, 2j + 1) of a block in its
                // column j.  Warps 7-10 and 11-14 each cover the four lane
                // quarters, for the first and the second half of the blocks.
                const unsigned char* src = packed_in_slot(slot);
                const int qd = warp & 3;                  // lane quarter this warp may access
                const int i = 32 * qd + lane;             // A row
                const int grp = (warp - kWarpC) >> 2;
                if (cq >= 2) {   // the MMAs have read what this buffer held two stages ago
                    wait_bar(&S.tma_empty[cq & 1u], ((cq >> 1) - 1) & 1u, S, flags);
                    if (*(volatile int*)&S.abort_flag) break;
                    tmem_fence_after_sync();
                }
                const uint32_t tb = tmem + ((uint32_t)(32 * qd) << 16) + kTmA + (cq & 1u) * kTmAStride;
#pragma unroll 1
                for (int h = 0; h < KBq / 2; ++h)
                    q4_block_to_tmem(src, tb, i, grp * (KBq / 2) + h, qch, ph_a);
                tmem_wait_st();
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&S.raw_empty[r]);
                    mbar_arrive(&S.cfull[slot]);
                }
                ++cq;
                rq.next(nraw);
                continue;
            }
            const unsigned char* src = raw_slot(r);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (kb >= KB) break;
                unsigned char* dstA = ring + (size_t)slot * slot_bytes + kb * kWBytes;
                const int ci = kb >> 1;                           // chunk of this block within the stage
                const int half = KB > 1 ? (kb & 1) : half1;       // 64-column half of that chunk
#pragma unroll
                for (int it = 0; it < 1024 / (kConvWarps * 32); ++it) {   // 128 rows x 8 units
                    const int k = it * (kConvWarps * 32) + ct;
                    const int i = k >> 3, u = k & 7;
                    // phase A: W_gate's chunk ci, or W_up's (after W_gate's qch)
                    const unsigned char* ch = ph_a ? src + (((i >> 3) & 1) * qch + ci) * kQ4A : src + ci * kQ4B;
                    const int srow = ph_a ? 8 * (i >> 4) + (i & 7) : i;
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(ch + srow * 64 + half * 32 + u * 4);
                    const __nv_bfloat16 sc = *reinterpret_cast<const __nv_bfloat16*>(ch + rows * 64 + srow * 2);
                    *reinterpret_cast<uint4*>(dstA + i * 128 + ((u ^ (i & 7)) << 4)) =
                        decode_q4_row8(w, __bfloat162bfloat162(sc));
                }
            }
            fence_proxy_async_shared();   // the tensor core reads the stage through the async proxy
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&S.raw_empty[r]);    // this warp has read the packed chunks
                mbar_arrive(&S.cfull[slot]);     // and written its rows of the stage
            }
            rq.next(nraw);
        }
    } else {
        // ------------------------------- epilogue --------------------------------
        const int tid = threadIdx.x;   // 0..127
        if (early) {
            wait_bar(&S.meta_full, 0, S, flags);   // token masks and first pairs
            grid_dependency_wait();                // the pairs' tokens come from the routing kernel
        }

        __nv_bfloat16* hb = static_cast<__nv_bfloat16*>(A.hbuf);
        const int i = 32 * warp + lane;                    // this thread's D row (tensor-memory lane)
        const uint32_t lane_addr = (uint32_t)(32 * warp) << 16;
        uint32_t nm = 0;   // meetings of the four warps so far (parity of epi_bar)
        uint32_t np = 0;   // phase-B tiles handed to warp 15
        // hands a finished phase-B tile (or the end, ntok = -1) to warp 15,
        // with the token of the tile's pair `tid` (looked up before the tile's
        // accumulator was ready, so warp 15 need not wait for the lookup)
        auto hand_over = [&](int pair0, int ntok, int rb, int tok) {
            const int slot = (int)(np % kNQ);
            if (np >= kNQ) wait_bar(&S.nt_empty[slot], ((np / kNQ) - 1) & 1, S, flags);
            if (tid < ntok) S.nt_tok[slot][tid] = (uint8_t)tok;
            if (tid == 0) S.nt_info[slot] = make_int4(pair0, ntok, rb, 0);
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.nt_full[slot]);
            ++np;
        };
        for (int n = 0;; ++n) {
            const int q = n % kQ;
            wait_bar(&S.tq_full[q], (n / kQ) & 1, S, flags);
            if (aborted(S)) break;
            const int tile = S.tq[q];
            if (tile < 0) break;
            const bool ph_a = tile < TA;
            const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, X, Tn, nmax);
            const int b = n % kAcc;
            const int ngroups = (ph_a && whole) ? nwb >> 4 : (T.ntok + 15) >> 4;   // 16-column groups of D
            // phase B: the token of pair `tid` of the tile, loaded while the MMAs run
            const int my_tok = !ph_a && tid < T.ntok ? A.perm[T.off + nmax * T.c + tid] / A.kslots : -1;
            wait_bar(&S.acc_full[b], (n / kAcc) & 1, S, flags);
            if (aborted(S)) break;
            tmem_fence_after_sync();
            if (ph_a) {
                // D row i = (2g + m) * 8 + r holds gate (m = 0) or up (m = 1) row
                // 8g + r of the tile, or the reverse when the map starts at W_up;
                // the partner row is 8 lanes away in the same warp.
                const int m = (i >> 3) & 1;
                const int frow = 64 * T.rb + 8 * (i >> 4) + (i & 7);
                const uint64_t tmask = whole ? X.tokmask[T.a] : 0ull;
                const bool swap = A.gu_swap && X.ex_slot[T.a] >= 0;   // INT4 stages hold the gate rows first
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
                        // column j: batch token j (whole batches) or the chunk's j-th pair
                        const bool keep = whole ? ((tmask >> j) & 1ull) != 0 : j < T.ntok;
                        if (m == 0 && keep) {
                            const size_t pos = whole ? (size_t)T.off + __popcll(tmask & ((1ull << j) - 1ull))
                                                     : (size_t)T.off + nmax * T.c + j;
                            hb[pos * F + frow] = __float2bfloat16_rn(silu_f(gs) * us);
                        }
                    }
                }
                // All four warps wait for each meeting's phase, so no warp can
                // arrive for the next meeting before this one completes.
                epi_meet(S, nm, flags, lane);
                if (tid == 0)   // all four warps have stored: release the chunk's counter
                    red_release_gpu_add(&A.hdone[X.chunk_off[T.a] + T.c], 1u);
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
                // the tile's y rows are stored: warp 15 counts its tokens down
                hand_over(T.off + nmax * T.c, T.ntok, T.rb, my_tok);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.tq_empty[q]);
        }
        hand_over(0, -1, 0, -1);   // no more tiles
    }

    // ---- combine: one warp per (token, 128 rows of d) ----
    // Item it goes to CTA it mod G; the idle INT4 converter warps take the
    // first items of a CTA, the epilogue warps the last.  The warp waits
    // until every y slice of its rows is stored (the counter is zero,
    // acquire), sums the kept weights times the y rows in slot order, and
    // sets the counter back to the token's kept slots for the next launch.
    // Tokens that keep no expert find zero at once and get rows of zeros.
    {
        if (early) grid_dependency_wait();   // slot positions, weights and counters come from the routing kernel
        // converters 0-7, producers and MMA 8-10, count-down warp 11, epilogue 12-15
        const int widx = warp == kWarpN ? kConvWarps + 3
                       : warp >= kWarpC ? warp - kWarpC
                       : warp >= kWarpW ? kConvWarps + warp - kWarpW : kConvWarps + 4 + warp;
        const int nitems = A.B * rbB;
        const int ks = A.kslots;
        const float4* y4 = reinterpret_cast<const float4*>(A.ybuf);
        uint2* out2 = static_cast<uint2*>(A.out);
        for (int it = (int)blockIdx.x + (int)G * widx; it < nitems; it += (int)G * (kThreads / 32)) {
            const int tok = it / rbB, r0 = (it - tok * rbB) * kM + 4 * lane;
            uint32_t* c = &A.ycnt[it];
            // the first eight slots' positions and weights (routing results) before the wait
            int pos0[8];
            float wv0[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                pos0[u] = u < ks ? A.pos_of[tok * ks + u] : -1;
                wv0[u] = u < ks ? A.w[tok * ks + u] : 0.f;
            }
            if (lane == 0) wait_zero(c, S, flags);
            __syncwarp();
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 0; s0 < ks; s0 += 8) {
                int pos[8];
                float wv[8];
                float4 yv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int sl = s0 + u;
                    pos[u] = s0 == 0 ? pos0[u] : sl < ks ? A.pos_of[tok * ks + sl] : -1;
                    wv[u] = s0 == 0 ? wv0[u] : sl < ks ? A.w[tok * ks + sl] : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    yv[u] = (pos[u] >= 0 && r0 < d) ? __ldcg(y4 + ((size_t)pos[u] * d + r0) / 4)
                                                    : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 8; ++u) {   // slot order
                    const float wu = pos[u] >= 0 ? wv[u] : 0.f;
                    acc.x += wu * yv[u].x;
                    acc.y += wu * yv[u].y;
                    acc.z += wu * yv[u].z;
                    acc.w += wu * yv[u].w;
                }
            }
            if (r0 < d) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
                out2[((size_t)tok * d + r0) / 4] =
                    make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
            }
            __syncwarp();
            if (lane == 0) *c = (uint32_t)A.nused[tok];
        }
    }

    // ---- release the tensor memory ----
    // After a wait gave up, stages may have been issued that no MMA waited
    // for: give their TMA copies (a few, each landing within microseconds)
    // a bounded 20 us to land before the CTA's shared memory is released.
    if (aborted(S)) {
        const long long t0 = clock64();
        while (clock64() - t0 < 40000) __nanosleep(1000);
    }
    tmem_fence_before_sync();
    __syncthreads();
    // This CTA is done with every counter and buffer of the workspace: the
    // next kernel in the stream may be scheduled (it still waits for this
    // grid's completion before it reads anything).  The counters are zeroed
    // by the next routing kernel, so no grid-wide reset (and no fence under
    // a memory system still saturated by other CTAs' streams) ends the
    // kernel.
    grid_launch_dependents();
    if (warp == kWarpM) {
        tmem_fence_after_sync();
        tmem_dealloc(tmem, tmem_cols);
    }
}

}  // namespace

cudaError_t launch_ffn_tc(const FfnArgs& a_in, const CUtensorMap* maps, int num_sms, cudaStream_t s) {
    // All the shared memory a CTA may have: the stage ring takes what the
    // barriers, the per-expert tables and the INT4 slots leave.
    static int smem_optin[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!smem_optin[dev]) {
        int v = 0;
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
        for (auto* kern : {ffn_tc_kernel<false>, ffn_tc_kernel<true>}) {
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, v)) != cudaSuccess)
                return e;
            // The CTAs wait for one another, so the grid (one CTA per SM) must
            // be able to be resident at once: one CTA of this size has to fit an SM.
            int per_sm = 0;
            if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, (size_t)v)) != cudaSuccess)
                return e;
            if (per_sm < 1) return cudaErrorInvalidConfiguration;
        }
        smem_optin[dev] = v;
    }
    FfnArgs a = a_in;
    a.smem_bytes = smem_optin[dev];
    // the ring must hold two stages of the largest slot this launch can use
    const int kb = a.B <= 16 && a.n_cold == 0 ? a.kbs : a.kbl;
    const int nwb = a.B <= 16 ? 16 : (a.B + 15) & ~15;
    const size_t slot = (size_t)kb * (kWBytes + (a.B <= kWholeMax ? nwb : kNMax) * 128);
    if ((size_t)a.smem_bytes < 4096 + tabs_bytes(a.N) + (size_t)kRawReserve ||
        ring_bytes_for((size_t)a.smem_bytes, a.N, a.n_cold > 0) < 2 * slot)
        return cudaErrorInvalidConfiguration;
    // One CTA per SM (the shared-memory size allows no second one, so the
    // tensor memory is never contended); programmatic dependent launch lets
    // the CTAs allocate and prefetch while the routing kernel finishes.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)a.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, a.n_cold > 0 ? ffn_tc_kernel<true> : ffn_tc_kernel<false>, a, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5],
                              maps[6], maps[7], maps[8], maps[9], maps[10], maps[11], maps[12], maps[13], maps[14]);
}

}  // namespace moe
