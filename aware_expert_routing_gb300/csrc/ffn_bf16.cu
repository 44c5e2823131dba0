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
// Structure (one persistent CTA per SM, 7 warps):
//   * Work is a list of tiles.  Phase-A tile (expert a, 16 rows of d_ff,
//     token chunk c) computes h = silu(W_gate x) * (W_up x) for those rows
//     and up to 16 tokens and writes h (bf16) to the workspace.  Phase-B
//     tile (expert a, 64 rows of d, chunk c) computes y = W_down h (fp32).
//     The list holds every phase-A tile, then every phase-B tile, each in
//     active-expert order.  CTA b starts with tile b and claims each next
//     tile from one grid-wide counter, so the tiles are taken in list order
//     and all CTAs finish within about one tile of each other.  The weight
//     warp claims the tiles and posts them to a 16-entry shared-memory
//     queue that the other warps read; the epilogue warp frees the entries.
//   * A phase-B tile needs the h rows of its token chunk: the epilogue
//     warp counts each finished phase-A tile on the chunk's counter, and
//     the operand warp waits for that count before it loads h.  All
//     phase-A tiles precede all phase-B tiles in the list and wait on
//     nothing later, so these waits always end.
//   * Phase-A operands.  Batches of up to 16 tokens: every expert's tile
//     multiplies the whole batch (two 8-row boxes straight from the hidden
//     states, no copy), and the epilogue keeps the columns of the tokens
//     routed to the expert.  Larger batches: the CTAs first copy the hidden
//     states into an expert-grouped buffer (row p = the token of pair p; CTA
//     b copies rows b, b+G, ...) and each raises its own flag; the operand
//     warp waits for all flags before its first phase-A tile.
//   * A stage of the 7-deep shared-memory ring holds 256 K-columns of the
//     weight tile (16 KB: 16 gate + 16 up rows, or 32 down rows) and the matching
//     columns of the tokens' operand rows (up to 16 rows, 8 KB), all loaded
//     by TMA with the 128-byte swizzle through 3D views of the matrices, so
//     a stage is one or two weight operations plus one per 8 tokens (the
//     TMA unit's cost per operation, not per byte, limits small boxes).
//     Warp 4 issues the weight loads and never waits for another CTA.
//     Weights read once are marked L2 evict-first; an expert with more than
//     16 tokens is read once per 16-token pass, the passes are neighbours in
//     the list (so they run at about the same time on different SMs), and
//     its weights use the normal L2 policy so the repeat reads hit L2.
//     Warp 5 issues the operand loads.  Both producers arrive on the
//     stage's full barrier.
//   * Warps 0-3 are consumers: warp w owns the w-th 64-column block of each
//     stage and runs warp-level bf16 tensor-core MMAs with the weight rows as
//     the M side and the tokens as the N side (8 tokens per MMA column
//     tile), accumulating in fp32.  Both operands are read from shared
//     memory with 16-byte loads; the K index inside each 64-column block is
//     permuted identically for both operands (k-step s, k-slot pair 2t and
//     2t+8 map to columns 16t+4s and 16t+4s+2) so every lane reads 32
//     contiguous bytes and the swizzle keeps the reads conflict free.
//   * At the end of a tile the four consumer warps leave their partial sums
//     in a double-buffered shared-memory area and signal without waiting;
//     warp 6, the epilogue warp, adds them in warp order and writes h
//     (SwiGLU) or y, then frees the buffer.  The consumers only wait when
//     they are two tiles ahead of it.
//   * After its last tile every CTA arrives at a grid-wide counter; once
//     all have arrived, each CTA combines its slice of the output four
//     columns at a time, out_i = sum over slots (in slot order) of
//     w_is * y_is.
//   * The last CTA to finish resets the counters for the next launch.
//   * Mixed precision (DynaExq page, section 3.2: hot experts in high
//     precision, cold experts INT4).  An INT4 expert's matrices are packed as
//     chunks of (16 or 32 rows) x 256 columns: 128 bytes of 4-bit codes per
//     row, then the rows' bf16 scales of the two 128-column groups.  Its
//     tiles have the same geometry as bf16 tiles; a stage is one 1D bulk
//     copy per matrix.  The consumer decodes a code pair into bf16 exactly
//     ((nibbles | 0x4300) is 128 + q + 8; subtracting 136 leaves q),
//     multiplies the integers on the tensor cores, and scales each row's
//     fp32 partial sum of the 64-column block (one 128-column group) by the
//     group scale, so q*s is never rounded.
// Every result is computed in a fixed order, so runs are bit-reproducible.
#include "common.cuh"

namespace moe {

namespace {

constexpr int kCW = 4;                    // consumer warps
constexpr int kWarpW = kCW;               // weight producer warp
constexpr int kWarpO = kCW + 1;           // operand producer warp
constexpr int kWarpE = kCW + 2;           // epilogue warp
constexpr int kThreads = (kCW + 3) * 32;
// Named barriers: 1 consumers (gather), 2/3 partial sums of buffer 0/1 are
// ready, 4/5 buffer 0/1 is free again, 6 consumers + epilogue warp.
constexpr uint32_t kBarGather = 1, kBarFull0 = 2, kBarFree0 = 4, kBarEnd = 6;
constexpr uint32_t kRedThreads = (kCW + 1) * 32;
constexpr int kNT = 2;                    // MMA column tiles (8 tokens each) per pass
constexpr int kChunk = 8 * kNT;           // tokens per tile pass
constexpr int kWBytes = 16384;            // weight part of a stage
constexpr int kOBytes = kNT * 4096;       // operand part: kNT boxes of 8 rows x 4 column blocks
constexpr int kSlotBytes = kWBytes + kOBytes;
constexpr int kStages = 7;
constexpr int kQ = 16;                    // tile queue entries
constexpr int kRed = 4 * 4 * kNT * 32;    // partial sums per warp per tile (up to 4 M-tiles)
constexpr long long kWaitCycles = 4000000000LL;   // about two seconds

struct Smem {
    float red[2][kCW][kRed];         // double-buffered per-warp partial sums
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tq_full[kQ];            // tile queue: entry posted by the weight producer
    uint64_t tq_empty[kQ];           // entry released by the epilogue warp
    int tq[kQ];                      // tile index, or -1 once the list is exhausted
    int red_tile[2];                 // tile whose partial sums are in red[b], or -1 (no more tiles)
    int chunk_off[MOE_MAX_EXPERTS + 1];
    uint32_t ex_info[MOE_MAX_EXPERTS];  // active index -> id | cnt << 10 | first pair << 19
    uint16_t tokmask[MOE_MAX_EXPERTS];  // active index -> tokens routed to it (batches of <= 16)
    int ex_slot[MOE_MAX_EXPERTS];       // active index -> bf16 row block (>= 0) or -1 - INT4 expert
    int abort_flag;
    int last_flag;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kSlotBytes + sizeof(Smem);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct Tile {
    int a, e, rb, c, off, ntok, nch, slot;
};

constexpr int kQ4ChunkA = 16 * 128 + 16 * 4;   // INT4 chunk of W_gate / W_up: 16 rows x 256 columns
constexpr int kQ4ChunkB = 32 * 128 + 32 * 4;   // INT4 chunk of W_down: 32 rows x 256 columns

// Tile t of a phase with rbn row blocks per (expert, chunk); shared memory only.
__device__ __forceinline__ Tile decode_tile(int t, int rbn, const Smem& S, int Tn) {
    const int* chunk_off = S.chunk_off;
    int lo = 0, hi = Tn - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] * rbn <= t) lo = mid; else hi = mid - 1;
    }
    Tile T;
    T.a = lo;
    const uint32_t info = S.ex_info[lo];
    T.e = info & 1023u;
    const int cnt = (info >> 10) & 511u;
    T.off = info >> 19;
    T.nch = chunk_off[lo + 1] - chunk_off[lo];
    T.slot = S.ex_slot[lo];
    const int r = t - chunk_off[lo] * rbn;
    T.rb = r / T.nch;
    T.c = r - T.rb * T.nch;
    T.ntok = min(kChunk, cnt - kChunk * T.c);
    return T;
}

__device__ __forceinline__ void give_up(Smem& S, uint32_t* flags) {
    *(volatile int*)&S.abort_flag = 1;
    raise_flag(flags, kFlagTimeout);
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

__device__ __forceinline__ uint4 lds16(const unsigned char* p) {
    return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ void unpack8(uint32_t (&r)[8], uint4 a, uint4 b) {
    r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
    r[4] = b.x; r[5] = b.y; r[6] = b.z; r[7] = b.w;
}

// Row `row` of a 128-byte-swizzled box: the lane's columns [16*t4, 16*t4+16).
__device__ __forceinline__ void load_row(const unsigned char* box, int row, int t4, uint32_t (&r)[8]) {
    const int sw = row & 7;
    unpack8(r, lds16(box + row * 128 + (((2 * t4) ^ sw) << 4)),
            lds16(box + row * 128 + (((2 * t4 + 1) ^ sw) << 4)));
}

// Two independent 16-row weight blocks (rows r0/r1 and q0/q1) times the same
// token block, the four k-steps of a 64-column block, chains interleaved.
__device__ __forceinline__ void mma_pair(float (&acc0)[4], float (&acc1)[4], const uint32_t (&r0)[8],
                                         const uint32_t (&r1)[8], const uint32_t (&q0)[8],
                                         const uint32_t (&q1)[8], const uint32_t (&xb)[8]) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        mma_bf16_16816(acc0, r0[2 * s], r1[2 * s], r0[2 * s + 1], r1[2 * s + 1], xb[2 * s], xb[2 * s + 1]);
        mma_bf16_16816(acc1, q0[2 * s], q1[2 * s], q0[2 * s + 1], q1[2 * s + 1], xb[2 * s], xb[2 * s + 1]);
    }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }

// Eight codes (one packed word) -> four bf16x2 A-fragment words, exact:
// (w >> 4p) & 0x000f000f | 0x43004300 is the pair (128 + c0, 128 + c1) with
// c = q + 8; subtracting 136 leaves (q0, q1).
__device__ __forceinline__ void decode_q4(uint32_t w, uint32_t* r) {
    const __nv_bfloat162 off = __floats2bfloat162_rn(136.f, 136.f);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t v;
        asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(v) : "r"(w >> (4 * p)), "r"(0x000f000fu), "r"(0x43004300u));
        const __nv_bfloat162 q = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v), off);
        r[p] = *reinterpret_cast<const uint32_t*>(&q);
    }
}

// Row `row` of an INT4 chunk (rows of 128 code bytes): the lane's 16 columns
// of the 64-column block `blk` as eight A-fragment words.
__device__ __forceinline__ void load_row_q4(const unsigned char* chunk, int row, int blk, int t4, uint32_t (&r)[8]) {
    const uint2 w = *reinterpret_cast<const uint2*>(chunk + row * 128 + blk * 32 + t4 * 8);
    decode_q4(w.x, r);
    decode_q4(w.y, r + 4);
}

__device__ __forceinline__ float q4_scale(const unsigned char* chunk, int rows, int row, int blk) {
    const __nv_bfloat16 s = *reinterpret_cast<const __nv_bfloat16*>(chunk + rows * 128 + (row * 2 + (blk >> 1)) * 2);
    return __bfloat162float(s);
}

// Consumer side of one tile: wait for each stage, multiply, release it.
// M-blocks: phase A = (gate rows 0-15, up rows 0-15) at byte offsets 0 and
// 8192 of the weight part (acc[0], acc[1]); phase B: stage s holds rows
// 32 * (s & 1) .. + 31 of the tile's 64 down rows for the K block s >> 1,
// as one 32-row box whose row halves are 2048 bytes apart (acc[2 (s & 1)],
// acc[2 (s & 1) + 1]).
template <bool PHASE_A>
__device__ __forceinline__ void consume_tile(const unsigned char* ring, Smem& S, uint32_t* flags, int nstage,
                                             int K, int NT, bool q4, uint32_t& it, float (&acc)[4][kNT][4]) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j = 0; j < kNT; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][j][q] = 0.f;
    for (int s = 0; s < nstage; ++s, ++it) {
        const int slot = it % kStages;
        const int kb = PHASE_A ? s : s >> 1;       // K block of 256 columns
        const bool hi = !PHASE_A && (s & 1);       // phase B: rows 32-63 of the tile
        const int kq = min(4, (K - 256 * kb) / 64);
        wait_bar(&S.full[slot], (it / kStages) & 1, S, flags);
        if (w < kq && q4) {
            // INT4 chunk(s): phase A gate at 0 and up at 8192 (16 rows each);
            // phase B one 32-row chunk.  Integer products into tmp, then each
            // row's partial sum is scaled by its group scale.
            const unsigned char* st = ring + (size_t)slot * kSlotBytes;
            const unsigned char* op = st + kWBytes + w * 1024;
            const unsigned char* c0p = st;
            const unsigned char* c1p = PHASE_A ? st + 8192 : st;
            const int rows = PHASE_A ? 16 : 32;
            const int r1 = PHASE_A ? 0 : 16;
            uint32_t a0[8], a1[8], c0[8], c1[8];
            load_row_q4(c0p, g, w, t4, a0);
            load_row_q4(c0p, g + 8, w, t4, a1);
            load_row_q4(c1p, r1 + g, w, t4, c0);
            load_row_q4(c1p, r1 + g + 8, w, t4, c1);
            const float s00 = q4_scale(c0p, rows, g, w), s01 = q4_scale(c0p, rows, g + 8, w);
            const float s10 = q4_scale(c1p, rows, r1 + g, w), s11 = q4_scale(c1p, rows, r1 + g + 8, w);
#pragma unroll
            for (int j = 0; j < kNT; ++j)
                if (j < NT) {
                    uint32_t X[8];
                    load_row(op + j * 4096, g, t4, X);
                    float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_pair(t0, t1, a0, a1, c0, c1, X);
                    float (&u0)[4] = hi ? acc[2][j] : acc[0][j];
                    float (&u1)[4] = hi ? acc[3][j] : acc[1][j];
                    u0[0] += s00 * t0[0];
                    u0[1] += s00 * t0[1];
                    u0[2] += s01 * t0[2];
                    u0[3] += s01 * t0[3];
                    u1[0] += s10 * t1[0];
                    u1[1] += s10 * t1[1];
                    u1[2] += s11 * t1[2];
                    u1[3] += s11 * t1[3];
                }
        } else if (w < kq) {
            const unsigned char* st = ring + (size_t)slot * kSlotBytes;
            const unsigned char* op = st + kWBytes + w * 1024;
            const unsigned char* b0 = PHASE_A ? st + w * 2048 : st + w * 4096;
            const unsigned char* b1 = PHASE_A ? st + 8192 + w * 2048 : st + w * 4096;
            const int r1 = PHASE_A ? 0 : 16;
            uint32_t a0[8], a1[8], c0[8], c1[8];
            load_row(b0, g, t4, a0);
            load_row(b0, g + 8, t4, a1);
            load_row(b1, r1 + g, t4, c0);
            load_row(b1, r1 + g + 8, t4, c1);
#pragma unroll
            for (int j = 0; j < kNT; ++j)
                if (j < NT) {
                    uint32_t X[8];
                    load_row(op + j * 4096, g, t4, X);
                    if (hi) mma_pair(acc[2][j], acc[3][j], a0, a1, c0, c1, X);
                    else mma_pair(acc[0][j], acc[1][j], a0, a1, c0, c1, X);
                }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
ffn_bf16_kernel(const FfnArgs A, const __grid_constant__ CUtensorMap tm_gate,
                const __grid_constant__ CUtensorMap tm_up, const __grid_constant__ CUtensorMap tm_down,
                const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_h,
                const __grid_constant__ CUtensorMap tm_hid) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* ring = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem& S = *reinterpret_cast<Smem*>(ring + (size_t)kStages * kSlotBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = A.d, F = A.F;
    uint32_t* flags = &A.hdr->flags;
    const uint32_t G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], 2);        // weight producer + operand producer
            mbar_init(&S.empty[i], kCW);
        }
        for (int i = 0; i < kQ; ++i) {
            mbar_init(&S.tq_full[i], 1);
            mbar_init(&S.tq_empty[i], 1);
        }
        fence_barrier_init();
        S.abort_flag = 0;
    }
    grid_dependency_wait();      // routing comes from the preceding kernel
    int Tn = *A.T;
    if (Tn < 0 || Tn > A.N) {
        if (threadIdx.x == 0 && blockIdx.x == 0) raise_flag(flags, kFlagBadIndex);
        Tn = 0;
    }
    if (warp == 0) {   // per-expert metadata and chunk offsets of the active experts
        int run = 0;
        if (lane == 0) S.chunk_off[0] = 0;
        for (int a0 = 0; a0 < Tn; a0 += 32) {
            const int a = a0 + lane;
            int nch = 0;
            if (a < Tn) {
                const uint32_t info = A.exinfo[a];   // written by the routing kernel
                const int e = info & 1023u;
                const int cnt = (info >> 10) & 511u;
                S.ex_info[a] = info;
                S.tokmask[a] = (uint16_t)A.exinfo[A.N + a];
                int sl = A.slot ? A.slot[e] : e;
                if (sl >= A.n_hot || -1 - sl >= A.n_cold) {   // out of range: flag it, read expert 0
                    raise_flag(flags, kFlagBadIndex);
                    sl = A.n_hot > 0 ? 0 : -1;
                }
                S.ex_slot[a] = sl;
                nch = (cnt + kChunk - 1) / kChunk;
            }
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
    const bool small_b = A.B <= kChunk;   // phase-A operands: the whole batch from the hidden states
    if (warp == kWarpW && lane == 0) {
        prefetch_tensormap(&tm_gate);
        prefetch_tensormap(&tm_up);
        prefetch_tensormap(&tm_down);
    }
    if (warp == kWarpO && lane == 0) {
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_hid);
        prefetch_tensormap(&tm_h);
    }
    __syncthreads();

    // Tiles: phase A (expert, 16 rows of d_ff, chunk) first, then phase B
    // (expert, 64 rows of d, chunk), both in active-expert order.
    const int rbA = F / 16, rbB = d / 64;
    const int SA = (d + 255) / 256, SB = (F + 255) / 256;
    const int TA = S.chunk_off[Tn] * rbA;
    const int Ttot = TA + S.chunk_off[Tn] * rbB;

    if (warp == kWarpW) {
        // ---------------------------- weight producer ----------------------------
        // Claims the CTA's tiles (its first tile is its block index, the
        // others come from one grid-wide counter, so the tiles are taken in
        // list order and every CTA runs until the list is exhausted), posts
        // each to the tile queue and streams its weights.
        if (lane == 0) {
            const uint64_t pol_once = l2_evict_first_policy();
            const uint64_t pol_keep = l2_evict_normal_policy();
            uint32_t it = 0;
            const size_t q4_mat_a = (size_t)(F / 16) * (d / 256) * kQ4ChunkA;   // bytes of one INT4 W_gate / W_up
            const size_t q4_mat_b = (size_t)(d / 32) * (F / 256) * kQ4ChunkB;   // bytes of one INT4 W_down
            // claims run two tiles ahead so that the atomic's latency is hidden
            int next0 = (int)blockIdx.x;
            int next1 = next0 < Ttot ? (int)G + (int)atomicAdd(&A.hdr->next_tile, 1u) : Ttot;
            for (int n = 0;; ++n) {
                const int q = n % kQ;
                if (n >= kQ) wait_bar(&S.tq_empty[q], ((n / kQ) - 1) & 1, S, flags);
                const int tile = next0 < Ttot ? next0 : -1;
                S.tq[q] = tile;
                mbar_arrive(&S.tq_full[q]);
                if (tile < 0) break;
                next0 = next1;
                next1 = next1 < Ttot ? (int)G + (int)atomicAdd(&A.hdr->next_tile, 1u) : Ttot;
                if (tile < TA) {
                    const Tile T = decode_tile(tile, rbA, S, Tn);
                    const int row = T.slot * F + 16 * T.rb;
                    const uint64_t pol = T.nch > 1 ? pol_keep : pol_once;
                    for (int s = 0; s < SA; ++s, ++it) {
                        const int slot = it % kStages;
                        if (it >= kStages) wait_bar(&S.empty[slot], ((it / kStages) - 1) & 1, S, flags);
                        unsigned char* dst = ring + (size_t)slot * kSlotBytes;
                        if (T.slot >= 0) {
                            mbar_arrive_expect_tx(&S.full[slot], kWBytes);   // column blocks past d are zero-filled
                            tma_load_3d(dst, &tm_gate, 0, row, 4 * s, &S.full[slot], pol);
                            tma_load_3d(dst + 8192, &tm_up, 0, row, 4 * s, &S.full[slot], pol);
                        } else {
                            const size_t off = (size_t)(-1 - T.slot) * q4_mat_a +
                                               ((size_t)T.rb * (d / 256) + s) * kQ4ChunkA;
                            mbar_arrive_expect_tx(&S.full[slot], 2 * kQ4ChunkA);
                            bulk_load(dst, A.q_gate + off, kQ4ChunkA, &S.full[slot], pol);
                            bulk_load(dst + 8192, A.q_up + off, kQ4ChunkA, &S.full[slot], pol);
                        }
                    }
                } else {
                    const Tile T = decode_tile(tile - TA, rbB, S, Tn);
                    const int row = T.slot * d + 64 * T.rb;
                    const uint64_t pol = T.nch > 1 ? pol_keep : pol_once;
                    for (int s = 0; s < 2 * SB; ++s, ++it) {   // K block s >> 1, row half s & 1
                        const int slot = it % kStages;
                        if (it >= kStages) wait_bar(&S.empty[slot], ((it / kStages) - 1) & 1, S, flags);
                        if (T.slot >= 0) {
                            mbar_arrive_expect_tx(&S.full[slot], kWBytes);
                            tma_load_3d(ring + (size_t)slot * kSlotBytes, &tm_down, 0, row + 32 * (s & 1), 4 * (s >> 1),
                                        &S.full[slot], pol);
                        } else {
                            const size_t off = (size_t)(-1 - T.slot) * q4_mat_b +
                                               ((size_t)(2 * T.rb + (s & 1)) * (F / 256) + (s >> 1)) * kQ4ChunkB;
                            mbar_arrive_expect_tx(&S.full[slot], kQ4ChunkB);
                            bulk_load(ring + (size_t)slot * kSlotBytes, A.q_down + off, kQ4ChunkB, &S.full[slot], pol);
                        }
                    }
                }
            }
            // Every issued stage is consumed before the consumers reach the
            // end, so no copy is in flight when the CTA exits.
        }
        __syncwarp();
    } else if (warp == kWarpO) {
        // ---------------------------- operand producer ---------------------------
        const uint64_t pol = l2_evict_last_policy();
        uint32_t it = 0;
        bool gathered = small_b;
        for (int n = 0;; ++n) {
            const int q = n % kQ;
            wait_bar(&S.tq_full[q], (n / kQ) & 1, S, flags);
            const int tile = S.tq[q];
            if (tile < 0) break;
            const bool ph_a = tile < TA;
            const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, S, Tn);
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
                const int nt = (ph_a && small_b) ? (A.B + 7) >> 3 : (T.ntok + 7) >> 3;
                const int row0 = (ph_a && small_b) ? 0 : T.off + kChunk * T.c;
                const CUtensorMap* map = ph_a ? (small_b ? &tm_hid : &tm_x) : &tm_h;
                const int ns = ph_a ? SA : 2 * SB;
                for (int s = 0; s < ns; ++s, ++it) {
                    const int slot = it % kStages;
                    const int kb = ph_a ? s : s >> 1;   // phase B: both row halves use the same h columns
                    if (it >= kStages) wait_bar(&S.empty[slot], ((it / kStages) - 1) & 1, S, flags);
                    mbar_arrive_expect_tx(&S.full[slot], nt * 4096);
                    unsigned char* dst = ring + (size_t)slot * kSlotBytes + kWBytes;
                    for (int j = 0; j < nt; ++j)
                        tma_load_3d(dst + j * 4096, map, 0, row0 + 8 * j, 4 * kb, &S.full[slot], pol);
                }
            }
            __syncwarp();
        }
    } else if (warp < kCW) {
        // ------------------------------- consumers -------------------------------
        const int w = warp, tid = threadIdx.x;

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
            for (int v0 = 0; v0 < nvec; v0 += 8 * kCW * 32) {
                uint4 val[8];
                size_t dst[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = v0 + u * kCW * 32 + tid;
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
            named_barrier(kBarGather, kCW * 32);
            if (tid == 0) {
                __threadfence();
                atomicExch(&A.gflag[blockIdx.x], 1u);
            }
        }

        // Every tile: multiply, leave the partial sums and the tile index,
        // signal the epilogue warp; after the last tile hand over -1.  The
        // epilogue warp follows this sequence, so both sides always agree
        // on the number of hand-offs.
        uint32_t it = 0;
        float acc[4][kNT][4];
        int n = 0;
        for (;; ++n) {
            const int q = n % kQ;
            wait_bar(&S.tq_full[q], (n / kQ) & 1, S, flags);
            const int tile = S.tq[q];
            const int buf = n & 1;
            if (tile < 0) {
                if (n >= 2) named_barrier(kBarFree0 + buf, kRedThreads);
                if (tid == 0) S.red_tile[buf] = -1;
                named_barrier_arrive(kBarFull0 + buf, kRedThreads);
                break;
            }
            const bool ph_a = tile < TA;
            const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, S, Tn);
            const int NT = (ph_a && small_b) ? (A.B + 7) >> 3 : (T.ntok + 7) >> 3;
            if (ph_a) consume_tile<true>(ring, S, flags, SA, d, NT, T.slot < 0, it, acc);
            else consume_tile<false>(ring, S, flags, 2 * SB, F, NT, T.slot < 0, it, acc);
            if (n >= 2) named_barrier(kBarFree0 + buf, kRedThreads);
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int j = 0; j < kNT; ++j)
                    if (j < NT && (m < 2 || !ph_a))
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq)
                            S.red[buf][w][(m * kNT + j) * 128 + lane * 4 + qq] = acc[m][j][qq];
            if (tid == 0) S.red_tile[buf] = tile;
            named_barrier_arrive(kBarFull0 + buf, kRedThreads);
        }
        // the epilogue warp frees the buffer of the last tile once more
        if (n >= 1) named_barrier(kBarFree0 + ((n + 1) & 1), kRedThreads);
        named_barrier(kBarEnd, kRedThreads);
    } else {
        // ------------------------------- epilogue warp ------------------------------
        __nv_bfloat16* hb = static_cast<__nv_bfloat16*>(A.hbuf);
        for (int n = 0;; ++n) {
            const int buf = n & 1;
            named_barrier(kBarFull0 + buf, kRedThreads);
            const int tile = S.red_tile[buf];
            if (tile < 0) break;
            const bool ph_a = tile < TA;
            const Tile T = decode_tile(ph_a ? tile : tile - TA, ph_a ? rbA : rbB, S, Tn);
            const int NT = (ph_a && small_b) ? (A.B + 7) >> 3 : (T.ntok + 7) >> 3;
            const uint32_t tmask = small_b ? S.tokmask[T.a] : 0u;
            const float* red = &S.red[buf][0][0];
            if (ph_a) {
                // element l = j*128 + lane*4 + q of the gate partials (up at +kNT*128)
                for (int l = lane; l < NT * 128; l += 32) {
                    const int j = l >> 7, ln = (l >> 2) & 31, qq = l & 3;
                    const int nn = 8 * j + 2 * (ln & 3) + (qq & 1);
                    // column nn: the tile's nn-th token, or batch token nn
                    const bool keep = small_b ? ((tmask >> nn) & 1u) != 0 : nn < T.ntok;
                    if (keep) {
                        float gs = 0.f, us = 0.f;
#pragma unroll
                        for (int ww = 0; ww < kCW; ++ww) {   // warp order
                            gs += red[ww * kRed + l];
                            us += red[ww * kRed + kNT * 128 + l];
                        }
                        const int row = (ln >> 2) + 8 * (qq >> 1);
                        const size_t pos = small_b ? (size_t)T.off + __popc(tmask & ((1u << nn) - 1u))
                                                   : (size_t)T.off + kChunk * T.c + nn;
                        hb[pos * F + 16 * T.rb + row] = __float2bfloat16_rn(silu_f(gs) * us);
                    }
                }
            } else {
                for (int l = lane; l < 4 * kNT * 128; l += 32) {
                    const int m = l / (kNT * 128), j = (l >> 7) % kNT, ln = (l >> 2) & 31, qq = l & 3;
                    const int nn = 8 * j + 2 * (ln & 3) + (qq & 1);
                    if (j < NT && nn < T.ntok) {
                        float ys = 0.f;
#pragma unroll
                        for (int ww = 0; ww < kCW; ++ww) ys += red[ww * kRed + l];
                        const int row = 16 * m + (ln >> 2) + 8 * (qq >> 1);
                        const size_t pos = (size_t)T.off + kChunk * T.c + nn;
                        A.ybuf[pos * d + 64 * T.rb + row] = ys;
                    }
                }
            }
            named_barrier_arrive(kBarFree0 + buf, kRedThreads);
            __syncwarp();
            if (lane == 0) {
                if (ph_a) {   // these h rows are written
                    __threadfence();
                    atomicAdd(&A.hdone[S.chunk_off[T.a] + T.c], 1u);
                }
                mbar_arrive(&S.tq_empty[n % kQ]);   // tile n came from queue entry n
            }
        }
        // Every CTA arrives after its last tile; once all have, the output is combined.
        if (lane == 0) {
            __threadfence();
            atomicAdd(&A.hdr->b_done, 1u);
            wait_counter(&A.hdr->b_done, G, S, flags);
            __threadfence();
        }
        __syncwarp();
        named_barrier(kBarEnd, kRedThreads);
    }

    // ---- combine: each CTA a slice of the output, four columns at a time ----
    if (warp < kCW || warp == kWarpE) {
        const int ctid = warp < kCW ? (int)threadIdx.x : kCW * 32 + lane;
        const int d4 = d / 4;
        const long long total = (long long)A.B * d4;
        const long long o0 = total * blockIdx.x / G, o1 = total * (blockIdx.x + 1) / G;
        const float4* y4 = reinterpret_cast<const float4*>(A.ybuf);
        uint2* out = static_cast<uint2*>(A.out);
        for (long long o = o0 + ctid; o < o1; o += kRedThreads) {
            const int i = (int)(o / d4), c4 = (int)(o - (long long)i * d4);
            float4 acc2 = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 0; s0 < A.kslots; s0 += 8) {
                float4 yv[8];
                float wv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int sl = s0 + u;
                    const int pos = sl < A.kslots ? A.pos_of[i * A.kslots + sl] : -1;
                    wv[u] = pos >= 0 ? A.w[i * A.kslots + sl] : 0.f;
                    yv[u] = pos >= 0 ? __ldcg(y4 + (size_t)pos * d4 + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {   // slot order
                    acc2.x += wv[u] * yv[u].x;
                    acc2.y += wv[u] * yv[u].y;
                    acc2.z += wv[u] * yv[u].z;
                    acc2.w += wv[u] * yv[u].w;
                }
            }
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc2.x, acc2.y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(acc2.z, acc2.w);
            out[o] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
        }
    }

    // ---- the last CTA resets the counters for the next launch ----
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(&A.hdr->ctas_done, 1u);
        S.last_flag = (old + 1 == G);
    }
    __syncthreads();
    if (S.last_flag) {
        __threadfence();
        for (int i = threadIdx.x; i < (int)G; i += kThreads) A.gflag[i] = 0;
        for (int i = threadIdx.x; i < S.chunk_off[Tn]; i += kThreads) A.hdone[i] = 0;
    }
    if (S.last_flag && threadIdx.x == 0) {
        A.hdr->next_tile = 0;
        A.hdr->b_done = 0;
        A.hdr->ctas_done = 0;
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
    // One CTA per SM (the shared-memory size allows no second one), so the
    // whole grid becomes resident once the preceding kernel has left its SM;
    // the grid-wide counters wait only on CTAs that never wait on anything
    // launched after them.  Programmatic dependent launch lets the CTAs start
    // their prologue while the routing kernel finishes.
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
    return cudaLaunchKernelEx(&cfg, ffn_bf16_kernel, a, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5]);
}

size_t ffn_bf16_smem_bytes() { return kSmemBytes; }

}  // namespace moe
