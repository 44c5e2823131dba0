// common.cuh -- internal definitions shared by the kernels of the library:
// argument structs, the workspace layout and inline-PTX wrappers for
// sm_103a (mbarrier, TMA, warp-level bf16 MMA, cluster shared memory).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr uint32_t kFlagNonFinite = MOE_FLAG_NONFINITE_SCORE;
constexpr uint32_t kFlagTimeout = MOE_FLAG_WAIT_TIMEOUT;
constexpr uint32_t kFlagBadIndex = MOE_FLAG_BAD_INDEX;

// ---------------------------------------------------------------------------
// Workspace layout.  Offsets are 256-byte aligned; the header holds the flag
// word and the counters that the expert kernel uses to order its two phases.
// ---------------------------------------------------------------------------
struct WsHeader {
    uint32_t flags;        // MOE_FLAG_* raised by kernels
    uint32_t unused0;
    // Two sets of the expert kernel's counters.  Routing call r on a
    // workspace zeroes set (r + 1) % 2, which the expert call of routing
    // r - 1 used, and the expert call of routing r uses set r % 2, which
    // routing r - 1 zeroed (the host zeroes a set itself before an expert
    // call that repeats one on the same routing).  So the expert kernel ends
    // without a grid-wide reset, and the routing kernel's zeroing is not
    // ordered against anything it publishes.
    uint32_t next_tile[2]; // expert kernel: tiles claimed beyond each CTA's first
    uint32_t gathered[2];  // expert kernel: CTAs that copied their rows of the grouped hidden states
    uint32_t pad[58];
    // routing kernel (OEA, batches of up to 32): S_base, word j (experts
    // 32j ... 32j + 31, one bit each) in the low half and the epoch of the
    // routing call in the high half, each stored at once with release
    uint64_t union_words[32];
};
static_assert(sizeof(WsHeader) == 512, "the header is two 256-byte blocks");

// Per-chunk counters of one set (hdone): at most N + B * kslots / 16 + 1
// token chunks of the largest launch.
constexpr int kHdoneSet = MOE_MAX_EXPERTS + MOE_MAX_TOKENS * MOE_MAX_SLOTS / 16 + 1;

struct WsLayout {
    size_t header, hdone, exinfo, pos_of, nused, ycnt, logits, hbuf, ybuf, xperm, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int kMaxGrid = 1024;   // largest grid of the persistent expert kernel

// B, N, d, kslots, F: see moe.h.  elt = bytes per element of the FFN width
// buffer H (bf16 or fp32).
inline WsLayout ws_layout(int B, int N, int d, int kslots, int F, int h_elt) {
    WsLayout L;
    size_t o = 0;
    L.header = o; o += align256(sizeof(WsHeader));
    L.hdone = o;  o += align256(sizeof(uint32_t) * 2 * (size_t)kHdoneSet);   // two sets, per token chunk
    L.exinfo = o; o += align256(sizeof(uint32_t) * 3 * N);   // per active expert: info, token mask (2 words)
    L.pos_of = o; o += align256(sizeof(int32_t) * (size_t)B * kslots + 4);
    L.nused = o;  o += align256(sizeof(int32_t) * (size_t)B + 4);                  // kept slots per token
    L.ycnt = o;   o += align256(sizeof(uint32_t) * (size_t)B * ((d + 127) / 128) + 4);   // per (token, 128 rows of d)
    L.logits = o; o += align256(sizeof(float) * (size_t)B * N + 4);
    L.hbuf = o;   o += align256((size_t)B * kslots * F * h_elt);
    L.ybuf = o;   o += align256(sizeof(float) * (size_t)B * kslots * d);
    L.xperm = o;  o += align256((size_t)B * kslots * d * h_elt);
    L.total = o;
    return L;
}

// ---------------------------------------------------------------------------
// Kernel argument structs.
// ---------------------------------------------------------------------------
struct RouterArgs {
    const void* x;          // [B][d]
    const void* w;          // [N][d]
    const float* bias;      // [N] or null
    float* logits;          // [B][N]
    int B, N, d;
    int ks;                 // cluster size along K
};

struct RouteArgs {
    const float* logits;    // [B][N]
    int B, B_valid, N, k, mode, k0, maxP, kmax, kslots;
    float p;
    int32_t* idx;           // [B][kslots]
    float* w;               // [B][kslots]
    int32_t* T;
    int32_t* active;        // [N]
    int32_t* counts;        // [N]
    int32_t* offsets;       // [N+1]
    int32_t* perm;          // [B*kslots]
    int32_t* pos_of;        // [B*kslots]
    int32_t* n_base;        // [B] or null
    uint32_t* exinfo;       // [3][N]: active expert a -> id | cnt << 10 | first pair << 19; tokens 0-31, 32-63 (B <= 64)
    int32_t* nused;         // [B] kept slots of each token
    uint32_t* ycnt;         // [B][rbd] set to nused: the expert kernel counts each row block's y slices down
    int rbd;                // row blocks of 128 in d
    uint32_t* flags;
    // OEA, batches of up to 64 tokens: S_base (one bit per expert), published
    // with `epoch` once phase 1 is done, so the expert kernel can start on
    // the activated experts' weights before the routing ends.
    uint64_t* uwords;       // [32] epoch << 32 | word, or null: not published
    uint32_t epoch;         // nonzero, distinct per routing call on this workspace
    // the expert kernel's counter set this call zeroes (see WsHeader): the
    // header's next_tile[s] and gathered[s], and hdone [kHdoneSet] of set s
    uint32_t* clr_next;
    uint32_t* clr_gathered;
    uint32_t* clr_hdone;
};

struct FfnArgs {
    const void* x;          // [B][d] hidden
    const int32_t* T;
    const int32_t* active;
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* perm;
    const int32_t* pos_of;
    const uint32_t* exinfo; // [3][N] written by the routing kernel
    const int32_t* idx;     // [B][kslots] routing experts
    const float* w;         // [B][kslots] routing weights
    void* hbuf;             // [pairs][F]
    float* ybuf;            // [pairs][d]
    void* xperm;            // [pairs][d] hidden states grouped by expert
    void* out;              // [B][d]
    uint32_t* hdone;        // [token chunks] phase-A tiles of the chunk whose h rows are written (this launch's set)
    uint32_t* next_tile;    // this launch's set of the header counters
    uint32_t* gathered;
    const int32_t* nused;   // [B] kept slots of each token (routing kernel)
    uint32_t* ycnt;         // [B][ceil(d / 128)] y slices still missing; the last writer combines
    WsHeader* hdr;
    const void* w_gate;     // [N][F][d]   (fp32 path)
    const void* w_up;
    const void* w_down;     // [N][d][F]
    const int32_t* slot;    // [N] or null: >= 0 bf16 expert, < 0: -1 - INT4 expert
    const uint8_t* q_gate;  // INT4 experts, packed (see moe.h)
    const uint8_t* q_up;
    const uint8_t* q_down;
    int B, N, d, F, kslots;
    int n_hot, n_cold;
    int gu_fused;           // tcgen05 kernel: W_gate and W_up through one interleaving 5D map
    int gu_swap;            // that map starts at W_up (the lower address): up rows come first
    int kbs;                // tcgen05 kernel: 64-column blocks per stage for batches of up to 16 tokens
    int kbl;                // tcgen05 kernel: 64-column blocks per stage for larger batches
    int smem_bytes;         // tcgen05 kernel: dynamic shared memory of the launch (set by the launcher)
    // OEA, batches of up to 64 tokens: the routing kernel's early S_base
    // (RouteArgs::uwords) and the epoch of the routing call that this launch
    // follows; epoch 0: wait for the whole routing instead.
    const uint64_t* uwords;
    uint32_t epoch;
    // Bound of every wait in the expert kernel, in SM clock cycles (about
    // 2000 per microsecond); a wait that runs longer gives up and raises
    // MOE_FLAG_WAIT_TIMEOUT.
    long long wait_cycles;
};

// Bound of in-kernel waits set with moe_set_wait_timeout_us, in cycles.
long long wait_cycles_now();

// Launchers (defined in the .cu files).
cudaError_t launch_router(const RouterArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s);
// Router scores and routing in one cluster launch (bf16, up to 32 tokens,
// N <= 128); launch_router + launch_route otherwise.
bool route_fused_supported(int dtype, int B, int N, int kslots);
cudaError_t launch_route_fused(const RouterArgs& r, const RouteArgs& a, cudaStream_t s);
// tcgen05 expert kernel (bf16 weights).  maps[0..6]: W_gate/W_up
// interleaved 8 rows at a time (5D, gu_fused) or W_gate alone (8-row
// boxes), the same again (not read), W_up (8-row boxes), W_down (128-row
// boxes), gathered hidden states and h (16-row boxes) and the hidden states
// (the whole batch of up to 64 tokens in one box), all one 64-column block
// wide; maps[7..10]: the 5D gate/up map (or W_gate's 8-row map), W_down,
// the hidden states (as wide as the launch's stages) and h with boxes kbs
// blocks wide (batches of up to 16 tokens); maps[11..12]: the 5D gate/up
// map (or W_gate's) and W_down with boxes kbl blocks wide (larger batches);
// maps[13..14]: W_up's 8-row map kbs, then kbl blocks wide (read when
// W_gate and W_up cannot share the 5D map).
cudaError_t launch_ffn_tc(const FfnArgs& a, const CUtensorMap* maps, int num_sms, cudaStream_t s);
cudaError_t launch_ffn_f32(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_synth(void* dst, int dtype, uint64_t n, uint64_t start, uint64_t seed,
                         float scale, cudaStream_t s);
cudaError_t launch_pack_int4(const void* w, int rows, int cols, int rb, void* out, cudaStream_t s);

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void raise_flag(uint32_t* flags, uint32_t bits) {
    atomicOr(flags, bits);
}

// mbarrier ------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait: gives up after `limit` polls (each poll may suspend the
// thread for a hardware-defined interval), returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit = (1u << 24)) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// TMA ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1),
          "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
          "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            int c4, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
          "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---- 5th-generation tensor cores (tcgen05) and tensor memory ------------
// Shared-memory matrix descriptor for a K-major operand stored as rows of
// 128 bytes (64 bf16) with the 128-byte swizzle, 8-row groups 1024 bytes
// apart (the image a TMA box with CU_TENSOR_MAP_SWIZZLE_128B and a 64-column
// inner extent leaves at a 1024-byte aligned address).  Fields: start
// address >> 4 (bits 0-13), leading byte offset >> 4 (16-29, unused by this
// layout), stride byte offset >> 4 (32-45), descriptor version 1 (46-47),
// layout 2 = 128-byte swizzle (61-63).  The K offset inside the 128-byte
// row is added to the start address.
__device__ __forceinline__ uint64_t umma_sdesc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// The same with the 8-row groups `sbo` bytes apart (a multiple of 1024
// below 256 KB): an operand whose 1024-byte swizzle atoms are interleaved
// with those of other K blocks.
__device__ __forceinline__ uint64_t umma_sdesc_sw128_sbo(uint32_t saddr, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), bf16 A and B (bits 7-9, 10-12 = 1), both K-major, N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A * B^T for one K=16 step, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A * B^T for one K=16 step with A read from tensor memory:
// row m of A in lane m, K pairs in 32-bit columns (the lower K in the low
// half), 8 columns per step, from column a_tmem & 0xffff.
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Whole warp: lane l stores 16 consecutive 32-bit columns of TMEM lane
// (taddr >> 16) + l, from column taddr & 0xffff.  tmem_wait_st() completes
// the warp's stores.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                   "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Arrive (once) on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tmem_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole warp: allocate `cols` TMEM columns (a power of two >= 32); the base
// address is written to *dst in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(dst)), "r"(cols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

// Whole warp: lane l receives 16 consecutive fp32 columns of TMEM lane
// (taddr >> 16) + l, starting at column taddr & 0xffff.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 1D bulk copy global -> shared (both addresses 16-byte aligned, bytes a
// multiple of 16), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Orders this thread's earlier generic-proxy accesses (and what it has
// acquired) before its later async-proxy (TMA) accesses of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Warp-level MMA: D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col) ------
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Cluster ----------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(raddr) : "memory");
    return v;
}

// Stores v at the address of `local` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ void st_dsmem_f32(float* local, uint32_t rank, float v) {
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(raddr), "f"(v) : "memory");
}

// Global memory ordering -------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its memory is visible / allow the next kernel in
// the stream to be scheduled now (it still waits for us before reading).
// Atomic add at GPU scope with release semantics (earlier writes this
// thread has made or observed are visible before it) and no result.
__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Relaxed 64-bit accesses at GPU scope (single-copy atomic, no fence): for
// words that carry their own tag, so that nothing else has to be ordered
// with them.
__device__ __forceinline__ void st_relaxed_gpu_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Atomic add at GPU scope with acquire and release semantics; returns the old value.
__device__ __forceinline__ uint32_t atom_acq_rel_gpu_add(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier for a subset of warps.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Arrive at a named barrier without waiting for it to complete.
__device__ __forceinline__ void named_barrier_arrive(uint32_t id, uint32_t threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

#endif  // __CUDACC__

}  // namespace moe
