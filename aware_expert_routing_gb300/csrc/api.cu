// api.cu -- the C ABI declared in include/moe.h: argument checks, workspace
// layout, TMA descriptor encoding and the launch sequence of the layer.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstddef>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <unordered_map>

#include "common.cuh"

using namespace moe;

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct Params {
    int B, B_valid, d, N, k, mode, k0, maxP, kmax, kslots, dtype;
    float p;
};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// k0 chosen from the batch (OEA page, section 7, implementation detail 2:
// piggybacking is redundant for a single token and pays only for
// non-trivial batches, where a larger, safer k0 suits smaller batches).
// At most one real token: OEA is off, i.e. k0 = k with top-p off, which
// routes exactly as plain top-k.  2..15 tokens: ceil(5k/8); 16 or more:
// ceil(3k/8) -- for k = 8 the page's two settings, 5 and 3, whose results
// it reports at 16 tokens.
int policy_k0(int B_valid, int k, float* p) {
    if (B_valid <= 1) {
        *p = 1.f;
        return k;
    }
    return B_valid < 16 ? (5 * k + 7) / 8 : (3 * k + 7) / 8;
}

moe_status resolve(const moe_route_params* in, Params& P) {
    if (!in) return fail(MOE_ERR_ARG, "params is NULL");
    P.B = in->B;
    P.B_valid = in->B_valid < 0 ? in->B : in->B_valid;
    P.d = in->d;
    P.N = in->N;
    P.k = in->k;
    P.mode = in->mode;
    P.dtype = in->dtype;
    P.k0 = in->k0;
    P.p = in->p;
    if (P.B < 0 || P.B > MOE_MAX_TOKENS) return fail(MOE_ERR_ARG, "B=%d outside 0..%d", P.B, MOE_MAX_TOKENS);
    if (P.B_valid > P.B) return fail(MOE_ERR_ARG, "B_valid=%d > B=%d", P.B_valid, P.B);
    if (P.d < 64 || P.d % 64 != 0 || P.d > 16384)
        return fail(MOE_ERR_ARG, "d=%d must be a multiple of 64 in 64..16384", P.d);
    if (P.N < 1 || P.N > MOE_MAX_EXPERTS) return fail(MOE_ERR_ARG, "N=%d outside 1..%d", P.N, MOE_MAX_EXPERTS);
    const int slot_cap = P.N < MOE_MAX_SLOTS ? P.N : MOE_MAX_SLOTS;
    if (P.k < 1 || P.k > slot_cap) return fail(MOE_ERR_ARG, "k=%d outside 1..%d", P.k, slot_cap);
    if (P.dtype != MOE_DTYPE_BF16 && P.dtype != MOE_DTYPE_F32) return fail(MOE_ERR_ARG, "unknown dtype %d", P.dtype);
    if (P.mode == MOE_MODE_TOPK) {
        P.k0 = P.k;
        P.p = 1.f;
        P.maxP = P.N;
        P.kmax = P.k;
        P.kslots = P.k;
    } else if (P.mode == MOE_MODE_OEA) {
        if (!(P.p > 0.f) || !(P.p <= 1.f)) return fail(MOE_ERR_ARG, "p=%g outside (0, 1]", (double)P.p);
        if (P.k0 <= 0) P.k0 = policy_k0(P.B_valid, P.k, &P.p);
        if (P.k0 < 1 || P.k0 > P.k) return fail(MOE_ERR_ARG, "k0=%d outside 1..k=%d", P.k0, P.k);
        P.maxP = (in->maxP <= 0 || in->maxP >= P.N) ? P.N : in->maxP;
        P.kmax = in->kmax <= 0 ? P.k : in->kmax;
        if (P.kmax < P.k0 || P.kmax > slot_cap)
            return fail(MOE_ERR_ARG, "kmax=%d outside k0..%d", P.kmax, slot_cap);
        P.kslots = P.kmax;
    } else {
        return fail(MOE_ERR_ARG, "unknown mode %d", P.mode);
    }
    return MOE_OK;
}

WsLayout layout(const Params& P, int F) {
    return ws_layout(P.B, P.N, P.d, P.kslots, F, P.dtype == MOE_DTYPE_BF16 ? 2 : 4);
}

moe_status check_ws(void* ws, size_t bytes, size_t need) {
    if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(MOE_ERR_WORKSPACE, "workspace not 256-byte aligned");
    if (bytes < need) return fail(MOE_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", bytes, need);
    return MOE_OK;
}

// Buffers sized by B may be NULL when B == 0.
moe_status check_routing(const moe_routing* r, bool for_route, int B) {
    if (!r) return fail(MOE_ERR_ARG, "routing is NULL");
    const void* req[] = {r->T, r->active, r->counts, r->offsets, r->expert_idx, r->weights, r->perm};
    for (int i = 0; i < 7; ++i) {
        const void* q = req[i];
        if (!q && (i < 4 || B > 0)) return fail(MOE_ERR_ARG, "a required routing buffer is NULL");
        if (!aligned(q, 4)) return fail(MOE_ERR_ARG, "routing buffer not 4-byte aligned");
    }
    if (for_route) {
        if (r->n_base && !aligned(r->n_base, 4)) return fail(MOE_ERR_ARG, "n_base not 4-byte aligned");
        if (r->logits && !aligned(r->logits, 4)) return fail(MOE_ERR_ARG, "logits not 4-byte aligned");
    }
    return MOE_OK;
}

// ---- TMA descriptors for the expert matrices (cached per weight set) -------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct MapKey {
    const void *g, *u, *dn;
    int N, F, d, dev;
    bool operator==(const MapKey& o) const {
        return g == o.g && u == o.u && dn == o.dn && N == o.N && F == o.F && d == o.d && dev == o.dev;
    }
};

std::mutex g_map_mu;

// Per workspace: the epoch of its last routing call, and whether the expert
// kernel's counters are fresh (zeroed by that routing call and not used
// since).  Each OEA routing launch of up to 32 tokens publishes its union of
// activated experts under a new epoch (never 0, distinct across all
// workspaces); the expert kernel that follows on the same workspace waits
// for that epoch, so a union left by an earlier call never passes for the
// current one.  Forgetting a workspace is safe: its next expert call then
// clears the counters itself and waits for the whole routing.
struct WsState {
    uint32_t epoch = 0;    // 0: no routing call recorded
    uint32_t routes = 0;   // routing calls recorded (their parity picks the counter sets)
    bool fresh = false;    // the expert counters of the last routing call are unused
    bool known = false;
};
std::mutex g_ws_mu;
std::unordered_map<const void*, WsState> g_ws;
uint32_t g_last_epoch = 0;

// The epoch the next routing call publishes under (recorded by
// routed() once that call's kernel has been launched).
uint32_t next_epoch() {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    return g_last_epoch + 1u == 0u ? 1u : g_last_epoch + 1u;
}

// A routing kernel was launched on `ws` (epoch e, or 0: none published).
void routed(const void* ws, uint32_t e) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if (g_ws.size() >= 4096 && !g_ws.count(ws)) g_ws.clear();
    WsState& st = g_ws[ws];
    st.epoch = e;
    st.routes += 1;
    st.fresh = true;
    st.known = true;
    if (e) g_last_epoch = e;
}

// The expert counter set used after routing call r (the one routing call
// r zeroes is the other).
int counter_set(uint32_t routes_before) { return (int)(routes_before & 1u); }

// Zeroes counter set `set` (both, if set < 0) of the workspace on `s`.
cudaError_t clear_counters(unsigned char* ws, const WsLayout& L, int set, cudaStream_t s) {
    WsHeader* h = reinterpret_cast<WsHeader*>(ws + L.header);
    for (int k = 0; k < 2; ++k) {
        if (set >= 0 && k != set) continue;
        cudaError_t e = cudaMemsetAsync(&h->next_tile[k], 0, sizeof(uint32_t), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(&h->gathered[k], 0, sizeof(uint32_t), s);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(ws + L.hdone + (size_t)k * kHdoneSet * sizeof(uint32_t), 0,
                                (size_t)kHdoneSet * sizeof(uint32_t), s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

WsState ws_state(const void* ws) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    const auto it = g_ws.find(ws);
    return it == g_ws.end() ? WsState{} : it->second;
}

// An expert kernel was launched on `ws`: its counters are used.
void experts_launched(const void* ws) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    const auto it = g_ws.find(ws);
    if (it != g_ws.end()) it->second.fresh = false;
}

// A row-major bf16 matrix [rows][cols] (cols a multiple of 64) viewed as 3D
// {64 columns, rows, cols/64 column blocks}: one box {64, box_rows, 4} moves
// 256 columns of box_rows rows and lands in shared memory as four
// consecutive 128-byte-swizzled [box_rows][64] blocks.  One TMA operation
// per 256 columns keeps the per-operation cost of the TMA unit off the
// critical path.
bool encode_3d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows,
               uint32_t box_blocks = 4) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64, box_rows, box_blocks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ---- tensor maps of the tcgen05 expert kernel
// W_gate and W_up ([rows][cols] each) interleaved 8 rows at a time through
// one 5D view {64 columns, 8 rows, 2 matrices, rows/8 row groups, cols/64
// column blocks}: one box {64, 8, 2, 8, kb} lands as kb consecutive blocks of
// 8 x {8 rows of the lower matrix, the same 8 rows of the other} = 128 rows
// x 64 columns.  The matrix
// stride is the distance between the two arrays, lower address first
// (*swap: W_up is the lower one).  Fails if the arrays coincide or lie 2^40
// bytes or more apart (the tensor-map stride limit).
bool encode_gate_up_5d(CUtensorMap* m, const void* g, const void* u, uint64_t cols, uint64_t rows, bool* swap,
                       uint32_t box_blocks = 1) {
    auto enc = get_encode();
    if (!enc) return false;
    const uintptr_t pg = reinterpret_cast<uintptr_t>(g), pu = reinterpret_cast<uintptr_t>(u);
    *swap = pu < pg;
    const uintptr_t lo = *swap ? pu : pg, hi = *swap ? pg : pu;
    const uint64_t delta = hi - lo;
    if (delta == 0 || delta % 16 != 0 || delta >= (1ull << 40) || rows % 8 != 0) return false;
    cuuint64_t dims[5] = {64, 8, 2, rows / 8, cols / 64};
    cuuint64_t strides[4] = {cols * 2, delta, 8 * cols * 2, 128};
    cuuint32_t box[5] = {64, 8, 2, 8, box_blocks};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, reinterpret_cast<void*>(lo), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Blocks of 64 columns per stage for batches of up to 16 tokens: the most
// of 4, 2, 1 that divides both d / 64 and d_ff / 64.
int small_batch_blocks(int d, int F) {
    for (int kb = 4; kb > 1; kb >>= 1)
        if ((d / 64) % kb == 0 && (F / 64) % kb == 0) return kb;
    return 1;
}

// Blocks per stage for larger batches (token rows of up to 128 per stage
// share the ring): 2 where d / 64 and d_ff / 64 are even, else 1.
int large_batch_blocks(int d, int F) { return ((d / 64) % 2 == 0 && (F / 64) % 2 == 0) ? 2 : 1; }

struct TcMapEntry {
    MapKey key;
    // gate/up 5D (or W_gate 8-row boxes), W_up 8-row boxes, W_down 128-row boxes
    // (one block wide); gate/up 5D (or W_gate 8-row boxes) and W_down as many
    // blocks wide as small batches use, then as many as larger batches use;
    // W_up 8-row boxes as wide as small, then as larger batches use (read
    // when W_gate and W_up cannot share the 5D map)
    CUtensorMap maps[9];
    bool fused, swap, used;
};
TcMapEntry g_tc_maps[64];
int g_tc_next = 0;

moe_status tc_expert_maps(const void* g, const void* u, const void* dn, int N, int F, int d, int dev,
                          CUtensorMap* out, bool* fused, bool* swap) {
    std::lock_guard<std::mutex> lk(g_map_mu);
    MapKey key{g, u, dn, N, F, d, dev};
    for (auto& e : g_tc_maps)
        if (e.used && e.key == key) {
            memcpy(out, e.maps, sizeof e.maps);
            *fused = e.fused;
            *swap = e.swap;
            return MOE_OK;
        }
    TcMapEntry& e = g_tc_maps[g_tc_next];
    g_tc_next = (g_tc_next + 1) % 64;
    e.key = key;
    e.used = false;
    e.swap = false;
    e.fused = encode_gate_up_5d(&e.maps[0], g, u, d, (uint64_t)N * F, &e.swap);
    if (!e.fused) {   // two maps, 8-row boxes (used when W_gate and W_up cannot share one map)
        e.swap = false;
        if (!encode_3d(&e.maps[0], g, d, (uint64_t)N * F, 8, 1))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (W_gate)");
    }
    if (!encode_3d(&e.maps[1], u, d, (uint64_t)N * F, 8, 1) || !encode_3d(&e.maps[2], dn, F, (uint64_t)N * d, 128, 1))
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (W_up / W_down)");
    const uint32_t kb = (uint32_t)small_batch_blocks(d, F);
    const uint32_t kbl = (uint32_t)large_batch_blocks(d, F);
    bool swap4 = false;
    if (e.fused) {
        if (!encode_gate_up_5d(&e.maps[3], g, u, d, (uint64_t)N * F, &swap4, kb) ||
            !encode_gate_up_5d(&e.maps[5], g, u, d, (uint64_t)N * F, &swap4, kbl))
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (W_gate / W_up, wide boxes)");
        e.maps[7] = e.maps[1];   // not read
        e.maps[8] = e.maps[1];
    } else if (!encode_3d(&e.maps[3], g, d, (uint64_t)N * F, 8, kb) ||
               !encode_3d(&e.maps[5], g, d, (uint64_t)N * F, 8, kbl) ||
               !encode_3d(&e.maps[7], u, d, (uint64_t)N * F, 8, kb) ||
               !encode_3d(&e.maps[8], u, d, (uint64_t)N * F, 8, kbl)) {
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (W_gate / W_up, 8-row wide boxes)");
    }
    if (!encode_3d(&e.maps[4], dn, F, (uint64_t)N * d, 128, kb) || !encode_3d(&e.maps[6], dn, F, (uint64_t)N * d, 128, kbl))
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (W_down, wide boxes)");
    e.used = true;
    memcpy(out, e.maps, sizeof e.maps);
    *fused = e.fused;
    *swap = e.swap;
    return MOE_OK;
}

// Workspace maps of the tcgen05 kernel: expert-grouped hidden states and h
// (16-row boxes), and the hidden states themselves (one box holds the whole
// batch of up to 64 tokens, rounded up to 16 rows; rows past B read as
// zeros); then the hidden states with boxes as wide as the launch's stages
// and h with boxes kb blocks wide (batches of up to 16 tokens).
struct TcOpEntry {
    const void* ws;
    const void* hidden;
    int pairs, B, d, F, dev;
    bool q4;   // a launch with INT4 experts: stages of kbl blocks at every batch size
    CUtensorMap maps[5];
    bool used;
};
TcOpEntry g_tc_ops[32];
int g_tc_ops_next = 0;

moe_status tc_operand_maps(unsigned char* ws, const WsLayout& L, const void* hidden, int pairs, int B, int d, int F,
                           int dev, bool q4, CUtensorMap* out) {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (auto& e : g_tc_ops)
        if (e.used && e.ws == ws && e.hidden == hidden && e.pairs == pairs && e.B == B && e.d == d && e.F == F &&
            e.dev == dev && e.q4 == q4) {
            memcpy(out, e.maps, sizeof e.maps);
            return MOE_OK;
        }
    TcOpEntry& e = g_tc_ops[g_tc_ops_next];
    g_tc_ops_next = (g_tc_ops_next + 1) % 32;
    e.used = false;
    e.ws = ws;
    e.hidden = hidden;
    e.pairs = pairs;
    e.B = B;
    e.d = d;
    e.F = F;
    e.dev = dev;
    e.q4 = q4;
    const uint32_t kb = (uint32_t)small_batch_blocks(d, F);
    // the whole batch of up to 64 tokens as one box (rows past B read as
    // zeros), as wide as the launch's stages
    const uint32_t nwb = B <= 64 ? (uint32_t)(B <= 16 ? 16 : (B + 15) & ~15) : 16u;
    const uint32_t kbw = B <= 16 && !q4 ? kb : (uint32_t)large_batch_blocks(d, F);
    if (!encode_3d(&e.maps[0], ws + L.xperm, d, pairs, 16, 1) || !encode_3d(&e.maps[1], ws + L.hbuf, F, pairs, 16, 1) ||
        !encode_3d(&e.maps[2], hidden, d, B, nwb, 1) || !encode_3d(&e.maps[3], hidden, d, B, nwb, kbw) ||
        !encode_3d(&e.maps[4], ws + L.hbuf, F, pairs, 16, kb))
        return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (operands)");
    e.used = true;
    memcpy(out, e.maps, sizeof e.maps);
    return MOE_OK;
}

int num_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace

namespace {
// Bound of every in-kernel wait (moe_set_wait_timeout_us), microseconds.
constexpr uint32_t kDefaultWaitUs = 2000000u;
std::atomic<uint32_t> g_wait_us{kDefaultWaitUs};
}  // namespace

namespace moe {
// SM cycles per microsecond assumed for the wait bound: the GB300's SM
// clock is at most 2.07 GHz, so a bound of t microseconds lasts at least
// about t microseconds.
long long wait_cycles_now() { return (long long)g_wait_us.load() * 2000LL; }

// Records `message` as this thread's last error and returns `status`.
moe_status report_error(moe_status status, const char* message) { return fail(status, "%s", message); }
}  // namespace moe

namespace {
// The mixed-precision expert descriptor (slot table and INT4 images).
moe_status check_mixed(const moe_mixed_experts* mixed, const Params& P, int d_ff) {
    if (P.dtype != MOE_DTYPE_BF16) return fail(MOE_ERR_ARG, "mixed experts need bf16 activations");
    if (P.d % 128 != 0 || d_ff % 128 != 0) return fail(MOE_ERR_ARG, "mixed experts need d and d_ff multiples of 128");
    if (!mixed->slot || !aligned(mixed->slot, 4)) return fail(MOE_ERR_ARG, "mixed->slot is NULL or misaligned");
    if (mixed->n_hot < 1 || mixed->n_cold < 0) return fail(MOE_ERR_ARG, "need n_hot >= 1 and n_cold >= 0");
    const void* q[] = {mixed->q_gate, mixed->q_up, mixed->q_down};
    for (const void* p : q)
        if ((mixed->n_cold > 0 && !p) || !aligned(p, 16))
            return fail(MOE_ERR_ARG, "an INT4 image is NULL or not 16-byte aligned");
    return MOE_OK;
}

moe_status expert_ffn_impl(const void* hidden, const void* w_gate, const void* w_up, const void* w_down,
                           const moe_mixed_experts* mixed, int32_t d_ff, const moe_route_params* params,
                           const moe_routing* routing, void* out, void* workspace, size_t workspace_bytes,
                           moe_stream_t stream) {
    Params P;
    moe_status st = resolve(params, P);
    if (st != MOE_OK) return st;
    if ((st = check_routing(routing, false, P.B)) != MOE_OK) return st;
    if (d_ff < 64 || d_ff % 64 != 0 || d_ff > 16384)
        return fail(MOE_ERR_ARG, "d_ff=%d must be a multiple of 64 in 64..16384", d_ff);
    const int n_hot = mixed ? mixed->n_hot : P.N;
    if (mixed && (st = check_mixed(mixed, P, d_ff)) != MOE_OK) return st;
    const void* req[] = {w_gate, w_up, w_down, hidden, out};
    for (int i = 0; i < 5; ++i) {
        if (!req[i] && (i < 3 || P.B > 0)) return fail(MOE_ERR_ARG, "a tensor pointer is NULL");
        if (!aligned(req[i], 16)) return fail(MOE_ERR_ARG, "a tensor pointer is not 16-byte aligned");
    }
    const WsLayout L = layout(P, d_ff);
    if ((st = check_ws(workspace, workspace_bytes, L.total)) != MOE_OK) return st;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    FfnArgs a{};
    a.x = hidden;
    a.T = routing->T;
    a.active = routing->active;
    a.counts = routing->counts;
    a.offsets = routing->offsets;
    a.perm = routing->perm;
    a.pos_of = reinterpret_cast<const int32_t*>(ws + L.pos_of);
    a.idx = routing->expert_idx;
    a.exinfo = reinterpret_cast<const uint32_t*>(ws + L.exinfo);
    a.w = routing->weights;
    a.hbuf = ws + L.hbuf;
    a.ybuf = reinterpret_cast<float*>(ws + L.ybuf);
    a.xperm = ws + L.xperm;
    a.out = out;
    a.hdone = reinterpret_cast<uint32_t*>(ws + L.hdone);
    a.nused = reinterpret_cast<const int32_t*>(ws + L.nused);
    a.ycnt = reinterpret_cast<uint32_t*>(ws + L.ycnt);
    a.hdr = reinterpret_cast<WsHeader*>(ws + L.header);
    a.uwords = a.hdr->union_words;
    const WsState wst = ws_state(workspace);
    // the early start serves OEA routing of batches of up to 64 tokens, right
    // after the routing call (counters fresh)
    a.epoch = P.B <= 64 && P.mode == MOE_MODE_OEA && wst.fresh ? wst.epoch : 0u;
    const int cset = counter_set(wst.routes > 0 ? wst.routes - 1 : 0u);
    a.hdone = reinterpret_cast<uint32_t*>(ws + L.hdone) + (size_t)cset * kHdoneSet;
    a.next_tile = &a.hdr->next_tile[cset];
    a.gathered = &a.hdr->gathered[cset];
    a.w_gate = w_gate;
    a.w_up = w_up;
    a.w_down = w_down;
    a.slot = mixed ? mixed->slot : nullptr;
    a.q_gate = mixed ? static_cast<const uint8_t*>(mixed->q_gate) : nullptr;
    a.q_up = mixed ? static_cast<const uint8_t*>(mixed->q_up) : nullptr;
    a.q_down = mixed ? static_cast<const uint8_t*>(mixed->q_down) : nullptr;
    a.n_hot = n_hot;
    a.n_cold = mixed ? mixed->n_cold : 0;
    a.B = P.B;
    a.N = P.N;
    a.d = P.d;
    a.F = d_ff;
    a.kslots = P.kslots;
    a.wait_cycles = wait_cycles_now();

    cudaError_t e;
    if (P.dtype == MOE_DTYPE_F32) {
        e = launch_ffn_f32(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "fp32 expert launch");
        return MOE_OK;
    }
    if (P.B == 0) return MOE_OK;   // nothing to compute or write
    if (!wst.fresh) {
        // another expert call used this counter set since the routing call
        // (or no routing call is recorded): zero it here
        if ((e = clear_counters(ws, L, cset, s)) != cudaSuccess)
            return cuda_fail(e, "clearing the expert kernel's counters");
    }
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int sms = num_sms();
    if (sms <= 0) return fail(MOE_ERR_CUDA, "cannot query the SM count");
    if (sms > kMaxGrid) sms = kMaxGrid;
    {   // the tcgen05 expert kernel (bf16 experts, and INT4 experts through its converter warps)
        CUtensorMap maps[15];
        bool fused = false, swap = false;
        CUtensorMap wm[9], om[5];
        if ((st = tc_expert_maps(w_gate, w_up, w_down, n_hot, d_ff, P.d, dev, wm, &fused, &swap)) != MOE_OK) return st;
        if ((st = tc_operand_maps(ws, L, hidden, P.B * P.kslots, P.B, P.d, d_ff, dev, a.n_cold > 0, om)) != MOE_OK)
            return st;
        maps[0] = wm[0];                       // gate/up 5D, or W_gate
        maps[1] = wm[0];                       // not read (the kernel takes W_gate's 8-row map from maps[0])
        maps[2] = wm[1];                       // W_up
        maps[3] = wm[2];                       // W_down
        maps[4] = om[0];                       // grouped hidden states
        maps[5] = om[1];                       // h
        maps[6] = om[2];                       // hidden states
        maps[7] = wm[3];                       // gate/up 5D, kb blocks wide
        maps[8] = wm[4];                       // W_down, kb blocks wide
        maps[9] = om[3];                       // hidden states, kb blocks wide
        maps[10] = om[4];                      // h, kb blocks wide
        maps[11] = wm[5];                      // gate/up 5D, 2 blocks wide (larger batches)
        maps[12] = wm[6];                      // W_down, 2 blocks wide (larger batches)
        maps[13] = wm[7];                      // W_up 8-row boxes, kb blocks wide (read when not fused)
        maps[14] = wm[8];                      // W_up 8-row boxes, 2 blocks wide (read when not fused)
        a.gu_fused = fused ? 1 : 0;
        a.gu_swap = swap ? 1 : 0;
        a.kbs = small_batch_blocks(P.d, d_ff);
        a.kbl = large_batch_blocks(P.d, d_ff);
        e = launch_ffn_tc(a, maps, sms, s);
        if (e != cudaSuccess) return cuda_fail(e, "expert kernel launch");
        experts_launched(workspace);
        return MOE_OK;
    }

}
}  // namespace

extern "C" {

int32_t moe_num_slots(const moe_route_params* params) {
    Params P;
    if (resolve(params, P) != MOE_OK) return -1;
    return P.kslots;
}

int32_t moe_layer_launches(const moe_route_params* params, int32_t d_ff) {
    Params P;
    if (resolve(params, P) != MOE_OK) return -1;
    if (d_ff <= 0 || d_ff % 64 != 0 || d_ff > 16384) return -1;
    int32_t n = route_fused_supported(P.dtype, P.B, P.N, P.kslots) ? 1 : (P.B > 0 ? 2 : 1);
    if (P.B > 0) n += P.dtype == MOE_DTYPE_F32 ? 3 : 1;
    return n;
}

size_t moe_workspace_bytes(const moe_route_params* params, int32_t d_ff) {
    Params P;
    if (resolve(params, P) != MOE_OK) return 0;
    if (d_ff < 0 || d_ff % 64 != 0 || d_ff > 16384) return 0;
    const WsLayout L = layout(P, d_ff);
    return d_ff == 0 ? L.hbuf : L.total;
}

moe_status moe_route(const void* hidden, const void* w_router, const float* router_bias,
                     const moe_route_params* params, const moe_routing* routing, void* workspace,
                     size_t workspace_bytes, moe_stream_t stream) {
    Params P;
    moe_status st = resolve(params, P);
    if (st != MOE_OK) return st;
    if ((st = check_routing(routing, true, P.B)) != MOE_OK) return st;
    if ((!hidden && P.B > 0) || !w_router) return fail(MOE_ERR_ARG, "hidden or w_router is NULL");
    if (!aligned(hidden, 16) || !aligned(w_router, 16)) return fail(MOE_ERR_ARG, "hidden/w_router not 16-byte aligned");
    if (router_bias && !aligned(router_bias, 4)) return fail(MOE_ERR_ARG, "router_bias not 4-byte aligned");
    const WsLayout L = layout(P, 0);
    if ((st = check_ws(workspace, workspace_bytes, L.hbuf)) != MOE_OK) return st;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    RouterArgs ra{};
    ra.x = hidden;
    ra.w = w_router;
    ra.bias = router_bias;
    ra.logits = routing->logits ? routing->logits : reinterpret_cast<float*>(ws + L.logits);
    ra.B = P.B;
    ra.N = P.N;
    ra.d = P.d;
    // batches of up to 32 tokens (bf16, N <= 128): scores and routing in one cluster launch
    const bool fused = route_fused_supported(P.dtype, P.B, P.N, P.kslots);
    cudaError_t e = fused ? cudaSuccess : launch_router(ra, P.dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "router launch");

    RouteArgs a{};
    a.logits = ra.logits;
    a.B = P.B;
    a.B_valid = P.B_valid;
    a.N = P.N;
    a.k = P.k;
    a.mode = P.mode;
    a.k0 = P.k0;
    a.maxP = P.maxP;
    a.kmax = P.kmax;
    a.kslots = P.kslots;
    a.p = P.p;
    a.idx = routing->expert_idx;
    a.w = routing->weights;
    a.T = routing->T;
    a.active = routing->active;
    a.counts = routing->counts;
    a.offsets = routing->offsets;
    a.perm = routing->perm;
    a.pos_of = reinterpret_cast<int32_t*>(ws + L.pos_of);
    a.n_base = routing->n_base;
    a.exinfo = reinterpret_cast<uint32_t*>(ws + L.exinfo);
    a.nused = reinterpret_cast<int32_t*>(ws + L.nused);
    a.ycnt = reinterpret_cast<uint32_t*>(ws + L.ycnt);
    a.rbd = (P.d + 127) / 128;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws + L.header);
    a.flags = &hdr->flags;
    const WsState wst = ws_state(workspace);
    if (!wst.known) {   // the counter sets' state is not recorded: zero both
        if ((e = clear_counters(ws, L, -1, s)) != cudaSuccess)
            return cuda_fail(e, "clearing the expert kernel's counters");
    }
    const int clr = 1 - counter_set(wst.routes);   // the set the previous expert call used
    a.clr_next = &hdr->next_tile[clr];
    a.clr_gathered = &hdr->gathered[clr];
    a.clr_hdone = reinterpret_cast<uint32_t*>(ws + L.hdone) + (size_t)clr * kHdoneSet;
    if (P.B <= 64 && P.mode == MOE_MODE_OEA) {   // it publishes S_base after phase 1 (and the cluster's union)
        a.uwords = hdr->union_words;
        a.epoch = next_epoch();
    }
    e = fused ? launch_route_fused(ra, a, s) : launch_route(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    routed(workspace, a.epoch);   // an expert call on this workspace now waits for it
    return MOE_OK;
}

moe_status moe_expert_ffn(const void* hidden, const void* w_gate, const void* w_up, const void* w_down,
                          int32_t d_ff, const moe_route_params* params, const moe_routing* routing, void* out,
                          void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return expert_ffn_impl(hidden, w_gate, w_up, w_down, nullptr, d_ff, params, routing, out, workspace,
                           workspace_bytes, stream);
}

moe_status moe_expert_ffn_mixed(const void* hidden, const void* w_gate, const void* w_up, const void* w_down,
                                const moe_mixed_experts* mixed, int32_t d_ff, const moe_route_params* params,
                                const moe_routing* routing, void* out, void* workspace, size_t workspace_bytes,
                                moe_stream_t stream) {
    if (!mixed) return fail(MOE_ERR_ARG, "mixed is NULL");
    return expert_ffn_impl(hidden, w_gate, w_up, w_down, mixed, d_ff, params, routing, out, workspace,
                           workspace_bytes, stream);
}

moe_status moe_decode_layer(const void* hidden, const void* w_router, const float* router_bias,
                            const void* w_gate, const void* w_up, const void* w_down, int32_t d_ff,
                            const moe_route_params* params, const moe_routing* routing, void* out,
                            void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    moe_status st = moe_route(hidden, w_router, router_bias, params, routing, workspace, workspace_bytes, stream);
    if (st != MOE_OK) return st;
    return moe_expert_ffn(hidden, w_gate, w_up, w_down, d_ff, params, routing, out, workspace, workspace_bytes,
                          stream);
}

moe_status moe_decode_layer_mixed(const void* hidden, const void* w_router, const float* router_bias,
                                  const void* w_gate, const void* w_up, const void* w_down,
                                  const moe_mixed_experts* mixed, int32_t d_ff, const moe_route_params* params,
                                  const moe_routing* routing, void* out, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream) {
    if (!mixed) return fail(MOE_ERR_ARG, "mixed is NULL");
    Params P;
    moe_status st = resolve(params, P);
    if (st != MOE_OK) return st;
    if ((st = check_mixed(mixed, P, d_ff)) != MOE_OK) return st;   // before the routing launches
    if ((st = moe_route(hidden, w_router, router_bias, params, routing, workspace, workspace_bytes, stream)) != MOE_OK)
        return st;
    return expert_ffn_impl(hidden, w_gate, w_up, w_down, mixed, d_ff, params, routing, out, workspace,
                           workspace_bytes, stream);
}

moe_status moe_device_status(void* workspace, moe_stream_t stream, uint32_t* flags) {
    if (!workspace || !aligned(workspace, 256)) return fail(MOE_ERR_WORKSPACE, "bad workspace");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t f = 0;
    WsHeader* h = static_cast<WsHeader*>(workspace);
    cudaError_t e = cudaMemcpyAsync(&f, &h->flags, sizeof f, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(&h->flags, 0, sizeof f, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device flags");
    if (flags) *flags = f;
    if (f) return fail(MOE_ERR_DEVICE_CHECK, "device flags 0x%x", f);
    return MOE_OK;
}

moe_status moe_synth_normal(void* dst, int32_t dtype, uint64_t n, uint64_t start, uint64_t seed, float scale,
                            moe_stream_t stream) {
    if (!dst && n) return fail(MOE_ERR_ARG, "dst is NULL");
    if (dtype != MOE_DTYPE_BF16 && dtype != MOE_DTYPE_F32) return fail(MOE_ERR_ARG, "unknown dtype %d", dtype);
    if (!std::isfinite(scale)) return fail(MOE_ERR_ARG, "scale is not finite");
    cudaError_t e = launch_synth(dst, dtype, n, start, seed, scale, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "synth launch");
    return MOE_OK;
}

moe_status moe_pack_int4(const void* w, int32_t rows, int32_t cols, int32_t rb, void* out, moe_stream_t stream) {
    if (!w || !out || !aligned(w, 16) || !aligned(out, 16))
        return fail(MOE_ERR_ARG, "w and out must be non-NULL and 16-byte aligned");
    if (rows < 1 || cols < 128 || cols % 128 != 0) return fail(MOE_ERR_ARG, "need rows >= 1 and cols a multiple of 128");
    if (rb < 8 || rb % 8 != 0 || rows % rb != 0)
        return fail(MOE_ERR_ARG, "rb=%d must be a multiple of 8 that divides rows=%d", rb, rows);
    cudaError_t e = launch_pack_int4(w, rows, cols, rb, out, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "INT4 pack launch");
    return MOE_OK;
}

moe_status moe_set_wait_timeout_us(uint32_t microseconds) {
    g_wait_us.store(microseconds ? microseconds : kDefaultWaitUs);
    return MOE_OK;
}

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_ARG: return "MOE_ERR_ARG";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    }
    return "unknown status";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
