// residency.cu -- the runtime that moves experts between bf16 and INT4
// versions while the layer keeps running (DynaExq page, sections 2-3).
//
//   * Stable handles (section 2.2 / 3.2): the slot table of the mixed
//     expert kernel.  slot[e] >= 0 resolves expert e to bf16 slot slot[e] of
//     the high-precision pool, slot[e] < 0 to its INT4 image -1 - slot[e];
//     the kernels read the table at every call, so a version switch needs
//     no change of kernel arguments.
//   * Pools (section 2.3): the caller's bf16 pool of n_hot expert slots (a
//     fixed-size free list of slots, so the budget can never be exceeded)
//     and INT4 images of all N experts, which stay resident: the low-
//     precision version every handle can fall back to.
//   * Hotness and selection (section 2.5 / 3.5): the routing's per-expert
//     counts are added up on the device at every call; every update_every
//     calls a snapshot is copied to the caller's pinned host buffer and the
//     accumulator cleared (on the compute stream, without waiting); once the
//     snapshot has arrived, S <- alpha S + (1 - alpha) c, and the best
//     outsider replaces the weakest member of the bf16 set while its score
//     exceeds the member's by more than the margin (hysteresis).
//   * Transitions (section 2.4 / 3.4): a demotion redirects the handle to
//     the INT4 image on the compute stream first (redirect, then reclaim);
//     the freed slot is refilled for the promoted expert by an asynchronous
//     copy of its bf16 weights from the caller's pinned host memory on a
//     migration stream, which waits for the redirect.  Its completion event
//     is polled, and only then is the handle pointed at the new slot
//     (publish after completion), so no kernel ever reads a partly copied
//     version.  At most max_inflight copies are in flight (backpressure);
//     the rest wait in a queue.  A new selection runs only when no
//     transition is pending.
#include <cstring>
#include <deque>
#include <new>
#include <vector>

#include "common.cuh"

namespace moe {
moe_status report_error(moe_status status, const char* message);
}

namespace {

__global__ void accumulate_counts_kernel(uint32_t* acc, const int32_t* counts, int N) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e < N) acc[e] += (uint32_t)counts[e];
}

__global__ void set_slot_kernel(int32_t* slot, int e, int32_t value) { slot[e] = value; }

enum State : int32_t { kLo = 0, kHi = 1, kPromoting = 2 };

struct Swap {
    int promote, demote;
};

struct Pending {
    int expert, slot;
    cudaEvent_t done;
};

}  // namespace

struct moe_residency {
    moe_residency_config cfg;
    std::vector<double> S;            // hotness
    std::vector<int32_t> state;       // per expert
    std::vector<int32_t> slot_of;     // expert -> bf16 slot, or -1
    std::vector<int32_t> owner;       // bf16 slot -> expert
    std::deque<Swap> queue;           // selected swaps not yet issued
    std::vector<Pending> inflight;    // promotions whose copy is in flight
    std::vector<cudaEvent_t> free_events;
    cudaStream_t mig = nullptr;
    cudaEvent_t snap_done = nullptr;
    bool snap_pending = false;
    uint64_t calls = 0, updates = 0, promotions = 0, demotions = 0;
};

namespace {

moe_status fail(moe_status s, const char* msg) { return moe::report_error(s, msg); }

moe_status cuda_fail(cudaError_t e) { return moe::report_error(MOE_ERR_CUDA, cudaGetErrorString(e)); }

cudaEvent_t take_event(moe_residency* r) {
    if (!r->free_events.empty()) {
        cudaEvent_t ev = r->free_events.back();
        r->free_events.pop_back();
        return ev;
    }
    cudaEvent_t ev = nullptr;
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    return ev;
}

// Points the handles of the promoted experts whose copies have completed at
// their new slots (on the compute stream).  `wait`: block on the copies.
moe_status publish(moe_residency* r, cudaStream_t s, bool wait) {
    for (size_t k = 0; k < r->inflight.size();) {
        Pending& p = r->inflight[k];
        cudaError_t q = wait ? cudaEventSynchronize(p.done) : cudaEventQuery(p.done);
        if (q == cudaErrorNotReady) {
            ++k;
            continue;
        }
        if (q != cudaSuccess) return cuda_fail(q);
        set_slot_kernel<<<1, 1, 0, s>>>(r->cfg.slot, p.expert, p.slot);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
        r->state[p.expert] = kHi;
        r->free_events.push_back(p.done);
        r->inflight[k] = r->inflight.back();
        r->inflight.pop_back();
    }
    return MOE_OK;
}

// Issues queued swaps while fewer than max_inflight copies are in flight.
moe_status issue(moe_residency* r, cudaStream_t s) {
    const moe_residency_config& c = r->cfg;
    const size_t mat = (size_t)c.d_ff * c.d * 2;   // bytes of one bf16 matrix
    while (!r->queue.empty() && (int)r->inflight.size() < c.max_inflight) {
        const Swap w = r->queue.front();
        const int slot = r->slot_of[w.demote];
        // redirect the demoted expert's handle to its INT4 image, then reclaim its slot
        set_slot_kernel<<<1, 1, 0, s>>>(c.slot, w.demote, -1 - w.demote);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
        cudaEvent_t redirected = take_event(r), done = take_event(r);
        if (!redirected || !done) return fail(MOE_ERR_CUDA, "cudaEventCreate failed");
        if ((e = cudaEventRecord(redirected, s)) != cudaSuccess) return cuda_fail(e);
        r->state[w.demote] = kLo;
        r->slot_of[w.demote] = -1;
        r->demotions++;
        // the promoted expert's bf16 weights into the slot, once no kernel can read the old contents
        if ((e = cudaStreamWaitEvent(r->mig, redirected, 0)) != cudaSuccess) return cuda_fail(e);
        const size_t src = (size_t)w.promote * mat, dst = (size_t)slot * mat;
        const unsigned char* hg = static_cast<const unsigned char*>(c.host_gate);
        const unsigned char* hu = static_cast<const unsigned char*>(c.host_up);
        const unsigned char* hd = static_cast<const unsigned char*>(c.host_down);
        if ((e = cudaMemcpyAsync(static_cast<unsigned char*>(c.hot_gate) + dst, hg + src, mat,
                                 cudaMemcpyHostToDevice, r->mig)) != cudaSuccess ||
            (e = cudaMemcpyAsync(static_cast<unsigned char*>(c.hot_up) + dst, hu + src, mat,
                                 cudaMemcpyHostToDevice, r->mig)) != cudaSuccess ||
            (e = cudaMemcpyAsync(static_cast<unsigned char*>(c.hot_down) + dst, hd + src, mat,
                                 cudaMemcpyHostToDevice, r->mig)) != cudaSuccess ||
            (e = cudaEventRecord(done, r->mig)) != cudaSuccess)
            return cuda_fail(e);
        r->free_events.push_back(redirected);   // reusable once recorded again later
        r->owner[slot] = w.promote;
        r->slot_of[w.promote] = slot;
        r->state[w.promote] = kPromoting;
        r->promotions++;
        r->inflight.push_back(Pending{w.promote, slot, done});
        r->queue.pop_front();
    }
    return MOE_OK;
}

}  // namespace

extern "C" {

int32_t moe_residency_select(const double* S, int32_t N, double margin, uint8_t* in_hot, int32_t* promote,
                             int32_t* demote) {
    if (!S || !in_hot || N < 1) return -1;
    int32_t n = 0;
    for (;;) {
        int o = -1, i = -1;
        double so = 0.0, si = 0.0;
        for (int e = 0; e < N; ++e) {
            if (in_hot[e]) {
                if (i < 0 || S[e] <= si) { i = e; si = S[e]; }   // weakest member, ties to the higher id
            } else if (o < 0 || S[e] > so) {
                o = e; so = S[e];                                // best outsider, ties to the lower id
            }
        }
        if (o < 0 || i < 0 || !(so > si + margin)) return n;
        in_hot[o] = 1;
        in_hot[i] = 0;
        if (promote) promote[n] = o;
        if (demote) demote[n] = i;
        ++n;
    }
}

moe_status moe_residency_create(const moe_residency_config* cfg, const int32_t* initial_hot,
                                moe_residency** out, moe_stream_t stream) {
    if (!cfg || !initial_hot || !out) return fail(MOE_ERR_ARG, "cfg, initial_hot and out are required");
    const moe_residency_config& c = *cfg;
    if (c.N < 2 || c.N > MOE_MAX_EXPERTS || c.n_hot < 1 || c.n_hot >= c.N || c.d < 128 || c.d % 128 ||
        c.d_ff < 128 || c.d_ff % 128)
        return fail(MOE_ERR_ARG, "need 1 <= n_hot < N <= 1024 and d, d_ff multiples of 128");
    if (!(c.alpha >= 0.0 && c.alpha < 1.0) || !(c.margin >= 0.0) || c.update_every < 1 || c.max_inflight < 1)
        return fail(MOE_ERR_ARG, "need 0 <= alpha < 1, margin >= 0, update_every >= 1, max_inflight >= 1");
    const void* req[] = {c.slot, c.counts_acc, c.snapshot, c.hot_gate, c.hot_up, c.hot_down,
                         c.host_gate, c.host_up, c.host_down};
    for (const void* p : req)
        if (!p) return fail(MOE_ERR_ARG, "a buffer of the configuration is NULL");
    std::vector<uint8_t> seen(c.N, 0);
    for (int k = 0; k < c.n_hot; ++k) {
        const int e = initial_hot[k];
        if (e < 0 || e >= c.N || seen[e]) return fail(MOE_ERR_ARG, "initial_hot must hold n_hot distinct experts");
        seen[e] = 1;
    }
    moe_residency* r = new (std::nothrow) moe_residency();
    if (!r) return fail(MOE_ERR_ARG, "out of host memory");
    r->cfg = c;
    r->S.assign(c.N, 0.0);
    r->state.assign(c.N, kLo);
    r->slot_of.assign(c.N, -1);
    r->owner.assign(c.n_hot, -1);
    std::vector<int32_t> table(c.N);
    for (int e = 0; e < c.N; ++e) table[e] = -1 - e;   // INT4 image of every expert
    for (int k = 0; k < c.n_hot; ++k) {
        const int e = initial_hot[k];
        r->state[e] = kHi;
        r->slot_of[e] = k;
        r->owner[k] = e;
        table[e] = k;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamCreateWithFlags(&r->mig, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->snap_done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c.slot, table.data(), sizeof(int32_t) * c.N, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(c.counts_acc, 0, sizeof(uint32_t) * c.N, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);   // the table above lives on this call's stack
    if (e != cudaSuccess) {
        moe_residency_destroy(r);
        return cuda_fail(e);
    }
    *out = r;
    return MOE_OK;
}

moe_status moe_residency_observe(moe_residency* r, const int32_t* counts, moe_stream_t stream) {
    if (!r || !counts) return fail(MOE_ERR_ARG, "residency and counts are required");
    const moe_residency_config& c = r->cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    accumulate_counts_kernel<<<(c.N + 127) / 128, 128, 0, s>>>(c.counts_acc, counts, c.N);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    r->calls++;
    moe_status st = publish(r, s, false);
    if (st != MOE_OK) return st;
    if (r->snap_pending) {   // a snapshot of the counts is on its way to the host
        e = cudaEventQuery(r->snap_done);
        if (e == cudaSuccess) {
            r->snap_pending = false;
            const uint32_t* cnt = static_cast<const uint32_t*>(c.snapshot);
            for (int k = 0; k < c.N; ++k) r->S[k] = c.alpha * r->S[k] + (1.0 - c.alpha) * (double)cnt[k];
            r->updates++;
            if (r->queue.empty() && r->inflight.empty()) {   // nothing pending: select
                std::vector<uint8_t> hot(c.N);
                for (int k = 0; k < c.N; ++k) hot[k] = r->state[k] != kLo;
                std::vector<int32_t> pro(c.N), dem(c.N);
                const int n = moe_residency_select(r->S.data(), c.N, c.margin, hot.data(), pro.data(), dem.data());
                for (int k = 0; k < n; ++k) r->queue.push_back(Swap{pro[k], dem[k]});
            }
        } else if (e != cudaErrorNotReady) {
            return cuda_fail(e);
        }
    }
    if ((st = issue(r, s)) != MOE_OK) return st;
    if (!r->snap_pending && r->calls % (uint64_t)c.update_every == 0) {
        // this interval's counts to the host, then a fresh interval
        e = cudaMemcpyAsync(c.snapshot, c.counts_acc, sizeof(uint32_t) * c.N, cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(c.counts_acc, 0, sizeof(uint32_t) * c.N, s);
        if (e == cudaSuccess) e = cudaEventRecord(r->snap_done, s);
        if (e != cudaSuccess) return cuda_fail(e);
        r->snap_pending = true;
    }
    return MOE_OK;
}

moe_status moe_residency_flush(moe_residency* r, moe_stream_t stream) {
    if (!r) return fail(MOE_ERR_ARG, "residency is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (;;) {
        moe_status st = publish(r, s, true);
        if (st != MOE_OK) return st;
        if (r->queue.empty()) break;
        if ((st = issue(r, s)) != MOE_OK) return st;
    }
    return MOE_OK;
}

moe_status moe_residency_query(const moe_residency* r, int32_t* state, double* scores, uint64_t* stats) {
    if (!r) return fail(MOE_ERR_ARG, "residency is NULL");
    const int N = r->cfg.N;
    if (state) memcpy(state, r->state.data(), sizeof(int32_t) * N);
    if (scores) memcpy(scores, r->S.data(), sizeof(double) * N);
    if (stats) {
        stats[0] = r->calls;
        stats[1] = r->updates;
        stats[2] = r->promotions;
        stats[3] = r->demotions;
        stats[4] = r->queue.size() + r->inflight.size();
    }
    return MOE_OK;
}

moe_status moe_residency_destroy(moe_residency* r) {
    if (!r) return MOE_OK;
    if (r->mig) cudaStreamSynchronize(r->mig);
    for (Pending& p : r->inflight) cudaEventDestroy(p.done);
    for (cudaEvent_t ev : r->free_events) cudaEventDestroy(ev);
    if (r->snap_done) cudaEventDestroy(r->snap_done);
    if (r->mig) cudaStreamDestroy(r->mig);
    delete r;
    return MOE_OK;
}

}  // extern "C"
