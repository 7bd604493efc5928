// Expert cache with miss fetch and background admission (gist.science "Which
// expert misses are worth waiting for?", method section: a miss that is the
// router's first choice, or whose gate weight reaches 0.15, is worth waiting
// for and is fetched; any other miss is served by a resident stand-in; the
// gate mass substituted for an expert accumulates and admits it to the cache
// in the background at a threshold (0.5 on the page); eviction goes by
// routing frequency).
//
// The cache of one layer is a device pool of S + k expert slots in the layout
// of moe_experts_t: slots 0..S-1 hold the cached experts, slots S..S+k-1 are
// transient, for a fetched miss that cannot enter the cache because every
// cached expert is in use by the token. The full set of E experts stays in
// host memory (pinned, reached by the copy engines over NVLink-C2C on GB300).
//
//   moe_cache_plan    host: one token's decisions at one layer, on the router's
//                     fp32 probabilities, with the rules of moe_replay (same
//                     ranking, stand-in choice, frequency eviction, admission)
//                     plus the slot each routed slot is served from
//   moe_pool_fetch    copies experts from host memory into pool slots
//                     (one cudaMemcpyAsync per tensor of each expert)
//   moe_cached_layer  one token through one layer: router on the GPU, the
//                     probabilities to the host, the plan, the synchronous
//                     fetches, the decode of the served experts from the pool,
//                     and the admissions on a copy stream behind the decode
//
// Staged slot table (xyznot.com "The Other Half of the Memory Wall", glossary:
// "staged decode", "incremental sticky-slot stack"; method: "prediction-as-
// routing"): the prerouter's prediction for the next token is staged into a
// pool of fixed slots (at least 2k: double buffering) before that token runs,
// rewriting only the slots whose expert changed.
//   moe_stage_plan        host: slots of one step's predicted experts (a staged
//                         expert keeps its slot, any other takes the lowest
//                         slot held by neither this step's experts nor the
//                         step in flight) and the loads
//   moe_stage_prediction  the predicted ids to the host, the plan, the loads
//                         and the slot ids on a copy stream, an event when done
#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <vector>

#include "moe_route.h"

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxK = 32;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// The cached expert to evict: lowest frequency, lower id on ties, not in use
// (a scan of the S slots).
int victim(const moe_cache_t* c, const std::vector<uint8_t>& in_use) {
    int best = -1;
    for (int sl = 0; sl < c->S; sl++) {
        const int e = c->expert_of[sl];
        if (in_use[e]) continue;
        if (best < 0 || c->freq[e] < c->freq[best] || (c->freq[e] == c->freq[best] && e < best)) best = e;
    }
    return best;
}

// e takes the slot of a victim; returns the slot, or -1 when nothing can go.
int enter(moe_cache_t* c, const std::vector<uint8_t>& in_use, int e) {
    const int v = victim(c, in_use);
    if (v < 0) return -1;
    const int s = c->slot_of[v];
    c->slot_of[v] = -1;
    c->slot_of[e] = s;
    c->expert_of[s] = e;
    return s;
}

bool cache_ok(const moe_cache_t* c) {
    return c && c->E >= 1 && c->S >= 1 && c->S <= c->E && c->k >= 1 && c->k <= kMaxK && c->k <= c->E &&
           c->slot_of && c->expert_of && c->freq && c->acc;
}

bool policy_ok(const moe_replay_policy_t* p) {
    if (!p) return false;
    if (p->policy != MOE_POLICY_FETCH_ALL && p->policy != MOE_POLICY_THRESHOLD &&
        p->policy != MOE_POLICY_FIRST_CHOICE)
        return false;
    return p->threshold >= 0.f && p->admit_mass >= 0.f;
}

bool step_ok(const moe_cache_step_t* s) {
    return s && s->expert && s->slot && s->w && s->flag && s->fetch_expert && s->fetch_slot && s->admit_expert &&
           s->admit_slot;
}

// Bytes of one expert's matrix in a [E][rows][cols] tensor: 0 gate/up codes,
// 1 gate/up scales, 2 down codes, 3 down scales.
size_t expert_bytes(const moe_experts_t* x, int which) {
    const bool i8 = x->q == MOE_Q_INT8_SYM_B32;
    const size_t sb = x->s_dtype == MOE_F16 ? 2 : 4;
    const size_t D = (size_t)x->D, F = (size_t)x->F;
    switch (which) {
        case 0: return F * (i8 ? D : D / 2);
        case 1: return F * (D / 32) * sb;
        case 2: return D * (i8 ? F : F / 2);
        default: return D * (F / 32) * sb;
    }
}

bool experts_ok(const moe_experts_t* x) {
    return x && x->E >= 1 && x->D >= 32 && x->D % 32 == 0 && x->F >= 32 && x->F % 32 == 0 &&
           (x->q == MOE_Q_INT8_SYM_B32 || x->q == MOE_Q_INT4_SYM_B32) &&
           (x->s_dtype == MOE_F32 || x->s_dtype == MOE_F16) && x->gate_q && x->gate_s && x->up_q && x->up_s &&
           x->down_q && x->down_s;
}

bool same_format(const moe_experts_t* a, const moe_experts_t* b) {
    return a->D == b->D && a->F == b->F && a->q == b->q && a->s_dtype == b->s_dtype;
}

// The copies of expert e (host) into slot s (pool), in stream order.
cudaError_t copy_expert(const moe_experts_t* host, const moe_experts_t* pool, int e, int s, cudaStream_t st) {
    const void* src[6] = {host->gate_q, host->gate_s, host->up_q, host->up_s, host->down_q, host->down_s};
    const void* dst[6] = {pool->gate_q, pool->gate_s, pool->up_q, pool->up_s, pool->down_q, pool->down_s};
    const int kind[6] = {0, 1, 0, 1, 2, 3};
    for (int i = 0; i < 6; i++) {
        const size_t n = expert_bytes(host, kind[i]);
        cudaError_t err = cudaMemcpyAsync(static_cast<char*>(const_cast<void*>(dst[i])) + (size_t)s * n,
                                          static_cast<const char*>(src[i]) + (size_t)e * n, n,
                                          cudaMemcpyHostToDevice, st);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

struct CachedLayout {
    size_t route, decode, probs, idx, w, slot, slot_w, total;
};

CachedLayout cached_layout(int E, int S, int k, int D, int F) {
    CachedLayout L = {};
    const size_t rb = moe_workspace_bytes(MOE_OP_ROUTE, 1, k, E, D, F);
    const size_t db = moe_workspace_bytes(MOE_OP_DECODE, 1, k, S + k, D, F);
    if (!rb || !db) return L;
    size_t o = 0;
    L.route = o;
    o += up(rb);
    L.decode = o;
    o += up(db);
    L.probs = o;
    o += up(sizeof(float) * (size_t)E);
    L.idx = o;
    o += up(sizeof(int32_t) * (size_t)k);
    L.w = o;
    o += up(sizeof(float) * (size_t)k);
    L.slot = o;
    o += up(sizeof(int32_t) * (size_t)k);
    L.slot_w = o;
    o += up(sizeof(float) * (size_t)k);
    L.total = o;
    return L;
}

}  // namespace

extern "C" moe_status_t moe_cache_plan(moe_cache_t* c, const float* p, const moe_replay_policy_t* pol,
                                       moe_cache_step_t* st) {
    if (!cache_ok(c) || !p || !policy_ok(pol) || !step_ok(st)) return MOE_ERR_INVALID_ARG;
    const int E = c->E, S = c->S, k = c->k;
    // the slot table must map the S slots one to one onto S cached experts
    for (int e = 0; e < E; e++)
        if (c->slot_of[e] < -1 || c->slot_of[e] >= S || (c->slot_of[e] >= 0 && c->expert_of[c->slot_of[e]] != e))
            return MOE_ERR_INVALID_ARG;
    for (int sl = 0; sl < S; sl++)
        if (c->expert_of[sl] < 0 || c->expert_of[sl] >= E || c->slot_of[c->expert_of[sl]] != sl)
            return MOE_ERR_INVALID_ARG;
    const bool admit = pol->admit_mass > 0.f && std::isfinite(pol->admit_mass);
    const double beta = pol->admit_mass, thr = pol->threshold;

    std::vector<int> idx(k);
    std::vector<double> w(k);
    std::vector<uint8_t> taken(E, 0), in_use(E, 0);
    // 1. top-k in one pass over the experts in id order, keeping the best k
    //    sorted by probability; an expert enters or moves up only past strictly
    //    smaller values, so equal values keep the lower id first
    int n = 0;
    float kth = 0.f;  // the k-th best so far, once k are kept
    for (int e = 0; e < E; e++) {
        const float v = p[e];
        if (n == k && !(v > kth)) continue;
        int pos = n < k ? n++ : k - 1;
        while (pos > 0 && v > p[idx[pos - 1]]) {
            idx[pos] = idx[pos - 1];
            pos--;
        }
        idx[pos] = e;
        if (n == k) kth = p[idx[k - 1]];
    }
    for (int r = 0; r < k; r++) taken[idx[r]] = 1;
    double sum = 0.0;
    for (int r = 0; r < k; r++) sum += (double)p[idx[r]];
    for (int r = 0; r < k; r++) w[r] = sum > 0.0 ? (double)p[idx[r]] / sum : 0.0;
    // 2. frequencies; the routed experts are in use
    for (int r = 0; r < k; r++) {
        c->freq[idx[r]] += 1;
        in_use[idx[r]] = 1;
    }
    // 3. the slots in rank order
    st->mass = 0.0;
    st->n_fetch = 0;
    st->n_admit = 0;
    for (int r = 0; r < k; r++) {
        const int e = idx[r];
        st->w[r] = (float)w[r];
        st->expert[r] = e;
        if (c->slot_of[e] >= 0) {
            st->slot[r] = c->slot_of[e];
            st->flag[r] = 0;
            continue;
        }
        bool want;
        if (pol->policy == MOE_POLICY_FETCH_ALL) want = true;
        else if (pol->policy == MOE_POLICY_FIRST_CHOICE) want = r == 0;
        else want = r == 0 || w[r] >= thr;
        int rep = -1;  // the stand-in: the most probable cached expert not taken, lower id on ties
        if (!want)
            for (int sl = 0; sl < S; sl++) {
                const int cand = c->expert_of[sl];
                if (taken[cand]) continue;
                if (rep < 0 || p[cand] > p[rep] || (p[cand] == p[rep] && cand < rep)) rep = cand;
            }
        if (rep < 0) {  // fetched: into a victim's slot, else into the transient slot S + r
            const int s = enter(c, in_use, e);
            st->slot[r] = s >= 0 ? s : S + r;
            st->flag[r] = s < 0 ? 4 : 1;
            st->fetch_expert[st->n_fetch] = e;
            st->fetch_slot[st->n_fetch] = st->slot[r];
            st->n_fetch++;
            continue;
        }
        taken[rep] = 1;
        in_use[rep] = 1;
        st->expert[r] = rep;
        st->slot[r] = c->slot_of[rep];
        st->flag[r] = 2;
        st->mass += w[r];
        c->acc[e] += w[r];
        if (admit && c->acc[e] >= beta && c->slot_of[e] < 0) {
            const int s = enter(c, in_use, e);
            if (s >= 0) {
                st->admit_expert[st->n_admit] = e;
                st->admit_slot[st->n_admit] = s;
                st->n_admit++;
                c->acc[e] = 0.0;
            }
        }
    }
    return MOE_OK;
}

extern "C" moe_status_t moe_pool_fetch(const moe_experts_t* host, const moe_experts_t* pool, int n,
                                       const int32_t* experts, const int32_t* slots, void* stream) {
    if (!experts_ok(host) || !experts_ok(pool) || !same_format(host, pool) || n < 0) return MOE_ERR_INVALID_ARG;
    if (n > 0 && (!experts || !slots)) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < n; i++)
        if (experts[i] < 0 || experts[i] >= host->E || slots[i] < 0 || slots[i] >= pool->E) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < n; i++)
        if (copy_expert(host, pool, experts[i], slots[i], static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return MOE_ERR_CUDA;
    return MOE_OK;
}

extern "C" size_t moe_cache_workspace_bytes(int E, int S, int k, int D, int F, size_t* host_bytes) {
    if (E < 1 || S < 1 || S > E || k < 1 || k > kMaxK || k > E) return 0;
    const CachedLayout L = cached_layout(E, S, k, D, F);
    if (host_bytes) *host_bytes = L.total ? sizeof(float) * (size_t)E + 2 * sizeof(int32_t) * (size_t)k : 0;
    return L.total;
}

extern "C" moe_status_t moe_cached_layer(const moe_router_t* router, const moe_experts_t* host,
                                         const moe_experts_t* pool, moe_cache_t* cache,
                                         const moe_replay_policy_t* policy, const void* x, moe_dtype_t x_dtype,
                                         float* y, void* x_next, moe_cache_step_t* step, void* host_scratch,
                                         void* workspace, size_t ws_bytes, void* stream, void* copy_stream,
                                         void* ev_issued, void* ev_copied) {
    if (!router || !cache_ok(cache) || !policy_ok(policy) || !step_ok(step) || !host_scratch) return MOE_ERR_INVALID_ARG;
    if (!experts_ok(host) || !experts_ok(pool) || !same_format(host, pool)) return MOE_ERR_INVALID_ARG;
    const int E = cache->E, S = cache->S, k = cache->k;
    if (router->E != E || router->k != k || router->D != host->D || host->E != E || pool->E != S + k)
        return MOE_ERR_INVALID_ARG;
    if (copy_stream && (!ev_issued || !ev_copied)) return MOE_ERR_INVALID_ARG;
    const CachedLayout L = cached_layout(E, S, k, host->D, host->F);
    if (!L.total) return MOE_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & (kAlign - 1)) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* h_probs = static_cast<float*>(host_scratch);
    int32_t* h_slot = reinterpret_cast<int32_t*>(h_probs + E);
    float* h_w = reinterpret_cast<float*>(h_slot + k);

    // router on the GPU; its fp32 probabilities decide on the host
    float* d_probs = reinterpret_cast<float*>(ws + L.probs);
    moe_status_t stt = moe_route(router, x, x_dtype, 1, reinterpret_cast<int32_t*>(ws + L.idx),
                                 reinterpret_cast<float*>(ws + L.w), d_probs, ws + L.route, L.decode - L.route, stream);
    if (stt != MOE_OK) return stt;
    if (cudaMemcpyAsync(h_probs, d_probs, sizeof(float) * E, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    stt = moe_check_status(ws + L.route, stream);  // waits for the stream
    if (stt != MOE_OK) return stt;
    stt = moe_cache_plan(cache, h_probs, policy, step);
    if (stt != MOE_OK) return stt;
    // earlier admissions land before any fetch or decode of this call
    if (copy_stream && cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(ev_copied), 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    stt = moe_pool_fetch(host, pool, step->n_fetch, step->fetch_expert, step->fetch_slot, stream);
    if (stt != MOE_OK) return stt;
    for (int r = 0; r < k; r++) {
        h_slot[r] = step->slot[r];
        h_w[r] = step->w[r];
    }
    int32_t* d_slot = reinterpret_cast<int32_t*>(ws + L.slot);
    float* d_w = reinterpret_cast<float*>(ws + L.slot_w);
    if (cudaMemcpyAsync(d_slot, h_slot, sizeof(int32_t) * k, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(d_w, h_w, sizeof(float) * k, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    // admissions: their slots are used by no work of this token, and every
    // earlier use of them is already on the stream
    if (step->n_admit > 0 && copy_stream) {
        cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
        if (cudaEventRecord(static_cast<cudaEvent_t>(ev_issued), s) != cudaSuccess ||
            cudaStreamWaitEvent(cs, static_cast<cudaEvent_t>(ev_issued), 0) != cudaSuccess)
            return MOE_ERR_CUDA;
        stt = moe_pool_fetch(host, pool, step->n_admit, step->admit_expert, step->admit_slot, copy_stream);
        if (stt != MOE_OK) return stt;
        if (cudaEventRecord(static_cast<cudaEvent_t>(ev_copied), cs) != cudaSuccess) return MOE_ERR_CUDA;
    }
    stt = moe_decode(pool, x, x_dtype, 1, k, d_slot, d_w, y, x_next, ws + L.decode, L.probs - L.decode, stream);
    if (stt != MOE_OK) return stt;
    if (step->n_admit > 0 && !copy_stream)
        return moe_pool_fetch(host, pool, step->n_admit, step->admit_expert, step->admit_slot, stream);
    return MOE_OK;
}

namespace {

bool stage_ok(const moe_stage_t* st) {
    return st && st->E >= 1 && st->k >= 1 && st->k <= kMaxK && st->n_slots >= 2 * st->k && st->slot_of &&
           st->expert_of && st->in_flight;
}

}  // namespace

extern "C" moe_status_t moe_stage_plan(moe_stage_t* st, const int32_t* ids, int32_t* slot, int32_t* load_expert,
                                       int32_t* load_slot, int* n_load) {
    if (!stage_ok(st) || !ids || !slot || !load_expert || !load_slot || !n_load) return MOE_ERR_INVALID_ARG;
    const int E = st->E, NS = st->n_slots, k = st->k;
    for (int r = 0; r < k; r++)
        if (ids[r] < 0 || ids[r] >= E || st->in_flight[r] < -1 || st->in_flight[r] >= NS) return MOE_ERR_INVALID_ARG;
    // the slot table must be a consistent partial map
    for (int e = 0; e < E; e++)
        if (st->slot_of[e] < -1 || st->slot_of[e] >= NS || (st->slot_of[e] >= 0 && st->expert_of[st->slot_of[e]] != e))
            return MOE_ERR_INVALID_ARG;
    for (int sl = 0; sl < NS; sl++)
        if (st->expert_of[sl] < -1 || st->expert_of[sl] >= E ||
            (st->expert_of[sl] >= 0 && st->slot_of[st->expert_of[sl]] != sl))
            return MOE_ERR_INVALID_ARG;
    // slots this step may not take: the in-flight step's, and those of this
    // step's experts that are staged already
    std::vector<uint8_t> locked(NS, 0);
    for (int r = 0; r < k; r++) {
        if (st->in_flight[r] >= 0) locked[st->in_flight[r]] = 1;
        if (st->slot_of[ids[r]] >= 0) locked[st->slot_of[ids[r]]] = 1;
    }
    int n = 0, next_free = 0;
    for (int r = 0; r < k; r++) {
        const int e = ids[r];
        if (st->slot_of[e] >= 0) {  // staged (possibly by an earlier slot of this step)
            slot[r] = st->slot_of[e];
            continue;
        }
        while (next_free < NS && locked[next_free]) next_free++;
        if (next_free == NS) return MOE_ERR_INVALID_ARG;  // cannot happen with 2k slots
        const int s = next_free;
        const int old = st->expert_of[s];
        if (old >= 0) st->slot_of[old] = -1;
        st->expert_of[s] = e;
        st->slot_of[e] = s;
        locked[s] = 1;
        slot[r] = s;
        load_expert[n] = e;
        load_slot[n] = s;
        n++;
    }
    for (int r = 0; r < k; r++) st->in_flight[r] = slot[r];
    *n_load = n;
    return MOE_OK;
}

extern "C" moe_status_t moe_stage_prediction(moe_stage_t* st, const moe_experts_t* host, const moe_experts_t* pool,
                                             const int32_t* pred_idx, int32_t* slot_idx, int32_t* host_scratch,
                                             int32_t* slot, int32_t* load_expert, int32_t* load_slot, int* n_load,
                                             void* stream, void* copy_stream, void* ev_staged) {
    if (!stage_ok(st) || !pred_idx || !slot_idx || !host_scratch || !slot || !load_expert || !load_slot || !n_load)
        return MOE_ERR_INVALID_ARG;
    if (!experts_ok(host) || !experts_ok(pool) || !same_format(host, pool) || host->E != st->E ||
        pool->E != st->n_slots)
        return MOE_ERR_INVALID_ARG;
    if (copy_stream && !ev_staged) return MOE_ERR_INVALID_ARG;
    const int k = st->k;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStream_t cs = copy_stream ? static_cast<cudaStream_t>(copy_stream) : s;
    int32_t* h_ids = host_scratch;
    int32_t* h_slot = host_scratch + k;
    // the prediction, and every earlier decode that read a slot, are done after this
    if (cudaMemcpyAsync(h_ids, pred_idx, sizeof(int32_t) * k, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    moe_status_t stt = moe_stage_plan(st, h_ids, slot, load_expert, load_slot, n_load);
    if (stt != MOE_OK) return stt;
    for (int r = 0; r < k; r++) h_slot[r] = slot[r];
    if (cudaMemcpyAsync(slot_idx, h_slot, sizeof(int32_t) * k, cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return MOE_ERR_CUDA;
    stt = moe_pool_fetch(host, pool, *n_load, load_expert, load_slot, copy_stream ? copy_stream : stream);
    if (stt != MOE_OK) return stt;
    if (copy_stream && cudaEventRecord(static_cast<cudaEvent_t>(ev_staged), cs) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}
