/*
 * moe_route.h -- C ABI of the routed-expert MoE layer for GB300 (sm_103a).
 *
 * One Mixture-of-Experts FFN layer that reads only the weights of the experts
 * each token is routed to:
 *
 *   router   logits = x . Wr^T + bias, fp32 softmax, top-k (lowest index first
 *            among equal probabilities), weights renormalised over the k
 *            (lilting.ch "observing the Qwen MoE router", section "hooking the
 *            router": gate -> softmax(precise) -> top-k indices)
 *   experts  for every routed (token t, slot r) with e = idx[t][r]:
 *              h = silu(Gate_e x_t) * (Up_e x_t),   o = Down_e h
 *            y[t] = sum_r w[t][r] * o_{t,r}, summed over r in a fixed order
 *            (Qiita "custom Metal gather_qmm": section 4, routing indices are an
 *            input of the kernel and unrouted experts are never fetched;
 *            section 7, gate/up share x, down takes each slot's own activation)
 *   weights  symmetric int8 or int4 codes with one scale per block of 32
 *            consecutive input elements ("sym8", same write-up, section 6),
 *            stacked as [E][rows][cols] with cols contiguous (the MLX
 *            (num_experts, output_dims, input_dims) layout of the lilting.ch
 *            article, section "warm-up vs mmap cache")
 *
 * Conventions for every entry point:
 *  - All array arguments are DEVICE pointers owned by the caller; descriptor
 *    structs are host memory read during the call only. The library allocates
 *    nothing and keeps no state between calls; it is reentrant as long as two
 *    concurrent calls do not share a workspace.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued asynchronously; outputs are valid once the stream reaches
 *    them. Two calls decide on the host and wait for their stream once:
 *    moe_cached_layer (for the router's probabilities) and
 *    moe_stage_prediction (for the predicted ids). The host-code calls
 *    (moe_replay, moe_cache_plan, moe_stage_plan) take host arrays only. Launches use programmatic dependent launch between the library's
 *    own kernels, so they can be captured into a CUDA graph.
 *  - Synchronous argument checks return MOE_ERR_INVALID_ARG / MOE_ERR_WORKSPACE
 *    / MOE_ERR_UNSUPPORTED before anything is launched. A failed launch returns
 *    MOE_ERR_CUDA. Problems found on the device (an expert id outside [0, E),
 *    a wait that ran out) are written to the workspace's status word -- the
 *    offending access is skipped, never performed -- and are read back by
 *    moe_check_status().
 *  - Workspace: `ws_bytes` >= moe_workspace_bytes(op, ...). It must be zeroed
 *    once before its first use (cudaMemset). Its header holds a launch sequence
 *    number that keeps growing from call to call; do not clear it afterwards.
 *  - Calls of up to 7 tokens run a persistent kernel (one launch per token)
 *    with one CTA per SM whose CTAs wait on one another (bounded waits, about
 *    30 ms by default, see moe_set_wait_limit). It needs every SM of the
 *    device: a kernel running at the same time on another stream can hold SMs
 *    until a wait runs out, in which case the call records
 *    MOE_ERR_DEVICE_TIMEOUT and its outputs are not valid. Do not run other
 *    kernels concurrently with these calls.
 *  - Alignment: every pointer 16-byte aligned; D and F multiples of 32, so
 *    every int8 row (D or F bytes) and int4 row (D/2 or F/2 bytes) starts on a
 *    16-byte boundary.
 *  - No exception crosses this boundary.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,    /* valid but not implemented combination */
    MOE_ERR_CUDA = 3,           /* a CUDA launch or copy failed */
    MOE_ERR_BAD_INDEX = 4,      /* device: expert id outside [0, E) (access skipped) */
    MOE_ERR_DEVICE_TIMEOUT = 5, /* device: a bounded wait ran out */
    MOE_ERR_WORKSPACE = 6       /* workspace missing or too small */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_F16 = 2 } moe_dtype_t;

typedef enum {
    MOE_Q_INT8_SYM_B32 = 0, /* int8 codes in [-127, 127], one scale per 32 codes */
    MOE_Q_INT4_SYM_B32 = 1  /* int4 codes in [-7, 7], two per byte: element 2j in the
                               low nibble of byte j, 2j+1 in the high nibble */
} moe_qfmt_t;

/* Router of one layer. W is [E][D] in w_dtype (MOE_F32 or MOE_BF16), D contiguous.
 * bias is [E] fp32 or NULL. norm_topk = 1 renormalises the k chosen
 * probabilities to sum to 1, 0 returns them as they are. */
typedef struct {
    int E, D, k;
    moe_dtype_t w_dtype;
    const void* W;
    const float* bias;
    int norm_topk;
} moe_router_t;

/* Experts of one layer, all [E][rows][cols] with cols contiguous:
 *   gate_q, up_q  [E][F][D]   (int4: [E][F][D/2] bytes)     gate_s, up_s [E][F][D/32]
 *   down_q        [E][D][F]   (int4: [E][D][F/2] bytes)     down_s       [E][D][F/32]
 * scales in s_dtype (MOE_F32 or MOE_F16). */
typedef struct {
    int E, D, F;
    moe_qfmt_t q;
    moe_dtype_t s_dtype;
    const void *gate_q, *gate_s, *up_q, *up_s, *down_q, *down_s;
} moe_experts_t;

/* Operation ids for moe_workspace_bytes. */
enum {
    MOE_OP_ROUTE = 0,
    MOE_OP_DECODE = 1,
    MOE_OP_LAYER = 2,         /* also moe_layer_stack (with T = 1) */
    MOE_OP_PREFILL = 3,
    MOE_OP_LAYER_RESIDENT = 4, /* moe_layer_resident */
    MOE_OP_SHARED = 5,         /* moe_shared_lora: D, F = the shared expert's d_ff; k, E unused (pass 1) */
    MOE_OP_PREROUTE = 6        /* moe_preroute: D, E, k, F = the head's hidden width H */
};

/*
 * Bytes of workspace an operation needs for T tokens (T >= 1). Returns 0 for an
 * invalid combination. For MOE_OP_DECODE / MOE_OP_LAYER with T >= 2 this covers
 * the grouped products (see moe_decode).
 */
size_t moe_workspace_bytes(int op, int T, int k, int E, int D, int F);

/*
 * Router: logits, fp32 softmax and top-k for T tokens.
 *   x      [T][D] in x_dtype (MOE_F32 or MOE_BF16)
 *   idx    [T][k] int32 out: expert ids, most probable first; equal fp32
 *          probabilities are ordered by lower expert id
 *   w      [T][k] fp32 out: routing weights (see norm_topk)
 *   probs  [T][E] fp32 out, or NULL: the full softmax
 * Source: lilting.ch "observing the Qwen MoE router", section "hooking the router".
 */
moe_status_t moe_route(const moe_router_t* router, const void* x, moe_dtype_t x_dtype, int T,
                       int32_t* idx, float* w, float* probs, void* workspace, size_t ws_bytes,
                       void* stream);

/*
 * Residency substitution (gist.science "Which expert misses are worth waiting
 * for?", method section). Slots are visited in rank order; a routed expert that
 * is not resident is kept (fetched) if it is the token's first choice or its
 * weight is >= threshold, otherwise it is replaced by the resident expert of
 * highest probability that is neither among the token's k routed experts nor
 * already used as a replacement (ties: lower id); the replacement keeps the
 * slot's weight.
 *   probs     [T][E] fp32 (from moe_route)   idx_in, w_in [T][k]   resident [E] uint8
 *   threshold 0.15 (the pages' rule); 0 = fetch every miss; +inf = first-choice rule
 *   idx_out, w_out [T][k] out (may alias idx_in / w_in)
 *   sub_flag  [T][k] uint8 out: 0 resident, 1 miss kept, 2 substituted,
 *             3 miss kept because no resident candidate was left
 *   sub_mass  [T] fp32 out: sum of the weights of substituted slots
 */
moe_status_t moe_substitute(int T, int E, int k, const float* probs, const int32_t* idx_in,
                            const float* w_in, const uint8_t* resident, float threshold,
                            int32_t* idx_out, float* w_out, uint8_t* sub_flag, float* sub_mass,
                            void* stream);

/*
 * Routed experts for T tokens given the routing (Qiita "custom Metal
 * gather_qmm", sections 4 and 7): only experts named in idx are read.
 *   x       [T][D] in x_dtype (MOE_F32 or MOE_BF16)
 *   idx, w  [T][k] routing (int32 ids in [0, E), fp32 weights)
 *   y       [T][D] fp32 out
 *   x_next  [T][D] in x_dtype out, or NULL: x + y rounded to x_dtype (residual)
 * T <= 7 runs one persistent single-token kernel per token (integer dot
 * products, fp32 accumulation; an expert shared by tokens is read once per
 * token). T >= 8 with D % 128 == 0, F % 64 == 0, D <= 8192 and E <= 1024 runs
 * the same grouped tensor-core products as moe_prefill, reading each distinct
 * expert once (fp16 operands with exact per-token power-of-two scaling, fp32
 * accumulation); other shapes run CUDA-core kernels. Ids outside [0, E) are skipped and reported by
 * moe_check_status as MOE_ERR_BAD_INDEX.
 */
moe_status_t moe_decode(const moe_experts_t* experts, const void* x, moe_dtype_t x_dtype, int T,
                        int k, const int32_t* idx, const float* w, float* y, void* x_next,
                        void* workspace, size_t ws_bytes, void* stream);

/*
 * One whole layer for T tokens: moe_route followed by moe_decode, with the
 * router's outputs handed to the expert kernels on the device.
 *   idx, w  [T][k] out    probs [T][E] out or NULL    y, x_next as moe_decode
 * T <= 7 runs one single-token layer launch per token (as moe_decode). Past
 * that (or for a shape the single-token kernel cannot run), with bf16 x and
 * router weights and E % 128 == 0, the logits come from the tensor cores (fp32
 * accumulation in another order than moe_route; probabilities may differ in
 * the last bits).
 */
moe_status_t moe_layer(const moe_router_t* router, const moe_experts_t* experts, const void* x,
                       moe_dtype_t x_dtype, int T, int32_t* idx, float* w, float* probs,
                       float* y, void* x_next, void* workspace, size_t ws_bytes, void* stream);

/*
 * One whole layer with residency substitution between the router and the
 * experts (gist.science "Which expert misses are worth waiting for?", method
 * section; the rule of moe_substitute): the router's top-k, then each missed
 * expert is kept if it is the token's first choice or its weight is >=
 * threshold, and otherwise replaced by the best resident expert; the experts
 * read are the substituted ones.
 *   resident   [E] uint8 (1 = resident)         threshold as moe_substitute
 *   idx, w     [T][k] out: the router's top-k and weights (weights are kept by
 *              a replacement)                   probs [T][E] out or NULL
 *   idx_used   [T][k] out: the experts read     sub_flag [T][k], sub_mass [T]
 *              out, as moe_substitute
 *   y, x_next  as moe_decode
 * T <= 7 runs the whole layer, substitution included, in one single-token
 * launch per token; more tokens run moe_layer's kernels with moe_substitute's
 * kernel between routing and experts. Workspace: MOE_OP_LAYER_RESIDENT.
 */
moe_status_t moe_layer_resident(const moe_router_t* router, const moe_experts_t* experts, const void* x,
                                moe_dtype_t x_dtype, int T, const uint8_t* resident, float threshold,
                                int32_t* idx, float* w, float* probs, int32_t* idx_used, uint8_t* sub_flag,
                                float* sub_mass, float* y, void* x_next, void* workspace, size_t ws_bytes,
                                void* stream);

/*
 * A stack of nlayers (<= 64) single-token layers in ONE launch of the
 * single-token layer kernel: layer l+1 starts only when every CTA has written
 * layer l's y and x_next. All layers share E, D, F, k, the quantisation, the
 * scale and router dtypes and norm_topk.
 *   routers, experts   host arrays [nlayers] of descriptors
 *   x        host array [nlayers] of device pointers, each [D] in x_dtype.
 *            chain = 1: layer 0 reads x[0] and layer l > 0 reads layer l-1's
 *            x + y (the residual stream; x[l > 0] is ignored). chain = 0: layer l
 *            reads x[l] (independent tokens), still after layer l-1 is done.
 *   idx, w   host arrays [nlayers] of device pointers to [k] outputs
 *   y        host array [nlayers] of device pointers to [D] fp32 outputs
 *   x_next   host array [nlayers] of device pointers to [D] outputs (x + y in
 *            x_dtype) or NULL entries; the whole array may be NULL (chained
 *            layers hand their output to the next layer through the workspace)
 * The host arrays are read during the call only. Workspace: MOE_OP_LAYER with
 * T = 1. Shapes the single-token kernel cannot run return MOE_ERR_UNSUPPORTED.
 */
moe_status_t moe_layer_stack(int nlayers, const moe_router_t* routers, const moe_experts_t* experts,
                             const void* const* x, moe_dtype_t x_dtype, int chain, int32_t* const* idx,
                             float* const* w, float* const* y, void* const* x_next, void* workspace,
                             size_t ws_bytes, void* stream);

/*
 * moe_layer_stack with residency substitution in every layer (gist.science
 * "Which expert misses are worth waiting for?", method section; the rule of
 * moe_substitute, decided in the kernel between the top-k and the experts).
 *   resident   host array [nlayers] of device pointers to [E] uint8 masks
 *   threshold  shared by the layers
 *   idx, w     as moe_layer_stack: the router's top-k and weights
 *   idx_used   host array [nlayers] of device pointers to [k] int32 outputs:
 *              the experts read
 *   sub_flag   host array [nlayers] of device pointers to [k] uint8 outputs
 *   sub_mass   host array [nlayers] of device pointers to one fp32 output
 * Every entry is required. Workspace: MOE_OP_LAYER with T = 1.
 */
moe_status_t moe_layer_stack_resident(int nlayers, const moe_router_t* routers, const moe_experts_t* experts,
                                      const void* const* x, moe_dtype_t x_dtype, int chain,
                                      const uint8_t* const* resident, float threshold, int32_t* const* idx,
                                      float* const* w, int32_t* const* idx_used, uint8_t* const* sub_flag,
                                      float* const* sub_mass, float* const* y, void* const* x_next,
                                      void* workspace, size_t ws_bytes, void* stream);

/*
 * Router-logit replay simulator (host code, no GPU): gist.science "Which
 * expert misses are worth waiting for?", method section (the C++ tool that
 * replays router outputs to compare policies, estimating the time per token
 * and the cache state; the fetch-all, 0.15 and first-choice rules; background
 * admission of substituted experts; frequency-based eviction).
 * Per token and layer: the top-k of the layer's probabilities (descending,
 * lower id on equal values; weights renormalised over the k in double); each
 * routed expert's frequency grows by one; slots in rank order: a resident
 * expert is a hit; a miss the policy fetches is a synchronous fetch and enters
 * the cache; another miss is substituted by the resident expert of highest
 * probability neither routed nor already chosen (lower id on ties), its weight
 * adds to the token's substituted mass and to the missed expert's accumulated
 * mass, and at admit_mass the expert enters the cache in the background (its
 * accumulation restarts); a miss with no candidate left is fetched. An expert
 * entering the cache evicts the resident expert of lowest frequency (lower id
 * on ties) that the token does not use in that layer; with none it is used
 * without entering. Time per token = sum over layers of t_layer_us +
 * (synchronous fetches) * t_fetch_us.
 *   probs        host [N][L][E] fp32: the router's probabilities per token and layer
 *   resident     host [L][E] uint8 in/out: the cache (its size per layer is kept)
 *   freq         host [L][E] int32 in/out: routing counts (zero for a fresh replay)
 *   acc          host [L][E] double in/out: accumulated substituted mass
 *   t_token_us, fetches, substituted, sub_mass, admissions
 *                host [N] out: estimated time, synchronous fetches, substituted
 *                slots, substituted mass and background admissions of each
 *                token, summed over its layers
 * Returns MOE_ERR_INVALID_ARG for bad sizes, pointers or policy values.
 */
typedef enum {
    MOE_POLICY_FETCH_ALL = 0,   /* every miss is fetched */
    MOE_POLICY_THRESHOLD = 1,   /* a miss is fetched if first choice or weight >= threshold */
    MOE_POLICY_FIRST_CHOICE = 2 /* only a first-choice miss is fetched */
} moe_policy_t;

typedef struct {
    moe_policy_t policy;
    float threshold;   /* MOE_POLICY_THRESHOLD (0.15 on the page) */
    float admit_mass;  /* background admission threshold (0.5 on the page); 0 = none */
    double t_layer_us; /* compute time of one layer */
    double t_fetch_us; /* time of one synchronous expert fetch */
} moe_replay_policy_t;

moe_status_t moe_replay(int N, int L, int E, int k, const float* probs, const moe_replay_policy_t* policy,
                        uint8_t* resident, int32_t* freq, double* acc, double* t_token_us, int32_t* fetches,
                        int32_t* substituted, double* sub_mass, int32_t* admissions);

/*
 * Prefill of T tokens: router, then the (token, slot) assignments grouped by
 * expert (histogram, exclusive scan, stable permutation), a grouped matrix
 * product per expert on the tensor cores, and the weighted un-permute.
 *   y          [T][D] fp32 out
 *   idx, w     [T][k] out, or NULL
 *   counts     [E] int32 out, or NULL: assignments per expert
 *   perm       [T*k] int32 out, or NULL: assignment id t*k+r at each grouped
 *              position (experts ascending, (t, r) order inside an expert)
 */
moe_status_t moe_prefill(const moe_router_t* router, const moe_experts_t* experts, const void* x,
                         moe_dtype_t x_dtype, int T, float* y, int32_t* idx, float* w,
                         int32_t* counts, int32_t* perm, void* workspace, size_t ws_bytes,
                         void* stream);

/* Shared expert of a MoE block with its recovery LoRA kept unmerged. Base
 * weights as one expert of moe_experts_t (no E dimension):
 *   gate_q, up_q [F][D] (int4: [F][D/2] bytes), gate_s, up_s [F][D/32]
 *   down_q       [D][F] (int4: [D][F/2] bytes), down_s       [D][F/32]
 * Adapters in lora_dtype (MOE_BF16 or MOE_F32), rank r (0 = none, A/B unused):
 *   gate_A, up_A [r][D], down_A [r][F]; gate_B, up_B [F][r], down_B [D][r]
 * lora_scale is alpha / r. */
typedef struct {
    int D, F, r;
    moe_qfmt_t q;
    moe_dtype_t s_dtype;
    const void *gate_q, *gate_s, *up_q, *up_s, *down_q, *down_s;
    moe_dtype_t lora_dtype;
    const void *gate_A, *gate_B, *up_A, *up_B, *down_A, *down_B;
    float lora_scale;
} moe_shared_t;

/*
 * Shared expert with an unmerged LoRA for T tokens (xyznot.com "The Other Half
 * of the Memory Wall", method section "unmerged adapter execution": the
 * quantised base is kept and the low-rank delta runs in parallel,
 * P(v) = dq(W) v + (alpha/r) B (A v), on the shared expert's projections):
 *   g = Gate(x_t), u = Up(x_t), h = silu(g) * u, o = Down(h)
 *   y[t] = o            (accumulate = 0)
 *   y[t] = y[t] + o     (accumulate = 1: adds the shared expert to a routed
 *                        output computed earlier on the same stream)
 *   x   [T][D] in x_dtype (MOE_F32 or MOE_BF16);  y [T][D] fp32
 * D and F multiples of 32, 0 <= r <= 64. Workspace: moe_workspace_bytes(
 * MOE_OP_SHARED, T, 1, 1, D, F). Four launches (two when r = 0).
 */
moe_status_t moe_shared_lora(const moe_shared_t* shared, const void* x, moe_dtype_t x_dtype, int T,
                             float* y, int accumulate, void* workspace, size_t ws_bytes, void* stream);

/* Prerouter head held by layer N that predicts layer N+1's routing. w_dtype
 * (MOE_BF16 or MOE_F32) is the type of fc1, fc2 and L:
 *   fc1 [H][D+2E], b1 [H] fp32 or NULL, fc2 [E][H], L [E][D+2E], bias [E] fp32 or NULL
 * E is the number of experts of layer N+1, k its routed experts per token;
 * norm_topk as in moe_router_t. */
typedef struct {
    int D, E, H, k;
    moe_dtype_t w_dtype;
    const void* fc1;
    const float* b1;
    const void* fc2;
    const void* L;
    const float* bias;
    int norm_topk;
} moe_prerouter_t;

/*
 * Prerouter for T tokens (xyznot.com "The Other Half of the Memory Wall",
 * method section "prerouter head architecture", glossary "prediction-as-
 * routing"). Input of the head: f = [x ; hot(cur) ; hot(prev)], hot(S)[e] = 1
 * when e is one of the ids S (a repeated id counts once, a negative id is an
 * absent entry, e.g. no previous token):
 *   logits = fc2 gelu(fc1 f + b1) + L f + bias,  gelu(z) = z/2 (1 + erf(z/sqrt 2))
 * then the router's fp32 softmax and top-k. The prediction is meant to be used
 * as the next layer's routing: idx/w go to moe_decode as they are.
 *   x          [T][D] in x_dtype (MOE_F32 or MOE_BF16)
 *   cur, prev  [T][k] int32: the current and previous tokens' routing ids
 *   idx, w     [T][k] out: predicted experts (most probable first, equal fp32
 *              probabilities by lower id) and their weights
 *   probs      [T][E] fp32 out, or NULL
 * D and H multiples of 32; E a multiple of 4, at most 1024; k <= 32. An id
 * >= E in cur/prev is recorded as MOE_ERR_BAD_INDEX (moe_check_status) and
 * skipped. Workspace: moe_workspace_bytes(MOE_OP_PREROUTE, T, k, E, D, H).
 */
moe_status_t moe_preroute(const moe_prerouter_t* head, const void* x, moe_dtype_t x_dtype, int T,
                          const int32_t* cur, const int32_t* prev, int32_t* idx, float* w, float* probs,
                          void* workspace, size_t ws_bytes, void* stream);

/* Expert cache of one layer. The experts live in host memory (all E, in the
 * layout of moe_experts_t); a device pool (moe_experts_t with E = S + k) holds
 * the S cached experts in slots 0..S-1, and slots S..S+k-1 are transient, for
 * a fetched miss that cannot enter the cache. The state is host memory owned
 * by the caller, and it is updated in place:
 *   slot_of   [E] int32: slot of expert e, or -1 (not cached)
 *   expert_of [S] int32: expert held by slot s (every slot holds one)
 *   freq      [E] int32: times the layer's router chose e
 *   acc       [E] double: routing weight substituted for e since its last admission */
typedef struct {
    int E, S, k;
    int32_t* slot_of;
    int32_t* expert_of;
    int32_t* freq;
    double* acc;
} moe_cache_t;

/* One token's decisions at one layer; every array is the caller's, [k] long.
 *   expert, slot  the expert serving each routed slot (a resident stand-in for
 *                 a substituted one) and the pool slot it is read from
 *   w             the routing weight of each routed slot
 *   flag          0 hit; 1 fetched and cached; 2 substituted; 4 fetched
 *                 into its transient slot (every cached expert in use; a
 *                 miss left without a stand-in always ends here, as stand-ins
 *                 and evictions come from the same cached experts); 3 is
 *                 not used
 *   fetch_*       the n_fetch synchronous fetches (expert, slot)
 *   admit_*       the n_admit background admissions (expert, slot)
 *   mass          routing weight served by stand-ins */
typedef struct {
    int32_t* expert;
    int32_t* slot;
    float* w;
    uint8_t* flag;
    int32_t *fetch_expert, *fetch_slot;
    int32_t *admit_expert, *admit_slot;
    int n_fetch, n_admit;
    double mass;
} moe_cache_step_t;

/*
 * Host code: the decisions of one token at one layer from the router's fp32
 * probabilities `probs` [E] (host), with the rules of moe_replay (gist.science
 * "Which expert misses are worth waiting for?", method section): top-k by
 * probability (lower id on equal values), weights over their sum; every
 * routed expert's frequency grows by one; in rank order a cached expert is a
 * hit, a miss the policy keeps is fetched (entering the cache in the slot of
 * the least frequent cached expert the token does not use, lower id on ties,
 * or its transient slot S + r when there is none), any other miss is served by
 * the cached expert of highest probability that is neither routed nor already
 * a stand-in (fetched when there is none) and its weight accumulates for the
 * missed expert, which is admitted (same eviction) once the accumulation
 * reaches policy->admit_mass (0 or +inf: never). policy->t_layer_us and
 * t_fetch_us are not used. The slot table must be consistent (checked).
 */
moe_status_t moe_cache_plan(moe_cache_t* cache, const float* probs, const moe_replay_policy_t* policy,
                            moe_cache_step_t* step);

/*
 * Copies n experts from host memory into pool slots: expert experts[i] of
 * `host` into slot slots[i] of `pool` (same D, F, formats), one
 * cudaMemcpyAsync per tensor, in stream order. Pinned host memory makes the
 * copies asynchronous (copy engines over NVLink-C2C on GB300); pageable
 * memory works but the host waits. experts/slots are host arrays.
 */
moe_status_t moe_pool_fetch(const moe_experts_t* host, const moe_experts_t* pool, int n,
                            const int32_t* experts, const int32_t* slots, void* stream);

/* Workspace bytes of moe_cached_layer (0 for an invalid shape); *host_bytes,
 * if not NULL, receives the size of its host scratch. */
size_t moe_cache_workspace_bytes(int E, int S, int k, int D, int F, size_t* host_bytes);

/*
 * One token (T = 1) through a layer whose experts are cached (the miss fetch
 * and background admission of the gist.science page, method section):
 *   1. the router on the GPU (moe_route), its probabilities copied to
 *      host_scratch, the stream waited for;
 *   2. moe_cache_plan on the host (`step` receives the decisions);
 *   3. the synchronous fetches into the pool on `stream`, after every earlier
 *      admission has landed;
 *   4. moe_decode of the served experts from the pool: y [T][D] fp32 (and
 *      x_next = x + y in x's dtype if x_next is not NULL);
 *   5. the admissions: on copy_stream, started once the work already on
 *      `stream` before the decode is done (ev_issued) and announced by
 *      ev_copied, which the next call waits for; with copy_stream NULL they
 *      follow the decode on `stream`.
 * host_scratch: host memory of the size moe_cache_workspace_bytes gives
 * (pinned for asynchronous copies), untouched by the caller until `stream` has
 * passed the call. ev_issued/ev_copied: cudaEvent_t (required with a
 * copy_stream). Workspace: moe_cache_workspace_bytes, zeroed once. The call
 * returns after step 2 has run, with steps 3-5 enqueued. A status other than
 * MOE_OK returned after step 2 leaves the slot table ahead of the pool: copy
 * expert_of[s] into every slot s with moe_pool_fetch before the next call.
 */
moe_status_t moe_cached_layer(const moe_router_t* router, const moe_experts_t* host, const moe_experts_t* pool,
                              moe_cache_t* cache, const moe_replay_policy_t* policy, const void* x,
                              moe_dtype_t x_dtype, float* y, void* x_next, moe_cache_step_t* step,
                              void* host_scratch, void* workspace, size_t ws_bytes, void* stream,
                              void* copy_stream, void* ev_issued, void* ev_copied);

/* Staged slot table: a pool of n_slots >= 2k expert slots (moe_experts_t with
 * E = n_slots) holding the experts predicted for the coming step. Host state
 * owned by the caller, updated in place:
 *   slot_of   [E] int32: slot of expert e, or -1
 *   expert_of [n_slots] int32: expert in slot s, or -1 (empty)
 *   in_flight [k] int32: the slots the previous step's decode reads (-1: none) */
typedef struct {
    int E, n_slots, k;
    int32_t* slot_of;
    int32_t* expert_of;
    int32_t* in_flight;
} moe_stage_t;

/*
 * Host code: the slots of one step's predicted experts ids [k] (host), for
 * the staged decode and the incremental sticky-slot stack of xyznot.com "The
 * Other Half of the Memory Wall" (glossary): an expert already staged keeps
 * its slot; any other takes the lowest slot that holds neither one of this
 * step's experts nor one the step in flight reads, and is listed as a load
 * (load_expert/load_slot, n_load of them; only changed slots are rewritten).
 * A repeated id maps to one slot. slot [k] receives each id's slot and becomes
 * the new in_flight.
 */
moe_status_t moe_stage_plan(moe_stage_t* stage, const int32_t* ids, int32_t* slot, int32_t* load_expert,
                            int32_t* load_slot, int* n_load);

/*
 * Stages a prediction (prediction-as-routing: the prerouter's ids for the
 * next step, pred_idx [k] on the device, e.g. moe_preroute's idx of one
 * token): copies the ids to host_scratch ([2k] int32, pinned for asynchronous
 * copies) and waits for `stream`; plans (moe_stage_plan: slot, loads); then,
 * on copy_stream (NULL: on `stream`), copies the slot ids to slot_idx [k]
 * (device) and the loaded experts from `host` into their `pool` slots, and
 * records ev_staged (a cudaEvent_t, required with a copy_stream). The decode
 * of that step is moe_decode on `pool` with idx = slot_idx and the predicted
 * weights, on a stream made to wait for ev_staged. Use two slot_idx buffers
 * in turn, as the decode of the step in flight still reads the other one.
 */
moe_status_t moe_stage_prediction(moe_stage_t* stage, const moe_experts_t* host, const moe_experts_t* pool,
                                  const int32_t* pred_idx, int32_t* slot_idx, int32_t* host_scratch, int32_t* slot,
                                  int32_t* load_expert, int32_t* load_slot, int* n_load, void* stream,
                                  void* copy_stream, void* ev_staged);

/*
 * moe_layer for ONE token (T = 1) without a workspace: no counterpart in the
 * pages; it exists for callers that cannot allocate device memory where they
 * run a layer (a frozen or captured memory pool, a host runtime whose
 * allocator is out of reach, an embedding that hands over only its input and
 * output buffers). Its scratch is a static device array inside the library of
 * 270,592 bytes (header + E tagged logits + k*F tagged activations),
 * held by every GPU that loads the library until the process exits. Limits:
 * E <= 1024 and k*F <= 32768 (beyond them: MOE_ERR_WORKSPACE); router weights
 * in the dtype of x; shapes the single-token kernel cannot run (k > 32 among
 * them) return MOE_ERR_UNSUPPORTED. Nothing is allocated: the first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) and caches
 * it, so make that first call before any stream capture. `stream` must belong
 * to the current device (MOE_ERR_INVALID_ARG otherwise). Every call on a device
 * shares the array, which keeps the previous call's contents (the status word
 * is cleared at the start of each call); calls whose execution overlaps on the
 * GPU, e.g. on two streams, race and must be avoided. Device-side conditions
 * (an expert id out of range, a wait that ran out because another kernel held
 * SMs) are not reported by this entry point, and outputs after such a
 * condition are not valid. An idx entry of -1 marks a slot the call could not
 * route (a wait that ran out before the routing was complete), so check that
 * every idx entry lies in [0, E) before using y; the converse does not hold, and
 * a caller that needs to detect every such condition uses moe_layer with a
 * workspace and moe_check_status. Arguments as moe_layer with T = 1.
 */
moe_status_t moe_layer_noalloc(const moe_router_t* router, const moe_experts_t* experts, const void* x,
                               moe_dtype_t x_dtype, int32_t* idx, float* w, float* probs, float* y,
                               void* x_next, void* stream);

/*
 * Waits for `stream`, reads the workspace's device status word, resets it to
 * zero and returns it (MOE_OK if no device-side problem was recorded).
 */
moe_status_t moe_check_status(void* workspace, void* stream);

/*
 * Sets the longest time, in clock64 cycles, that any bounded wait of a kernel
 * using this workspace spins before it records MOE_ERR_DEVICE_TIMEOUT and lets
 * the call finish (outputs then not valid); 0 restores the default (2^26
 * cycles, about 30 ms at 2 GHz). Enqueued on `stream`; it stays set for later
 * calls on the workspace. A short limit detects a stalled layer sooner; the
 * library's tests use it to make a wait run out on purpose.
 */
moe_status_t moe_set_wait_limit(void* workspace, unsigned long long cycles, void* stream);

/* Static description of a status code. */
const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ROUTE_H */
