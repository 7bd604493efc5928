// Router-logit replay simulator (host code).
//
// gist.science "Which expert misses are worth waiting for?", method section:
// a C++ tool replays router outputs to compare fetch/substitution policies
// quickly, estimating the time per token and the state of the expert cache.
// The policies are the ones the page tests: fetch every miss, the 0.15 rule
// (fetch a miss that is the first choice or has gate weight >= 0.15, else
// substitute it), the first-choice rule, and background admission (the gate
// mass a substituted expert accumulates admits it to the cache at a threshold,
// 0.5 on the page), with frequency-based eviction.
//
// Per token, per layer, in layer order:
//   1. top-k of the layer's fp32 probabilities (descending, lower id on equal
//      values); weights w_r = p_r / sum of the k (double, slot order);
//   2. each routed expert's routing count (its frequency) grows by one;
//   3. slots in rank order: a resident expert is a hit; a miss the policy
//      fetches is a synchronous fetch and enters the cache; any other miss is
//      substituted by the resident expert of highest probability that is
//      neither routed nor already chosen (lower id on equal values), its weight
//      adds to the token's substituted mass and to the missed expert's
//      accumulated mass, and when that reaches the admission threshold the
//      expert enters the cache in the background (its accumulation restarts);
//      a miss with no resident candidate is fetched;
//   4. time += t_layer + fetches * t_fetch.
// An expert entering the cache evicts the resident expert with the lowest
// frequency (lower id on equal values) among those the token does not use in
// this layer (routed or chosen as a replacement); with no such expert it is
// used without entering. The state (residency, frequencies, accumulated mass)
// is the caller's, so a replay can be resumed.
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <vector>

#include "moe_route.h"

namespace {

// One layer's cache: the caller's residency flags, frequencies and
// accumulated mass, plus the list of resident experts (kept in step with the
// flags, in no particular order) so that stand-in and eviction searches visit
// the residents only.
struct LayerState {
    uint8_t* res;
    int32_t* freq;
    double* acc;
    std::vector<int> list;  // resident experts
    std::vector<int> pos;   // position of e in list, or -1
};

// The resident expert to evict: lowest frequency, lower id on ties, not in use.
int victim(const LayerState& s, const std::vector<uint8_t>& in_use) {
    int best = -1;
    for (const int e : s.list) {
        if (in_use[e]) continue;
        if (best < 0 || s.freq[e] < s.freq[best] || (s.freq[e] == s.freq[best] && e < best)) best = e;
    }
    return best;
}

// e enters the cache (evicting a victim); returns false when nothing can go.
bool enter(LayerState& s, const std::vector<uint8_t>& in_use, int e) {
    const int v = victim(s, in_use);
    if (v < 0) return false;
    const int at = s.pos[v];
    s.list[at] = e;
    s.pos[e] = at;
    s.pos[v] = -1;
    s.res[v] = 0;
    s.res[e] = 1;
    return true;
}

}  // namespace

extern "C" moe_status_t moe_replay(int N, int L, int E, int k, const float* probs, const moe_replay_policy_t* pol,
                                   uint8_t* resident, int32_t* freq, double* acc, double* t_token_us,
                                   int32_t* fetches, int32_t* substituted, double* sub_mass,
                                   int32_t* admissions) {
    if (N < 0 || L < 1 || E < 1 || k < 1 || k > E || !pol || !resident || !freq || !acc) return MOE_ERR_INVALID_ARG;
    if (N > 0 && (!probs || !t_token_us || !fetches || !substituted || !sub_mass || !admissions))
        return MOE_ERR_INVALID_ARG;
    if (pol->policy != MOE_POLICY_FETCH_ALL && pol->policy != MOE_POLICY_THRESHOLD &&
        pol->policy != MOE_POLICY_FIRST_CHOICE)
        return MOE_ERR_INVALID_ARG;
    if (!(pol->threshold >= 0.f) || !(pol->admit_mass >= 0.f) || !(pol->t_layer_us >= 0.0) ||
        !(pol->t_fetch_us >= 0.0))
        return MOE_ERR_INVALID_ARG;
    const bool admit = pol->admit_mass > 0.f && std::isfinite(pol->admit_mass);
    const double beta = pol->admit_mass, thr = pol->threshold;

    std::vector<LayerState> layers(L);
    for (int l = 0; l < L; l++) {
        LayerState& s = layers[l];
        s.res = resident + (size_t)l * E;
        s.freq = freq + (size_t)l * E;
        s.acc = acc + (size_t)l * E;
        s.pos.assign(E, -1);
        for (int e = 0; e < E; e++)
            if (s.res[e]) {
                s.pos[e] = (int)s.list.size();
                s.list.push_back(e);
            }
    }
    std::vector<int> idx(k), used;
    std::vector<double> w(k);
    std::vector<uint8_t> taken(E, 0), in_use(E, 0);
    used.reserve(2 * (size_t)k);
    for (int t = 0; t < N; t++) {
        double time = 0.0, mass = 0.0;
        int nf = 0, ns = 0, na = 0;
        for (int l = 0; l < L; l++) {
            const float* p = probs + ((size_t)t * L + l) * E;
            LayerState& s = layers[l];
            // 1. top-k in one pass over the experts in id order, keeping the
            //    best k sorted by probability; an expert enters or moves up
            //    only past strictly smaller values, so equal values keep the
            //    lower id first
            int n = 0;
            float kth = 0.f;  // the k-th best so far, once k are kept
            for (int e = 0; e < E; e++) {
                const float v = p[e];
                if (n == k && !(v > kth)) continue;
                int at = n < k ? n++ : k - 1;
                while (at > 0 && v > p[idx[at - 1]]) {
                    idx[at] = idx[at - 1];
                    at--;
                }
                idx[at] = e;
                if (n == k) kth = p[idx[k - 1]];
            }
            double sum = 0.0;
            for (int r = 0; r < k; r++) sum += (double)p[idx[r]];
            for (int r = 0; r < k; r++) w[r] = sum > 0.0 ? (double)p[idx[r]] / sum : 0.0;
            // 2. frequencies; the routed experts are taken and in use (the
            //    flags set here are cleared again at the end of the layer)
            used.clear();
            for (int r = 0; r < k; r++) {
                s.freq[idx[r]] += 1;
                taken[idx[r]] = 1;
                in_use[idx[r]] = 1;
                used.push_back(idx[r]);
            }
            // 3. the slots in rank order
            int lf = 0;
            for (int r = 0; r < k; r++) {
                const int e = idx[r];
                if (s.res[e]) continue;
                bool fetch;
                if (pol->policy == MOE_POLICY_FETCH_ALL) fetch = true;
                else if (pol->policy == MOE_POLICY_FIRST_CHOICE) fetch = r == 0;
                else fetch = r == 0 || w[r] >= thr;
                int rep = -1;  // the stand-in: the most probable resident not taken, lower id on ties
                if (!fetch) {
                    for (const int c : s.list)
                        if (!taken[c] && (rep < 0 || p[c] > p[rep] || (p[c] == p[rep] && c < rep))) rep = c;
                    if (rep < 0) fetch = true;  // no resident candidate left: the miss is kept
                }
                if (fetch) {
                    lf++;
                    enter(s, in_use, e);
                    continue;
                }
                taken[rep] = 1;
                in_use[rep] = 1;
                used.push_back(rep);
                ns++;
                mass += w[r];
                s.acc[e] += w[r];
                if (admit && s.acc[e] >= beta && !s.res[e]) {
                    if (enter(s, in_use, e)) {
                        na++;
                        s.acc[e] = 0.0;
                    }
                }
            }
            for (const int e : used) taken[e] = in_use[e] = 0;
            nf += lf;
            time += pol->t_layer_us + lf * pol->t_fetch_us;
        }
        t_token_us[t] = time;
        fetches[t] = nf;
        substituted[t] = ns;
        sub_mass[t] = mass;
        admissions[t] = na;
    }
    return MOE_OK;
}
