// Test scaffolding: plain double-precision stand-ins for the library calls
// csrc/cache.cu composes (moe_route, moe_decode, moe_check_status,
// moe_workspace_bytes), so that cache.cu's own logic can run on the CPU. They
// compute the definitions directly: router logits, softmax; dequantised
// SwiGLU experts combined with the given weights.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include "moe_route.h"
static float bf(uint16_t b) { uint32_t u = (uint32_t)b << 16; float f; std::memcpy(&f, &u, 4); return f; }
static float hf(uint16_t h) {
    uint32_t s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    float v = e == 0 ? std::ldexp((float)m, -24) : std::ldexp((float)(m | 1024), (int)e - 25);
    return s ? -v : v;
}
static double act(const void* x, moe_dtype_t t, size_t i) {
    return t == MOE_BF16 ? bf(((const uint16_t*)x)[i]) : ((const float*)x)[i];
}
extern "C" size_t moe_workspace_bytes(int, int, int k, int E, int, int) { return 1024 + 64 * (size_t)(E + k); }
extern "C" moe_status_t moe_check_status(void*, void*) { return MOE_OK; }
extern "C" moe_status_t moe_route(const moe_router_t* r, const void* x, moe_dtype_t xt, int T, int32_t* idx, float* w,
                                  float* probs, void*, size_t, void*) {
    for (int t = 0; t < T; t++) {
        std::vector<double> l(r->E);
        double mx = -1e300;
        for (int e = 0; e < r->E; e++) {
            double a = r->bias ? r->bias[e] : 0.0;
            for (int d = 0; d < r->D; d++)
                a += act(r->W, r->w_dtype, (size_t)e * r->D + d) * act(x, xt, (size_t)t * r->D + d);
            l[e] = a;
            mx = std::fmax(mx, a);
        }
        double s = 0;
        for (int e = 0; e < r->E; e++) s += std::exp(l[e] - mx);
        for (int e = 0; e < r->E; e++) probs[(size_t)t * r->E + e] = (float)(std::exp(l[e] - mx) / s);
        for (int q = 0; q < r->k; q++) { idx[(size_t)t * r->k + q] = q; w[(size_t)t * r->k + q] = 0.f; }
    }
    return MOE_OK;
}
static double dq(const moe_experts_t* x, const void* codes, const void* sc, int rows, int cols, int e, int n, int c) {
    size_t rb = x->q == MOE_Q_INT8_SYM_B32 ? cols : cols / 2;
    const uint8_t* row = (const uint8_t*)codes + ((size_t)e * rows + n) * rb;
    int q;
    if (x->q == MOE_Q_INT8_SYM_B32) q = (int8_t)row[c];
    else { int nib = (c & 1) ? row[c >> 1] >> 4 : row[c >> 1] & 15; q = nib >= 8 ? nib - 16 : nib; }
    size_t si = ((size_t)e * rows + n) * (cols / 32) + c / 32;
    double s = x->s_dtype == MOE_F16 ? hf(((const uint16_t*)sc)[si]) : ((const float*)sc)[si];
    return q * s;
}
extern "C" moe_status_t moe_decode(const moe_experts_t* x, const void* xin, moe_dtype_t xt, int T, int k,
                                   const int32_t* idx, const float* w, float* y, void*, void*, size_t, void*) {
    const int D = x->D, F = x->F;
    for (int t = 0; t < T; t++) {
        std::vector<double> acc(D, 0.0), h(F);
        for (int r = 0; r < k; r++) {
            int e = idx[t * k + r];
            if (e < 0 || e >= x->E) return MOE_ERR_BAD_INDEX;
            for (int n = 0; n < F; n++) {
                double g = 0, u = 0;
                for (int c = 0; c < D; c++) {
                    double v = act(xin, xt, (size_t)t * D + c);
                    g += dq(x, x->gate_q, x->gate_s, F, D, e, n, c) * v;
                    u += dq(x, x->up_q, x->up_s, F, D, e, n, c) * v;
                }
                h[n] = g / (1 + std::exp(-g)) * u;
            }
            for (int d = 0; d < D; d++) {
                double o = 0;
                for (int n = 0; n < F; n++) o += dq(x, x->down_q, x->down_s, D, F, e, d, n) * h[n];
                acc[d] += w[t * k + r] * o;
            }
        }
        for (int d = 0; d < D; d++) y[(size_t)t * D + d] = (float)acc[d];
    }
    return MOE_OK;
}
