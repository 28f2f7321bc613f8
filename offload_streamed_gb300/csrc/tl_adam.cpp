// tl_adam.cpp -- the optimizer update that runs on the host CPU, beside the
// DRAM that holds the optimizer state.
//
// The Adam update is elementwise: about a dozen FLOPs against the fp32 master
// weight, both moments and the gradient read and written, an arithmetic
// intensity near 0.5 FLOP/byte that no GPU link could hide, so it runs on the
// CPU next to its data (tm_zero_infinity, "Applying the test: which state can
// live where"; the state is the fp32 master weight, first and second moment,
// 12 bytes per parameter: gpu_zero_sharding, "The architecture: every piece
// explained").  The update itself is Adam (Kingma & Ba) with bias correction
// and decoupled weight decay (Loshchilov & Hutter), in fp32:
//     m <- b1 m + (1 - b1) g
//     v <- b2 v + (1 - b2) g^2
//     p <- p - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps) - lr wd p
// and the bf16 weights the next forward streams are the new p rounded to
// nearest even.
#include "tl_adam.h"

#include <cmath>
#include <cstring>

namespace tl {

uint16_t f32_to_bf16(float x) {
    uint32_t u;
    std::memcpy(&u, &x, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) return uint16_t((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}

static inline float bf16_to_f32(uint16_t h) {
    const uint32_t u = uint32_t(h) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
}

void accumulate_rows(const Block& b, bool overwrite, int64_t r0, int64_t r1) {
    for (int64_t r = r0; r < r1; ++r) {
        float* acc = b.acc + r * b.ld;
        const uint16_t* g = b.grad + r * b.ld;
        if (overwrite)
            for (int64_t c = 0; c < b.cols; ++c) acc[c] = bf16_to_f32(g[c]);
        else
            for (int64_t c = 0; c < b.cols; ++c) acc[c] += bf16_to_f32(g[c]);
    }
}

void adam_rows(const Block& b, const AdamHyper& hp, int64_t step, bool use_acc, int64_t r0, int64_t r1) {
    // bias corrections in double, once per call
    const double bc1 = 1.0 - std::pow(double(hp.beta1), double(step));
    const double bc2 = 1.0 - std::pow(double(hp.beta2), double(step));
    const float step_size = float(double(hp.lr) / bc1);
    const float inv_sqrt_bc2 = float(1.0 / std::sqrt(bc2));
    const float b1 = hp.beta1, b2 = hp.beta2, c1 = 1.f - hp.beta1, c2 = 1.f - hp.beta2;
    const float eps = hp.eps, decay = hp.lr * hp.weight_decay;
    for (int64_t r = r0; r < r1; ++r) {
        const int64_t o = r * b.ld;
        float* p = b.master + o;
        float* m = b.m + o;
        float* v = b.v + o;
        const uint16_t* g16 = b.grad + o;
        const float* acc = use_acc ? b.acc + o : nullptr;
        uint16_t* w = b.w + o;
        for (int64_t c = 0; c < b.cols; ++c) {
            const float g = acc ? acc[c] + bf16_to_f32(g16[c]) : bf16_to_f32(g16[c]);
            const float mn = b1 * m[c] + c1 * g;
            const float vn = b2 * v[c] + c2 * (g * g);
            const float denom = std::sqrt(vn) * inv_sqrt_bc2 + eps;
            const float pn = p[c] - step_size * (mn / denom) - decay * p[c];
            m[c] = mn;
            v[c] = vn;
            p[c] = pn;
            w[c] = f32_to_bf16(pn);
        }
    }
}

}  // namespace tl
