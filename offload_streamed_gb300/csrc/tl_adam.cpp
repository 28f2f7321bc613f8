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

// f32_to_bf16 without branches, so that a row's loop vectorizes: the same
// bits for every input (NaN keeps its payload's top and is made quiet).
static inline uint16_t f32_to_bf16_row(float x) {
    uint32_t u;
    std::memcpy(&u, &x, sizeof u);
    const uint32_t rounded = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    const bool nan = (u & 0x7FFFFFFFu) > 0x7F800000u;
    return uint16_t(nan ? ((u >> 16) | 0x0040u) : rounded);
}

// One row of the update: every element takes the same operations in the same
// order, with no branch, so the compiler vectorizes the row (sqrt included:
// this unit is built with -fno-math-errno; v is a sum of squares, never
// negative, so sqrt would never have set errno anyway).
template <bool ACC>
static void adam_row(float* __restrict p, float* __restrict m, float* __restrict v, const uint16_t* __restrict g16,
                     const float* __restrict acc, uint16_t* __restrict w, int64_t n, float b1, float c1, float b2,
                     float c2, float step_size, float inv_sqrt_bc2, float eps, float decay) {
    for (int64_t c = 0; c < n; ++c) {
        float g = bf16_to_f32(g16[c]);
        if (ACC) g = acc[c] + g;
        const float mn = b1 * m[c] + c1 * g;
        const float vn = b2 * v[c] + c2 * (g * g);
        const float denom = std::sqrt(vn) * inv_sqrt_bc2 + eps;
        const float pn = p[c] - step_size * (mn / denom) - decay * p[c];
        m[c] = mn;
        v[c] = vn;
        p[c] = pn;
        w[c] = f32_to_bf16_row(pn);
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
        if (use_acc)
            adam_row<true>(b.master + o, b.m + o, b.v + o, b.grad + o, b.acc + o, b.w + o, b.cols, b1, c1, b2, c2,
                           step_size, inv_sqrt_bc2, eps, decay);
        else
            adam_row<false>(b.master + o, b.m + o, b.v + o, b.grad + o, nullptr, b.w + o, b.cols, b1, c1, b2, c2,
                            step_size, inv_sqrt_bc2, eps, decay);
    }
}

}  // namespace tl
