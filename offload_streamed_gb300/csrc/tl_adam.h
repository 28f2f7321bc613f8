// tl_adam.h -- internal: the host-side Adam update and gradient accumulation
// applied per weight tile (host memory, CPU threads).
#pragma once
#include <cstdint>

namespace tl {

struct AdamHyper {
    float lr = 1e-3f, beta1 = 0.9f, beta2 = 0.999f, eps = 1e-8f, weight_decay = 0.f;
};

// A 2-D block of `rows` rows of `cols` elements, `ld` elements apart, in each
// of the parameter arrays (fp32 master / first / second moment / gradient
// accumulator, bf16 weights and gradient).  Arrays not used may be null.
struct Block {
    float* master = nullptr;
    float* m = nullptr;
    float* v = nullptr;
    float* acc = nullptr;           // fp32 gradient accumulator (or null)
    const uint16_t* grad = nullptr; // bf16 gradient (this backward's dW)
    uint16_t* w = nullptr;          // bf16 weights written from the new master
    int64_t rows = 0, cols = 0, ld = 0;
};

// acc = grad (overwrite) or acc += grad, rows [r0, r1) of the block.
void accumulate_rows(const Block& b, bool overwrite, int64_t r0, int64_t r1);

// One Adam step (number `step` >= 1) on rows [r0, r1) of the block.  The
// gradient is grad (bf16), or acc + grad when use_acc.  See adam_update in
// tl_adam.cpp for the formula.
void adam_rows(const Block& b, const AdamHyper& hp, int64_t step, bool use_acc, int64_t r0, int64_t r1);

// fp32 -> bf16 bits, round to nearest even (NaN kept NaN).
uint16_t f32_to_bf16(float x);

}  // namespace tl
