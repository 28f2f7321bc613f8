// tl_optimizer.h -- internal: the host worker that applies gradient
// accumulation and the Adam update tile by tile, as each tile's dW lands in
// host memory, while the GPU goes on with the backward.
#pragma once
#include "tl_adam.h"

#include <cuda_runtime.h>

#include <string>
#include <vector>

namespace tl {

class Optimizer;

// tiles[g] describes tile g of the handle (its block in every parameter
// array); threads <= 0 uses every hardware thread.
Optimizer* optimizer_new(const std::vector<Block>& tiles, const AdamHyper& hp, int threads);
// Waits for every submitted job, stops the threads.
void optimizer_delete(Optimizer* o);

// Queue one job over the tiles in `order`: for each, wait (host) for
// ev_dw[g] (its dW is in host memory) and, for a step, ev_w[g] (the last read
// of its W by the GPU is done), then accumulate (step = false) or run the
// Adam step (step = true, using the accumulator when one was filled since
// the last step).  Returns false if the optimizer has failed.
bool optimizer_submit(Optimizer* o, bool step, const std::vector<int>& order, const std::vector<cudaEvent_t>& ev_w,
                      const std::vector<cudaEvent_t>& ev_dw);

// Block until every submitted step has updated tile g (its W, master and
// moments), or every submitted job has read tile g's dW, or all jobs are
// done.  False on timeout or failure (see optimizer_error).
bool optimizer_wait_update(Optimizer* o, int g, double timeout_s);
bool optimizer_wait_read(Optimizer* o, int g, double timeout_s);
bool optimizer_wait_all(Optimizer* o, double timeout_s);
// Steps submitted so far.
int64_t optimizer_steps(const Optimizer* o);
// Host seconds spent in accumulation and update work.
double optimizer_busy_seconds(const Optimizer* o);
std::string optimizer_error(const Optimizer* o);

}  // namespace tl
