// tl_stats.cpp -- the engine's sampled per-launch and per-copy timing: the
// event ring each call records into, its harvest into per-call spans and
// sums, and the stats / trace / timing entry points built on it.
#include "tl_engine.h"

#include <cstring>

namespace tl {

tl_status create_phase(tl_handle* h, Phase& p, int n, bool backward) {
    p.backward = backward;
    p.ring.resize(kTimingRing);
    for (auto& c : p.ring) {
        c.dx_at.assign(size_t(n), 0);
        TL_TRY(h, cudaEventCreate(&c.start));
        TL_TRY(h, cudaEventCreate(&c.end));
        for (int k = 0; k < 8; ++k) {
            if (!backward && (k == 2 || k == 3 || k == 6 || k == 7)) continue;
            c.ev[k].assign(size_t(n), nullptr);
            for (auto& e : c.ev[k]) TL_TRY(h, cudaEventCreate(&e));
        }
    }
    return TL_OK;
}

void destroy_phase(Phase& p) {
    for (auto& c : p.ring) {
        if (c.start) cudaEventDestroy(c.start);
        if (c.end) cudaEventDestroy(c.end);
        for (auto& v : c.ev)
            for (auto e : v)
                if (e) cudaEventDestroy(e);
    }
    p.ring.clear();
}

float span_ms(cudaEvent_t a, cudaEvent_t b) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) {
        cudaGetLastError();
        return 0.f;
    }
    return ms;
}

tl_status harvest(tl_handle* h, Phase& p, CallSlot& c, int n) {
    if (!c.pending) return TL_OK;
    TL_TRY(h, cudaEventSynchronize(c.end));
    c.total = span_ms(c.start, c.end);
    c.gemm1 = c.gemm2 = c.h2d = c.d2h = 0;
    if (!c.timed) {  // only counted: the sums describe the timed calls
        c.pending = false;
        c.harvested = true;
        p.sum_calls += 1;
        return TL_OK;
    }
    c.h2d_max = 0;
    for (int i = 0; i < n; ++i) {
        if (i < c.nk) {
            c.gemm1 += span_ms(c.ev[0][i], c.ev[1][i]);
            if (p.backward) c.gemm2 += span_ms(c.ev[2][i], c.ev[3][i]);
        }
        const float copy = span_ms(c.ev[4][i], c.ev[5][i]);
        c.h2d += copy;
        c.h2d_max = std::max(c.h2d_max, copy);
        if (p.backward) c.d2h += span_ms(c.ev[6][i], c.ev[7][i]);
    }
    c.pending = false;
    c.harvested = true;
    p.sum_calls += 1;
    p.sum_timed += 1;
    p.sum_total += c.total;
    p.sum_gemm1 += c.gemm1;
    p.sum_gemm2 += c.gemm2;
    p.sum_h2d += c.h2d;
    p.sum_d2h += c.d2h;
    return TL_OK;
}

tl_status harvest_all(tl_handle* h, Phase& p) {
    for (auto& c : p.ring) {
        tl_status st = harvest(h, p, c, h->n_total);
        if (st != TL_OK) return st;
    }
    return TL_OK;
}

// Slot for the next call of phase p (harvesting the call that used it last).
CallSlot* begin_call(tl_handle* h, Phase& p, tl_status* st) {
    CallSlot& c = p.ring[p.calls % kTimingRing];
    *st = harvest(h, p, c, h->n_total);
    if (*st != TL_OK) return nullptr;
    c.timed = p.calls % uint64_t(h->timing_every) == 0;
    return &c;
}

void end_call(Phase& p, CallSlot& c) {
    c.pending = true;
    c.harvested = false;
    if (c.timed) p.last = int(p.calls % kTimingRing);
    p.calls += 1;
}

}  // namespace tl

using namespace tl;

extern "C" {

tl_status tiled_linear_get_trace(tl_handle* h, int32_t backward, tl_trace_event* out, int32_t capacity,
                                 int32_t* count) {
    if (!h || !count || capacity < 0 || (capacity > 0 && !out)) return TL_ERR_INVALID;
    *count = 0;
    DeviceGuard guard(h->device);
    Phase& p = backward ? h->bwd : h->fwd;
    tl_status st = harvest_all(h, p);
    if (st != TL_OK) return st;
    if (p.last < 0) return TL_OK;
    const CallSlot& c = p.ring[size_t(p.last)];
    int32_t n = 0;
    auto add = [&](int32_t kind, int32_t tile, cudaEvent_t a, cudaEvent_t b) {
        const float t0 = span_ms(c.start, a), t1 = span_ms(c.start, b);
        if (n < capacity) out[n] = tl_trace_event{kind, tile, t0, t1};
        ++n;
    };
    const int NT = h->n_total;
    for (int j = 0; j < c.nk; ++j) {
        const int tile = backward ? NT - 1 - j : j;
        add(backward ? TL_TRACE_DW_GEMM : TL_TRACE_FWD_GEMM, tile, c.ev[0][j], c.ev[1][j]);
        if (backward && c.dx_at[size_t(j)]) add(TL_TRACE_DX_GEMM, tile, c.ev[2][j], c.ev[3][j]);
    }
    for (int j = 0; j < NT; ++j) {
        const int tile = backward ? NT - 1 - j : j;
        if (!backward || j >= c.reused) add(TL_TRACE_H2D, tile, c.ev[4][j], c.ev[5][j]);  // reused: no copy
        if (backward) add(TL_TRACE_D2H, tile, c.ev[6][j], c.ev[7][j]);
    }
    *count = n;
    return TL_OK;
}

tl_status tiled_linear_get_stats(tl_handle* h, void* out_v) {
    if (!h || !out_v) return TL_ERR_INVALID;
    tl_stats* out = static_cast<tl_stats*>(out_v);
    std::memset(out, 0, sizeof(*out));
    DeviceGuard guard(h->device);
    out->n_tiles = h->n_total;
    out->depth = h->d;
    tl_status st = harvest_all(h, h->fwd);
    if (st == TL_OK) st = harvest_all(h, h->bwd);
    if (st != TL_OK) return st;
    if (h->fwd.last >= 0) {
        const CallSlot& c = h->fwd.ring[h->fwd.last];
        out->fwd_valid = 1;
        out->fwd_total_ms = c.total;
        out->fwd_gemm_ms = c.gemm1;
        out->fwd_h2d_ms = c.h2d;
        out->fwd_wait_ms = c.total - c.gemm1;
        out->fwd_h2d_bytes = c.h2d_bytes;
        out->fwd_launches = c.launches;
        out->depth = c.depth;
        out->fwd_h2d_max_ms = c.h2d_max;
    }
    if (h->bwd.last >= 0) {
        const CallSlot& c = h->bwd.ring[h->bwd.last];
        out->bwd_valid = 1;
        out->bwd_total_ms = c.total;
        out->bwd_gemm_ms = c.gemm1 + c.gemm2;
        out->bwd_dw_gemm_ms = c.gemm1;
        out->bwd_dx_gemm_ms = c.gemm2;
        out->bwd_h2d_ms = c.h2d;
        out->bwd_d2h_ms = c.d2h;
        out->bwd_wait_ms = c.total - c.gemm1 - c.gemm2;
        out->bwd_h2d_bytes = c.h2d_bytes;
        out->bwd_d2h_bytes = c.d2h_bytes;
        out->bwd_launches = c.launches;
        out->bwd_reused_tiles = c.reused;
    }
    out->fwd_calls = h->fwd.sum_calls;
    out->sum_fwd_total_ms = h->fwd.sum_total;
    out->sum_fwd_gemm_ms = h->fwd.sum_gemm1;
    out->sum_fwd_h2d_ms = h->fwd.sum_h2d;
    out->bwd_calls = h->bwd.sum_calls;
    out->sum_bwd_total_ms = h->bwd.sum_total;
    out->sum_bwd_dw_gemm_ms = h->bwd.sum_gemm1;
    out->sum_bwd_dx_gemm_ms = h->bwd.sum_gemm2;
    out->sum_bwd_h2d_ms = h->bwd.sum_h2d;
    out->sum_bwd_d2h_ms = h->bwd.sum_d2h;
    out->sum_bwd_gemm_ms = h->bwd.sum_gemm1 + h->bwd.sum_gemm2;
    out->staging_slots = h->nstage;
    out->fwd_timed_calls = h->fwd.sum_timed;
    out->bwd_timed_calls = h->bwd.sum_timed;
    out->timing_every = h->timing_every;
    int32_t word = 0;
    TL_TRY(h, cudaMemcpy(&word, h->err_dev, sizeof(word), cudaMemcpyDeviceToHost));
    if (word != 0)
        return fail(h, TL_ERR_TIMEOUT,
                    "a kernel's bounded wait timed out (error bits " + std::to_string(word) + ")");
    return h->sticky;
}

tl_status tiled_linear_set_timing(tl_handle* h, int32_t every) {
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    if (every < 1) return fail(h, TL_ERR_INVALID, "every must be >= 1");
    h->timing_every = every;
    return TL_OK;
}

tl_status tiled_linear_reset_stats(tl_handle* h) {
    if (!h) return TL_ERR_INVALID;
    DeviceGuard guard(h->device);
    tl_status st = harvest_all(h, h->fwd);
    if (st == TL_OK) st = harvest_all(h, h->bwd);
    if (st != TL_OK) return st;
    for (Phase* p : {&h->fwd, &h->bwd}) {
        p->sum_calls = 0;
        p->sum_timed = 0;
        p->sum_total = p->sum_gemm1 = p->sum_gemm2 = p->sum_h2d = p->sum_d2h = 0;
    }
    return TL_OK;
}

}  // extern "C"
