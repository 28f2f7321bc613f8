// tl_hooks.cpp -- entry points of the two subsystems that hook into the
// engine's fetch and write-back: the host optimizer (gradient accumulation
// and the Adam step on the CPU, tile by tile as each dW lands; tl_optimizer)
// and the file tier (W and dW in files, moved through pinned host slots with
// direct I/O; tl_filetier).
#include "tl_engine.h"
#include "tl_adam.h"
#include "tl_unbound_error.h"

#include <cmath>
#include <cstring>
#include <new>

struct tl_optimizer {
    tl_handle* h = nullptr;
    bool has_acc = false;
};

namespace tl {

void detach_optimizer(tl_handle* h) {
    if (h->opt_owner) {
        h->opt_owner->h = nullptr;
        h->opt_owner = nullptr;
    }
    if (!h->opt) return;
    tl::optimizer_delete(h->opt);  // waits for the submitted jobs
    h->opt = nullptr;
    for (auto* v : {&h->opt_ev_w, &h->opt_ev_dw}) {
        for (auto e : *v)
            if (e) cudaEventDestroy(e);
        v->clear();
    }
    h->opt_have_bwd = false;
}


}  // namespace tl

using namespace tl;

extern "C" {

tl_status tiled_linear_create_file(tl_handle** out, int64_t K, int64_t M, int32_t N, int32_t d, const char* w_path,
                                   const char* dw_path, int32_t host_slots, int32_t io_threads, void* workspace_dev,
                                   size_t workspace_bytes, int device) {
    std::string bad;
    if (!w_path || !dw_path || !w_path[0] || !dw_path[0]) bad = "null or empty file path";
    else if (host_slots < 2 || host_slots > 64) bad = "host_slots must be in 2..64";
    else if (io_threads < 1 || io_threads > 64) bad = "io_threads must be in 1..64";
    else if (check_shape(K, M, N, d).empty() && (K * (M / N) * 2) % 4096)
        bad = "a tile (K * M/N * 2 bytes) must be a multiple of 4096 bytes for direct I/O";
    if (!bad.empty()) {
        tl::set_unbound_error(bad);
        if (out) *out = nullptr;
        return TL_ERR_INVALID;
    }
    FileArgs fa;
    fa.w_path = w_path;
    fa.dw_path = dw_path;
    fa.host_slots = host_slots;
    fa.io_threads = io_threads;
    return create_ops(out, {one_op(K, M, N, nullptr, nullptr, TL_LAYOUT_TILE_MAJOR)}, d, workspace_dev,
                      workspace_bytes, device, true, &fa);
}

tl_status tiled_linear_file_sync(tl_handle* h) {
    if (!h) return TL_ERR_STATE;
    if (!h->tier) return fail(h, TL_ERR_INVALID, "the handle keeps W and dW in host memory");
    std::string why;
    if (!h->tier->sync(&why)) return fail(h, TL_ERR_IO, "file tier: " + why);
    return TL_OK;
}

tl_status tiled_linear_file_stats(const tl_handle* h, tl_file_stats* out) {
    if (!h || !out) return TL_ERR_INVALID;
    if (!h->tier) return TL_ERR_INVALID;
    const tl::FileTierStats st = h->tier->stats();
    std::memset(out, 0, sizeof(*out));
    out->read_bytes = st.read_bytes;
    out->write_bytes = st.write_bytes;
    out->read_seconds = st.read_s;
    out->write_seconds = st.write_s;
    out->fetch_wait_seconds = st.fetch_wait_s;
    out->writeback_wait_seconds = st.writeback_wait_s;
    out->host_slots = h->tier->host_slots();
    out->io_threads = h->tier->io_threads();
    return TL_OK;
}

static std::string adam_config_error(const tl_adam_config* c) {
    if (!c) return "null config";
    if (!(c->lr >= 0.f) || !std::isfinite(c->lr)) return "lr must be finite and >= 0";
    if (!(c->beta1 >= 0.f && c->beta1 < 1.f) || !(c->beta2 >= 0.f && c->beta2 < 1.f))
        return "beta1 and beta2 must be in [0, 1)";
    if (!(c->eps > 0.f) || !std::isfinite(c->eps)) return "eps must be finite and > 0";
    if (!(c->weight_decay >= 0.f) || !std::isfinite(c->weight_decay)) return "weight_decay must be finite and >= 0";
    return {};
}

static tl::AdamHyper hyper(const tl_adam_config* c) {
    tl::AdamHyper hp;
    hp.lr = c->lr;
    hp.beta1 = c->beta1;
    hp.beta2 = c->beta2;
    hp.eps = c->eps;
    hp.weight_decay = c->weight_decay;
    return hp;
}

tl_status tiled_linear_adam_update(const tl_adam_config* cfg, int64_t step, int64_t n, float* master, float* m,
                                   float* v, const float* grad_acc, const void* grad_bf16, void* w_bf16) {
    if (!adam_config_error(cfg).empty() || step < 1 || n < 0) return TL_ERR_INVALID;
    if (n == 0) return TL_OK;
    if (!master || !m || !v || !grad_bf16 || !w_bf16) return TL_ERR_INVALID;
    tl::Block b;
    b.master = master;
    b.m = m;
    b.v = v;
    b.acc = const_cast<float*>(grad_acc);
    b.grad = static_cast<const uint16_t*>(grad_bf16);
    b.w = static_cast<uint16_t*>(w_bf16);
    b.rows = 1;
    b.cols = n;
    b.ld = n;
    tl::adam_rows(b, hyper(cfg), step, grad_acc != nullptr, 0, 1);
    return TL_OK;
}

tl_status tiled_linear_optimizer_create(tl_optimizer** out, tl_handle* h, const tl_adam_config* cfg,
                                        float* const* master, float* const* m, float* const* v,
                                        float* const* grad_acc) {
    if (!out) return TL_ERR_INVALID;
    *out = nullptr;
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    const std::string bad = adam_config_error(cfg);
    if (!bad.empty()) return fail(h, TL_ERR_INVALID, "optimizer config: " + bad);
    if (h->tier) return fail(h, TL_ERR_INVALID, "the host optimizer needs W and dW in host memory");
    if (h->opt) return fail(h, TL_ERR_STATE, "the handle already has an optimizer");
    if (!master || !m || !v) return fail(h, TL_ERR_INVALID, "null master, m or v array");
    std::vector<tl::Block> tiles;
    for (size_t l = 0; l < h->ops.size(); ++l) {
        const Op& o = h->ops[l];
        if (!master[l] || !m[l] || !v[l] || (grad_acc && !grad_acc[l]))
            return fail(h, TL_ERR_INVALID, "null parameter array for operator " + std::to_string(l));
        for (int i = 0; i < o.s.N; ++i) {
            const bool tm = o.layout == TL_LAYOUT_TILE_MAJOR;
            const size_t off = tm ? size_t(i) * size_t(o.s.K) * size_t(o.s.Mi) : size_t(i) * size_t(o.s.Mi);
            tl::Block b;
            b.master = master[l] + off;
            b.m = m[l] + off;
            b.v = v[l] + off;
            b.acc = grad_acc ? grad_acc[l] + off : nullptr;
            b.grad = reinterpret_cast<const uint16_t*>(o.dw_host) + off;
            b.w = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(o.w_host)) + off;
            b.rows = o.s.K;
            b.cols = o.s.Mi;
            b.ld = tm ? o.s.Mi : o.s.M;
            tiles.push_back(b);
        }
    }
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return fail(h, TL_ERR_CUDA, "cudaSetDevice failed");
    auto* o = new (std::nothrow) tl_optimizer();
    if (!o) return fail(h, TL_ERR_INVALID, "out of host memory");
    h->opt_ev_w.assign(size_t(h->n_total), nullptr);
    h->opt_ev_dw.assign(size_t(h->n_total), nullptr);
    for (auto* vv : {&h->opt_ev_w, &h->opt_ev_dw})
        for (auto& e : *vv)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
                detach_optimizer(h);
                delete o;
                return fail(h, TL_ERR_CUDA, "optimizer event creation failed");
            }
    try {
        h->opt = tl::optimizer_new(tiles, hyper(cfg), cfg->threads);
    } catch (const std::exception& e) {
        detach_optimizer(h);
        delete o;
        return fail(h, TL_ERR_INVALID, std::string("optimizer threads: ") + e.what());
    }
    h->opt_have_bwd = false;
    h->opt_owner = o;
    o->h = h;
    o->has_acc = grad_acc != nullptr;
    *out = o;
    return TL_OK;
}

static tl_status optimizer_submit_job(tl_optimizer* o, bool step) {
    if (!o || !o->h || !o->h->opt) return TL_ERR_STATE;
    tl_handle* h = o->h;
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    if (!step && !o->has_acc) return fail(h, TL_ERR_INVALID, "accumulate needs a gradient accumulator");
    if (!h->opt_have_bwd) return fail(h, TL_ERR_STATE, "no backward since the last optimizer call");
    if (!tl::optimizer_submit(h->opt, step, h->opt_order, h->opt_ev_w, h->opt_ev_dw))
        return fail(h, TL_ERR_TIMEOUT, tl::optimizer_error(h->opt));
    h->opt_have_bwd = false;
    return TL_OK;
}

tl_status tiled_linear_optimizer_accumulate(tl_optimizer* o) { return optimizer_submit_job(o, false); }
tl_status tiled_linear_optimizer_step(tl_optimizer* o) { return optimizer_submit_job(o, true); }

tl_status tiled_linear_optimizer_wait(tl_optimizer* o) {
    if (!o || !o->h || !o->h->opt) return TL_ERR_STATE;
    if (!tl::optimizer_wait_all(o->h->opt, kOptWaitSeconds))
        return fail(o->h, TL_ERR_TIMEOUT, tl::optimizer_error(o->h->opt));
    return TL_OK;
}

tl_status tiled_linear_optimizer_stats(const tl_optimizer* o, int64_t* steps, double* busy_seconds) {
    if (!o || !o->h || !o->h->opt) return TL_ERR_STATE;
    if (steps) *steps = tl::optimizer_steps(o->h->opt);
    if (busy_seconds) *busy_seconds = tl::optimizer_busy_seconds(o->h->opt);
    return TL_OK;
}

tl_status tiled_linear_optimizer_destroy(tl_optimizer* o) {
    if (!o) return TL_OK;
    tl_status st = TL_OK;
    if (o->h && o->h->opt) {
        if (!tl::optimizer_error(o->h->opt).empty()) st = TL_ERR_TIMEOUT;
        DeviceGuard guard(o->h->device);
        detach_optimizer(o->h);
    }
    delete o;
    return st;
}

}  // extern "C"
