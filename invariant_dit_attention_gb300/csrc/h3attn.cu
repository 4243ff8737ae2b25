// h3attn.cu -- the C ABI (include/h3attn.h): argument checks, workspace, launches.
//
// Strict contract of the "ws1_full_h3_transformer" page (RL-Kernel PR #571),
// Scope / Known limitations: unsupported shapes, dtypes and devices are
// rejected with an error code, never run through another path.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/h3attn.h"
#include "common.cuh"
#include "host.cuh"

using namespace h3;

static constexpr int kMaxEvents = 4096;

// What the rotated rows q^ / k^ in a handle's workspace were computed from.
struct RowsKey {
    const void *q, *k, *wq, *wk, *pos[3], *seg;
    int n, S;
};

struct h3attn_ctx {
    h3attn_config cfg;
    int device;
    RopeTable rope;
    Workspace ws;
    int max_tiles64;
    unsigned* host_err;  // pinned
    void* allocs[40];
    int nalloc;
    // stage timing (instrumentation)
    int timing;
    cudaEvent_t* events;  // kMaxEvents, created on first use
    int ev_used;
    int ev_stage[kMaxEvents / 2];
    // test hook: a stall requested for the next forward / backward / QKV call
    StallRequest stall;
    // samples of the last backward call (its per-(sample, head) weight-gradient
    // partials stay in the workspace), 0 before the first
    int last_bwd_samples;
    // the inputs whose q^ / k^ rows the workspace holds (packed key order), if any
    RowsKey hat_key;
    bool hat_valid;
};

namespace {

bool same_rows(const RowsKey& a, const RowsKey& b) {
    return a.q == b.q && a.k == b.k && a.wq == b.wq && a.wk == b.wk && a.pos[0] == b.pos[0] &&
           a.pos[1] == b.pos[1] && a.pos[2] == b.pos[2] && a.seg == b.seg && a.n == b.n && a.S == b.S;
}
RowsKey rows_key(const Problem& p) {
    return RowsKey{p.q, p.k, p.wq, p.wk, {p.seq.pos_t, p.seq.pos_h, p.seq.pos_w}, p.seq.seg, p.seq.n, p.seq.S};
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

template <class T>
bool ws_alloc(h3attn_ctx* h, T** p, size_t bytes) {
    void* d = nullptr;
    if (h->nalloc >= (int)(sizeof h->allocs / sizeof h->allocs[0])) return false;
    if (cudaMalloc(&d, bytes < 256 ? 256 : bytes) != cudaSuccess) return false;
    h->allocs[h->nalloc++] = d;
    *p = reinterpret_cast<T*>(d);
    return true;
}

void free_ctx(h3attn_ctx* h) {
    if (h->events) {
        for (int i = 0; i < kMaxEvents; ++i) cudaEventDestroy(h->events[i]);
        free(h->events);
    }
    for (int i = 0; i < h->nalloc; ++i) cudaFree(h->allocs[i]);
    if (h->host_err) cudaFreeHost(h->host_err);
    free(h);
}

// Checks shared by forward and backward.
h3attn_status check_common(h3attn_t h, const void* q, const void* k, const void* v, const float* wq,
                           const float* wk, const int32_t* const pos_ids[3], const int32_t* seg,
                           int num_samples, int total_tokens) {
    if (!h) return H3ATTN_ERR_INVALID_ARG;
    if (total_tokens < 0 || num_samples < 0) return H3ATTN_ERR_INVALID_ARG;
    if (total_tokens == 0) return H3ATTN_OK;
    if (num_samples < 1 || num_samples > total_tokens) return H3ATTN_ERR_INVALID_ARG;
    if (total_tokens > h->cfg.max_tokens || num_samples > h->cfg.max_samples) return H3ATTN_ERR_CAPACITY;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(wq) || !aligned16(wk))
        return H3ATTN_ERR_INVALID_ARG;
    if (!pos_ids || !aligned4(pos_ids[0]) || !aligned4(pos_ids[1]) || !aligned4(pos_ids[2]) || !aligned4(seg))
        return H3ATTN_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return H3ATTN_ERR_CUDA;
    if (dev != h->device) return H3ATTN_ERR_INVALID_ARG;
    return H3ATTN_OK;
}

Problem make_problem(h3attn_t h, const void* q, const void* k, const void* v, const float* wq, const float* wk,
                     const int32_t* const pos_ids[3], const int32_t* seg, int n, int S) {
    Problem p;
    p.q = reinterpret_cast<const __nv_bfloat16*>(q);
    p.k = reinterpret_cast<const __nv_bfloat16*>(k);
    p.v = reinterpret_cast<const __nv_bfloat16*>(v);
    p.wq = wq;
    p.wk = wk;
    p.seq.seg = seg;
    p.seq.pos_t = pos_ids[0];
    p.seq.pos_h = pos_ids[1];
    p.seq.pos_w = pos_ids[2];
    p.seq.n = n;
    p.seq.S = S;
    p.H = h->cfg.num_heads;
    p.eps = h->cfg.eps;
    p.scale = h->cfg.softmax_scale;
    p.stall = h->stall;
    return p;
}

// The problem in canonical order: same samples; q and k read through the order's
// map, v and the positions gathered.
Problem canonical_problem(h3attn_t h, const Problem& p) {
    Problem c = p;
    const Workspace& ws = h->ws;
    c.v = ws.rows_c[0];
    c.rowmap = ws.perm;
    c.seq.pos_t = ws.pos_c;
    c.seq.pos_h = ws.pos_c + h->cfg.max_tokens;
    c.seq.pos_w = ws.pos_c + 2 * (size_t)h->cfg.max_tokens;
    return c;
}

// Clears the handle's stall request when the call that read it returns.
struct StallClear {
    h3attn_ctx* h;
    ~StallClear() { h->stall = StallRequest{}; }
};

// Runs one stage's launches, bracketed by events when stage timing is on.
template <class F>
cudaError_t stage(h3attn_ctx* h, int which, cudaStream_t s, F&& launch) {
    const bool rec = h->timing && h->events && h->ev_used + 2 <= kMaxEvents;
    if (rec && cudaEventRecord(h->events[h->ev_used], s) != cudaSuccess) return cudaErrorUnknown;
    cudaError_t e = launch();
    if (e != cudaSuccess) return e;
    if (rec) {
        if (cudaEventRecord(h->events[h->ev_used + 1], s) != cudaSuccess) return cudaErrorUnknown;
        h->ev_stage[h->ev_used / 2] = which;
        h->ev_used += 2;
    }
    return cudaSuccess;
}

}  // namespace

extern "C" {

const char* h3attn_status_string(h3attn_status s) {
    switch (s) {
        case H3ATTN_OK: return "ok";
        case H3ATTN_ERR_INVALID_ARG: return "invalid argument";
        case H3ATTN_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case H3ATTN_ERR_CAPACITY: return "exceeds the handle's capacity";
        case H3ATTN_ERR_CUDA: return "CUDA error";
        case H3ATTN_ERR_TIMEOUT: return "on-device wait timed out";
    }
    return "unknown status";
}

h3attn_status h3attn_create(const h3attn_config* cfg, h3attn_t* out) {
    if (!cfg || !out) return H3ATTN_ERR_INVALID_ARG;
    *out = nullptr;
    if (cfg->num_heads < 1 || cfg->max_tokens < 1 || cfg->max_samples < 1) return H3ATTN_ERR_INVALID_ARG;
    if (!(cfg->eps >= 0.f) || !(cfg->rope_theta > 0.f) || !(cfg->softmax_scale >= 0.f)) return H3ATTN_ERR_INVALID_ARG;
    if (cfg->key_order != H3ATTN_KEY_ORDER_PACKED && cfg->key_order != H3ATTN_KEY_ORDER_CANONICAL)
        return H3ATTN_ERR_INVALID_ARG;
    if (cfg->store_ds != 0 && cfg->store_ds != 1) return H3ATTN_ERR_INVALID_ARG;
    if (cfg->reuse_qk_hat != 0 && cfg->reuse_qk_hat != 1) return H3ATTN_ERR_INVALID_ARG;
    {
        const long long t128 = ((long long)cfg->max_tokens + 127) / 128;
        if (cfg->store_ds && (long long)cfg->num_heads * t128 * (t128 + cfg->max_samples) * 128 >= (1LL << 31))
            return H3ATTN_ERR_CAPACITY;  // TMA row coordinates of the stored blocks are 32-bit
    }
    if (cfg->head_dim != kD || cfg->rope_pairing != 0) return H3ATTN_ERR_UNSUPPORTED;
    if ((long)cfg->max_tokens * cfg->num_heads * kD >= (1L << 40)) return H3ATTN_ERR_CAPACITY;
    RopeTable rt;
    if (!build_rope_table(cfg->rope_sections, cfg->rope_theta, rt)) return H3ATTN_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return H3ATTN_ERR_CUDA;
    {
        const cudaError_t pe = prepare_device();
        if (pe != cudaSuccess) return pe == cudaErrorNotSupported ? H3ATTN_ERR_UNSUPPORTED : H3ATTN_ERR_CUDA;
    }

    h3attn_ctx* h = static_cast<h3attn_ctx*>(calloc(1, sizeof(h3attn_ctx)));
    if (!h) return H3ATTN_ERR_CUDA;
    h->cfg = *cfg;
    if (h->cfg.softmax_scale == 0.f) h->cfg.softmax_scale = 1.0f / sqrtf((float)kD);
    h->device = dev;
    h->rope = rt;
    const size_t H = cfg->num_heads, T = cfg->max_tokens, N = cfg->max_samples;
    h->max_tiles64 = (int)((T + 63) / 64 + N);
    Workspace& ws = h->ws;
    bool ok = ws_alloc(h, &ws.qhat, T * H * kD * 2) && ws_alloc(h, &ws.khat, T * H * kD * 2) &&
              ws_alloc(h, &ws.delta, T * H * 4) && ws_alloc(h, &ws.dqhat32, T * H * kD * 4) &&
              ws_alloc(h, &ws.dkhat32, T * H * kD * 4) && ws_alloc(h, &ws.rope_cs, T * 2 * kD * 4) &&
              ws_alloc(h, &ws.dwq_part, (size_t)h->max_tiles64 * H * kD * 4) &&
              ws_alloc(h, &ws.dwk_part, (size_t)h->max_tiles64 * H * kD * 4) &&
              ws_alloc(h, &ws.dwq_sample, N * kD * 4) && ws_alloc(h, &ws.dwk_sample, N * kD * 4) &&
              ws_alloc(h, &ws.dwq_head, N * H * kD * 4) && ws_alloc(h, &ws.dwk_head, N * H * kD * 4) &&
              ws_alloc(h, &ws.plan.order, N * 4) && ws_alloc(h, &ws.plan.rank_of, N * 4) &&
              ws_alloc(h, &ws.plan.cum64, (N + 1) * 4) && ws_alloc(h, &ws.plan.cum128, (N + 1) * 4) &&
              ws_alloc(h, &ws.plan.cum256, (N + 1) * 4) && ws_alloc(h, &ws.plan.cumsq, (N + 1) * 4) &&
              ws_alloc(h, &ws.plan.err, 4);
    if (ok) ok = ws_alloc(h, &ws.keys, T * 16);
    if (ok && cfg->store_ds) {
        // sum over samples of tiles^2 <= (largest tiles) * (sum of tiles) <= ceil(T/128) (ceil(T/128) + N)
        const long long t128 = ((long long)T + 127) / 128;
        ws.ds_blocks = (long long)H * t128 * (t128 + (long long)N);
        ok = ws_alloc(h, &ws.ds, (size_t)ws.ds_blocks * 128 * kD * 2);
    }
    if (ok && cfg->key_order == H3ATTN_KEY_ORDER_CANONICAL) {
        ok = ws_alloc(h, &ws.perm, T * 4) && ws_alloc(h, &ws.pos_c, 3 * T * 4) && ws_alloc(h, &ws.lse_c, T * H * 4);
        for (int t = 0; ok && t < 4; ++t) ok = ws_alloc(h, &ws.rows_c[t], T * H * kD * 2);
    }
    if (ok) ok = cudaMemset(ws.plan.err, 0, 4) == cudaSuccess;
    if (ok) ok = cudaMallocHost(&h->host_err, 4) == cudaSuccess;
    if (ok) ok = cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        free_ctx(h);
        return H3ATTN_ERR_CUDA;
    }
    *out = h;
    return H3ATTN_OK;
}

h3attn_status h3attn_destroy(h3attn_t h) {
    if (!h) return H3ATTN_OK;
    cudaDeviceSynchronize();
    free_ctx(h);
    return H3ATTN_OK;
}

h3attn_status h3attn_forward(h3attn_t h, const h3attn_bf16* q, const h3attn_bf16* k, const h3attn_bf16* v,
                             const float* q_norm_w, const float* k_norm_w, const int32_t* const pos_ids[3],
                             const int32_t* seg_offsets, int num_samples, int total_tokens, h3attn_bf16* out,
                             float* lse, void* stream) {
    h3attn_status st = check_common(h, q, k, v, q_norm_w, k_norm_w, pos_ids, seg_offsets, num_samples, total_tokens);
    if (st != H3ATTN_OK || total_tokens == 0) return st;
    StallClear clear_stall{h};
    if (!aligned16(out) || (lse && !aligned4(lse))) return H3ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Problem p = make_problem(h, q, k, v, q_norm_w, k_norm_w, pos_ids, seg_offsets, num_samples, total_tokens);
    Workspace& ws = h->ws;
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
    if (h->cfg.key_order == H3ATTN_KEY_ORDER_CANONICAL) {
        h->hat_valid = false;  // q^ / k^ are held in this call's canonical order
        const Problem c = canonical_problem(h, p);
        const int S = total_tokens, H = p.H;
        const void* gsrc[1] = {v};
        void* gdst[1] = {ws.rows_c[0]};
        const int32_t* psrc[3] = {p.seq.pos_t, p.seq.pos_h, p.seq.pos_w};
        int32_t* pdst[3] = {const_cast<int32_t*>(c.seq.pos_t), const_cast<int32_t*>(c.seq.pos_h),
                            const_cast<int32_t*>(c.seq.pos_w)};
        const void* ssrc[1] = {ws.rows_c[1]};
        void* sdst[1] = {out};
        float* lc = lse ? ws.lse_c : nullptr;
        if (stage(h, kStagePlan, s, [&] { return launch_plan(p, ws, s); }) != cudaSuccess ||
            stage(h, kStageOrder, s, [&] {
                return launch_order(p, nullptr, ws.keys, ws.perm, ws.plan.err, s);
            }) != cudaSuccess ||
            stage(h, kStagePermute, s, [&] {
                return launch_permute(ws.perm, S, H, 1, gsrc, gdst, nullptr, nullptr, psrc, pdst, false, ws.plan.err, s);
            }) != cudaSuccess ||
            stage(h, kStagePrologue, s, [&] { return launch_prologue(c, ws, &h->rope, s); }) != cudaSuccess ||
            stage(h, kStageFwd, s, [&] { return launch_fwd(c, ws, ws.rows_c[1], lc, s); }) != cudaSuccess ||
            stage(h, kStagePermute, s, [&] {
                return launch_permute(ws.perm, S, H, 1, ssrc, sdst, lc, lse, nullptr, nullptr, true, ws.plan.err, s);
            }) != cudaSuccess)
            return H3ATTN_ERR_CUDA;
        return H3ATTN_OK;
    }
    h->hat_valid = false;
    if (stage(h, kStagePlan, s, [&] { return launch_plan(p, ws, s); }) != cudaSuccess ||
        stage(h, kStagePrologue, s, [&] { return launch_prologue(p, ws, &h->rope, s); }) != cudaSuccess ||
        stage(h, kStageFwd, s, [&] { return launch_fwd(p, ws, o, lse, s); }) != cudaSuccess)
        return H3ATTN_ERR_CUDA;
    h->hat_key = rows_key(p);
    h->hat_valid = true;
    return H3ATTN_OK;
}

h3attn_status h3attn_backward(h3attn_t h, const h3attn_bf16* q, const h3attn_bf16* k, const h3attn_bf16* v,
                              const float* q_norm_w, const float* k_norm_w, const int32_t* const pos_ids[3],
                              const int32_t* seg_offsets, int num_samples, int total_tokens, const h3attn_bf16* out,
                              const float* lse, const h3attn_bf16* dout, h3attn_bf16* dq, h3attn_bf16* dk,
                              h3attn_bf16* dv, float* dq_norm_w, float* dk_norm_w, float* dq_norm_w_per_sample,
                              float* dk_norm_w_per_sample, void* stream) {
    h3attn_status st = check_common(h, q, k, v, q_norm_w, k_norm_w, pos_ids, seg_offsets, num_samples, total_tokens);
    if (st != H3ATTN_OK) return st;
    StallClear clear_stall{h};
    if (!aligned4(dq_norm_w) || !aligned4(dk_norm_w)) return H3ATTN_ERR_INVALID_ARG;
    if ((dq_norm_w_per_sample && !aligned4(dq_norm_w_per_sample)) ||
        (dk_norm_w_per_sample && !aligned4(dk_norm_w_per_sample)))
        return H3ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (total_tokens == 0) {  // empty batch: the weight gradients are zero
        if (cudaMemsetAsync(dq_norm_w, 0, kD * 4, s) != cudaSuccess ||
            cudaMemsetAsync(dk_norm_w, 0, kD * 4, s) != cudaSuccess)
            return H3ATTN_ERR_CUDA;
        h->last_bwd_samples = 0;
        return H3ATTN_OK;
    }
    if (!aligned16(out) || !aligned4(lse) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return H3ATTN_ERR_INVALID_ARG;
    Problem p = make_problem(h, q, k, v, q_norm_w, k_norm_w, pos_ids, seg_offsets, num_samples, total_tokens);
    Workspace& ws = h->ws;
    const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(out);
    const __nv_bfloat16* dO = reinterpret_cast<const __nv_bfloat16*>(dout);
    __nv_bfloat16* gq = reinterpret_cast<__nv_bfloat16*>(dq);
    __nv_bfloat16* gk = reinterpret_cast<__nv_bfloat16*>(dk);
    __nv_bfloat16* gv = reinterpret_cast<__nv_bfloat16*>(dv);
    if (h->cfg.key_order == H3ATTN_KEY_ORDER_CANONICAL) {
        h->hat_valid = false;
        const Problem c = canonical_problem(h, p);
        const int S = total_tokens, H = p.H;
        const void* gsrc[2] = {v, dout};
        void* gdst[2] = {ws.rows_c[0], ws.rows_c[2]};
        const int32_t* psrc[3] = {p.seq.pos_t, p.seq.pos_h, p.seq.pos_w};
        int32_t* pdst[3] = {const_cast<int32_t*>(c.seq.pos_t), const_cast<int32_t*>(c.seq.pos_h),
                            const_cast<int32_t*>(c.seq.pos_w)};
        const void* ssrc[1] = {ws.rows_c[3]};
        void* sdst[1] = {dv};
        __nv_bfloat16 *doc = ws.rows_c[2], *dvc = ws.rows_c[3];
        // dq, dk and out are addressed through the order's map by the row kernels
        if (stage(h, kStagePlan, s, [&] { return launch_plan(p, ws, s); }) != cudaSuccess ||
            stage(h, kStageOrder, s, [&] { return launch_order(p, dO, ws.keys, ws.perm, ws.plan.err, s); }) != cudaSuccess ||
            stage(h, kStagePermute, s, [&] {
                return launch_permute(ws.perm, S, H, 2, gsrc, gdst, lse, ws.lse_c, psrc, pdst, false, ws.plan.err, s);
            }) != cudaSuccess ||
            stage(h, kStagePrologue, s, [&] { return launch_prologue(c, ws, &h->rope, s); }) != cudaSuccess ||
            stage(h, kStageDelta, s, [&] { return launch_bwd_delta(c, ws, o, doc, s); }) != cudaSuccess ||
            stage(h, kStageDkdv, s, [&] { return launch_bwd_dkdv(c, ws, ws.lse_c, doc, gk, dvc, s); }) != cudaSuccess ||
            stage(h, kStageDq, s, [&] { return launch_bwd_dq(c, ws, ws.lse_c, doc, &h->rope, gq, gk, s); }) != cudaSuccess ||
            stage(h, kStageRows, s, [&] { return launch_bwd_rows(c, ws, &h->rope, gq, gk, s); }) != cudaSuccess ||
            stage(h, kStageDw, s, [&] {
                return launch_bwd_dw(c, ws, dq_norm_w, dk_norm_w, dq_norm_w_per_sample, dk_norm_w_per_sample, s);
            }) != cudaSuccess ||
            stage(h, kStagePermute, s, [&] {
                return launch_permute(ws.perm, S, H, 1, ssrc, sdst, nullptr, nullptr, nullptr, nullptr, true,
                                      ws.plan.err, s);
            }) != cudaSuccess)
            return H3ATTN_ERR_CUDA;
        h->last_bwd_samples = num_samples;
        return H3ATTN_OK;
    }
    // q^ / k^ of these inputs are still in the workspace when the handle's last
    // forward computed them from the same tensors (and the caller allows reuse)
    const bool reuse = h->cfg.reuse_qk_hat && h->hat_valid && same_rows(h->hat_key, rows_key(p));
    h->hat_valid = false;
    if (stage(h, kStagePlan, s, [&] { return launch_plan(p, ws, s); }) != cudaSuccess ||
        (!reuse &&
         stage(h, kStagePrologue, s, [&] { return launch_prologue(p, ws, &h->rope, s); }) != cudaSuccess) ||
        stage(h, kStageDelta, s, [&] { return launch_bwd_delta(p, ws, o, dO, s); }) != cudaSuccess ||
        stage(h, kStageDkdv, s, [&] { return launch_bwd_dkdv(p, ws, lse, dO, gk, gv, s); }) != cudaSuccess ||
        stage(h, kStageDq, s, [&] { return launch_bwd_dq(p, ws, lse, dO, &h->rope, gq, gk, s); }) != cudaSuccess ||
        stage(h, kStageRows, s, [&] { return launch_bwd_rows(p, ws, &h->rope, gq, gk, s); }) != cudaSuccess ||
        stage(h, kStageDw, s, [&] {
            return launch_bwd_dw(p, ws, dq_norm_w, dk_norm_w, dq_norm_w_per_sample, dk_norm_w_per_sample, s);
        }) != cudaSuccess)
        return H3ATTN_ERR_CUDA;
    h->last_bwd_samples = num_samples;
    h->hat_key = rows_key(p);
    h->hat_valid = true;
    return H3ATTN_OK;
}

h3attn_status h3attn_qkv_forward(h3attn_t h, const h3attn_bf16* x, int in_features, const h3attn_bf16* w_qkv,
                                 const float* b_qkv, const float* q_norm_w, const float* k_norm_w,
                                 const int32_t* const pos_ids[3], const int32_t* seg_offsets, int num_samples,
                                 int total_tokens, h3attn_bf16* q, h3attn_bf16* k, h3attn_bf16* v, h3attn_bf16* out,
                                 float* lse, void* stream) {
    h3attn_status st = check_common(h, q, k, v, q_norm_w, k_norm_w, pos_ids, seg_offsets, num_samples, total_tokens);
    if (st != H3ATTN_OK) return st;
    StallClear clear_stall{h};
    if (in_features < 1) return H3ATTN_ERR_INVALID_ARG;
    if (in_features % 64 != 0 || h->cfg.key_order != H3ATTN_KEY_ORDER_PACKED) return H3ATTN_ERR_UNSUPPORTED;
    if (total_tokens == 0) return H3ATTN_OK;
    if (!aligned16(x) || !aligned16(w_qkv) || (b_qkv && !aligned16(b_qkv)) || !aligned16(out) ||
        (lse && !aligned4(lse)))
        return H3ATTN_ERR_INVALID_ARG;
    if ((long long)total_tokens * in_features >= (1LL << 40) ||
        (long long)3 * h->cfg.num_heads * kD * in_features >= (1LL << 40))
        return H3ATTN_ERR_CAPACITY;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Problem p = make_problem(h, q, k, v, q_norm_w, k_norm_w, pos_ids, seg_offsets, num_samples, total_tokens);
    Workspace& ws = h->ws;
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
    const __nv_bfloat16* wb = reinterpret_cast<const __nv_bfloat16*>(w_qkv);
    __nv_bfloat16* qb = reinterpret_cast<__nv_bfloat16*>(q);
    __nv_bfloat16* kb = reinterpret_cast<__nv_bfloat16*>(k);
    __nv_bfloat16* vb = reinterpret_cast<__nv_bfloat16*>(v);
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
    h->hat_valid = false;
    if (stage(h, kStagePlan, s, [&] { return launch_plan(p, ws, s); }) != cudaSuccess ||
        stage(h, kStageQkv, s, [&] {
            cudaError_t e = launch_rope_table(p, ws, &h->rope, s);
            return e != cudaSuccess ? e : launch_qkv(p, ws, &h->rope, xb, in_features, wb, b_qkv, qb, kb, vb, s);
        }) != cudaSuccess ||
        stage(h, kStageFwd, s, [&] { return launch_fwd(p, ws, o, lse, s); }) != cudaSuccess)
        return H3ATTN_ERR_CUDA;
    h->hat_key = rows_key(p);  // the epilogue wrote q^ / k^ of the q, k it produced
    h->hat_valid = true;
    return H3ATTN_OK;
}

h3attn_status h3attn_canonical_order(h3attn_t h, const h3attn_bf16* q, const h3attn_bf16* k, const h3attn_bf16* v,
                                     const h3attn_bf16* dout, const int32_t* const pos_ids[3],
                                     const int32_t* seg_offsets, int num_samples, int total_tokens, int32_t* perm,
                                     void* stream) {
    if (!h) return H3ATTN_ERR_INVALID_ARG;
    if (total_tokens < 0 || num_samples < 0) return H3ATTN_ERR_INVALID_ARG;
    if (total_tokens == 0) return H3ATTN_OK;
    if (num_samples < 1 || num_samples > total_tokens) return H3ATTN_ERR_INVALID_ARG;
    if (total_tokens > h->cfg.max_tokens || num_samples > h->cfg.max_samples) return H3ATTN_ERR_CAPACITY;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (dout && !aligned16(dout)) || !aligned4(perm))
        return H3ATTN_ERR_INVALID_ARG;
    if (!pos_ids || !aligned4(pos_ids[0]) || !aligned4(pos_ids[1]) || !aligned4(pos_ids[2]) || !aligned4(seg_offsets))
        return H3ATTN_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return H3ATTN_ERR_CUDA;
    if (dev != h->device) return H3ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Problem p = make_problem(h, q, k, v, nullptr, nullptr, pos_ids, seg_offsets, num_samples, total_tokens);
    if (launch_plan(p, h->ws, s) != cudaSuccess ||
        launch_order(p, reinterpret_cast<const __nv_bfloat16*>(dout), h->ws.keys, perm, h->ws.plan.err, s) !=
            cudaSuccess)
        return H3ATTN_ERR_CUDA;
    return H3ATTN_OK;
}

h3attn_status h3attn_set_stage_timing(h3attn_t h, int enable) {
    if (!h) return H3ATTN_ERR_INVALID_ARG;
    if (enable && !h->events) {
        h->events = static_cast<cudaEvent_t*>(calloc(kMaxEvents, sizeof(cudaEvent_t)));
        if (!h->events) return H3ATTN_ERR_CUDA;
        for (int i = 0; i < kMaxEvents; ++i)
            if (cudaEventCreate(&h->events[i]) != cudaSuccess) return H3ATTN_ERR_CUDA;
    }
    h->timing = enable ? 1 : 0;
    return H3ATTN_OK;
}

h3attn_status h3attn_stage_times(h3attn_t h, float* total_ms, int* launches, int n_stages) {
    if (!h || !total_ms || !launches || n_stages < 1) return H3ATTN_ERR_INVALID_ARG;
    for (int i = 0; i < n_stages; ++i) { total_ms[i] = 0.f; launches[i] = 0; }
    if (h->ev_used && cudaEventSynchronize(h->events[h->ev_used - 1]) != cudaSuccess) return H3ATTN_ERR_CUDA;
    for (int k = 0; k < h->ev_used / 2; ++k) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, h->events[2 * k], h->events[2 * k + 1]) != cudaSuccess) return H3ATTN_ERR_CUDA;
        const int st = h->ev_stage[k];
        if (st < n_stages) { total_ms[st] += ms; launches[st] += 1; }
    }
    h->ev_used = 0;
    return H3ATTN_OK;
}

h3attn_status h3attn_norm_weight_grad_partials(h3attn_t h, float* dq_norm_w_partials, float* dk_norm_w_partials,
                                               void* stream) {
    if (!h || !aligned4(dq_norm_w_partials) || !aligned4(dk_norm_w_partials)) return H3ATTN_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return H3ATTN_ERR_CUDA;
    if (dev != h->device) return H3ATTN_ERR_INVALID_ARG;
    const size_t bytes = (size_t)h->last_bwd_samples * h->cfg.num_heads * kD * 4;
    if (bytes == 0) return H3ATTN_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(dq_norm_w_partials, h->ws.dwq_head, bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(dk_norm_w_partials, h->ws.dwk_head, bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return H3ATTN_ERR_CUDA;
    return H3ATTN_OK;
}

h3attn_status h3attn_combine_norm_weight_grads(const float* partials, int num_samples, int num_heads,
                                               float* per_sample, float* total, void* stream) {
    if (num_samples < 0 || num_heads < 1 || !aligned4(total)) return H3ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (num_samples == 0) return cudaMemsetAsync(total, 0, kD * 4, s) == cudaSuccess ? H3ATTN_OK : H3ATTN_ERR_CUDA;
    if (!aligned4(partials) || !aligned4(per_sample)) return H3ATTN_ERR_INVALID_ARG;
    const cudaError_t pe = prepare_device();
    if (pe != cudaSuccess) return pe == cudaErrorNotSupported ? H3ATTN_ERR_UNSUPPORTED : H3ATTN_ERR_CUDA;
    return launch_dw_combine(partials, num_samples, num_heads, per_sample, total, s) == cudaSuccess ? H3ATTN_OK
                                                                                                      : H3ATTN_ERR_CUDA;
}

h3attn_status h3attn_debug_stall(h3attn_t h, int kernel, int role, long long budget_cycles) {
    if (!h) return H3ATTN_ERR_INVALID_ARG;
    if (kernel == 0) {
        h->stall = StallRequest{};
        return H3ATTN_OK;
    }
    if (kernel < H3ATTN_STALL_FWD || kernel > H3ATTN_STALL_QKV || role < H3ATTN_STALL_PRODUCER ||
        role > H3ATTN_STALL_CONSUMER || budget_cycles < 1)
        return H3ATTN_ERR_INVALID_ARG;
    h->stall.kernel = kernel;
    h->stall.role = role;
    h->stall.budget = budget_cycles;
    return H3ATTN_OK;
}

h3attn_status h3attn_device_status(h3attn_t h, void* stream) {
    if (!h) return H3ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(h->host_err, h->ws.plan.err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return H3ATTN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return H3ATTN_ERR_CUDA;
    const unsigned e = *h->host_err;
    if (e) {
        if (cudaMemsetAsync(h->ws.plan.err, 0, 4, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
            return H3ATTN_ERR_CUDA;
    }
    if (e & kErrTimeout) return H3ATTN_ERR_TIMEOUT;
    if (e & (kErrBadOffsets | kErrRange)) return H3ATTN_ERR_INVALID_ARG;
    return H3ATTN_OK;
}

}  // extern "C"
