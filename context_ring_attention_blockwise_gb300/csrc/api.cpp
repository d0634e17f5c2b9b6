// api.cpp -- the extern "C" entry points of libcpattn (declared in include/cpattn.h). Host
// code only: argument checks, workspace layout, stream/event ordering of the ring-step path,
// and kernel launches. Every compute step runs in the CUDA kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace cpattn {
std::string build_plan(Plan& p, int64_t T, int h, int n_kv, int d, int n_cp, int layout, int causal);
}

using cpattn::Plan;

namespace {
thread_local std::string g_err;
}

namespace cpattn {
// Record the message cpattn_last_error returns on this thread (for entry points in other files).
void set_last_error(const std::string& msg) { g_err = msg; }
}  // namespace cpattn

namespace {

cpattn_status_t fail(cpattn_status_t s, const std::string& msg) {
    g_err = msg;
    return s;
}

cpattn_status_t cuda_fail(int e, const char* what) {
    return fail(CPATTN_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString((cudaError_t)e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

Plan* as_plan(cpattn_plan_t p) { return reinterpret_cast<Plan*>(p); }

// A plan made by cpattn_ulysses_plan describes the per-rank problem of the head split and works
// only with the cpattn_ulysses_* calls; a ring plan does not work with those.
cpattn_status_t reject_ulysses(const Plan& p) {
    return p.u_ncp ? fail(CPATTN_ERR_INVALID, "a plan made by cpattn_ulysses_plan works only with the cpattn_ulysses_* calls")
                   : CPATTN_OK;
}

float resolve_scale(const Plan& p, float scale) {
    double s = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)p.d);
    return (float)(s * 1.4426950408889634);   // scores are exponentiated with exp2
}

cpattn_status_t check_ws(const Plan& p, int B, const void* ws, size_t ws_bytes, bool ring) {
    if (cpattn_status_t s = reject_ulysses(p)) return s;
    if (!ws) return fail(CPATTN_ERR_WORKSPACE, "workspace pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(ws) & 1023u) != 0) return fail(CPATTN_ERR_WORKSPACE, "workspace must be 1024-byte aligned");
    cpattn::WsLayout w = cpattn::ws_layout(p, B);
    size_t need = ring ? w.ring_end : w.fwd_end;
    if (ws_bytes < need)
        return fail(CPATTN_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes, got " +
                                              std::to_string(ws_bytes));
    return CPATTN_OK;
}

template <class T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// Reset the header, upload the tile order, place tokens and position ids. The order table goes
// to the device inside kernel parameters: nothing is allocated, nothing is staged from host
// memory, and no copy engine is involved (a host-to-device copy here would queue behind whatever
// large upload the caller has in flight on the same engine, delaying the whole forward).
cpattn_status_t prologue(Plan& p, int B, const void* q, const void* k, const void* v, const int32_t* pos, void* ws,
                         cudaStream_t st, const int32_t* lo = nullptr, bool v_f16 = true) {
    cpattn::WsLayout w = cpattn::ws_layout(p, B);
    int e = cudaMemsetAsync(at<char>(ws, w.header), 0, sizeof(uint32_t) * cpattn::kHeaderWords, st);
    if (e) return cuda_fail(e, "cudaMemsetAsync(header)");
    e = cudaMemsetAsync(at<char>(ws, w.counts), 0, w.sched + sizeof(uint32_t) * (1 + (size_t)p.n_cp) - w.counts, st);
    if (e) return cuda_fail(e, "cudaMemsetAsync(counts)");
    e = cpattn::launch_upload_i32(at<int32_t>(ws, w.order), p.order.data(), (int64_t)p.order.size(), st);
    if (e) return cuda_fail(e, "order upload kernel");
    cpattn::PermuteArgs a{};
    a.B = B; a.T = p.T; a.n = p.n; a.m = p.m; a.h = p.h; a.n_kv = p.n_kv; a.d = p.d; a.n_cp = p.n_cp;
    a.layout = p.layout; a.n_qt = p.n_qt;
    a.q = q; a.k = k; a.v = v; a.pos = pos;
    a.qL = at<char>(ws, w.qL); a.kL = at<char>(ws, w.kL); a.vL = at<char>(ws, w.vL);
    a.posL = at<int32_t>(ws, w.posL); a.tile_mm = at<int32_t>(ws, w.tile_mm);
    a.lo = lo; a.loL = at<int32_t>(ws, w.loL); a.tile_lo = at<int32_t>(ws, w.tile_lo);
    a.v_f16 = v_f16 ? 1 : 0;
    a.header = at<uint32_t>(ws, w.header);
    e = cpattn::launch_permute(a, st);
    if (e) return cuda_fail(e, "permute kernel");
    return CPATTN_OK;
}

cpattn_status_t check_inputs(const Plan& p, int B, const void* q, const void* k, const void* v, const int32_t* pos) {
    if (cpattn_status_t s = reject_ulysses(p)) return s;
    if (B <= 0) return fail(CPATTN_ERR_INVALID, "B must be positive");
    if (!q || !k || !v) return fail(CPATTN_ERR_INVALID, "q, k and v must be non-NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (pos && !aligned16(pos)))
        return fail(CPATTN_ERR_INVALID, "q, k, v and pos must be 16-byte aligned");
    if ((double)B * (double)p.T * p.h > 2.0e9) return fail(CPATTN_ERR_UNSUPPORTED, "B*T*h beyond 2e9 rows");
    return CPATTN_OK;
}

cpattn::AttnLaunch attn_args(const Plan& p, int B, float scale, void* ws) {
    cpattn::WsLayout w = cpattn::ws_layout(p, B);
    cpattn::AttnLaunch a{};
    a.B = B; a.T = p.T; a.n = p.n; a.m = p.m; a.h = p.h; a.n_kv = p.n_kv; a.d = p.d; a.n_cp = p.n_cp;
    a.layout = p.layout; a.causal = p.causal; a.n_qt = p.n_qt; a.pair_heads = p.pair_heads; a.n_grp = p.n_grp;
    a.sched = at<uint32_t>(ws, w.sched);
    a.unit_tiles = at<int32_t>(ws, w.unit_tiles);
    a.walk_tab = at<int32_t>(ws, w.walk_tab);
    a.walk_nz = at<unsigned long long>(ws, w.walk_nz);
    a.walk_bits = at<unsigned long long>(ws, w.walk_bits);
    a.order_scratch = at<int32_t>(ws, w.order_masked);
    a.scale_log2 = resolve_scale(p, scale);
    a.qL = at<char>(ws, w.qL);
    a.kv_k = at<char>(ws, w.kL); a.kv_v = at<char>(ws, w.vL);
    a.posL = at<int32_t>(ws, w.posL); a.tile_mm = at<int32_t>(ws, w.tile_mm); a.order = at<int32_t>(ws, w.order);
    a.counts = at<unsigned long long>(ws, w.counts);
    a.header = at<uint32_t>(ws, w.header);
    a.timeout_ns = 2000000000ull;
    a.reserved_sms = p.reserved_sms;
    return a;
}

// Zero the launch's work counter, then enqueue the persistent attention kernel.
int launch_attn(const cpattn::AttnLaunch& a, cudaStream_t st, std::string* why) {
    int e = cudaMemsetAsync(a.sched, 0, sizeof(uint32_t), st);
    if (e) return e;
    return cpattn::launch_attention(a, st, why);
}

}  // namespace

extern "C" {

const char* cpattn_last_error(void) { return g_err.c_str(); }

const char* cpattn_version(void) { return "cpattn 0.1 sm_103a"; }

cpattn_status_t cpattn_plan(int64_t T, int h, int n_kv, int d_k, int n_cp, cpattn_layout_t layout, int causal,
                            cpattn_plan_t* out) {
    if (!out) return fail(CPATTN_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (d_k != 64 && d_k != 128) return fail(CPATTN_ERR_UNSUPPORTED, "d_k must be 64 or 128");
    Plan* p = new Plan();
    std::string why = cpattn::build_plan(*p, T, h, n_kv, d_k, n_cp, (int)layout, causal);
    if (!why.empty()) {
        delete p;
        return fail(CPATTN_ERR_INVALID, why);
    }
    *out = reinterpret_cast<cpattn_plan_t>(p);
    return CPATTN_OK;
}

cpattn_status_t cpattn_plan_set_reserved_sms(cpattn_plan_t plan, int sms) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (sms < 0 || sms > 1024) return fail(CPATTN_ERR_INVALID, "reserved SMs must lie in 0..1024");
    p->reserved_sms = sms;
    return CPATTN_OK;
}

cpattn_status_t cpattn_plan_destroy(cpattn_plan_t plan) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    for (int i = 0; i < 2; ++i) {
        if (p->ev_step[i]) cudaEventDestroy(p->ev_step[i]);
        if (p->ev_copy[i]) cudaEventDestroy(p->ev_copy[i]);
    }
    if (p->ev_start) cudaEventDestroy(p->ev_start);
    for (int i = 0; i < 2; ++i) {
        if (p->bev_kv[i]) cudaEventDestroy(p->bev_kv[i]);
        if (p->bev_used[i]) cudaEventDestroy(p->bev_used[i]);
        if (p->bev_circ[i]) cudaEventDestroy(p->bev_circ[i]);
    }
    if (p->bev_ready) cudaEventDestroy(p->bev_ready);
    if (p->bev_start) cudaEventDestroy(p->bev_start);
    delete p;
    return CPATTN_OK;
}

cpattn_status_t cpattn_workspace_size(cpattn_plan_t plan, int B, size_t* bytes) {
    Plan* p = as_plan(plan);
    if (!p || !bytes || B <= 0) return fail(CPATTN_ERR_INVALID, "plan, bytes and B > 0 required");
    if (cpattn_status_t s = reject_ulysses(*p)) return s;
    *bytes = cpattn::ws_layout(*p, B).fwd_end;
    return CPATTN_OK;
}

cpattn_status_t cpattn_ring_workspace_size(cpattn_plan_t plan, int B, size_t* bytes) {
    Plan* p = as_plan(plan);
    if (!p || !bytes || B <= 0) return fail(CPATTN_ERR_INVALID, "plan, bytes and B > 0 required");
    if (cpattn_status_t s = reject_ulysses(*p)) return s;
    *bytes = cpattn::ws_layout(*p, B).ring_end;
    return CPATTN_OK;
}

cpattn_status_t cpattn_backward_workspace_size(cpattn_plan_t plan, int B, size_t* bytes) {
    Plan* p = as_plan(plan);
    if (!p || !bytes || B <= 0) return fail(CPATTN_ERR_INVALID, "plan, bytes and B > 0 required");
    if (cpattn_status_t s = reject_ulysses(*p)) return s;
    *bytes = cpattn::ws_layout(*p, B).bwd_end;
    return CPATTN_OK;
}

cpattn_status_t cpattn_backward_ring_workspace_size(cpattn_plan_t plan, int B, size_t* bytes) {
    Plan* p = as_plan(plan);
    if (!p || !bytes || B <= 0) return fail(CPATTN_ERR_INVALID, "plan, bytes and B > 0 required");
    if (cpattn_status_t s = reject_ulysses(*p)) return s;
    *bytes = cpattn::ws_layout(*p, B).bring_end;
    return CPATTN_OK;
}

cpattn_status_t cpattn_tile_shape(cpattn_plan_t plan, int* block_q, int* block_k) {
    if (!plan) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (block_q) *block_q = cpattn::kBlockQ;
    if (block_k) *block_k = cpattn::kBlockK;
    return CPATTN_OK;
}

cpattn_status_t cpattn_plan_counts(cpattn_plan_t plan, int B, int64_t* tiles_full, int64_t* tiles_diag,
                                   int64_t* tiles_skip, int64_t* pairs, int64_t* kv_bytes_recv,
                                   int64_t* half_units) {
    Plan* p = as_plan(plan);
    if (!p || B <= 0) return fail(CPATTN_ERR_INVALID, "plan and B > 0 required");
    if (cpattn_status_t s = reject_ulysses(*p)) return s;
    size_t nn = (size_t)p->n_cp * p->n_cp;
    if (tiles_full) std::memcpy(tiles_full, p->full.data(), nn * sizeof(int64_t));
    if (tiles_diag) std::memcpy(tiles_diag, p->diag.data(), nn * sizeof(int64_t));
    if (tiles_skip) std::memcpy(tiles_skip, p->skip.data(), nn * sizeof(int64_t));
    if (pairs) std::memcpy(pairs, p->pairs.data(), p->n_cp * sizeof(int64_t));
    if (half_units) std::memcpy(half_units, p->half_units.data(), p->n_cp * sizeof(int64_t));
    if (kv_bytes_recv)
        for (int r = 0; r < p->n_cp; ++r)
            kv_bytes_recv[r] = (int64_t)4 * B * p->n * p->n_kv * p->d * (p->n_cp - 1);
    return CPATTN_OK;
}

cpattn_status_t cpattn_backward_counts(cpattn_plan_t plan, int B, int64_t* bytes_recv) {
    Plan* p = as_plan(plan);
    if (!p || B <= 0 || !bytes_recv) return fail(CPATTN_ERR_INVALID, "plan, B > 0 and bytes_recv required");
    if (cpattn_status_t s = reject_ulysses(*p)) return s;
    // the other ranks' K and V blocks (bf16), and the circulating dK and dV blocks (fp32 partial
    // sums), which arrive n_cp times: the last hop returns a rank's own block
    const int64_t blk = (int64_t)B * p->n * p->n_kv * p->d;
    for (int r = 0; r < p->n_cp; ++r)
        bytes_recv[r] = (int64_t)(p->n_cp - 1) * 2 * blk * 2 + (int64_t)p->n_cp * 2 * blk * 4;
    return CPATTN_OK;
}

cpattn_status_t cpattn_forward(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                               const int32_t* pos, float scale, void* o, float* lse, void* ws, size_t ws_bytes,
                               cpattn_stream_t stream) {
    return cpattn::forward_with_workspace(plan, B, q, k, v, pos, scale, o, lse, ws, ws_bytes, stream);
}

}  // extern "C"

cpattn_status_t cpattn::forward_with_workspace(cpattn_plan_t plan, int B, const void* q, const void* k,
                                               const void* v, const int32_t* pos, float scale, void* o, float* lse,
                                               void* ws, size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    cpattn_status_t s = check_inputs(*p, B, q, k, v, pos);
    if (s) return s;
    if (!o || !lse || !aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_INVALID, "o and lse must be non-NULL and 16-byte aligned");
    if ((s = check_ws(*p, B, ws, ws_bytes, false))) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = prologue(*p, B, q, k, v, pos, ws, st, nullptr))) return s;
    cpattn::AttnLaunch a = attn_args(*p, B, scale, ws);
    a.fused = 1; a.step = 0; a.kv_by_holder = 0;
    a.o = o; a.lse = lse;
    std::string why;
    int e = launch_attn(a, st, &why);
    if (e) return why.empty() ? cuda_fail(e, "attention kernel") : fail(CPATTN_ERR_CUDA, why);
    return CPATTN_OK;
}

extern "C" {

namespace {
// The backward's launch arguments: every pointer into the workspace, the rest from the plan.
cpattn::BwdLaunch bwd_args(const Plan& p, int B, float scale, void* ws, const int32_t* lo) {
    cpattn::WsLayout w = cpattn::ws_layout(p, B);
    const size_t nu = (size_t)p.n_cp * p.n_qt;
    cpattn::BwdLaunch a{};
    a.B = B; a.T = p.T; a.n = p.n; a.m = p.m; a.h = p.h; a.n_kv = p.n_kv; a.d = p.d; a.n_cp = p.n_cp;
    a.layout = p.layout; a.causal = p.causal; a.n_qt = p.n_qt;
    a.scale = scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)p.d));
    a.qL = at<char>(ws, w.qL); a.kL = at<char>(ws, w.kL); a.vL = at<char>(ws, w.vL); a.doL = at<char>(ws, w.doL);
    a.nlse2L = at<float>(ws, w.lse2); a.nDL = at<float>(ws, w.Dl);
    a.posL = at<int32_t>(ws, w.posL); a.tile_mm = at<int32_t>(ws, w.tile_mm);
    a.order_q = at<int32_t>(ws, w.bwd_order); a.order_kv = a.order_q + nu;
    a.loL = lo ? at<int32_t>(ws, w.loL) : nullptr;
    a.tile_lo = lo ? at<int32_t>(ws, w.tile_lo) : nullptr;
    a.header = at<uint32_t>(ws, w.header);
    a.timeout_ns = 2000000000ull;
    return a;
}

// Checks, token placement, and the backward's side data in layout order (dO, -lse log2 e, -D)
// and unit orders: everything before the tcgen05 kernels. `need` is the workspace end required.
cpattn_status_t backward_prepare(Plan& p, int B, const void* q, const void* k, const void* v, const void* o,
                                 const float* lse, const void* dout, const int32_t* pos, const int32_t* lo, void* ws,
                                 size_t ws_bytes, size_t need, cudaStream_t st) {
    cpattn_status_t s = check_inputs(p, B, q, k, v, pos);
    if (s) return s;
    if (!o || !lse || !dout) return fail(CPATTN_ERR_INVALID, "o, lse and dout must be non-NULL");
    if (!aligned16(o) || !aligned16(lse) || !aligned16(dout))
        return fail(CPATTN_ERR_INVALID, "o, lse and dout must be 16-byte aligned");
    if (!ws) return fail(CPATTN_ERR_WORKSPACE, "workspace pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(ws) & 1023u) != 0) return fail(CPATTN_ERR_WORKSPACE, "workspace must be 1024-byte aligned");
    if (ws_bytes < need)
        return fail(CPATTN_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes, got " +
                                              std::to_string(ws_bytes));
    cpattn::WsLayout w = cpattn::ws_layout(p, B);
    if ((s = prologue(p, B, q, k, v, pos, ws, st, lo, false))) return s;   // the backward reads bf16 V
    cpattn::BwdPrepArgs pa{};
    pa.B = B; pa.T = p.T; pa.n = p.n; pa.m = p.m; pa.h = p.h; pa.d = p.d; pa.n_cp = p.n_cp;
    pa.layout = p.layout; pa.n_qt = p.n_qt;
    pa.o = o; pa.dout = dout; pa.lse = lse;
    pa.doL = at<char>(ws, w.doL); pa.nlse2L = at<float>(ws, w.lse2); pa.nDL = at<float>(ws, w.Dl);
    int e = 0;
    if (p.n % 128 != 0) {
        // the padding after a short last tile must hold finite values: zero both side tables
        const size_t padded = sizeof(float) * (size_t)p.n_cp * B * p.h * (size_t)p.n_qt * 128;
        e = cudaMemsetAsync(at<char>(ws, w.lse2), 0, padded, st);
        if (!e) e = cudaMemsetAsync(at<char>(ws, w.Dl), 0, padded, st);
        if (e) return cuda_fail(e, "cudaMemsetAsync(backward side tables)");
    }
    e = cpattn::launch_bwd_prep(pa, st);
    if (e) return cuda_fail(e, "backward prep kernel");
    const size_t nu = (size_t)p.n_cp * p.n_qt;
    e = cpattn::launch_upload_i32(at<int32_t>(ws, w.bwd_order), p.order_q.data(), (int64_t)nu, st);
    if (!e) e = cpattn::launch_upload_i32(at<int32_t>(ws, w.bwd_order) + nu, p.order_kv.data(), (int64_t)nu, st);
    if (e) return cuda_fail(e, "backward order upload kernel");
    return CPATTN_OK;
}

cpattn_status_t backward_impl(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, const int32_t* pos, const int32_t* lo, float scale,
                              void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!dq || !dk || !dv) return fail(CPATTN_ERR_INVALID, "o, lse, dout, dq, dk and dv must be non-NULL");
    if (!aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(CPATTN_ERR_INVALID, "o, lse, dout, dq, dk and dv must be 16-byte aligned");
    if (cpattn_status_t s0 = reject_ulysses(*p)) return s0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cpattn_status_t s = backward_prepare(*p, B, q, k, v, o, lse, dout, pos, lo, ws, ws_bytes,
                                         B > 0 ? cpattn::ws_layout(*p, B).bwd_end : 0, st);
    if (s) return s;
    cpattn::BwdLaunch a = bwd_args(*p, B, scale, ws, lo);
    a.dq = dq; a.dk = dk; a.dv = dv;
    std::string why;
    int e = cpattn::launch_backward(a, st, &why);
    if (e) return why.empty() ? cuda_fail(e, "backward kernels") : fail(CPATTN_ERR_CUDA, why);
    return CPATTN_OK;
}
}  // namespace

cpattn_status_t cpattn_backward(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dout, const int32_t* pos, float scale, void* dq, void* dk,
                                void* dv, void* ws, size_t ws_bytes, cpattn_stream_t stream) {
    return backward_impl(plan, B, q, k, v, o, lse, dout, pos, nullptr, scale, dq, dk, dv, ws, ws_bytes, stream);
}

cpattn_status_t cpattn_backward_masked(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                       const void* o, const float* lse, const void* dout, const int32_t* pos,
                                       const int32_t* lo, float scale, void* dq, void* dk, void* dv, void* ws,
                                       size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!p->causal) return fail(CPATTN_ERR_UNSUPPORTED, "a lower bound per query needs a causal plan");
    if (!lo || !aligned16(lo)) return fail(CPATTN_ERR_INVALID, "lo must be non-NULL and 16-byte aligned");
    return backward_impl(plan, B, q, k, v, o, lse, dout, pos, lo, scale, dq, dk, dv, ws, ws_bytes, stream);
}

cpattn_status_t cpattn_forward_masked(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                      const int32_t* pos, const int32_t* lo, float scale, void* o, float* lse, void* ws,
                                      size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!p->causal) return fail(CPATTN_ERR_UNSUPPORTED, "a lower bound per query needs a causal plan");
    if (p->n_qt > 65535) return fail(CPATTN_ERR_UNSUPPORTED, "a lower bound per query supports up to 65535 tiles per rank");
    if (!lo || !aligned16(lo)) return fail(CPATTN_ERR_INVALID, "lo must be non-NULL and 16-byte aligned");
    cpattn_status_t s = check_inputs(*p, B, q, k, v, pos);
    if (s) return s;
    if (!o || !lse || !aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_INVALID, "o and lse must be non-NULL and 16-byte aligned");
    if ((s = check_ws(*p, B, ws, ws_bytes, false))) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = prologue(*p, B, q, k, v, pos, ws, st, lo))) return s;
    cpattn::WsLayout w = cpattn::ws_layout(*p, B);
    cpattn::AttnLaunch a = attn_args(*p, B, scale, ws);
    a.fused = 1; a.step = 0; a.kv_by_holder = 0;
    a.o = o; a.lse = lse;
    a.loL = at<int32_t>(ws, w.loL); a.tile_lo = at<int32_t>(ws, w.tile_lo);
    std::string why;
    int e = launch_attn(a, st, &why);
    if (e) return why.empty() ? cuda_fail(e, "attention kernel") : fail(CPATTN_ERR_CUDA, why);
    return CPATTN_OK;
}

cpattn_status_t cpattn_forward_docs(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                    const int32_t* pos, const int32_t* doc, float scale, void* o, float* lse, void* ws,
                                    size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!doc || !aligned16(doc)) return fail(CPATTN_ERR_INVALID, "doc must be non-NULL and 16-byte aligned");
    cpattn_status_t s = check_inputs(*p, B, q, k, v, pos);
    if (s) return s;
    if (!o || !lse || !aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_INVALID, "o and lse must be non-NULL and 16-byte aligned");
    if ((s = check_ws(*p, B, ws, ws_bytes, false))) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the ids travel with the tokens like the lower bound does, with their range per tile
    if ((s = prologue(*p, B, q, k, v, pos, ws, st, doc))) return s;
    cpattn::WsLayout w = cpattn::ws_layout(*p, B);
    cpattn::AttnLaunch a = attn_args(*p, B, scale, ws);
    a.fused = 1; a.step = 0; a.kv_by_holder = 0;
    a.o = o; a.lse = lse;
    a.loL = at<int32_t>(ws, w.loL); a.tile_lo = at<int32_t>(ws, w.tile_lo); a.doc_ids = 1;
    std::string why;
    int e = launch_attn(a, st, &why);
    if (e) return why.empty() ? cuda_fail(e, "attention kernel") : fail(CPATTN_ERR_CUDA, why);
    return CPATTN_OK;
}

cpattn_status_t cpattn_attend(cpattn_plan_t plan, int B, float scale, void* o, float* lse, void* ws, size_t ws_bytes,
                              cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (B <= 0) return fail(CPATTN_ERR_INVALID, "B must be positive");
    if (!o || !lse || !aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_INVALID, "o and lse must be non-NULL and 16-byte aligned");
    cpattn_status_t s = check_ws(*p, B, ws, ws_bytes, false);
    if (s) return s;
    cpattn::AttnLaunch a = attn_args(*p, B, scale, ws);
    a.fused = 1; a.step = 0; a.kv_by_holder = 0;
    a.o = o; a.lse = lse;
    std::string why;
    int e = launch_attn(a, reinterpret_cast<cudaStream_t>(stream), &why);
    if (e) return why.empty() ? cuda_fail(e, "attention kernel") : fail(CPATTN_ERR_CUDA, why);
    return CPATTN_OK;
}

cpattn_status_t cpattn_permute(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                               const int32_t* pos, void* ws, size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    cpattn_status_t s = check_inputs(*p, B, q, k, v, pos);
    if (s) return s;
    if ((s = check_ws(*p, B, ws, ws_bytes, false))) return s;
    if ((s = prologue(*p, B, q, k, v, pos, ws, reinterpret_cast<cudaStream_t>(stream)))) return s;
    p->next_step = 0;
    p->ring_B = B;
    return CPATTN_OK;
}

cpattn_status_t cpattn_ring_step(cpattn_plan_t plan, int B, int step, float scale, void* ws, size_t ws_bytes,
                                 cpattn_stream_t compute, cpattn_stream_t copy) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (B <= 0) return fail(CPATTN_ERR_INVALID, "B must be positive");
    cpattn_status_t s = check_ws(*p, B, ws, ws_bytes, true);
    if (s) return s;
    if (step < 0 || step >= p->n_cp) return fail(CPATTN_ERR_INVALID, "step out of range");
    if (p->next_step != step)
        return fail(CPATTN_ERR_INVALID, "ring steps must follow cpattn_permute in order 0..n_cp-1 (expected step " +
                                            std::to_string(p->next_step) + ")");
    if (B != p->ring_B) return fail(CPATTN_ERR_INVALID, "B differs from the batch cpattn_permute placed");
    cudaStream_t cst = reinterpret_cast<cudaStream_t>(compute), xst = reinterpret_cast<cudaStream_t>(copy);
    int e;
    for (int i = 0; i < 2; ++i) {
        if (!p->ev_step[i] && (e = cudaEventCreateWithFlags(&p->ev_step[i], cudaEventDisableTiming))) return cuda_fail(e, "cudaEventCreate");
        if (!p->ev_copy[i] && (e = cudaEventCreateWithFlags(&p->ev_copy[i], cudaEventDisableTiming))) return cuda_fail(e, "cudaEventCreate");
    }
    if (!p->ev_start && (e = cudaEventCreateWithFlags(&p->ev_start, cudaEventDisableTiming))) return cuda_fail(e, "cudaEventCreate");
    cpattn::WsLayout w = cpattn::ws_layout(*p, B);
    const int slot = step & 1, nxt = (step + 1) & 1;
    const bool hop_in_kernel = xst == nullptr;   // no copy stream: the step's kernel moves the blocks
    if (step == 0) p->ring_hop_kernel = hop_in_kernel ? 1 : 0;
    else if (p->ring_hop_kernel != (hop_in_kernel ? 1 : 0))
        return fail(CPATTN_ERR_INVALID, "a ring pass keeps one kind of hop: a copy stream at every step, or none");
    const size_t blk = 2 * (size_t)B * p->n * p->n_kv * p->d;    // one rank's block, bytes
    const size_t all = blk * p->n_cp;

    if (hop_in_kernel) {
        // everything runs on the compute stream, in order: nothing to wait for
    } else if (step == 0) {   // the copy stream must see the permuted blocks
        if ((e = cudaEventRecord(p->ev_start, cst))) return cuda_fail(e, "cudaEventRecord");
        if ((e = cudaStreamWaitEvent(xst, p->ev_start, 0))) return cuda_fail(e, "cudaStreamWaitEvent");
    } else if ((e = cudaStreamWaitEvent(cst, p->ev_copy[slot], 0))) {
        return cuda_fail(e, "cudaStreamWaitEvent");
    }
    cpattn::AttnLaunch a = attn_args(*p, B, scale, ws);
    a.fused = 0; a.step = step;
    a.sched = at<uint32_t>(ws, w.sched) + 1 + step;
    if (step > 0) { a.kv_k = at<char>(ws, w.stageK[slot]); a.kv_v = at<char>(ws, w.stageV[slot]); }
    a.kv_by_holder = 1;
    a.o_run = at<float>(ws, w.o_run); a.lse_run = at<float>(ws, w.lse_run);
    a.l_run = a.lse_run + (size_t)B * p->T * p->h;
    if (hop_in_kernel && step + 1 < p->n_cp) {
        // Send right, receive left, inside this step's kernel: slot nxt of rank r <- the block
        // rank r-1 holds now (its idle warps copy while the attention runs).
        a.hop_src_k = step == 0 ? at<char>(ws, w.kL) : at<char>(ws, w.stageK[slot]);
        a.hop_src_v = step == 0 ? at<char>(ws, w.vL) : at<char>(ws, w.stageV[slot]);
        a.hop_dst_k = at<char>(ws, w.stageK[nxt]);
        a.hop_dst_v = at<char>(ws, w.stageV[nxt]);
        a.hop_words = (int64_t)(all / 16);
        a.hop_blk = (int64_t)(blk / 16);
    }
    std::string why;
    if ((e = launch_attn(a, cst, &why))) return why.empty() ? cuda_fail(e, "attention kernel") : fail(CPATTN_ERR_CUDA, why);
    if (!hop_in_kernel && (e = cudaEventRecord(p->ev_step[slot], cst))) return cuda_fail(e, "cudaEventRecord");

    if (!hop_in_kernel && step + 1 < p->n_cp) {
        // Send right, receive left: slot nxt of rank r <- the block rank r-1 holds now. Blocks
        // are rank-major, so the hop is two contiguous copies per tensor.
        if (step >= 1 && (e = cudaStreamWaitEvent(xst, p->ev_step[nxt], 0))) return cuda_fail(e, "cudaStreamWaitEvent");
        for (int t = 0; t < 2; ++t) {
            const char* src = (step == 0) ? at<char>(ws, t ? w.vL : w.kL) : at<char>(ws, t ? w.stageV[slot] : w.stageK[slot]);
            char* dst = at<char>(ws, t ? w.stageV[nxt] : w.stageK[nxt]);
            if (p->n_cp > 1 && (e = cudaMemcpyAsync(dst + blk, src, all - blk, cudaMemcpyDeviceToDevice, xst)))
                return cuda_fail(e, "cudaMemcpyAsync(ring hop)");
            if ((e = cudaMemcpyAsync(dst, src + all - blk, blk, cudaMemcpyDeviceToDevice, xst)))
                return cuda_fail(e, "cudaMemcpyAsync(ring hop)");
        }
        if ((e = cudaEventRecord(p->ev_copy[nxt], xst))) return cuda_fail(e, "cudaEventRecord");
    }
    p->next_step = step + 1;
    return CPATTN_OK;
}

cpattn_status_t cpattn_finalize(cpattn_plan_t plan, int B, void* o, float* lse, void* ws, size_t ws_bytes,
                                cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (B <= 0) return fail(CPATTN_ERR_INVALID, "B must be positive");
    if (!o || !lse || !aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_INVALID, "o and lse must be non-NULL and 16-byte aligned");
    cpattn_status_t s = check_ws(*p, B, ws, ws_bytes, true);
    if (s) return s;
    if (p->next_step != p->n_cp) return fail(CPATTN_ERR_INVALID, "finalize needs all n_cp ring steps first");
    if (B != p->ring_B) return fail(CPATTN_ERR_INVALID, "B differs from the batch cpattn_permute placed");
    cpattn::WsLayout w = cpattn::ws_layout(*p, B);
    cpattn::FinalizeArgs a{};
    a.B = B; a.T = p->T; a.n = p->n; a.m = p->m; a.h = p->h; a.d = p->d; a.n_cp = p->n_cp; a.layout = p->layout;
    a.o_run = at<float>(ws, w.o_run); a.lse_run = at<float>(ws, w.lse_run); a.o = o; a.lse = lse;
    a.l_run = a.lse_run + (size_t)B * p->T * p->h;
    int e = cpattn::launch_finalize(a, stream);
    if (e) return cuda_fail(e, "finalize kernel");
    p->next_step = -1;
    return CPATTN_OK;
}

// ---- the backward as ring steps ("What context parallelism communicates": each rank keeps the
// gradient of its own queries; the key/value gradient of a block travels with the block as a
// second circulating block and returns to its owner) -------------------------------------------

namespace {

// Send right, receive left between two rank-major slot arrays: slot `dst` of rank r <- the
// block of rank r - 1 in `src` (two contiguous copies per array).
int ring_hop(const char* src, char* dst, size_t blk, int n_cp, cudaStream_t st) {
    const size_t all = blk * (size_t)n_cp;
    int e = 0;
    if (n_cp > 1) e = cudaMemcpyAsync(dst + blk, src, all - blk, cudaMemcpyDeviceToDevice, st);
    if (!e) e = cudaMemcpyAsync(dst, src + all - blk, blk, cudaMemcpyDeviceToDevice, st);
    return e;
}

cpattn_status_t check_bring_ws(const Plan& p, int B, const void* ws, size_t ws_bytes) {
    if (cpattn_status_t s = reject_ulysses(p)) return s;
    if (B <= 0) return fail(CPATTN_ERR_INVALID, "B must be positive");
    if (!ws) return fail(CPATTN_ERR_WORKSPACE, "workspace pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(ws) & 1023u) != 0) return fail(CPATTN_ERR_WORKSPACE, "workspace must be 1024-byte aligned");
    const size_t need = cpattn::ws_layout(p, B).bring_end;
    if (ws_bytes < need)
        return fail(CPATTN_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes, got " +
                                              std::to_string(ws_bytes));
    return CPATTN_OK;
}

}  // namespace

cpattn_status_t cpattn_backward_begin(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                      const void* o, const float* lse, const void* dout, const int32_t* pos, void* ws,
                                      size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    cpattn_status_t s = check_bring_ws(*p, B, ws, ws_bytes);
    if (s) return s;
    s = backward_prepare(*p, B, q, k, v, o, lse, dout, pos, nullptr, ws, ws_bytes, cpattn::ws_layout(*p, B).bring_end,
                         reinterpret_cast<cudaStream_t>(stream));
    if (s) return s;
    p->next_bstep = 0;
    p->bring_B = B;
    return CPATTN_OK;
}

cpattn_status_t cpattn_backward_ring_step(cpattn_plan_t plan, int B, int step, float scale, void* ws, size_t ws_bytes,
                                          cpattn_stream_t compute, cpattn_stream_t copy) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    cpattn_status_t s = check_bring_ws(*p, B, ws, ws_bytes);
    if (s) return s;
    if (step < 0 || step >= p->n_cp) return fail(CPATTN_ERR_INVALID, "step out of range");
    if (p->next_bstep != step)
        return fail(CPATTN_ERR_INVALID, "backward ring steps must follow cpattn_backward_begin in order 0..n_cp-1 "
                                        "(expected step " + std::to_string(p->next_bstep) + ")");
    if (B != p->bring_B) return fail(CPATTN_ERR_INVALID, "B differs from the batch cpattn_backward_begin placed");
    cudaStream_t cst = reinterpret_cast<cudaStream_t>(compute), xst = reinterpret_cast<cudaStream_t>(copy);
    int e = 0;
    auto mk = [&](CUevent_st*& ev) { if (!ev && !e) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming); };
    for (int i = 0; i < 2; ++i) { mk(p->bev_kv[i]); mk(p->bev_used[i]); mk(p->bev_circ[i]); }
    mk(p->bev_ready);
    mk(p->bev_start);
    if (e) return cuda_fail(e, "cudaEventCreate");
    cpattn::WsLayout w = cpattn::ws_layout(*p, B);
    const int slot = step & 1, nxt = (step + 1) & 1;

    if (step == 0) {   // the copy stream must see the placed blocks
        if ((e = cudaEventRecord(p->bev_start, cst)) || (e = cudaStreamWaitEvent(xst, p->bev_start, 0)))
            return cuda_fail(e, "stream ordering");
    } else if ((e = cudaStreamWaitEvent(cst, p->bev_kv[slot], 0))) {   // this step's K, V have arrived
        return cuda_fail(e, "cudaStreamWaitEvent");
    }
    // dK/dV of the visiting blocks against this rank's queries, and this step's dQ
    cpattn::BwdLaunch a = bwd_args(*p, B, scale, ws, nullptr);
    a.step = step;
    if (step > 0) { a.kL = at<char>(ws, w.bstageK[slot]); a.vL = at<char>(ws, w.bstageV[slot]); }
    // step 0 starts the partial dK/dV sums; later steps add into the sums that arrived with the
    // blocks, so the dK/dV kernel waits for that hop and the dQ kernel runs first, overlapping it
    a.dk_f32 = at<float>(ws, w.circK[slot]);
    a.dv_f32 = at<float>(ws, w.circV[slot]);
    a.dq_run = at<float>(ws, w.dq_run);
    if (step > 0) { a.dkdv_add = 1; a.dkdv_after = p->bev_circ[slot]; }
    std::string why;
    if ((e = cpattn::launch_backward(a, cst, &why))) return why.empty() ? cuda_fail(e, "backward kernels") : fail(CPATTN_ERR_CUDA, why);
    if ((e = cudaEventRecord(p->bev_used[slot], cst))) return cuda_fail(e, "cudaEventRecord");
    if ((e = cudaEventRecord(p->bev_ready, cst))) return cuda_fail(e, "cudaEventRecord");

    // K, V for the next step: slot nxt of rank r <- the block rank r - 1 holds now (issued before
    // the gradient hop so that it overlaps this step's kernels)
    const size_t blk_kv = 2 * (size_t)B * p->n * p->n_kv * p->d, blk_g = 2 * blk_kv;   // bf16, fp32 bytes
    if (step + 1 < p->n_cp) {
        if (step >= 1 && (e = cudaStreamWaitEvent(xst, p->bev_used[nxt], 0))) return cuda_fail(e, "cudaStreamWaitEvent");
        for (int t = 0; t < 2; ++t) {
            const char* src = step == 0 ? at<char>(ws, t ? w.vL : w.kL) : at<char>(ws, t ? w.bstageV[slot] : w.bstageK[slot]);
            if ((e = ring_hop(src, at<char>(ws, t ? w.bstageV[nxt] : w.bstageK[nxt]), blk_kv, p->n_cp, xst)))
                return cuda_fail(e, "cudaMemcpyAsync(ring hop)");
        }
        if ((e = cudaEventRecord(p->bev_kv[nxt], xst))) return cuda_fail(e, "cudaEventRecord");
    }
    // the partial dK/dV sums move on with their blocks; after the last step this hop returns each
    // block's gradient to its owner
    if ((e = cudaStreamWaitEvent(xst, p->bev_ready, 0))) return cuda_fail(e, "cudaStreamWaitEvent");
    for (int t = 0; t < 2; ++t)
        if ((e = ring_hop(at<char>(ws, t ? w.circV[slot] : w.circK[slot]), at<char>(ws, t ? w.circV[nxt] : w.circK[nxt]),
                          blk_g, p->n_cp, xst)))
            return cuda_fail(e, "cudaMemcpyAsync(gradient hop)");
    if ((e = cudaEventRecord(p->bev_circ[nxt], xst))) return cuda_fail(e, "cudaEventRecord");
    p->next_bstep = step + 1;
    return CPATTN_OK;
}

cpattn_status_t cpattn_backward_finalize(cpattn_plan_t plan, int B, void* dq, void* dk, void* dv, void* ws,
                                         size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    cpattn_status_t s = check_bring_ws(*p, B, ws, ws_bytes);
    if (s) return s;
    if (!dq || !dk || !dv || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(CPATTN_ERR_INVALID, "dq, dk and dv must be non-NULL and 16-byte aligned");
    if (p->next_bstep != p->n_cp) return fail(CPATTN_ERR_INVALID, "backward finalize needs all n_cp ring steps first");
    if (B != p->bring_B) return fail(CPATTN_ERR_INVALID, "B differs from the batch cpattn_backward_begin placed");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cpattn::WsLayout w = cpattn::ws_layout(*p, B);
    const int home = p->n_cp & 1;   // the slot the returning gradients arrived in
    int e = cudaStreamWaitEvent(st, p->bev_circ[home], 0);
    if (e) return cuda_fail(e, "cudaStreamWaitEvent");
    if ((e = cpattn::launch_unpermute_f32(at<float>(ws, w.dq_run), dq, B, p->T, p->n, p->m, p->h, p->d, p->n_cp, p->layout, st)) ||
        (e = cpattn::launch_unpermute_f32(at<float>(ws, w.circK[home]), dk, B, p->T, p->n, p->m, p->n_kv, p->d, p->n_cp,
                                          p->layout, st)) ||
        (e = cpattn::launch_unpermute_f32(at<float>(ws, w.circV[home]), dv, B, p->T, p->n, p->m, p->n_kv, p->d, p->n_cp,
                                          p->layout, st)))
        return cuda_fail(e, "gradient unpermute kernel");
    p->next_bstep = -1;
    return CPATTN_OK;
}

// ---- Ulysses ("Ulysses, splitting by heads instead") ---------------------------------------

cpattn_status_t cpattn_ulysses_plan(int64_t T, int h, int n_kv, int d_k, int n_cp, int causal, cpattn_plan_t* out) {
    if (!out) return fail(CPATTN_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (d_k != 64 && d_k != 128) return fail(CPATTN_ERR_UNSUPPORTED, "d_k must be 64 or 128");
    if (n_cp < 1 || h < 1 || n_kv < 1 || T < 1) return fail(CPATTN_ERR_INVALID, "T, h, n_kv and n_cp must be positive");
    if (h % n_kv) return fail(CPATTN_ERR_INVALID, "h must be a multiple of n_kv");
    if (h % n_cp) return fail(CPATTN_ERR_INVALID, "Ulysses gives every rank whole heads: h must be a multiple of n_cp");
    if (n_kv % n_cp && n_cp % n_kv)
        return fail(CPATTN_ERR_INVALID, "the KV heads split evenly (n_cp divides n_kv) or are replicated evenly (n_kv divides n_cp)");
    if (T % n_cp) return fail(CPATTN_ERR_INVALID, "T must be a multiple of n_cp (equal token shards)");
    Plan* p = new Plan();
    const int hp = h / n_cp, nkvp = n_kv >= n_cp ? n_kv / n_cp : 1;
    std::string why = cpattn::build_plan(*p, T, hp, nkvp, d_k, 1, CPATTN_CONTIGUOUS, causal);
    if (!why.empty()) {
        delete p;
        return fail(CPATTN_ERR_INVALID, why);
    }
    p->u_ncp = n_cp; p->u_h = h; p->u_nkv = n_kv;
    *out = reinterpret_cast<cpattn_plan_t>(p);
    return CPATTN_OK;
}

namespace {
struct UlyssesWs {
    size_t inner, qs, ks, vs, os, end;
};
UlyssesWs ulysses_ws(const Plan& p, int B) {
    const size_t bp = (size_t)B * p.u_ncp;
    auto up = [](size_t x) { return (x + 1023) / 1024 * 1024; };
    UlyssesWs w{};
    w.inner = 0;
    w.qs = up(cpattn::ws_layout(p, (int)bp).fwd_end);
    const size_t qbytes = bp * (size_t)p.T * p.h * p.d * 2, kvbytes = bp * (size_t)p.T * p.n_kv * p.d * 2;
    w.ks = up(w.qs + qbytes);
    w.vs = up(w.ks + kvbytes);
    w.os = up(w.vs + kvbytes);
    w.end = up(w.os + qbytes);
    return w;
}
cpattn_status_t need_ulysses(const Plan* p) {
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!p->u_ncp) return fail(CPATTN_ERR_INVALID, "the cpattn_ulysses_* calls need a plan made by cpattn_ulysses_plan");
    return CPATTN_OK;
}
}  // namespace

cpattn_status_t cpattn_ulysses_workspace_size(cpattn_plan_t plan, int B, size_t* bytes) {
    Plan* p = as_plan(plan);
    if (cpattn_status_t s = need_ulysses(p)) return s;
    if (!bytes || B <= 0) return fail(CPATTN_ERR_INVALID, "bytes and B > 0 required");
    *bytes = ulysses_ws(*p, B).end;
    return CPATTN_OK;
}

cpattn_status_t cpattn_ulysses_counts(cpattn_plan_t plan, int B, int64_t* bytes_recv) {
    Plan* p = as_plan(plan);
    if (cpattn_status_t s = need_ulysses(p)) return s;
    if (!bytes_recv || B <= 0) return fail(CPATTN_ERR_INVALID, "bytes_recv and B > 0 required");
    // Per rank: the other ranks' n tokens of its hp query heads and of its nkvp KV heads (K and V)
    // in the first all-to-all, and its own n tokens of the other ranks' heads of the output in the
    // second; 2 bytes a number.
    const int64_t n = p->T / p->u_ncp, others = p->u_ncp - 1;
    const int64_t per = (int64_t)B * n * p->d * 2 * others * (2 * (int64_t)p->h + 2 * (int64_t)p->n_kv);
    for (int r = 0; r < p->u_ncp; ++r) bytes_recv[r] = per;
    return CPATTN_OK;
}

cpattn_status_t cpattn_ulysses_forward(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                       const int32_t* pos, float scale, void* o, float* lse, void* ws, size_t ws_bytes,
                                       cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (cpattn_status_t s = need_ulysses(p)) return s;
    if (B <= 0) return fail(CPATTN_ERR_INVALID, "B must be positive");
    if (!q || !k || !v || !o || !lse) return fail(CPATTN_ERR_INVALID, "q, k, v, o and lse must be non-NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || (pos && !aligned16(pos)))
        return fail(CPATTN_ERR_INVALID, "q, k, v, pos, o and lse must be 16-byte aligned");
    if ((double)B * (double)p->T * p->u_h > 2.0e9) return fail(CPATTN_ERR_UNSUPPORTED, "B*T*h beyond 2e9 rows");
    if (!ws) return fail(CPATTN_ERR_WORKSPACE, "workspace pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(ws) & 1023u) != 0) return fail(CPATTN_ERR_WORKSPACE, "workspace must be 1024-byte aligned");
    const UlyssesWs uw = ulysses_ws(*p, B);
    if (ws_bytes < uw.end)
        return fail(CPATTN_ERR_WORKSPACE, "workspace too small: need " + std::to_string(uw.end) + " bytes, got " +
                                              std::to_string(ws_bytes));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int Bp = B * p->u_ncp;
    cpattn::UlyssesArgs u{};
    u.B = B; u.T = p->T; u.h = p->u_h; u.n_kv = p->u_nkv; u.d = p->d; u.n_cp = p->u_ncp; u.hp = p->h; u.nkvp = p->n_kv;
    u.q = q; u.k = k; u.v = v;
    u.qs = at<char>(ws, uw.qs); u.ks = at<char>(ws, uw.ks); u.vs = at<char>(ws, uw.vs);
    u.os = at<char>(ws, uw.os); u.o = o;
    int e = cpattn::launch_ulysses_split(u, st);                       // first all-to-all
    if (e) return cuda_fail(e, "Ulysses all-to-all (split)");
    // every rank's exact attention over all T tokens of its heads: one problem of B n_cp batches;
    // its lse [B n_cp][hp][T] is the natural lse [B][h][T] already
    cpattn_status_t s = prologue(*p, Bp, u.qs, u.ks, u.vs, pos, ws, st);
    if (s) return s;
    cpattn::AttnLaunch a = attn_args(*p, Bp, scale, ws);
    a.fused = 1; a.step = 0; a.kv_by_holder = 0;
    a.o = at<char>(ws, uw.os); a.lse = lse;
    std::string why;
    e = launch_attn(a, st, &why);
    if (e) return why.empty() ? cuda_fail(e, "attention kernel") : fail(CPATTN_ERR_CUDA, why);
    e = cpattn::launch_ulysses_merge(u, st);                           // second all-to-all
    if (e) return cuda_fail(e, "Ulysses all-to-all (merge)");
    return CPATTN_OK;
}

cpattn_status_t cpattn_merge(int S, int64_t rows, int h, int d, const float* o_parts, const float* lse_parts,
                             void* o_bf16, float* lse, cpattn_stream_t stream) {
    if (S <= 0 || rows <= 0 || h <= 0 || d <= 0 || d % 8) return fail(CPATTN_ERR_INVALID, "S, rows, h > 0 and d a positive multiple of 8 required");
    if (!o_parts || !lse_parts || !o_bf16 || !lse) return fail(CPATTN_ERR_INVALID, "NULL pointer");
    if (!aligned16(o_parts) || !aligned16(o_bf16)) return fail(CPATTN_ERR_INVALID, "o_parts and o must be 16-byte aligned");
    int e = cpattn::launch_merge(S, rows, h, d, o_parts, lse_parts, o_bf16, lse, stream);
    if (e) return cuda_fail(e, "merge kernel");
    return CPATTN_OK;
}

// ---- the all-gather variant ("What context parallelism communicates": all-gather the keys and
// values so every rank holds the full K and V, then one ordinary attention pass for the local
// queries; the gather is exposed, ahead of the kernel) -----------------------------------------

namespace {

cpattn_status_t check_gather_ws(const Plan& p, int B, const void* ws, size_t ws_bytes) {
    if (cpattn_status_t s = reject_ulysses(p)) return s;
    if (B <= 0) return fail(CPATTN_ERR_INVALID, "B must be positive");
    if (!ws) return fail(CPATTN_ERR_WORKSPACE, "workspace pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(ws) & 1023u) != 0) return fail(CPATTN_ERR_WORKSPACE, "workspace must be 1024-byte aligned");
    const size_t need = cpattn::ws_layout(p, B).gather_end;
    if (ws_bytes < need)
        return fail(CPATTN_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes, got " +
                                              std::to_string(ws_bytes));
    if ((double)p.n_cp * p.n_cp * B * p.n_kv * (double)p.n > 2.0e9)
        return fail(CPATTN_ERR_UNSUPPORTED, "gathered key/value rows beyond 2e9");
    return CPATTN_OK;
}

// Every rank r receives the blocks of all other ranks: its gathered copy is the whole rank-major
// K (and V) of the layout, which on one GPU is one device-to-device copy per rank and tensor.
cpattn_status_t gather_kv(const Plan& p, int B, void* ws, cudaStream_t st) {
    const cpattn::WsLayout w = cpattn::ws_layout(p, B);
    const size_t all = 2 * (size_t)B * p.T * p.n_kv * p.d;
    for (int r = 0; r < p.n_cp; ++r)
        for (int t = 0; t < 2; ++t) {
            int e = cudaMemcpyAsync(at<char>(ws, t ? w.gV : w.gK) + r * all, at<char>(ws, t ? w.vL : w.kL), all,
                                    cudaMemcpyDeviceToDevice, st);
            if (e) return cuda_fail(e, "cudaMemcpyAsync(all-gather)");
        }
    return CPATTN_OK;
}

cpattn_status_t gather_attend(const Plan& p, int B, float scale, const int32_t* lo, void* o, float* lse, void* ws,
                              cudaStream_t st, int doc_ids = 0) {
    const cpattn::WsLayout w = cpattn::ws_layout(p, B);
    cpattn::AttnLaunch a = attn_args(p, B, scale, ws);
    a.fused = 1; a.step = 0; a.kv_by_holder = 0;
    a.kv_k = at<char>(ws, w.gK); a.kv_v = at<char>(ws, w.gV);
    a.kv_rank_rows = (int64_t)p.n_cp * B * p.n_kv * p.n;
    a.kv_rows = (uint64_t)p.n_cp * a.kv_rank_rows;
    a.o = o; a.lse = lse;
    if (lo) { a.loL = at<int32_t>(ws, w.loL); a.tile_lo = at<int32_t>(ws, w.tile_lo); a.doc_ids = doc_ids; }
    std::string why;
    int e = launch_attn(a, st, &why);
    if (e) return why.empty() ? cuda_fail(e, "attention kernel") : fail(CPATTN_ERR_CUDA, why);
    return CPATTN_OK;
}

}  // namespace

cpattn_status_t cpattn_allgather_workspace_size(cpattn_plan_t plan, int B, size_t* bytes) {
    Plan* p = as_plan(plan);
    if (!p || !bytes || B <= 0) return fail(CPATTN_ERR_INVALID, "plan, bytes and B > 0 required");
    if (cpattn_status_t s = reject_ulysses(*p)) return s;
    *bytes = cpattn::ws_layout(*p, B).gather_end;
    return CPATTN_OK;
}

cpattn_status_t cpattn_allgather_counts(cpattn_plan_t plan, int B, int64_t* bytes_recv) {
    Plan* p = as_plan(plan);
    if (!p || B <= 0 || !bytes_recv) return fail(CPATTN_ERR_INVALID, "plan, B > 0 and bytes_recv required");
    if (cpattn_status_t s = reject_ulysses(*p)) return s;
    // the other n_cp - 1 ranks' K and V blocks, 2 bytes a number
    for (int r = 0; r < p->n_cp; ++r)
        bytes_recv[r] = (int64_t)(p->n_cp - 1) * 2 * 2 * B * p->n * p->n_kv * p->d;
    return CPATTN_OK;
}

cpattn_status_t cpattn_allgather_forward(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                         const int32_t* pos, const int32_t* lo, float scale, void* o, float* lse,
                                         void* ws, size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    cpattn_status_t s = check_inputs(*p, B, q, k, v, pos);
    if (s) return s;
    if (!o || !lse || !aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_INVALID, "o and lse must be non-NULL and 16-byte aligned");
    if (lo) {
        if (!p->causal) return fail(CPATTN_ERR_UNSUPPORTED, "a lower bound per query needs a causal plan");
        if (p->n_qt > 65535) return fail(CPATTN_ERR_UNSUPPORTED, "a lower bound per query supports up to 65535 tiles per rank");
        if (!aligned16(lo)) return fail(CPATTN_ERR_INVALID, "lo must be 16-byte aligned");
    }
    if ((s = check_gather_ws(*p, B, ws, ws_bytes))) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = prologue(*p, B, q, k, v, pos, ws, st, lo))) return s;
    if ((s = gather_kv(*p, B, ws, st))) return s;
    return gather_attend(*p, B, scale, lo, o, lse, ws, st);
}

cpattn_status_t cpattn_allgather_forward_docs(cpattn_plan_t plan, int B, const void* q, const void* k,
                                              const void* v, const int32_t* pos, const int32_t* doc, float scale,
                                              void* o, float* lse, void* ws, size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!doc || !aligned16(doc)) return fail(CPATTN_ERR_INVALID, "doc must be non-NULL and 16-byte aligned");
    cpattn_status_t s = check_inputs(*p, B, q, k, v, pos);
    if (s) return s;
    if (!o || !lse || !aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_INVALID, "o and lse must be non-NULL and 16-byte aligned");
    if ((s = check_gather_ws(*p, B, ws, ws_bytes))) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = prologue(*p, B, q, k, v, pos, ws, st, doc))) return s;
    if ((s = gather_kv(*p, B, ws, st))) return s;
    return gather_attend(*p, B, scale, doc, o, lse, ws, st, 1);
}

cpattn_status_t cpattn_allgather_gather(cpattn_plan_t plan, int B, void* ws, size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    cpattn_status_t s = check_gather_ws(*p, B, ws, ws_bytes);
    if (s) return s;
    return gather_kv(*p, B, ws, reinterpret_cast<cudaStream_t>(stream));
}

cpattn_status_t cpattn_allgather_attend(cpattn_plan_t plan, int B, float scale, void* o, float* lse, void* ws,
                                        size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!o || !lse || !aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_INVALID, "o and lse must be non-NULL and 16-byte aligned");
    cpattn_status_t s = check_gather_ws(*p, B, ws, ws_bytes);
    if (s) return s;
    return gather_attend(*p, B, scale, nullptr, o, lse, ws, reinterpret_cast<cudaStream_t>(stream));
}

// ---- one process of a multi-process ring ("Pass them around a ring": each rank computes against
// the block it holds while it sends that block to its right neighbour and receives the next one
// from its left). A process holds R consecutive ranks rank0 .. rank0 + R - 1; the library does
// the per-step attention of its ranks and the moves between its own ranks' slots, and the caller
// moves the one block that crosses to the next process. ----------------------------------------

namespace {

cpattn_status_t check_dist(const Plan& p, int B, int rank0, int R, const void* ws, size_t ws_bytes, const void* slot,
                           size_t slot_bytes) {
    if (cpattn_status_t s = reject_ulysses(p)) return s;
    if (B <= 0) return fail(CPATTN_ERR_INVALID, "B must be positive");
    if (R <= 0 || rank0 < 0 || rank0 + R > p.n_cp)
        return fail(CPATTN_ERR_INVALID, "ranks rank0 .. rank0 + R - 1 must lie in 0 .. n_cp - 1");
    if ((double)B * R * (double)p.n * p.h > 2.0e9) return fail(CPATTN_ERR_UNSUPPORTED, "B*R*n*h beyond 2e9 rows");
    const cpattn::DistLayout w = cpattn::dist_layout(p, B, R);
    if (ws) {
        if ((reinterpret_cast<uintptr_t>(ws) & 1023u) != 0) return fail(CPATTN_ERR_WORKSPACE, "workspace must be 1024-byte aligned");
        if (ws_bytes < w.ws_end)
            return fail(CPATTN_ERR_WORKSPACE, "workspace too small: need " + std::to_string(w.ws_end) + " bytes, got " +
                                                  std::to_string(ws_bytes));
    }
    if (slot) {
        if ((reinterpret_cast<uintptr_t>(slot) & 1023u) != 0) return fail(CPATTN_ERR_WORKSPACE, "slot must be 1024-byte aligned");
        if (slot_bytes < w.slot_end)
            return fail(CPATTN_ERR_WORKSPACE, "slot too small: need " + std::to_string(w.slot_end) + " bytes, got " +
                                                  std::to_string(slot_bytes));
    }
    return CPATTN_OK;
}

cpattn_status_t check_dist_state(const Plan& p, int B, int rank0, int R) {
    if (p.dist_next < 0) return fail(CPATTN_ERR_INVALID, "cpattn_dist_begin must come first");
    if (B != p.dist_B || rank0 != p.dist_rank0 || R != p.dist_R)
        return fail(CPATTN_ERR_INVALID, "B, rank0 and R differ from what cpattn_dist_begin placed");
    return CPATTN_OK;
}

}  // namespace

cpattn_status_t cpattn_dist_sizes(cpattn_plan_t plan, int B, int R, size_t* ws_bytes, size_t* slot_bytes,
                                  size_t* region_offset, size_t* block_bytes) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (cpattn_status_t s = check_dist(*p, B, 0, R, nullptr, 0, nullptr, 0)) return s;
    const cpattn::DistLayout w = cpattn::dist_layout(*p, B, R);
    if (ws_bytes) *ws_bytes = w.ws_end;
    if (slot_bytes) *slot_bytes = w.slot_end;
    if (region_offset) {
        region_offset[0] = w.slot_k; region_offset[1] = w.slot_v;
        region_offset[2] = w.slot_pos; region_offset[3] = w.slot_tile;
    }
    if (block_bytes) {
        block_bytes[0] = w.blk_k; block_bytes[1] = w.blk_v;
        block_bytes[2] = w.blk_pos; block_bytes[3] = w.blk_tile;
    }
    return CPATTN_OK;
}

cpattn_status_t cpattn_dist_begin(cpattn_plan_t plan, int B, int rank0, int R, const void* q, const void* k,
                                  const void* v, const int32_t* pos, const int32_t* lo, void* ws, size_t ws_bytes,
                                  void* slot, size_t slot_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!ws || !slot) return fail(CPATTN_ERR_WORKSPACE, "workspace and slot must be non-NULL");
    cpattn_status_t s = check_dist(*p, B, rank0, R, ws, ws_bytes, slot, slot_bytes);
    if (s) return s;
    if (!q || !k || !v) return fail(CPATTN_ERR_INVALID, "q, k and v must be non-NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (pos && !aligned16(pos)) || (lo && !aligned16(lo)))
        return fail(CPATTN_ERR_INVALID, "q, k, v, pos and lo must be 16-byte aligned");
    if (lo && !p->causal) return fail(CPATTN_ERR_UNSUPPORTED, "a lower bound per query needs a causal plan");
    if (lo && p->n_qt > 65535) return fail(CPATTN_ERR_UNSUPPORTED, "a lower bound per query supports up to 65535 tiles per rank");
    const cpattn::DistLayout w = cpattn::dist_layout(*p, B, R);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int e = cudaMemsetAsync(at<char>(ws, w.header), 0, sizeof(uint32_t) * cpattn::kHeaderWords, st);
    if (!e) e = cudaMemsetAsync(at<char>(ws, w.counts), 0, w.sched + sizeof(uint32_t) * (1 + (size_t)R) - w.counts, st);
    if (e) return cuda_fail(e, "cudaMemsetAsync(header)");
    // the plan's longest-first order of row groups, restricted to this process's ranks
    std::vector<int32_t> order;
    order.reserve((size_t)R * p->n_grp);
    for (int32_t rg : p->order) {
        const int r = rg / p->n_grp;
        if (r >= rank0 && r < rank0 + R) order.push_back((r - rank0) * p->n_grp + rg % p->n_grp);
    }
    if ((e = cpattn::launch_upload_i32(at<int32_t>(ws, w.order), order.data(), (int64_t)order.size(), st)))
        return cuda_fail(e, "order upload kernel");
    // the process's tokens are rank-major in each rank's local order: placement is the identity
    // over R ranks, and default positions are the tokens' natural positions in the whole sequence
    cpattn::PermuteArgs a{};
    a.B = B; a.T = (int64_t)R * p->n; a.n = p->n; a.m = 0; a.h = p->h; a.n_kv = p->n_kv; a.d = p->d; a.n_cp = R;
    a.layout = CPATTN_CONTIGUOUS; a.n_qt = p->n_qt;
    a.q = q; a.k = k; a.v = v; a.pos = pos;
    a.qL = at<char>(ws, w.qL); a.kL = at<char>(slot, w.slot_k); a.vL = at<char>(slot, w.slot_v);
    a.posL = at<int32_t>(ws, w.posL); a.tile_mm = at<int32_t>(ws, w.tile_mm);
    // the queries' lower bounds stay with the queries: only the keys' positions travel
    a.lo = lo; a.loL = at<int32_t>(ws, w.loL); a.tile_lo = at<int32_t>(ws, w.tile_lo);
    a.dflt_ncp = p->n_cp; a.dflt_layout = p->layout; a.dflt_rank0 = rank0; a.dflt_m = p->m;
    a.v_f16 = 1;
    a.header = at<uint32_t>(ws, w.header);
    if ((e = cpattn::launch_permute(a, st))) return cuda_fail(e, "permute kernel");
    // each block carries its position tables with it around the ring
    e = cudaMemcpyAsync(at<char>(slot, w.slot_pos), at<char>(ws, w.posL), w.blk_pos * R, cudaMemcpyDeviceToDevice, st);
    if (!e)
        e = cudaMemcpyAsync(at<char>(slot, w.slot_tile), at<char>(ws, w.tile_mm), w.blk_tile * R,
                            cudaMemcpyDeviceToDevice, st);
    if (e) return cuda_fail(e, "cudaMemcpyAsync(position tables)");
    p->dist_next = 0; p->dist_B = B; p->dist_rank0 = rank0; p->dist_R = R; p->dist_lo = lo ? 1 : 0;
    return CPATTN_OK;
}

namespace {
// Local rank i + 1's block of regions x_begin..x_end - 1 in dst <- local rank i's in src (i < R - 1),
// and with wrap local rank 0's <- local rank R - 1's: device-to-device copies on st.
int shift_regions(const cpattn::DistLayout& w, const void* src_slot, void* dst_slot, int R, int wrap, cudaStream_t st,
                  int x_begin, int x_end) {
    const size_t off[4] = {w.slot_k, w.slot_v, w.slot_pos, w.slot_tile};
    const size_t blk[4] = {w.blk_k, w.blk_v, w.blk_pos, w.blk_tile};
    const char* src = static_cast<const char*>(src_slot);
    char* dst = static_cast<char*>(dst_slot);
    for (int x = x_begin; x < x_end; ++x) {
        int e = 0;
        // local rank i + 1 receives the block local rank i holds now
        if (R > 1) e = cudaMemcpyAsync(dst + off[x] + blk[x], src + off[x], blk[x] * (R - 1), cudaMemcpyDeviceToDevice, st);
        // a process holding the whole ring passes its last block to its own first rank
        if (!e && wrap)
            e = cudaMemcpyAsync(dst + off[x], src + off[x] + blk[x] * (R - 1), blk[x], cudaMemcpyDeviceToDevice, st);
        if (e) return e;
    }
    return 0;
}

// cpattn_dist_step, and with next_slot the shift into it: K and V by the step kernel's idle warps,
// the position tables by copies on the same stream after it.
cpattn_status_t dist_step_impl(cpattn_plan_t plan, int B, int rank0, int R, int step, float scale, const void* slot,
                               void* next_slot, int wrap, size_t slot_bytes, void* ws, size_t ws_bytes,
                               cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!ws || !slot) return fail(CPATTN_ERR_WORKSPACE, "workspace and slot must be non-NULL");
    cpattn_status_t s = check_dist(*p, B, rank0, R, ws, ws_bytes, slot, slot_bytes);
    if (s) return s;
    if (next_slot) {
        if (next_slot == slot) return fail(CPATTN_ERR_INVALID, "the two slots must differ");
        if ((s = check_dist(*p, B, 0, R, nullptr, 0, next_slot, slot_bytes))) return s;
    }
    if ((s = check_dist_state(*p, B, rank0, R))) return s;
    if (step != p->dist_next)
        return fail(CPATTN_ERR_INVALID, "ring steps must follow cpattn_dist_begin in order 0..n_cp-1 (expected step " +
                                            std::to_string(p->dist_next) + ")");
    const cpattn::DistLayout w = cpattn::dist_layout(*p, B, R);
    cpattn::AttnLaunch a{};
    a.B = B; a.T = p->T; a.n = p->n; a.m = p->m; a.h = p->h; a.n_kv = p->n_kv; a.d = p->d; a.n_cp = R;
    a.layout = p->layout; a.causal = p->causal; a.n_qt = p->n_qt; a.pair_heads = p->pair_heads; a.n_grp = p->n_grp;
    a.sched = at<uint32_t>(ws, w.sched);
    a.unit_tiles = at<int32_t>(ws, w.unit_tiles);
    a.walk_tab = at<int32_t>(ws, w.walk_tab);
    a.walk_nz = at<unsigned long long>(ws, w.walk_nz);
    a.scale_log2 = resolve_scale(*p, scale);
    // every local rank attends to the one block it holds: a one-step walk in which the block read
    // is the holder's own slot entry, with the position tables that travelled with it
    a.fused = 0; a.step = 0; a.first = step == 0 ? 1 : 0;
    a.qL = at<char>(ws, w.qL);
    a.kv_k = const_cast<char*>(static_cast<const char*>(slot) + w.slot_k);
    a.kv_v = const_cast<char*>(static_cast<const char*>(slot) + w.slot_v);
    a.kv_by_holder = 1;
    a.posL = at<int32_t>(ws, w.posL); a.tile_mm = at<int32_t>(ws, w.tile_mm);
    a.kposL = reinterpret_cast<const int32_t*>(static_cast<const char*>(slot) + w.slot_pos);
    a.ktile_mm = reinterpret_cast<const int32_t*>(static_cast<const char*>(slot) + w.slot_tile);
    a.order = at<int32_t>(ws, w.order);
    a.counts = at<unsigned long long>(ws, w.counts);
    a.o_run = at<float>(ws, w.o_run); a.lse_run = at<float>(ws, w.lse_run);
    a.l_run = a.lse_run + (size_t)B * R * p->n * p->h;
    if (p->dist_lo) { a.loL = at<int32_t>(ws, w.loL); a.tile_lo = at<int32_t>(ws, w.tile_lo); }
    a.header = at<uint32_t>(ws, w.header);
    a.timeout_ns = 2000000000ull;
    a.reserved_sms = p->reserved_sms;
    if (next_slot) {
        a.hop_src_k = static_cast<const char*>(slot) + w.slot_k;
        a.hop_src_v = static_cast<const char*>(slot) + w.slot_v;
        a.hop_dst_k = static_cast<char*>(next_slot) + w.slot_k;
        a.hop_dst_v = static_cast<char*>(next_slot) + w.slot_v;
        a.hop_words = (int64_t)(w.blk_k * R / 16);
        a.hop_blk = (int64_t)(w.blk_k / 16);
        a.hop_wrap = wrap ? 1 : 0;
    }
    std::string why;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int e = launch_attn(a, st, &why);
    if (e) return why.empty() ? cuda_fail(e, "attention kernel") : fail(CPATTN_ERR_CUDA, why);
    if (next_slot && (e = shift_regions(w, slot, next_slot, R, wrap, st, 2, 4))) return cuda_fail(e, "cudaMemcpyAsync(ring hop)");
    p->dist_next = step + 1;
    return CPATTN_OK;
}
}  // namespace

cpattn_status_t cpattn_dist_step(cpattn_plan_t plan, int B, int rank0, int R, int step, float scale,
                                 const void* slot, size_t slot_bytes, void* ws, size_t ws_bytes,
                                 cpattn_stream_t stream) {
    return dist_step_impl(plan, B, rank0, R, step, scale, slot, nullptr, 0, slot_bytes, ws, ws_bytes, stream);
}

cpattn_status_t cpattn_dist_step_shift(cpattn_plan_t plan, int B, int rank0, int R, int step, float scale,
                                       const void* slot, void* next_slot, int wrap, size_t slot_bytes, void* ws,
                                       size_t ws_bytes, cpattn_stream_t stream) {
    if (!next_slot) return fail(CPATTN_ERR_INVALID, "next_slot must be non-NULL");
    return dist_step_impl(plan, B, rank0, R, step, scale, slot, next_slot, wrap, slot_bytes, ws, ws_bytes, stream);
}

cpattn_status_t cpattn_dist_shift(cpattn_plan_t plan, int B, int R, const void* src_slot, void* dst_slot,
                                  size_t slot_bytes, int wrap, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!src_slot || !dst_slot) return fail(CPATTN_ERR_INVALID, "slots must be non-NULL");
    if (src_slot == dst_slot) return fail(CPATTN_ERR_INVALID, "the two slots must differ");
    cpattn_status_t s = check_dist(*p, B, 0, R, nullptr, 0, dst_slot, slot_bytes);
    if (s) return s;
    if ((s = check_dist(*p, B, 0, R, nullptr, 0, src_slot, slot_bytes))) return s;
    const cpattn::DistLayout w = cpattn::dist_layout(*p, B, R);
    const int e = shift_regions(w, src_slot, dst_slot, R, wrap, reinterpret_cast<cudaStream_t>(stream), 0, 4);
    if (e) return cuda_fail(e, "cudaMemcpyAsync(ring hop)");
    return CPATTN_OK;
}

cpattn_status_t cpattn_dist_finalize(cpattn_plan_t plan, int B, int rank0, int R, void* o, float* lse, void* ws,
                                     size_t ws_bytes, cpattn_stream_t stream) {
    Plan* p = as_plan(plan);
    if (!p) return fail(CPATTN_ERR_INVALID, "plan is NULL");
    if (!ws) return fail(CPATTN_ERR_WORKSPACE, "workspace must be non-NULL");
    cpattn_status_t s = check_dist(*p, B, rank0, R, ws, ws_bytes, nullptr, 0);
    if (s) return s;
    if ((s = check_dist_state(*p, B, rank0, R))) return s;
    if (p->dist_next != p->n_cp) return fail(CPATTN_ERR_INVALID, "finalize needs all n_cp ring steps first");
    if (!o || !lse || !aligned16(o) || !aligned16(lse)) return fail(CPATTN_ERR_INVALID, "o and lse must be non-NULL and 16-byte aligned");
    const cpattn::DistLayout w = cpattn::dist_layout(*p, B, R);
    cpattn::FinalizeArgs a{};
    a.B = B; a.T = (int64_t)R * p->n; a.n = p->n; a.m = 0; a.h = p->h; a.d = p->d; a.n_cp = R;
    a.layout = CPATTN_CONTIGUOUS;
    a.o_run = at<float>(ws, w.o_run); a.lse_run = at<float>(ws, w.lse_run); a.o = o; a.lse = lse;
    a.l_run = a.lse_run + (size_t)B * R * p->n * p->h;
    int e = cpattn::launch_finalize(a, stream);
    if (e) return cuda_fail(e, "finalize kernel");
    p->dist_next = -1;
    return CPATTN_OK;
}

cpattn_status_t cpattn_tile_counts(cpattn_plan_t plan, int B, const void* ws, int64_t* full, int64_t* diag) {
    Plan* p = as_plan(plan);
    if (!p || !ws || B <= 0) return fail(CPATTN_ERR_INVALID, "plan, ws and B > 0 required");
    cpattn::WsLayout w = cpattn::ws_layout(*p, B);
    const size_t nn = (size_t)p->n_cp * p->n_cp;
    std::vector<unsigned long long> buf(2 * nn);
    int e = cudaMemcpy(buf.data(), static_cast<const char*>(ws) + w.counts, sizeof(uint64_t) * 2 * nn,
                       cudaMemcpyDeviceToHost);
    if (e) return cuda_fail(e, "cudaMemcpy(counts)");
    for (size_t i = 0; i < nn; ++i) {
        if (full) full[i] = (int64_t)buf[2 * i];
        if (diag) diag[i] = (int64_t)buf[2 * i + 1];
    }
    return CPATTN_OK;
}

cpattn_status_t cpattn_check(cpattn_plan_t plan, const void* ws) {
    (void)plan;
    if (!ws) return fail(CPATTN_ERR_WORKSPACE, "workspace pointer is NULL");
    uint32_t hdr[2] = {0, 0};
    int e = cudaMemcpy(hdr, ws, sizeof(hdr), cudaMemcpyDeviceToHost);
    if (e) return cuda_fail(e, "cudaMemcpy(header)");
    if (hdr[cpattn::kErrFlags] & cpattn::kErrRangeFlag)
        return fail(CPATTN_ERR_INVALID, "v holds a value outside the fp16 range (|v| > 65504, inf or NaN): the "
                                        "forward's P V product runs in fp16; the outputs were not computed");
    if (hdr[cpattn::kErrFlags] & cpattn::kErrTimeoutFlag) {
        char buf[128];
        std::snprintf(buf, sizeof buf, "device wait timed out (wait site %u)", hdr[cpattn::kErrWhere]);
        return fail(CPATTN_ERR_TIMEOUT, buf);
    }
    return CPATTN_OK;
}

cpattn_status_t cpattn_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t timeout_ns, cpattn_stream_t stream) {
    if (!ws || ws_bytes < sizeof(uint32_t) * cpattn::kHeaderWords) return fail(CPATTN_ERR_WORKSPACE, "workspace too small");
    int e = cudaMemsetAsync(ws, 0, sizeof(uint32_t) * cpattn::kHeaderWords, reinterpret_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, "cudaMemsetAsync(header)");
    e = cpattn::launch_wait_selftest(static_cast<uint32_t*>(ws), timeout_ns, stream);
    if (e) return cuda_fail(e, "wait self-test kernel");
    return CPATTN_OK;
}

}  // extern "C"
