// internal.h -- plan, workspace layout and launcher declarations shared by the host code and
// the CUDA kernels of libcpattn. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/cpattn.h"

struct CUevent_st;

namespace cpattn {

constexpr int kBlockQ = 128;   // query rows per tile (the tcgen05 MMA M)
constexpr int kBlockK = 128;   // keys per tile (the QK^T MMA N, the PV MMA K)

// Workspace header words (uint32), written by kernels, read by cpattn_check.
enum HeaderWord : int { kErrFlags = 0, kErrWhere = 1, kHeaderWords = 64 };
enum ErrFlag : uint32_t { kErrTimeoutFlag = 1u, kErrRangeFlag = 2u };

// Byte offsets of the regions inside the caller's workspace, all 1024-aligned.
struct WsLayout {
    size_t header = 0;      // uint32[kHeaderWords]
    size_t posL = 0;        // int32 [n_cp][n]: position id of (rank, local index)
    size_t tile_mm = 0;     // int32x4 [n_cp][n_qt]: min, max position of each tile, min over the
                            // tiles from this one to the end of its block, max over the tiles
                            // from the start of its block to this one
    size_t order = 0;       // int32 [n_cp * n_qt]: (rank, q-tile) pairs, longest first
    size_t counts = 0;      // uint64 [n_cp][n_cp][2]: tiles computed per (rank, step), FULL / DIAG
    size_t sched = 0;       // uint32 [1 + n_cp]: work counters of the persistent kernel (fused, each step)
    size_t loL = 0;         // int32 [n_cp][n]: lowest visible key position of (rank, local index) (document masks)
    size_t tile_lo = 0;     // int32x4 [n_cp][n_qt]: min and max of loL over each query tile
    size_t unit_tiles = 0;  // int32 [n_cp * n_qt]: key tiles a unit of row group (r, group) visits in
                            // the current launch (written by the attention launch itself)
    size_t walk_tab = 0;    // int32 [n_cp * n_qt][n_cp]: document masks: visited key-tile range per row group and step
    size_t walk_nz = 0;     // uint64 [n_cp * n_qt]: document masks: the steps with visited tiles
    size_t walk_bits = 0;   // uint64 [n_cp * n_qt][n_cp][ceil(n_qt / 64)]: document ids: visited key tiles
    size_t order_masked = 0;  // int32 [n_cp * n_qt]: masks: row groups by the masked walk's tile counts
    size_t qL = 0;          // bf16 [n_cp][B][h][n][d]
    size_t kL = 0, vL = 0;  // bf16 [n_cp][B][n_kv][n][d]
    size_t fwd_end = 0;     // end of what cpattn_forward needs
    size_t stageK[2] = {0, 0}, stageV[2] = {0, 0};  // ring stage slots, same shape as kL
    size_t o_run = 0;       // fp32 [n_cp][B][h][n][d] running output, unnormalised (relative to m_run)
    size_t lse_run = 0;     // fp32 [n_cp][B][h][n] running maximum m_run (log2 units), then the same
                            // shape of running sums l_run
    size_t ring_end = 0;
    // all-gather variant (after fwd_end, overlapping the ring-step regions): every rank's gathered
    // copy of the whole K and V, [n_cp holder][n_cp source][B][n_kv][n][d] bf16 each
    size_t gK = 0, gV = 0, gather_end = 0;
    // backward (after fwd_end; the ring-step regions are not used by the backward)
    size_t doL = 0;         // bf16 [n_cp][B][h][n][d] output gradient in layout order
    size_t lse2 = 0;        // fp32 [n_cp][B][h][n_qt * 128] -lse * log2(e) of the forward (padding 0)
    size_t Dl = 0;          // fp32 [n_cp][B][h][n_qt * 128] -D = -<dO, O> of every query row (padding 0)
    size_t bwd_order = 0;   // int32 [2][n_cp * n_qt]: order_q, then order_kv
    size_t bwd_end = 0;
    // backward ring-step path (after bwd_end): K/V stage slots, the circulating fp32 dK/dV
    // partial sums (two slots), and the running fp32 dQ; all [n_cp][B][...][n][d] with the rank
    // index the block's current holder (dQ: its own rank)
    size_t bstageK[2] = {0, 0}, bstageV[2] = {0, 0};
    size_t circK[2] = {0, 0}, circV[2] = {0, 0};
    size_t dq_run = 0;
    size_t bring_end = 0;
};

struct Plan {
    int64_t T = 0, n = 0, m = 0;   // tokens, tokens per rank, zigzag chunk
    int h = 0, n_kv = 0, d = 0, n_cp = 0, layout = 0, causal = 0;
    int n_qt = 0;                   // tiles per rank block (query and key tiles have one size)
    int pair_heads = 0;             // a CTA pairs two heads of one KV group (else two adjacent q-tiles)
    int n_grp = 0;                  // row groups per rank: n_qt when pairing heads, ceil(n_qt / 2) otherwise
    std::vector<int32_t> order;     // (r * n_grp + group), longest first
    std::vector<int32_t> order_q;   // backward: (r * n_qt + q-tile), most visible key tiles first
    std::vector<int32_t> order_kv;  // backward: (r * n_qt + key tile), most visible query tiles first
    std::vector<int64_t> full, diag, skip;  // [n_cp][n_cp] by (rank, step), per (b, head)
    std::vector<int64_t> pairs;             // [n_cp]
    std::vector<int64_t> half_units;        // [n_cp]
    // ring-step path state (created on first use)
    CUevent_st* ev_step[2] = {nullptr, nullptr};
    CUevent_st* ev_copy[2] = {nullptr, nullptr};
    CUevent_st* ev_start = nullptr;
    int next_step = -1;             // step expected next on the ring path (-1: permute first)
    int ring_hop_kernel = 0;        // this pass's hops run in the step kernels (no copy stream)
    int ring_B = 0;                 // batch size cpattn_permute placed (the steps must use the same)
    // backward ring-step path state: K/V of a step arrived, a stage slot's kernels done, the
    // circulating partial ready to send (after the step's add), a partial arrived
    CUevent_st* bev_kv[2] = {nullptr, nullptr};
    CUevent_st* bev_used[2] = {nullptr, nullptr};
    CUevent_st* bev_ready = nullptr;
    CUevent_st* bev_circ[2] = {nullptr, nullptr};
    CUevent_st* bev_start = nullptr;
    int next_bstep = -1;            // step expected next on the backward ring path (-1: begin first)
    // multi-process ring (cpattn_dist_*): the step expected next and what cpattn_dist_begin placed
    int dist_next = -1, dist_B = 0, dist_rank0 = 0, dist_R = 0, dist_lo = 0;
    int bring_B = 0;                // batch size cpattn_backward_begin placed
    // Ulysses plans (cpattn_ulysses_plan): the attention above is the per-rank problem (T tokens,
    // h / u_ncp query heads, its KV heads, one rank); these are the outer shape. 0 otherwise.
    int u_ncp = 0, u_h = 0, u_nkv = 0;
    // SMs the persistent attention launches leave free (cpattn_plan_set_reserved_sms)
    int reserved_sms = 0;
};

// One-time set-up per device (kernel attributes), safe when several host threads drive several
// devices: f() runs under the lock until it succeeds once on a device; devices beyond the table
// run it on every call.
struct PerDeviceOnce {
    static constexpr int kMax = 64;
    std::mutex mu;
    bool done[kMax] = {};
    template <class F>
    int run(int dev, F&& f) {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 0 && dev < kMax && done[dev]) return 0;
        const int e = f();
        if (e == 0 && dev >= 0 && dev < kMax) done[dev] = true;
        return e;
    }
};

WsLayout ws_layout(const Plan& p, int B);

// One process of a multi-process ring holds R consecutive ranks: its workspace (query side and
// running state) and its key/value stage slot (the blocks it holds, with their position tables).
struct DistLayout {
    size_t header = 0, posL = 0, tile_mm = 0, order = 0, counts = 0, sched = 0, unit_tiles = 0, walk_tab = 0,
           walk_nz = 0, loL = 0, tile_lo = 0, qL = 0, o_run = 0, lse_run = 0, ws_end = 0;
    size_t slot_k = 0, slot_v = 0, slot_pos = 0, slot_tile = 0, slot_end = 0;   // offsets in a slot
    size_t blk_k = 0, blk_v = 0, blk_pos = 0, blk_tile = 0;                     // one rank's block, bytes
};
DistLayout dist_layout(const Plan& p, int B, int R);
void set_last_error(const std::string& msg);
int64_t token_of(const Plan& p, int r, int64_t j);   // natural token of (rank, local index)

// ---- kernels (enqueue only; return a cudaError_t as int) --------------------------------
struct PermuteArgs {
    int B, T_is_int; int64_t T, n, m; int h, n_kv, d, n_cp, layout, n_qt;
    const void* q; const void* k; const void* v; const int32_t* pos;
    void* qL; void* kL; void* vL; int32_t* posL; int32_t* tile_mm;
    const int32_t* lo; int32_t* loL; int32_t* tile_lo;   // optional per-query lower bound (NULL: none)
    // With pos NULL and dflt_ncp > 0, the position of (rank r, local index j) is its natural token
    // under a plan of dflt_ncp ranks and layout dflt_layout, for rank dflt_rank0 + r (the tokens
    // one process of a multi-process ring holds); otherwise it is the natural index here.
    int dflt_ncp = 0, dflt_layout = 0, dflt_rank0 = 0;
    int64_t dflt_m = 0;
    int v_f16 = 0;   // write V in fp16 (exact for |v| <= 65504) for the forward's fp16 P V product
    uint32_t* header = nullptr;   // v_f16: a value outside the fp16 range sets kErrRangeFlag here
};
int launch_permute(const PermuteArgs& a, void* stream);

struct AttnLaunch {
    int B; int64_t T, n, m; int h, n_kv, d, n_cp, layout, causal, n_qt, pair_heads, n_grp;
    uint32_t* sched;  // work counter of this launch (zeroed before the launch)
    int32_t* unit_tiles;  // [n_cp * n_grp] scratch: key tiles per row group for this launch
    int32_t* walk_tab;    // [n_cp * n_grp][n_cp] scratch (document masks)
    unsigned long long* walk_nz;  // [n_cp * n_grp] scratch (document masks)
    float scale_log2;
    int fused;        // 1: all ring steps, natural-order bf16 output; 0: one step, merge into running state
    int step;         // ring step (fused == 0)
    const void* qL; const void* kv_k; const void* kv_v;   // K/V base: kL/vL or a stage slot
    int kv_by_holder; // K/V rows indexed by the holder rank r instead of the source rank
    const int32_t* posL; const int32_t* tile_mm; const int32_t* order;
    const int32_t* loL; const int32_t* tile_lo;   // document-mask lower bounds, or NULL
    unsigned long long* counts;     // tiles computed per (rank, step, class)
    void* o; float* lse;            // fused outputs (natural order)
    float* o_run; float* lse_run;   // ring-step running state: O (unnormalised), maximum m_run
    float* l_run = nullptr;         //   and sum l_run (log2 units; see the attention kernel's epilogue)
    uint32_t* header;
    uint64_t timeout_ns;
    // Key-side position tables when they are not posL / tile_mm (indexed like them by the rank
    // whose block is read): the blocks held by one process of a multi-process ring carry their own.
    const int32_t* kposL = nullptr; const int32_t* ktile_mm = nullptr;
    int first = -1;            // ring step: write (1) or merge into (0) the running state; -1: step == 0
    int64_t kv_rank_rows = 0;  // all-gather: K/V rows between the gathered copies of consecutive ranks
    // ring step: the hop to the next step done by the kernel's idle warps (hop_words 16-byte words
    // per tensor, 0: none); word w of hop_src_* goes to (w + hop_blk) mod hop_words of hop_dst_*
    const void* hop_src_k = nullptr; const void* hop_src_v = nullptr;
    void* hop_dst_k = nullptr; void* hop_dst_v = nullptr;
    int64_t hop_words = 0, hop_blk = 0;
    int hop_wrap = 1;          // the last rank's block goes to rank 0 (0: rank 0's is left alone)
    uint64_t kv_rows = 0;      // rows the K/V tensor maps span (0: n_cp B n_kv n)
    int doc_ids = 0;           // loL / tile_lo hold document ids (else a per-query lower bound)
    int reserved_sms = 0;      // SMs the persistent grid leaves free for concurrent work
    int32_t* order_scratch = nullptr;  // masks: [n_cp * n_grp] row groups sorted by this launch's tile counts
    unsigned long long* walk_bits = nullptr;   // document ids: [n_cp * n_grp][n_cp][ceil(n_qt / 64)] scratch
};
int launch_attention(const AttnLaunch& a, void* stream, std::string* why);

struct FinalizeArgs {
    int B; int64_t T, n, m; int h, d, n_cp, layout;
    const float* o_run; const float* lse_run; const float* l_run; void* o; float* lse;
};
int launch_finalize(const FinalizeArgs& a, void* stream);

int launch_merge(int S, int64_t rows, int h, int d, const float* o_parts, const float* lse_parts, void* o,
                 float* lse, void* stream);

int launch_wait_selftest(uint32_t* header, uint64_t timeout_ns, void* stream);

// Copy n int32 values from host memory to dst by kernel parameters (no host staging buffer).
int launch_upload_i32(int32_t* dst, const int32_t* host, int64_t n, void* stream);

// cpattn_forward's body, on a given workspace (the caller's, or the allocation-free entry
// point's static scratch).
cpattn_status_t forward_with_workspace(cpattn_plan_t plan, int B, const void* q, const void* k, const void* v,
                                       const int32_t* pos, float scale, void* o, float* lse, void* ws,
                                       size_t ws_bytes, cpattn_stream_t stream);

// Ulysses all-to-alls: natural q [B][T][h][d], k/v [B][T][n_kv][d] to per-rank head shards
// qs [B n_cp][T][hp][d], ks/vs [B n_cp][T][nkvp][d] (batch b n_cp + r'), and the output os
// [B n_cp][T][hp][d] back to natural o [B][T][h][d].
struct UlyssesArgs {
    int B; int64_t T; int h, n_kv, d, n_cp, hp, nkvp;
    const void* q; const void* k; const void* v; void* qs; void* ks; void* vs;
    const void* os; void* o;
};
int launch_ulysses_split(const UlyssesArgs& a, void* stream);
int launch_ulysses_merge(const UlyssesArgs& a, void* stream);

struct BwdPrepArgs {
    int B; int64_t T, n, m; int h, d, n_cp, layout, n_qt;
    const void* o; const void* dout; const float* lse;   // natural order
    void* doL; float* nlse2L; float* nDL;                  // layout order
};
int launch_bwd_prep(const BwdPrepArgs& a, void* stream);

struct BwdLaunch {
    int B; int64_t T, n, m; int h, n_kv, d, n_cp, layout, causal, n_qt;
    float scale;
    const void* qL; const void* kL; const void* vL; const void* doL;
    const float* nlse2L; const float* nDL;
    const int32_t* posL; const int32_t* tile_mm;
    const int32_t* order_q; const int32_t* order_kv;   // longest-first unit orders
    const int32_t* loL; const int32_t* tile_lo;         // document-mask lower bounds, or NULL
    void* dq; void* dk; void* dv;                         // natural order, bf16
    uint32_t* header;
    uint64_t timeout_ns;
    // one ring step (step >= 0; -1: the whole walk, fused): K/V rows taken from kL/vL indexed by
    // the holder rank, the dK/dV contribution written as fp32 by holder (dk_f32, dv_f32) and dQ
    // added into the running fp32 dq_run (written at step 0)
    int step = -1;
    float* dk_f32 = nullptr; float* dv_f32 = nullptr; float* dq_run = nullptr;
    // dkdv_add: the dK/dV contribution is added into dk_f32 / dv_f32 (the partial sums) by
    // reductions instead of written; dkdv_after (a cudaEvent_t, or NULL): the dQ kernel is
    // launched first and the dK/dV kernel after a stream wait on this event
    int dkdv_add = 0;
    void* dkdv_after = nullptr;
};
int launch_backward(const BwdLaunch& a, void* stream, std::string* why);

// acc[i] += c[i] over n floats (16-byte aligned, n a multiple of 4)
// fp32 [n_cp][B][H][n][d] in layout order -> bf16 [B][T][H][d] in natural order
int launch_unpermute_f32(const float* src, void* dst, int B, int64_t T, int64_t n, int64_t m, int H, int d, int n_cp,
                         int layout, void* stream);

}  // namespace cpattn
