// plan.cpp -- host planning for the virtual-rank ring: token placement, block classes, work
// and byte counters, the longest-first order of query tiles and the workspace layout.
//
// Placement follows "Context and expert parallelism", section "The causal mask unbalances the
// sequence" (contiguous chunks; zigzag chunks r and 2n_cp-1-r; round-robin stripes), and
// "primitive-context-parallel", section "What it does" (rank i holds [i*N/cp, (i+1)*N/cp),
// read as half-open). The ring order follows "Pass them around a ring": each step a rank sends
// its block right and receives from the left, so at step s it holds the block of (r - s) mod n_cp.
#include <algorithm>
#include <climits>
#include <numeric>

#include "internal.h"

namespace cpattn {

int64_t token_of(const Plan& p, int r, int64_t j) {
    switch (p.layout) {
        case CPATTN_CONTIGUOUS: return (int64_t)r * p.n + j;
        case CPATTN_ZIGZAG: return j < p.m ? (int64_t)r * p.m + j : (int64_t)(2 * p.n_cp - 1 - r) * p.m + (j - p.m);
        default: return j * p.n_cp + r;
    }
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsLayout ws_layout(const Plan& p, int B) {
    WsLayout w;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + bytes, 1024); return at; };
    const size_t T = (size_t)p.T, d = (size_t)p.d;
    w.header = take(sizeof(uint32_t) * kHeaderWords);
    w.posL = take(sizeof(int32_t) * T);
    w.tile_mm = take(sizeof(int32_t) * 4 * (size_t)p.n_cp * p.n_qt);
    w.order = take(sizeof(int32_t) * (size_t)p.n_cp * p.n_qt);
    w.counts = take(sizeof(uint64_t) * 2 * (size_t)p.n_cp * p.n_cp);
    w.sched = take(sizeof(uint32_t) * (1 + (size_t)p.n_cp));
    w.loL = take(sizeof(int32_t) * T);
    w.tile_lo = take(sizeof(int32_t) * 4 * (size_t)p.n_cp * p.n_qt);
    w.unit_tiles = take(sizeof(int32_t) * (size_t)p.n_cp * p.n_qt);
    w.walk_tab = take(sizeof(int32_t) * (size_t)p.n_cp * p.n_qt * p.n_cp);
    w.walk_nz = take(sizeof(uint64_t) * (size_t)p.n_cp * p.n_qt);
    w.walk_bits = take(sizeof(uint64_t) * (size_t)p.n_cp * p.n_qt * p.n_cp * (((size_t)p.n_qt + 63) / 64));
    w.order_masked = take(sizeof(int32_t) * (size_t)p.n_cp * p.n_qt);
    w.qL = take(2 * (size_t)B * T * p.h * d);
    w.kL = take(2 * (size_t)B * T * p.n_kv * d);
    w.vL = take(2 * (size_t)B * T * p.n_kv * d);
    w.fwd_end = off;
    for (int s = 0; s < 2; ++s) {
        w.stageK[s] = take(2 * (size_t)B * T * p.n_kv * d);
        w.stageV[s] = take(2 * (size_t)B * T * p.n_kv * d);
    }
    w.o_run = take(4 * (size_t)B * T * p.h * d);
    w.lse_run = take(2 * 4 * (size_t)B * T * p.h);     // running maximum, then running sum
    w.ring_end = off;
    off = w.fwd_end;
    w.gK = take(2 * (size_t)p.n_cp * B * T * p.n_kv * d);
    w.gV = take(2 * (size_t)p.n_cp * B * T * p.n_kv * d);
    w.gather_end = off;
    // the backward reuses the forward regions and appends its own after them
    off = w.fwd_end;
    const size_t padded = (size_t)p.n_cp * B * p.h * (size_t)p.n_qt * 128;
    w.doL = take(2 * (size_t)B * T * p.h * d);
    w.lse2 = take(4 * padded);
    w.Dl = take(4 * padded);
    w.bwd_order = take(sizeof(int32_t) * 2 * (size_t)p.n_cp * p.n_qt);
    w.bwd_end = off;
    for (int s = 0; s < 2; ++s) {
        w.bstageK[s] = take(2 * (size_t)B * T * p.n_kv * d);
        w.bstageV[s] = take(2 * (size_t)B * T * p.n_kv * d);
    }
    for (int s = 0; s < 2; ++s) {
        w.circK[s] = take(4 * (size_t)B * T * p.n_kv * d);
        w.circV[s] = take(4 * (size_t)B * T * p.n_kv * d);
    }
    w.dq_run = take(4 * (size_t)B * T * p.h * d);
    w.bring_end = off;
    return w;
}

DistLayout dist_layout(const Plan& p, int B, int R) {
    DistLayout w;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + bytes, 1024); return at; };
    const size_t n = (size_t)p.n, d = (size_t)p.d, nq = (size_t)p.n_qt, ng = (size_t)p.n_grp;
    w.header = take(sizeof(uint32_t) * kHeaderWords);
    w.posL = take(sizeof(int32_t) * R * n);
    w.tile_mm = take(sizeof(int32_t) * 4 * R * nq);
    w.order = take(sizeof(int32_t) * R * ng);
    w.counts = take(sizeof(uint64_t) * 2 * R * R);
    w.sched = take(sizeof(uint32_t) * (1 + (size_t)R));
    w.unit_tiles = take(sizeof(int32_t) * R * ng);
    w.walk_tab = take(sizeof(int32_t) * R * ng * R);
    w.walk_nz = take(sizeof(uint64_t) * R * ng);
    w.loL = take(sizeof(int32_t) * R * n);
    w.tile_lo = take(sizeof(int32_t) * 4 * R * nq);
    w.qL = take(2 * (size_t)B * R * n * p.h * d);
    w.o_run = take(4 * (size_t)B * R * n * p.h * d);
    w.lse_run = take(2 * 4 * (size_t)B * R * n * p.h);     // running maximum, then running sum
    w.ws_end = off;
    w.blk_k = w.blk_v = 2 * (size_t)B * n * p.n_kv * d;
    w.blk_pos = sizeof(int32_t) * n;
    w.blk_tile = sizeof(int32_t) * 4 * nq;
    off = 0;
    w.slot_k = take(w.blk_k * R);
    w.slot_v = take(w.blk_v * R);
    w.slot_pos = take(w.blk_pos * R);
    w.slot_tile = take(w.blk_tile * R);
    w.slot_end = off;
    return w;
}

// Block classes from the position range of each tile: all keys at or before every query ->
// FULL; all keys after every query -> SKIP; otherwise the tile is partly visible (DIAG). For
// the mask "key u visible to query t iff pos[u] <= pos[t]" this is exact: every pair is visible
// iff max(kpos) <= min(qpos), none is iff min(kpos) > max(qpos).
static int classify(int causal, int64_t qmin, int64_t qmax, int64_t kmin, int64_t kmax) {
    if (!causal) return CPATTN_TILE_FULL;
    if (kmax <= qmin) return CPATTN_TILE_FULL;
    if (kmin > qmax) return CPATTN_TILE_SKIP;
    return CPATTN_TILE_DIAG;
}

std::string build_plan(Plan& p, int64_t T, int h, int n_kv, int d, int n_cp, int layout, int causal) {
    if (T <= 0 || h <= 0 || n_kv <= 0 || n_cp <= 0) return "T, h, n_kv and n_cp must be positive";
    if (h % n_kv) return "h must be a multiple of n_kv";
    if (layout < CPATTN_CONTIGUOUS || layout > CPATTN_STRIPED) return "unknown layout";
    if (T % n_cp) return "T must be a multiple of n_cp";
    if (layout == CPATTN_ZIGZAG && T % (2 * (int64_t)n_cp)) return "zigzag needs T to be a multiple of 2*n_cp";
    if (T > INT_MAX / 2) return "T must fit position ids in int32";
    p.T = T; p.h = h; p.n_kv = n_kv; p.d = d; p.n_cp = n_cp; p.layout = layout; p.causal = causal ? 1 : 0;
    p.n = T / n_cp;
    p.m = (layout == CPATTN_ZIGZAG) ? T / (2 * n_cp) : 0;
    p.n_qt = (int)((p.n + kBlockQ - 1) / kBlockQ);

    // position range of every (rank, tile), positions 0..T-1
    std::vector<int64_t> tmin((size_t)n_cp * p.n_qt, INT64_MAX), tmax((size_t)n_cp * p.n_qt, INT64_MIN);
    for (int r = 0; r < n_cp; ++r)
        for (int64_t j = 0; j < p.n; ++j) {
            int64_t t = token_of(p, r, j);
            size_t i = (size_t)r * p.n_qt + (size_t)(j / kBlockQ);
            tmin[i] = std::min(tmin[i], t);
            tmax[i] = std::max(tmax[i], t);
        }
    p.full.assign((size_t)n_cp * n_cp, 0);
    p.diag.assign((size_t)n_cp * n_cp, 0);
    p.skip.assign((size_t)n_cp * n_cp, 0);
    // A CTA computes two 128-row query tiles against each key tile: two heads of one KV group
    // when the group size is even, else two adjacent query tiles of one head.
    p.pair_heads = ((h / n_kv) % 2 == 0) ? 1 : 0;
    p.n_grp = p.pair_heads ? p.n_qt : (p.n_qt + 1) / 2;
    std::vector<int64_t> work((size_t)n_cp * p.n_grp, 0);  // key tiles a row group computes
    std::vector<int64_t> work_q((size_t)n_cp * p.n_qt, 0), work_kv((size_t)n_cp * p.n_qt, 0);
    for (int r = 0; r < n_cp; ++r)
        for (int s = 0; s < n_cp; ++s) {
            int src = ((r - s) % n_cp + n_cp) % n_cp;
            for (int qt = 0; qt < p.n_qt; ++qt) {
                size_t qi = (size_t)r * p.n_qt + qt;
                for (int kt = 0; kt < p.n_qt; ++kt) {
                    size_t ki = (size_t)src * p.n_qt + kt;
                    int c = classify(p.causal, tmin[qi], tmax[qi], tmin[ki], tmax[ki]);
                    size_t rs = (size_t)r * n_cp + s;
                    if (c == CPATTN_TILE_FULL) ++p.full[rs];
                    else if (c == CPATTN_TILE_DIAG) ++p.diag[rs];
                    else ++p.skip[rs];
                    if (c != CPATTN_TILE_SKIP) {
                        ++work_q[qi];
                        ++work_kv[ki];
                    }
                }
            }
            for (int grp = 0; grp < p.n_grp; ++grp) {
                const int q0 = p.pair_heads ? grp : 2 * grp;
                const int q1 = p.pair_heads ? grp : std::min(2 * grp + 1, p.n_qt - 1);
                for (int kt = 0; kt < p.n_qt; ++kt) {
                    size_t ki = (size_t)src * p.n_qt + kt;
                    int c0 = classify(p.causal, tmin[(size_t)r * p.n_qt + q0], tmax[(size_t)r * p.n_qt + q0],
                                      tmin[ki], tmax[ki]);
                    int c1 = classify(p.causal, tmin[(size_t)r * p.n_qt + q1], tmax[(size_t)r * p.n_qt + q1],
                                      tmin[ki], tmax[ki]);
                    if (c0 != CPATTN_TILE_SKIP || c1 != CPATTN_TILE_SKIP) ++work[(size_t)r * p.n_grp + grp];
                }
            }
        }
    // exact visible pairs: with positions 0..T-1 the query at natural token t sees t+1 keys
    p.pairs.assign(n_cp, 0);
    for (int r = 0; r < n_cp; ++r) {
        int64_t c = 0;
        for (int64_t j = 0; j < p.n; ++j) c += p.causal ? token_of(p, r, j) + 1 : T;
        p.pairs[r] = c;
    }
    // chunk-level half units: FULL chunk pair 2, partly visible 1
    p.half_units.assign(n_cp, 0);
    {
        int nchunks = (layout == CPATTN_ZIGZAG) ? 2 * n_cp : n_cp;
        int64_t cs = T / nchunks;
        auto crange = [&](int c, int64_t& lo, int64_t& hi) {
            if (layout == CPATTN_STRIPED) { lo = c; hi = c + (int64_t)n_cp * (cs - 1); }
            else { lo = (int64_t)c * cs; hi = lo + cs - 1; }
        };
        for (int r = 0; r < n_cp; ++r) {
            int mine[2] = {r, 2 * n_cp - 1 - r};
            int nm = (layout == CPATTN_ZIGZAG) ? 2 : 1;
            int64_t u = 0;
            for (int a = 0; a < nm; ++a) {
                int64_t qlo, qhi;
                crange(mine[a], qlo, qhi);
                for (int c = 0; c < nchunks; ++c) {
                    int64_t klo, khi;
                    crange(c, klo, khi);
                    int cls = classify(p.causal, qlo, qhi, klo, khi);
                    u += (cls == CPATTN_TILE_FULL) ? 2 : (cls == CPATTN_TILE_DIAG) ? 1 : 0;
                }
            }
            p.half_units[r] = u;
        }
    }
    // longest-first order of (rank, q-tile): the block scheduler starts the heaviest units first
    p.order.resize((size_t)n_cp * p.n_grp);
    std::iota(p.order.begin(), p.order.end(), 0);
    std::stable_sort(p.order.begin(), p.order.end(), [&](int32_t a, int32_t b) { return work[a] > work[b]; });
    // the backward launches one CTA per query tile (dQ) and per key tile (dK, dV), heaviest first
    p.order_q.resize((size_t)n_cp * p.n_qt);
    std::iota(p.order_q.begin(), p.order_q.end(), 0);
    std::stable_sort(p.order_q.begin(), p.order_q.end(), [&](int32_t a, int32_t b) { return work_q[a] > work_q[b]; });
    p.order_kv.resize((size_t)n_cp * p.n_qt);
    std::iota(p.order_kv.begin(), p.order_kv.end(), 0);
    std::stable_sort(p.order_kv.begin(), p.order_kv.end(), [&](int32_t a, int32_t b) { return work_kv[a] > work_kv[b]; });
    return "";
}

}  // namespace cpattn
