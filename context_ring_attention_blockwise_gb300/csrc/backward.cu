// backward.cu -- the backward pass of ring attention on sm_103a: the gradients of the forward
// with respect to Q, K and V ("Context and expert parallelism", section "What context
// parallelism communicates": each rank keeps the gradient of its own queries, and the key and
// value gradients travel back to their owners as a second circulating block of the ring).
//
// With P_tu = exp(s_tu - lse_t), dP_tu = <dO_t, v_u>, D_t = <dO_t, O_t> and
// dS_tu = P_tu (dP_tu - D_t):  dQ_t = scale sum_u dS_tu k_u,  dK_u = scale sum_t dS_tu q_t,
// dV_u = sum_t P_tu dO_t, the sums over t running over the query heads of the key's group.
//
// Three kernels:
//   bwd_prep_kernel   D_t from O and dO (fp32), and dO, -lse (as log2) and -D in layout order.
//   bwd_dkdv_kernel   one CTA per key tile (128 keys of one rank block, one KV head). It walks
//                     the query tiles in ring order -- the block's gradient visits rank src + s
//                     at step s -- and for every visible (query tile, query head of the group):
//                       S^T = K Q^T, dP^T = V dO^T          (tcgen05, SS form)
//                       P^T, dS^T elementwise (two warpgroups, 64 query columns each)
//                       dV += P^T dO, dK += dS^T Q          (tcgen05, TS form, P^T / dS^T in TMEM)
//                     dK and dV accumulate in tensor memory for the whole walk and are written
//                     once, to natural token order: the block arriving back at its owner.
//   bwd_dq_kernel     one CTA per query tile (128 queries of one rank, one head). It walks the
//                     key tiles like the forward and for each: S = Q K^T, dP = dO V^T, dS, then
//                     dQ += dS K (TS form, dS in TMEM).
// Both tcgen05 kernels: warp 0 loads tiles by TMA and publishes each step of the walk in a
// shared-memory ring; warp 1 owns tensor memory and one lane issues the MMAs; warps 4..11 are
// the elementwise warpgroups. All waits are bounded by the global timer like the forward's.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <string>

#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace cpattn {
namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr int kRing = 8;            // walk steps published ahead by the producer
constexpr int kNS = 2;              // stages of the streamed operand pair
constexpr float kLog2e = 1.4426950408889634f;

enum BwdSite : int { kBSiteStage = 101, kBSiteStageEmpty, kBSiteFixed, kBSiteSt, kBSiteP, kBSiteDone, kBSiteWalk,
                     kBSiteDrain };

struct BwdParams {
    int B, h, n_kv, g, n_cp, n_qt, causal, layout;
    int64_t n, m, T, n_pad;   // n_pad = n_qt * 128: row stride of nlse2L and nDL
    float scale, scale_log2;
    const int32_t* posL;
    const int4* tile_mm;
    const float* nlse2L;  // [n_cp][B][h][n_pad] -lse * log2(e) (tile starts 512-byte aligned; padding 0)
    const float* nDL;     // [n_cp][B][h][n_pad] -D (padding 0)
    const int32_t* loL;        // [n_cp][n] lowest visible key position per query (document masks), or NULL
    const int4* tile_lo;       // [n_cp][n_qt] (min, max) of loL over a query tile, or NULL
    const int32_t* order_q;    // (r * n_qt + qt), heaviest first
    const int32_t* order_kv;   // (src * n_qt + kt), heaviest first
    uint16_t* dq;         // natural [B,T,h,d]
    uint16_t* dk;         // natural [B,T,n_kv,d]
    uint16_t* dv;
    uint32_t* header;
    uint64_t timeout_ns;
    // One ring step (step >= 0) instead of the whole walk (-1). K and V rows are then indexed by
    // the rank holding the block at that step; dK/dV leave as this step's fp32 contribution
    // [holder][B][n_kv][n][d], written or added into the partial sums there, and dQ is added
    // into the running fp32 [r][B][h][n][d].
    int step;
    float* dk_f32;
    float* dv_f32;
    int dkdv_add;           // add the contribution into dk_f32 / dv_f32 by reductions
    float* dq_run;
};

struct BWaiter {
    volatile int* abort_flag;
    uint32_t* header;
    uint64_t timeout_ns;
    __device__ bool operator()(uint32_t bar, uint32_t parity, int site, bool honour_abort = true) const {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer();
        for (uint32_t it = 1;; ++it) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((it & 63u) == 0) {
                if (honour_abort && (*abort_flag || *(volatile uint32_t*)(header + kErrFlags))) {
                    *abort_flag = 1;
                    return false;
                }
                if (globaltimer() - t0 > timeout_ns) {
                    *abort_flag = 1;
                    atomicOr(header + kErrFlags, kErrTimeoutFlag);
                    atomicExch(header + kErrWhere, (uint32_t)site);
                    return false;
                }
            }
        }
    }
};

__device__ __forceinline__ int64_t natural_token(int layout, int r, int64_t j, int64_t n, int64_t m, int n_cp) {
    if (layout == CPATTN_CONTIGUOUS) return (int64_t)r * n + j;
    if (layout == CPATTN_ZIGZAG) return j < m ? (int64_t)r * m + j : (int64_t)(2 * n_cp - 1 - r) * m + (j - m);
    return j * n_cp + r;
}

// Tile classes from the position ranges of a query tile and a key tile (exact for the mask
// pos[u] <= pos[t]): SKIP if every key follows every query, FULL if every key precedes every
// query, DIAG otherwise.
// With document masks each query also has a lowest visible key position; ql = (min, max) of it
// over the query tile ((INT_MIN, INT_MIN) without): SKIP also when every key lies below every
// bound, FULL only when every key lies at or above every bound.
__device__ __forceinline__ int tile_class(int causal, int4 q, int2 ql, int4 k) {
    if (!causal) return CPATTN_TILE_FULL;
    if (k.x > q.y || k.y < ql.x) return CPATTN_TILE_SKIP;
    if (k.y <= q.x && k.x >= ql.y) return CPATTN_TILE_FULL;
    return CPATTN_TILE_DIAG;
}

template <bool LB>
__device__ __forceinline__ int2 tile_bound(const BwdParams& P, int r, int qt) {
    if (!LB) return make_int2(INT_MIN, INT_MIN);
    const int4 l4 = __ldg(P.tile_lo + r * P.n_qt + qt);
    return make_int2(l4.x, l4.y);
}

// ---- shared-memory layout and barriers (both tcgen05 kernels) --------------------------
// fixed pair: the CTA's own two tiles (K, V for dK/dV; Q, dO for dQ), loaded once;
// stream pair: the walked tiles (Q, dO for dK/dV; K, V for dQ), kNS stages;
// side: per stage 2 x 128 floats (-lse2 and -D of the query tile, dK/dV only), bulk-copied.
template <int D>
struct BCfg {
    static constexpr int PANELS = D / 64;
    static constexpr int PANEL_BYTES = 128 * 128;
    static constexpr int TILE = 128 * D * 2;
    static constexpr int OFF_F0 = 0, OFF_F1 = TILE;                 // fixed pair
    static constexpr int OFF_S = 2 * TILE;                          // stream: stage st, member m at + (2 st + m) TILE
    static constexpr int OFF_SIDE = OFF_S + 2 * kNS * TILE;         // float [kNS][2][128]
    static constexpr int OFF_BAR = OFF_SIDE + kNS * 2 * 128 * 4;
    static constexpr int NBAR = 8 + 2 * kNS + kRing;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int OFF_RING = (OFF_MISC + 64 + 15) / 16 * 16;   // int4 [kRing]
    static constexpr int SMEM_BYTES = OFF_RING + 16 * kRing + 1024;
    static_assert(OFF_S % 1024 == 0 && OFF_SIDE % 16 == 0 && OFF_BAR % 8 == 0 && OFF_RING % 16 == 0,
                  "shared-memory regions must keep their alignment");
    // a ring step's epilogue reuses the fixed pair as 4 KB of staging for each elementwise warp
    static_assert(OFF_F0 == 0 && OFF_F1 == TILE && 8 * 4096 <= 2 * TILE, "ring-step staging in the fixed pair");
    // tensor memory: two accumulators (A0, A1: dV and dK, or dQ), the score tile S and the dP
    // tile (128 columns each). The elementwise warps overwrite the first half of each warpgroup's
    // 64 columns of S with packed bf16 P and of dP with packed bf16 dS, the A operands of the
    // accumulating MMAs.
    static constexpr uint32_t COL_A0 = 0, COL_A1 = D, COL_S = 2 * D, COL_DP = 2 * D + 128;
    // dQ only: the CTA's fixed Q and dO tiles as packed bf16 rows (D / 2 columns each), where the
    // dK accumulator sits in the other kernel: the A operands of its score MMAs (TS form)
    static constexpr uint32_t COL_Q = D, COL_DO = D + D / 2;
    static_assert(2 * D + 2 * 128 <= 512, "tensor-memory columns");
};

// A walk step runs in two phases on the elementwise warps: P from S, then dS from dP (P stays in
// registers in between). The barriers follow them:
//   s_full   the score MMA of the step has completed          (MMA commit)
//   p_done   P has been read out of S (and, for dK/dV, packed back into it)  (8 warps)
//   dp_full  the dP MMA of the step has completed             (MMA commit)
//   ds_done  dS has been packed into the dP columns           (8 warps)
// The MMA issuer orders each step as  [p_done] dV or S(next) ... [ds_done] dK or dQ, dP(next),
// so the score MMA of the next step and the dP MMA overlap the elementwise phases.
template <int D>
struct BBars {
    uint32_t base;
    __device__ uint32_t at(int i) const { return base + 8u * (uint32_t)i; }
    __device__ uint32_t fixed_full() const { return at(0); }
    __device__ uint32_t s_full() const { return at(1); }
    __device__ uint32_t p_done() const { return at(2); }
    __device__ uint32_t dp_full() const { return at(3); }
    __device__ uint32_t ds_done() const { return at(4); }
    __device__ uint32_t spare() const { return at(5); }
    // every MMA of the CTA has completed: committed once, after the last one (a single phase, so
    // no waiter can mistake an older phase for it)
    __device__ uint32_t drain() const { return at(6); }
    __device__ uint32_t fixed_tmem() const { return at(7); }        // dQ: Q and dO copied into TMEM (8 warps)
    __device__ uint32_t st_full(int s) const { return at(8 + s); }
    __device__ uint32_t st_empty(int s) const { return at(8 + kNS + s); }
    __device__ uint32_t ring_full(int s) const { return at(8 + 2 * kNS + s); }
    __device__ void init() const {
        mbar_init(fixed_full(), 1);
        mbar_init(s_full(), 1);
        mbar_init(p_done(), 8);                 // one lane per elementwise warp
        mbar_init(dp_full(), 1);
        mbar_init(ds_done(), 8);
        mbar_init(spare(), 1);
        mbar_init(drain(), 1);
        mbar_init(fixed_tmem(), 8);
        for (int s = 0; s < kNS; ++s) {
            mbar_init(st_full(s), 1);
            mbar_init(st_empty(s), 1);
        }
        for (int s = 0; s < kRing; ++s) mbar_init(ring_full(s), 1);
    }
};

// A step of the walk, as published by the producer: x, y = rank and tile of the streamed tile,
// z = head (dK/dV) or source rank (dQ), w = class | mask << 2 | last << 3 | empty << 4.
constexpr int kFlagLast = 8, kFlagEmpty = 16;

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// =============================================================================================
// bwd_prep_kernel: one thread per 8 consecutive d of one (b, t, head) row. D_t is reduced over
// the row's d/8 threads with shuffles.
// =============================================================================================
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                                                       const float* __restrict__ lse, uint4* __restrict__ doL,
                                                       float* __restrict__ nlse2L, float* __restrict__ nDL, int B,
                                                       int64_t T, int64_t n, int64_t m, int64_t n_pad, int h, int d,
                                                       int n_cp, int layout) {
    const int cpr = d / 8;                       // 8 or 16 threads per row, aligned within the warp
    const int64_t total = (int64_t)B * T * h * cpr;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < total; base += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = base + threadIdx.x;
        const bool act = i < total;
        float part = 0.f;
        int c = 0;
        int64_t row = 0;
        if (act) {
            c = (int)(i % cpr);
            row = i / cpr;                        // (b, t, head)
            const uint4 a = __ldg(o + i), g = __ldg(dout + i);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                part += __uint_as_float(aw[e] << 16) * __uint_as_float(gw[e] << 16);
                part += __uint_as_float(aw[e] & 0xFFFF0000u) * __uint_as_float(gw[e] & 0xFFFF0000u);
            }
        }
        for (int off = cpr / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (!act) continue;
        const int hd = (int)(row % h);
        const int64_t bt = row / h;
        const int64_t t = bt % T;
        const int b = (int)(bt / T);
        int r;
        int64_t j;
        if (layout == CPATTN_CONTIGUOUS) { r = (int)(t / n); j = t - (int64_t)r * n; }
        else if (layout == CPATTN_ZIGZAG) {
            const int ch = (int)(t / m);
            if (ch < n_cp) { r = ch; j = t - (int64_t)ch * m; }
            else { r = 2 * n_cp - 1 - ch; j = m + (t - (int64_t)ch * m); }
        } else { r = (int)(t % n_cp); j = t / n_cp; }
        const int64_t lrow = (((int64_t)r * B + b) * h + hd) * n + j;
        doL[lrow * cpr + c] = __ldg(dout + i);
        if (c == 0) {
            const int64_t prow = (((int64_t)r * B + b) * h + hd) * n_pad + j;
            const float l = __ldg(lse + ((int64_t)b * h + hd) * T + t);
            nlse2L[prow] = -l * kLog2e;           // negated: the kernels add them in fused multiply-adds
            nDL[prow] = -part;
        }
    }
}

// ---- elementwise bodies -----------------------------------------------------------------
// 32 columns of one TMEM lane at a time, in packed fp32 pairs: x = s scale log2(e) - lse2,
// P = 2^x; later dS = P (dP - D). Masked chunks force x = -inf where the bit of the column is
// clear, which makes P = 0 and dS = 0 (dP and the side tables are finite, their padding zero).

// P of 32 columns; nl = -lse2 per column (dK/dV: the columns are queries, nl4 from shared
// memory) or per row (dQ: nl4 == nullptr, nl2 the row's pair).
template <bool MASKED>
__device__ __forceinline__ void p_chunk(const uint32_t (&sr)[32], const float4* nl4, uint64_t nl2, uint64_t c2,
                                        uint32_t vis_bits, float* pf) {
#pragma unroll
    for (int q2 = 0; q2 < 16; ++q2) {
        uint64_t nl = nl2;
        if (nl4) {
            const float4 l = nl4[q2 >> 1];
            nl = (q2 & 1) ? f2_pack(l.z, l.w) : f2_pack(l.x, l.y);
        }
        float x[2];
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * q2]), __uint_as_float(sr[2 * q2 + 1])), c2, nl), x[0], x[1]);
        if (MASKED) {
#pragma unroll
            for (int e = 0; e < 2; ++e) x[e] = ((vis_bits >> (2 * q2 + e)) & 1u) ? x[e] : -INFINITY;
        }
        pf[2 * q2] = ex2(x[0]);
        pf[2 * q2 + 1] = ex2(x[1]);
    }
}
__device__ __forceinline__ void pack_chunk(const float* v, uint32_t (&pk)[16]) {
#pragma unroll
    for (int q2 = 0; q2 < 16; ++q2) pk[q2] = pack_bf16(v[2 * q2], v[2 * q2 + 1]);
}
// dS = P (dP - D) of 32 columns, packed; nd = -D per column (nd4) or per row (nd2).
__device__ __forceinline__ void ds_chunk(const uint32_t (&dr)[32], const float* pf, const float4* nd4, uint64_t nd2,
                                         uint32_t (&pd)[16]) {
#pragma unroll
    for (int q2 = 0; q2 < 16; ++q2) {
        uint64_t nd = nd2;
        if (nd4) {
            const float4 d4 = nd4[q2 >> 1];
            nd = (q2 & 1) ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y);
        }
        const uint64_t t = f2_add(f2_pack(__uint_as_float(dr[2 * q2]), __uint_as_float(dr[2 * q2 + 1])), nd);
        float ds[2];
        f2_unpack(f2_mul(f2_pack(pf[2 * q2], pf[2 * q2 + 1]), t), ds[0], ds[1]);
        pd[q2] = pack_bf16(ds[0], ds[1]);
    }
}

// =============================================================================================
// bwd_dkdv_kernel
// =============================================================================================
template <int D, bool LB>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const BwdParams P) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
    const uint32_t ring = sb + C::OFF_RING;
    const BBars<D> bars{sb + C::OFF_BAR};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // unit: (b, kvh, src, kt), KV-head-major (the CTAs in flight share one head group's Q and dO
    // in L2), heaviest key tile first within a head
    const int n_tiles = P.n_cp * P.n_qt;
    const int bk = blockIdx.x / n_tiles;
    const int ut = __ldg(P.order_kv + blockIdx.x % n_tiles);
    const int kt = ut % P.n_qt, src = ut / P.n_qt;
    const int kvh = bk % P.n_kv, b = bk / P.n_kv;

    if (threadIdx.x == 0) *skip_flag = (int)*(volatile uint32_t*)(P.header + kErrFlags);
    __syncthreads();
    if (*skip_flag) return;
    if (threadIdx.x == 0) {
        bars.init();
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmDO);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const BWaiter wait{abort_flag, P.header, P.timeout_ns};
    const int4 kmm = __ldg(P.tile_mm + src * P.n_qt + kt);
    // rank whose slot holds this key block's K, V (and receives its dK/dV contribution): the
    // owner for the whole walk; at ring step s, rank src + s
    const int kvr = P.step >= 0 ? (src + P.step) % P.n_cp : src;
    const int s_lo = P.step >= 0 ? P.step : 0, s_hi = P.step >= 0 ? P.step + 1 : P.n_cp;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer: fixed K, V; walk (s, qt, head); stream Q, dO + side data
            const int krow = (int)((((int64_t)kvr * P.B + b) * P.n_kv + kvh) * P.n + (int64_t)kt * 128);
            mbar_arrive_expect_tx(bars.fixed_full(), 2 * C::TILE);
            for (int pn = 0; pn < C::PANELS; ++pn) {
                tma_load_2d(sb + C::OFF_F0 + pn * C::PANEL_BYTES, &tmK, bars.fixed_full(), pn * 64, krow);
                tma_load_2d(sb + C::OFF_F1 + pn * C::PANEL_BYTES, &tmV, bars.fixed_full(), pn * 64, krow);
            }
            int ns = 0;                 // steps published (each loads one stage, except an empty unit's)
            int nl = 0;                 // stages loaded
            bool ok = true;
            int pending = -1;           // the last visible (r, qt), published one step late so "last" is known
            int pend_r = 0, pend_qt = 0, pend_head = 0, pend_cls = 0, pend_mask = 0;
            auto publish = [&](int r, int qt, int head, int flags) -> bool {
                const int slot = ns % kRing;
                const int st = ns % kNS;
                if (!(flags & kFlagEmpty)) {
                    if (ns >= kNS && !wait(bars.st_empty(st), ((ns / kNS) - 1) & 1, kBSiteStageEmpty)) return false;
                    const int qrow = (int)((((int64_t)r * P.B + b) * P.h + head) * P.n + (int64_t)qt * 128);
                    mbar_arrive_expect_tx(bars.st_full(st), 2 * C::TILE + 2 * 512);
                    const uint32_t s0 = sb + C::OFF_S + (2 * st) * C::TILE, s1 = s0 + C::TILE;
                    for (int pn = 0; pn < C::PANELS; ++pn) {
                        tma_load_2d(s0 + pn * C::PANEL_BYTES, &tmQ, bars.st_full(st), pn * 64, qrow);
                        tma_load_2d(s1 + pn * C::PANEL_BYTES, &tmDO, bars.st_full(st), pn * 64, qrow);
                    }
                    const uint32_t side = sb + C::OFF_SIDE + st * 2 * 512;
                    const int64_t prow = (((int64_t)r * P.B + b) * P.h + head) * P.n_pad + (int64_t)qt * 128;
                    bulk_copy_g2s(side, P.nlse2L + prow, 512, bars.st_full(st));
                    bulk_copy_g2s(side + 512, P.nDL + prow, 512, bars.st_full(st));
                    ++nl;
                }
                st_shared_v4(ring + 16u * (uint32_t)slot, (uint32_t)r, (uint32_t)qt, (uint32_t)head, (uint32_t)flags);
                mbar_arrive(bars.ring_full(slot));
                ++ns;
                return true;
            };
            for (int s = s_lo; s < s_hi && ok; ++s) {
                const int r = (src + s) % P.n_cp;         // the block's gradient is at rank src + s at step s
                // Causal: the query tiles whose positions all precede the key tile's first one see
                // none of it, and they are the tiles before the first whose running maximum (.w,
                // non-decreasing) reaches it: start there (binary search, exact for any positions).
                int qt0 = 0;
                if (P.causal) {
                    int lo = 0, hi = P.n_qt;
                    while (lo < hi) {
                        const int mid = (lo + hi) >> 1;
                        if (__ldg(P.tile_mm + r * P.n_qt + mid).w < kmm.x) lo = mid + 1;
                        else hi = mid;
                    }
                    qt0 = lo;
                }
                for (int qt = qt0; qt < P.n_qt && ok; ++qt) {
                    const int4 qmm = __ldg(P.tile_mm + r * P.n_qt + qt);
                    const int cls = tile_class(P.causal, qmm, tile_bound<LB>(P, r, qt), kmm);
                    if (cls == CPATTN_TILE_SKIP) continue;
                    const int qshort = (qt == P.n_qt - 1) && (P.n % 128) != 0;
                    const int kshort = (kt == P.n_qt - 1) && (P.n % 128) != 0;
                    const int mask = (cls != CPATTN_TILE_FULL) || qshort || kshort;
                    for (int hi = 0; hi < P.g && ok; ++hi) {
                        if (pending >= 0) ok = publish(pend_r, pend_qt, pend_head, pend_cls | (pend_mask << 2));
                        pending = 1;
                        pend_r = r; pend_qt = qt; pend_head = kvh * P.g + hi; pend_cls = cls; pend_mask = mask;
                    }
                }
            }
            if (ok) {
                if (pending >= 0) ok = publish(pend_r, pend_qt, pend_head, pend_cls | (pend_mask << 2) | kFlagLast);
                else ok = publish(0, 0, 0, kFlagEmpty | kFlagLast);
            }
            // wait (bounded) until every stage we filled has been consumed or, after an abort,
            // has landed, before the CTA may exit
            // the CTA exits only after its own copies have landed (bounded waits)
            const int first = nl > kNS ? nl - kNS : 0;
            for (int i = first; i < nl; ++i) wait(bars.st_full(i % kNS), (i / kNS) & 1, kBSiteStage, false);
            wait(bars.fixed_full(), 0, kBSiteFixed, false);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issue. Per walked query tile (stage st):
            //   S^T = K Q^T into S and dP^T = V dO^T into dP           (SS form)
            //   dV += P^T dO once P^T is packed into S                 (TS form)
            //   dK += dS^T Q once dS^T is packed into dP                (TS form)
            // issued as  [p_done] dV(i), S(i+1), [ds_done] dK(i), dP(i+1): the score MMAs of the next
            // tile run while the elementwise warps work on this one. MMAs run in issue order, so
            // S(i+1) cannot overwrite P^T before dV(i) has read it, nor dP(i+1) dS^T before dK(i).
            constexpr uint32_t kIdSS = idesc_bf16(128, 128, 0, 0);   // A = K or V, B = Q or dO (K-major)
            constexpr uint32_t kIdTS = idesc_bf16(128, D, 0, 1);     // A = P^T / dS^T (TMEM), B = dO / Q (MN-major)
            const uint32_t sK = sb + C::OFF_F0, sV = sb + C::OFF_F1;
            const uint32_t tdV = tmem + C::COL_A0, tdK = tmem + C::COL_A1, tS = tmem + C::COL_S, tDP = tmem + C::COL_DP;
            auto score = [&](uint32_t d, uint32_t a, uint32_t b) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::PANEL_BYTES + (kk & 3) * 32;
                    mma_bf16_ss(d, desc_sw128(a + off, 16, 1024), desc_sw128(b + off, 16, 1024), kIdSS, kk > 0);
                }
            };
            // packed P^T / dS^T: the 64 queries of warpgroup w in columns 64 w .. 64 w + 31 of their
            // buffer, so query 16 kk .. 16 kk + 15 sits at 64 (kk / 4) + 8 (kk % 4)
            auto accumulate = [&](uint32_t d, uint32_t a_t, uint32_t b, bool first) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(d, a_t + 64 * (kk >> 2) + 8 * (kk & 3), desc_sw128(b + kk * 2048, C::PANEL_BYTES, 1024),
                                kIdTS, (first && kk == 0) ? 0u : 1u);
            };
            auto sQ_of = [&](int st) { return sb + C::OFF_S + (2 * st) * C::TILE; };
            bool ok = wait(bars.fixed_full(), 0, kBSiteFixed);
            int4 e = make_int4(0, 0, 0, kFlagEmpty);
            if (ok) ok = wait(bars.ring_full(0), 0, kBSiteWalk);
            if (ok) e = ld_shared_v4(ring);
            if (ok && !(e.w & kFlagEmpty)) {
                ok = wait(bars.st_full(0), 0, kBSiteStage);
                if (ok) {
                    tc_fence_after();
                    score(tS, sK, sQ_of(0));
                    mma_commit(bars.s_full());
                    score(tDP, sV, sQ_of(0) + C::TILE);
                    mma_commit(bars.dp_full());
                }
            }
            int step = 0;
            while (ok && !(e.w & kFlagEmpty)) {
                const int st = step % kNS, st1 = (step + 1) % kNS;
                const bool last = (e.w & kFlagLast) != 0;
                if (!wait(bars.p_done(), step & 1, kBSiteP)) break;
                tc_fence_after();
                accumulate(tdV, tS, sQ_of(st) + C::TILE, step == 0);
                int4 nx = e;
                if (!last) {
                    const int n1 = step + 1;
                    if (!wait(bars.ring_full(n1 % kRing), (n1 / kRing) & 1, kBSiteWalk)) break;
                    nx = ld_shared_v4(ring + 16u * (uint32_t)(n1 % kRing));
                    if (!wait(bars.st_full(st1), (n1 / kNS) & 1, kBSiteStage)) break;
                    tc_fence_after();
                    score(tS, sK, sQ_of(st1));
                    mma_commit(bars.s_full());
                }
                if (!wait(bars.ds_done(), step & 1, kBSiteP)) break;
                tc_fence_after();
                accumulate(tdK, tDP, sQ_of(st), step == 0);
                mma_commit(bars.st_empty(st));
                if (!last) {
                    score(tDP, sV, sQ_of(st1) + C::TILE);
                    mma_commit(bars.dp_full());
                }
                ++step;
                if (last) break;
                e = nx;
            }
            mma_commit(bars.drain());
            wait(bars.drain(), 0, kBSiteDrain, false);
        }
    } else if (warp >= 4) {
        // ---------------- elementwise: warpgroup wg takes query columns 64 wg .. 64 wg + 63,
        // in two chunks of 32
        const int wg = (warp - 4) >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;                      // key row of the tile (TMEM lane)
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const int64_t jk = (int64_t)kt * 128 + row;               // local key index on rank src
        const bool key_valid = jk < P.n;
        const int kpos = key_valid ? __ldg(P.posL + (int64_t)src * P.n + jk) : INT_MAX;
        const uint64_t c2 = f2_pack(P.scale_log2, P.scale_log2);
        const uint32_t xs = tmem + lane_base + C::COL_S + 64 * wg, xd = tmem + lane_base + C::COL_DP + 64 * wg;
        bool ok = true;
        int step = 0;
        int n_steps = 0;
        for (;;) {
            const int slot = step % kRing, st = step % kNS;
            ok = __all_sync(0xffffffffu, wait(bars.ring_full(slot), (step / kRing) & 1, kBSiteWalk));
            if (!ok) break;
            const int4 e = ld_shared_v4(ring + 16u * (uint32_t)slot);
            if (e.w & kFlagEmpty) break;
            const int qt = e.y, tmask = (e.w >> 2) & 1;
            int qvalid = 128;
            if (qt == P.n_qt - 1 && (P.n % 128) != 0) qvalid = (int)(P.n - (int64_t)qt * 128);
            const int64_t qoff = (int64_t)e.x * P.n + (int64_t)qt * 128;   // positions of the query tile
            const int32_t* qposg = P.posL + qoff;
            // Which queries of each chunk this row is seen by: all on unmasked tiles (no branch in
            // the element loop), else by position, one bit per query column. Computed before the
            // scores are ready.
            uint32_t vis[2] = {0xffffffffu, 0xffffffffu};
            if (tmask) {
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int c0 = 64 * wg + 32 * ch;
                    uint32_t bits = 0u;
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const int col = c0 + 4 * q4;
                        int4 qp4 = make_int4(INT_MIN, INT_MIN, INT_MIN, INT_MIN);
                        if (col + 3 < qvalid && ((qoff + col) & 3) == 0) {   // 16-byte aligned: one vector load
                            qp4 = __ldg(reinterpret_cast<const int4*>(qposg + col));
                        } else {
                            if (col < qvalid) qp4.x = __ldg(qposg + col);
                            if (col + 1 < qvalid) qp4.y = __ldg(qposg + col + 1);
                            if (col + 2 < qvalid) qp4.z = __ldg(qposg + col + 2);
                            if (col + 3 < qvalid) qp4.w = __ldg(qposg + col + 3);
                        }
                        const int qp[4] = {qp4.x, qp4.y, qp4.z, qp4.w};
                        int ql[4] = {INT_MIN, INT_MIN, INT_MIN, INT_MIN};
                        if (LB) {
                            const int32_t* qlog = P.loL + qoff;
#pragma unroll
                            for (int e4 = 0; e4 < 4; ++e4)
                                if (col + e4 < qvalid) ql[e4] = __ldg(qlog + col + e4);
                        }
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const bool vis_q = key_valid && col + e4 < qvalid && (!P.causal || kpos <= qp[e4]) &&
                                               (!LB || kpos >= ql[e4]);
                            bits |= (vis_q ? 1u : 0u) << (4 * q4 + e4);
                        }
                    }
                    vis[ch] = bits;
                }
            }
            const float4* nl4 = reinterpret_cast<const float4*>(smem + C::OFF_SIDE + st * 2 * 512) + 16 * wg;   // -lse2
            const float4* nd4 = nl4 + 32;                                                                       // -D
            // phase 1: P^T from S^T, kept in registers, packed back into S for dV += P^T dO
            ok = __all_sync(0xffffffffu, wait(bars.s_full(), step & 1, kBSiteSt));
            if (!ok) break;
            tc_fence_after();
            float pf[64];
            {
                uint32_t sa[32], sb2[32];
                tmem_ld32_nw(xs, sa);
                tmem_ld32_nw(xs + 32, sb2);
                tmem_ld_wait2(sa, sb2);
                if (tmask) {
                    p_chunk<true>(sa, nl4, 0, c2, vis[0], pf);
                    p_chunk<true>(sb2, nl4 + 8, 0, c2, vis[1], pf + 32);
                } else {
                    p_chunk<false>(sa, nl4, 0, c2, 0u, pf);
                    p_chunk<false>(sb2, nl4 + 8, 0, c2, 0u, pf + 32);
                }
                uint32_t pk[16];
                pack_chunk(pf, pk);
                tmem_st16(xs, pk);
                pack_chunk(pf + 32, pk);
                tmem_st16(xs + 16, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.p_done());
            // phase 2: dS^T = P^T (dP^T - D), packed into dP for dK += dS^T Q
            ok = __all_sync(0xffffffffu, wait(bars.dp_full(), step & 1, kBSiteSt));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t dr[32], pd[16];
                tmem_ld32(xd + 32 * ch, dr);
                ds_chunk(dr, pf + 32 * ch, nd4 + 8 * ch, 0, pd);
                tmem_st16(xd + 16 * ch, pd);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.ds_done());
            ++step;
            ++n_steps;
            if (e.w & kFlagLast) break;
        }
        // epilogue: wait for the last accumulating MMAs, then write dK (scaled) and dV
        if (ok && n_steps > 0) {
            ok = __all_sync(0xffffffffu, wait(bars.drain(), 0, kBSiteDone));
            if (ok) tc_fence_after();
        }
        // tcgen05.ld is a warp-wide instruction: every lane loads, and only the lanes of valid
        // keys store (the last key tile of a block may be short)
        if (ok && P.dk_f32) {
            // One ring step: this step's contribution, fp32, in the holder's slot: written (step
            // 0 starts the partial sums), or added into the partial sums that arrived with the
            // blocks by fire-and-forget reductions (one per element and step, ordered by the
            // launches: deterministic); an empty walk adds nothing.
            // The rows go through this warp's 4 KB of the fixed-pair region (free once the last
            // MMA has drained), as in the dQ kernel: whole 128-byte row segments per reduction.
            const int64_t jk0 = (int64_t)kt * 128 + quarter * 32;      // the warp's first key row
            const int64_t krow0 = (((int64_t)kvr * P.B + b) * P.n_kv + kvh) * P.n + jk0;
            const uint32_t stg = sb + C::OFF_F0 + (uint32_t)(warp - 4) * 4096u;
            // An empty walk waited for no MMA, so nothing yet says the fixed pair's load has
            // landed: wait for it before its region is reused.
            bool staged = n_steps > 0 || !P.dkdv_add;
            if (staged && n_steps == 0) staged = __all_sync(0xffffffffu, wait(bars.fixed_full(), 0, kBSiteFixed));
#pragma unroll
            for (int which = 0; which < 2 && staged; ++which) {
                const uint32_t col0 = (which ? C::COL_A1 : C::COL_A0) + (uint32_t)(wg * (D / 2));
                const float mul = which ? P.scale : 1.0f;
                float* g = which ? P.dk_f32 : P.dv_f32;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t t[32];
                    if (n_steps > 0) {
                        tmem_ld32(tmem + lane_base + col0 + c * 32, t);
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; ++q) t[q] = 0u;
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_shared_v4(stg + (lane * 8 + (q ^ (lane & 7))) * 16, __float_as_uint(__uint_as_float(t[4 * q]) * mul),
                                     __float_as_uint(__uint_as_float(t[4 * q + 1]) * mul),
                                     __float_as_uint(__uint_as_float(t[4 * q + 2]) * mul),
                                     __float_as_uint(__uint_as_float(t[4 * q + 3]) * mul));
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = i * 4 + (lane >> 3), q = lane & 7;
                        const int4 x = ld_shared_v4(stg + (rr * 8 + (q ^ (rr & 7))) * 16);
                        if (jk0 + rr < P.n) {
                            float* dst = g + (krow0 + rr) * D + wg * (D / 2) + c * 32 + q * 4;
                            if (P.dkdv_add)
                                red_add_v4_f32(dst, __int_as_float(x.x), __int_as_float(x.y), __int_as_float(x.z), __int_as_float(x.w));
                            else *reinterpret_cast<int4*>(dst) = x;
                        }
                    }
                    __syncwarp();
                }
            }
        } else if (ok) {
            const int64_t tn = key_valid ? natural_token(P.layout, src, jk, P.n, P.m, P.n_cp) : 0;
            uint4* gk = reinterpret_cast<uint4*>(P.dk + (((int64_t)b * P.T + tn) * P.n_kv + kvh) * D);
            uint4* gv = reinterpret_cast<uint4*>(P.dv + (((int64_t)b * P.T + tn) * P.n_kv + kvh) * D);
            // each warpgroup writes half of the columns of both gradients
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                const uint32_t col0 = (which ? C::COL_A1 : C::COL_A0) + (uint32_t)(wg * (D / 2));
                const float mul = which ? P.scale : 1.0f;
                uint4* g = which ? gk : gv;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t t[32];
                    if (n_steps > 0) {
                        tmem_ld32(tmem + lane_base + col0 + c * 32, t);
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; ++q) t[q] = 0u;
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 v;
                        v.x = pack_bf16(__uint_as_float(t[8 * q4 + 0]) * mul, __uint_as_float(t[8 * q4 + 1]) * mul);
                        v.y = pack_bf16(__uint_as_float(t[8 * q4 + 2]) * mul, __uint_as_float(t[8 * q4 + 3]) * mul);
                        v.z = pack_bf16(__uint_as_float(t[8 * q4 + 4]) * mul, __uint_as_float(t[8 * q4 + 5]) * mul);
                        v.w = pack_bf16(__uint_as_float(t[8 * q4 + 6]) * mul, __uint_as_float(t[8 * q4 + 7]) * mul);
                        if (key_valid) g[(wg * (D / 2) + c * 32) / 8 + q4] = v;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// =============================================================================================
// bwd_dq_kernel
// =============================================================================================
template <int D, bool LB>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const BwdParams P) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
    const uint32_t ring = sb + C::OFF_RING;
    const BBars<D> bars{sb + C::OFF_BAR};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // unit: (b, head, r, qt), KV-head-major (the CTAs in flight share one head's K and V in L2):
    // per (b, KV head), the query tiles heaviest first, the group's query heads of a tile together
    const int n_tiles = P.n_cp * P.n_qt;
    const int per_bk = n_tiles * P.g;
    const int bk = blockIdx.x / per_bk, rem = blockIdx.x % per_bk;
    const int uq = __ldg(P.order_q + rem / P.g);
    const int qt = uq % P.n_qt, r = uq / P.n_qt;
    const int b = bk / P.n_kv, head = (bk % P.n_kv) * P.g + rem % P.g;
    const int kvh = head / P.g;

    if (threadIdx.x == 0) *skip_flag = (int)*(volatile uint32_t*)(P.header + kErrFlags);
    __syncthreads();
    if (*skip_flag) return;
    if (threadIdx.x == 0) {
        bars.init();
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmDO);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const BWaiter wait{abort_flag, P.header, P.timeout_ns};
    const int4 qmm = __ldg(P.tile_mm + r * P.n_qt + qt);
    const int2 qlb = tile_bound<LB>(P, r, qt);
    const int qrow0 = (int)((((int64_t)r * P.B + b) * P.h + head) * P.n + (int64_t)qt * 128);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer: fixed Q, dO; walk the key tiles in ring order
            mbar_arrive_expect_tx(bars.fixed_full(), 2 * C::TILE);
            for (int pn = 0; pn < C::PANELS; ++pn) {
                tma_load_2d(sb + C::OFF_F0 + pn * C::PANEL_BYTES, &tmQ, bars.fixed_full(), pn * 64, qrow0);
                tma_load_2d(sb + C::OFF_F1 + pn * C::PANEL_BYTES, &tmDO, bars.fixed_full(), pn * 64, qrow0);
            }
            int ns = 0, nl = 0;         // steps published, stages loaded
            bool ok = true;
            int pending = -1, pend_src = 0, pend_kt = 0, pend_flags = 0;
            auto publish = [&](int srcr, int ktt, int flags) -> bool {
                const int slot = ns % kRing, st = ns % kNS;
                if (!(flags & kFlagEmpty)) {
                    if (ns >= kNS && !wait(bars.st_empty(st), ((ns / kNS) - 1) & 1, kBSiteStageEmpty)) return false;
                    // one ring step: the visiting block sits in rank r's slot
                    const int kvr = P.step >= 0 ? r : srcr;
                    const int krow = (int)((((int64_t)kvr * P.B + b) * P.n_kv + kvh) * P.n + (int64_t)ktt * 128);
                    mbar_arrive_expect_tx(bars.st_full(st), 2 * C::TILE);
                    const uint32_t s0 = sb + C::OFF_S + (2 * st) * C::TILE, s1 = s0 + C::TILE;
                    for (int pn = 0; pn < C::PANELS; ++pn) {
                        tma_load_2d(s0 + pn * C::PANEL_BYTES, &tmK, bars.st_full(st), pn * 64, krow);
                        tma_load_2d(s1 + pn * C::PANEL_BYTES, &tmV, bars.st_full(st), pn * 64, krow);
                    }
                    ++nl;
                }
                st_shared_v4(ring + 16u * (uint32_t)slot, (uint32_t)srcr, (uint32_t)ktt, 0u, (uint32_t)flags);
                mbar_arrive(bars.ring_full(slot));
                ++ns;
                return true;
            };
            const int s_lo = P.step >= 0 ? P.step : 0, s_hi = P.step >= 0 ? P.step + 1 : P.n_cp;
            for (int s = s_lo; s < s_hi && ok; ++s) {
                const int srcr = (r - s + P.n_cp) % P.n_cp;     // the block rank r holds at step s
                for (int ktt = 0; ktt < P.n_qt && ok; ++ktt) {
                    const int4 kmm = __ldg(P.tile_mm + srcr * P.n_qt + ktt);
                    // causal: this key tile and every later one of the block start after every
                    // query (suffix minimum .z): none of the rest is visible
                    if (P.causal && kmm.z > qmm.y) break;
                    const int cls = tile_class(P.causal, qmm, qlb, kmm);
                    if (cls == CPATTN_TILE_SKIP) continue;
                    const int qshort = (qt == P.n_qt - 1) && (P.n % 128) != 0;
                    const int kshort = (ktt == P.n_qt - 1) && (P.n % 128) != 0;
                    const int mask = (cls != CPATTN_TILE_FULL) || qshort || kshort;
                    if (pending >= 0) ok = publish(pend_src, pend_kt, pend_flags);
                    pending = 1;
                    pend_src = srcr; pend_kt = ktt; pend_flags = cls | (mask << 2);
                }
            }
            if (ok) {
                if (pending >= 0) ok = publish(pend_src, pend_kt, pend_flags | kFlagLast);
                else ok = publish(0, 0, kFlagEmpty | kFlagLast);
            }
            // the CTA exits only after its own copies have landed (bounded waits)
            const int first = nl > kNS ? nl - kNS : 0;
            for (int i = first; i < nl; ++i) wait(bars.st_full(i % kNS), (i / kNS) & 1, kBSiteStage, false);
            wait(bars.fixed_full(), 0, kBSiteFixed, false);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issue. Per walked key tile (stage st):
            //   S = Q K^T into S and dP = dO V^T into dP               (TS form, Q and dO in TMEM)
            //   dQ += dS K once dS is packed into dP                   (TS form)
            // issued as  [p_done] S(i+1), [ds_done] dQ(i), dP(i+1): the next score MMA starts as soon
            // as the elementwise warps hold P(i) in registers.
            // The score MMAs take Q and dO from tensor memory (TS form), so only K and V are read
            // from shared memory, which the stage loads also write.
            constexpr uint32_t kIdX = idesc_bf16(128, 128, 0, 0);    // A = Q or dO (TMEM), B = K or V (K-major)
            constexpr uint32_t kIdTS = idesc_bf16(128, D, 0, 1);     // A = dS (TMEM), B = K (MN-major)
            const uint32_t tQ = tmem + C::COL_Q, tDO = tmem + C::COL_DO;
            const uint32_t tdQ = tmem + C::COL_A0, tS = tmem + C::COL_S, tDP = tmem + C::COL_DP;
            auto score = [&](uint32_t d, uint32_t a_t, uint32_t b) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * C::PANEL_BYTES + (kk & 3) * 32;
                    mma_bf16_ts(d, a_t + 8 * kk, desc_sw128(b + off, 16, 1024), kIdX, kk > 0);
                }
            };
            auto sK_of = [&](int st) { return sb + C::OFF_S + (2 * st) * C::TILE; };
            bool ok = wait(bars.fixed_tmem(), 0, kBSiteFixed);
            int4 e = make_int4(0, 0, 0, kFlagEmpty);
            if (ok) ok = wait(bars.ring_full(0), 0, kBSiteWalk);
            if (ok) e = ld_shared_v4(ring);
            if (ok && !(e.w & kFlagEmpty)) {
                ok = wait(bars.st_full(0), 0, kBSiteStage);
                if (ok) {
                    tc_fence_after();
                    score(tS, tQ, sK_of(0));
                    mma_commit(bars.s_full());
                    score(tDP, tDO, sK_of(0) + C::TILE);
                    mma_commit(bars.dp_full());
                }
            }
            int step = 0;
            while (ok && !(e.w & kFlagEmpty)) {
                const int st = step % kNS, st1 = (step + 1) % kNS;
                const bool last = (e.w & kFlagLast) != 0;
                if (!wait(bars.p_done(), step & 1, kBSiteP)) break;
                int4 nx = e;
                if (!last) {
                    const int n1 = step + 1;
                    if (!wait(bars.ring_full(n1 % kRing), (n1 / kRing) & 1, kBSiteWalk)) break;
                    nx = ld_shared_v4(ring + 16u * (uint32_t)(n1 % kRing));
                    if (!wait(bars.st_full(st1), (n1 / kNS) & 1, kBSiteStage)) break;
                    tc_fence_after();
                    score(tS, tQ, sK_of(st1));
                    mma_commit(bars.s_full());
                }
                if (!wait(bars.ds_done(), step & 1, kBSiteP)) break;
                tc_fence_after();
                // dS packed like P^T in the dK/dV kernel: keys 16 kk .. 16 kk + 15 at 64 (kk / 4) + 8 (kk % 4)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(tdQ, tDP + 64 * (kk >> 2) + 8 * (kk & 3),
                                desc_sw128(sK_of(st) + kk * 2048, C::PANEL_BYTES, 1024), kIdTS,
                                (step > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bars.st_empty(st));
                if (!last) {
                    score(tDP, tDO, sK_of(st1) + C::TILE);
                    mma_commit(bars.dp_full());
                }
                ++step;
                if (last) break;
                e = nx;
            }
            mma_commit(bars.drain());
            wait(bars.drain(), 0, kBSiteDrain, false);
        }
    } else if (warp >= 4) {
        // ---------------- elementwise: warpgroup wg takes key columns 64 wg .. 64 wg + 63, in two
        // chunks of 32
        const int wg = (warp - 4) >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;                      // query row of the tile (TMEM lane)
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const int64_t jq = (int64_t)qt * 128 + row;
        const bool q_valid = jq < P.n;
        const int64_t lrow = (((int64_t)r * P.B + b) * P.h + head) * P.n_pad + jq;
        const int qpos = q_valid ? __ldg(P.posL + (int64_t)r * P.n + jq) : INT_MIN;
        const float nl = q_valid ? __ldg(P.nlse2L + lrow) : INFINITY;
        const bool row_live = q_valid && nl != INFINITY;      // a row that sees some key
        // a row that sees no key gets x = -inf everywhere: P = 0 and dS = 0
        const uint64_t nl2 = row_live ? f2_pack(nl, nl) : f2_pack(-INFINITY, -INFINITY);
        const float nd = row_live ? __ldg(P.nDL + lrow) : 0.f;
        const uint64_t nd2 = f2_pack(nd, nd);
        const uint64_t c2 = f2_pack(P.scale_log2, P.scale_log2);
        const int qlo = (LB && q_valid) ? __ldg(P.loL + (int64_t)r * P.n + jq) : INT_MIN;
        const uint32_t xs = tmem + lane_base + C::COL_S + 64 * wg, xd = tmem + lane_base + C::COL_DP + 64 * wg;
        // The fixed tiles into tensor memory: warpgroup 0 copies Q, warpgroup 1 dO, each thread its
        // row. Row r of a 128-byte-swizzled panel holds its 16-byte chunk j at chunk j ^ (r % 8).
        bool ok = __all_sync(0xffffffffu, wait(bars.fixed_full(), 0, kBSiteFixed));
        if (ok) {
            const uint8_t* tile = smem + (wg == 0 ? C::OFF_F0 : C::OFF_F1);
            uint32_t rw[D / 2];
#pragma unroll
            for (int pn = 0; pn < C::PANELS; ++pn)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 v = *reinterpret_cast<const uint4*>(tile + pn * C::PANEL_BYTES + row * 128 + ((j ^ (row & 7)) << 4));
                    rw[32 * pn + 4 * j] = v.x;
                    rw[32 * pn + 4 * j + 1] = v.y;
                    rw[32 * pn + 4 * j + 2] = v.z;
                    rw[32 * pn + 4 * j + 3] = v.w;
                }
            const uint32_t dst = tmem + lane_base + (wg == 0 ? C::COL_Q : C::COL_DO);
            if constexpr (D == 128) tmem_st64(dst, rw);
            else tmem_st32(dst, rw);
            tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.fixed_tmem());
        int step = 0, n_steps = 0;
        for (;;) {
            const int slot = step % kRing;
            ok = __all_sync(0xffffffffu, wait(bars.ring_full(slot), (step / kRing) & 1, kBSiteWalk));
            if (!ok) break;
            const int4 e = ld_shared_v4(ring + 16u * (uint32_t)slot);
            if (e.w & kFlagEmpty) break;
            const int srcr = e.x, ktt = e.y, tmask = (e.w >> 2) & 1;
            int kvalid = 128;
            if (ktt == P.n_qt - 1 && (P.n % 128) != 0) kvalid = (int)(P.n - (int64_t)ktt * 128);
            const int64_t kbase = (int64_t)srcr * P.n + (int64_t)ktt * 128;
            // Which keys of each chunk this row sees: all of them on unmasked tiles, else by
            // position (keys beyond a short block are never seen), one bit per key column.
            // Computed before the scores are ready.
            uint32_t vis[2] = {0u, 0u};
            if (tmask && row_live) {
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int c0 = 64 * wg + 32 * ch;
                    uint32_t bits = 0u;
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        const int col = c0 + 4 * q4;
                        int4 kp4 = make_int4(INT_MAX, INT_MAX, INT_MAX, INT_MAX);
                        if (col + 3 < kvalid && ((kbase + col) & 3) == 0) {   // 16-byte aligned: one vector load
                            kp4 = __ldg(reinterpret_cast<const int4*>(P.posL + kbase + col));
                        } else {
                            if (col < kvalid) kp4.x = __ldg(P.posL + kbase + col);
                            if (col + 1 < kvalid) kp4.y = __ldg(P.posL + kbase + col + 1);
                            if (col + 2 < kvalid) kp4.z = __ldg(P.posL + kbase + col + 2);
                            if (col + 3 < kvalid) kp4.w = __ldg(P.posL + kbase + col + 3);
                        }
                        const int kp[4] = {kp4.x, kp4.y, kp4.z, kp4.w};
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const bool vis_k = col + e4 < kvalid && (!P.causal || kp[e4] <= qpos) && (!LB || kp[e4] >= qlo);
                            bits |= (vis_k ? 1u : 0u) << (4 * q4 + e4);
                        }
                    }
                    vis[ch] = bits;
                }
            }
            // phase 1: P from S, kept in registers; S is free for the next key tile's scores
            ok = __all_sync(0xffffffffu, wait(bars.s_full(), step & 1, kBSiteSt));
            if (!ok) break;
            tc_fence_after();
            float pf[64];
            {
                uint32_t sa[32], sb2[32];
                tmem_ld32_nw(xs, sa);
                tmem_ld32_nw(xs + 32, sb2);
                tmem_ld_wait2(sa, sb2);
                if (tmask) {
                    p_chunk<true>(sa, nullptr, nl2, c2, vis[0], pf);
                    p_chunk<true>(sb2, nullptr, nl2, c2, vis[1], pf + 32);
                } else {
                    p_chunk<false>(sa, nullptr, nl2, c2, 0u, pf);
                    p_chunk<false>(sb2, nullptr, nl2, c2, 0u, pf + 32);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.p_done());
            // phase 2: dS = P (dP - D), packed into dP for dQ += dS K
            ok = __all_sync(0xffffffffu, wait(bars.dp_full(), step & 1, kBSiteSt));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t dr[32], pd[16];
                tmem_ld32(xd + 32 * ch, dr);
                ds_chunk(dr, pf + 32 * ch, nullptr, nd2, pd);
                tmem_st16(xd + 16 * ch, pd);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.ds_done());
            ++step;
            ++n_steps;
            if (e.w & kFlagLast) break;
        }
        if (ok && n_steps > 0) {
            ok = __all_sync(0xffffffffu, wait(bars.drain(), 0, kBSiteDone));
            if (ok) tc_fence_after();
        }
        // warp-wide TMEM loads; only the lanes of valid query rows store
        if (ok && P.dq_run) {
            // One ring step: add this step's dQ into the running fp32 rows of rank r (step 0
            // writes). The additions are fire-and-forget reductions, one per element and step (the
            // steps are ordered by their launches, so the sum is deterministic): no read of the
            // running rows to wait on. A later step with nothing visible adds nothing.
            // The rows go through this warp's 4 KB of the fixed-pair region (free once the last
            // MMA has drained), 16-byte pieces XOR-swizzled by row, so that each reduction moves a
            // whole 128-byte row segment: 8 lanes per row, 4 rows per instruction.
            const int64_t jq0 = (int64_t)qt * 128 + quarter * 32;      // the warp's first query row
            const int64_t qrow0 = (((int64_t)r * P.B + b) * P.h + head) * P.n + jq0;
            const uint32_t stg = sb + C::OFF_F0 + (uint32_t)(warp - 4) * 4096u;
#pragma unroll
            for (int c = 0; c < D / 64 && (n_steps > 0 || P.step == 0); ++c) {
                uint32_t t[32];
                if (n_steps > 0) {
                    tmem_ld32(tmem + lane_base + C::COL_A0 + wg * (D / 2) + c * 32, t);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) t[q] = 0u;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_shared_v4(stg + (lane * 8 + (q ^ (lane & 7))) * 16,
                                 __float_as_uint(__uint_as_float(t[4 * q]) * P.scale),
                                 __float_as_uint(__uint_as_float(t[4 * q + 1]) * P.scale),
                                 __float_as_uint(__uint_as_float(t[4 * q + 2]) * P.scale),
                                 __float_as_uint(__uint_as_float(t[4 * q + 3]) * P.scale));
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = i * 4 + (lane >> 3), q = lane & 7;
                    const int4 x = ld_shared_v4(stg + (rr * 8 + (q ^ (rr & 7))) * 16);
                    if (jq0 + rr < P.n) {
                        float* dst = P.dq_run + (qrow0 + rr) * D + wg * (D / 2) + c * 32 + q * 4;
                        if (P.step > 0) red_add_v4_f32(dst, __int_as_float(x.x), __int_as_float(x.y), __int_as_float(x.z), __int_as_float(x.w));
                        else *reinterpret_cast<int4*>(dst) = x;
                    }
                }
                __syncwarp();
            }
        } else if (ok) {
            const int64_t tn = q_valid ? natural_token(P.layout, r, jq, P.n, P.m, P.n_cp) : 0;
            uint4* g = reinterpret_cast<uint4*>(P.dq + (((int64_t)b * P.T + tn) * P.h + head) * D);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t t[32];
                if (n_steps > 0) {
                    tmem_ld32(tmem + lane_base + C::COL_A0 + wg * (D / 2) + c * 32, t);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) t[q] = 0u;
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 v;
                    v.x = pack_bf16(__uint_as_float(t[8 * q4 + 0]) * P.scale, __uint_as_float(t[8 * q4 + 1]) * P.scale);
                    v.y = pack_bf16(__uint_as_float(t[8 * q4 + 2]) * P.scale, __uint_as_float(t[8 * q4 + 3]) * P.scale);
                    v.z = pack_bf16(__uint_as_float(t[8 * q4 + 4]) * P.scale, __uint_as_float(t[8 * q4 + 5]) * P.scale);
                    v.w = pack_bf16(__uint_as_float(t[8 * q4 + 6]) * P.scale, __uint_as_float(t[8 * q4 + 7]) * P.scale);
                    if (q_valid) g[(wg * (D / 2) + c * 32) / 8 + q4] = v;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, bool LB>
int launch_bwd_d(const BwdLaunch& a, cudaStream_t st, std::string* why) {
    using C = BCfg<D>;
    static PerDeviceOnce attr_once;
    int dev = 0;
    cudaGetDevice(&dev);
    const int ea = attr_once.run(dev, [&]() -> int {
        cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_kernel<D, LB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(bwd_dq_kernel<D, LB>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        return (int)e;
    });
    if (ea) return ea;
    CUtensorMap tq, tdo, tk, tv;
    const uint64_t qrows = (uint64_t)a.n_cp * a.B * a.h * a.n, kvrows = (uint64_t)a.n_cp * a.B * a.n_kv * a.n;
    if (!make_map(&tq, a.qL, qrows, D) || !make_map(&tdo, a.doL, qrows, D) || !make_map(&tk, a.kL, kvrows, D) ||
        !make_map(&tv, a.vL, kvrows, D)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point unavailable or bad tensor shape)";
        return (int)cudaErrorInvalidValue;
    }
    BwdParams P{};
    P.B = a.B; P.h = a.h; P.n_kv = a.n_kv; P.g = a.h / a.n_kv; P.n_cp = a.n_cp; P.n_qt = a.n_qt;
    P.causal = a.causal; P.layout = a.layout; P.n = a.n; P.m = a.m; P.T = a.T; P.n_pad = (int64_t)a.n_qt * 128;
    P.scale = a.scale; P.scale_log2 = a.scale * kLog2e;
    P.posL = a.posL; P.tile_mm = reinterpret_cast<const int4*>(a.tile_mm);
    P.nlse2L = a.nlse2L; P.nDL = a.nDL; P.order_q = a.order_q; P.order_kv = a.order_kv;
    P.loL = a.loL; P.tile_lo = reinterpret_cast<const int4*>(a.tile_lo);
    P.dq = static_cast<uint16_t*>(a.dq); P.dk = static_cast<uint16_t*>(a.dk); P.dv = static_cast<uint16_t*>(a.dv);
    P.header = a.header; P.timeout_ns = a.timeout_ns;
    P.step = a.step; P.dk_f32 = a.dk_f32; P.dv_f32 = a.dv_f32; P.dq_run = a.dq_run; P.dkdv_add = a.dkdv_add;
    const int64_t kv_units = (int64_t)a.B * a.n_kv * a.n_cp * a.n_qt, q_units = (int64_t)a.B * a.h * a.n_cp * a.n_qt;
    if (kv_units > INT_MAX || q_units > INT_MAX) {
        *why = "too many work units";
        return (int)cudaErrorInvalidValue;
    }
    int e = 0;
    if (a.dkdv_after) {
        // the dK/dV kernel adds into partial sums that are still arriving: dQ first, then wait
        bwd_dq_kernel<D, LB><<<(int)q_units, kThreads, C::SMEM_BYTES, st>>>(tq, tdo, tk, tv, P);
        if ((e = (int)cudaGetLastError())) return e;
        if ((e = (int)cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(a.dkdv_after), 0))) return e;
        bwd_dkdv_kernel<D, LB><<<(int)kv_units, kThreads, C::SMEM_BYTES, st>>>(tq, tdo, tk, tv, P);
        return (int)cudaGetLastError();
    }
    bwd_dkdv_kernel<D, LB><<<(int)kv_units, kThreads, C::SMEM_BYTES, st>>>(tq, tdo, tk, tv, P);
    if ((e = (int)cudaGetLastError())) return e;
    bwd_dq_kernel<D, LB><<<(int)q_units, kThreads, C::SMEM_BYTES, st>>>(tq, tdo, tk, tv, P);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_bwd_prep(const BwdPrepArgs& a, void* stream) {
    const int64_t work = (int64_t)a.B * a.T * a.h * (a.d / 8);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (work + 255) / 256, cap = (int64_t)sms * 8;
    bwd_prep_kernel<<<(int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.dout), a.lse, static_cast<uint4*>(a.doL), a.nlse2L,
        a.nDL, a.B, a.T, a.n, a.m, (int64_t)a.n_qt * 128, a.h, a.d, a.n_cp, a.layout);
    return (int)cudaGetLastError();
}

int launch_backward(const BwdLaunch& a, void* stream, std::string* why) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool lb = a.loL != nullptr;   // document masks
    if (a.d == 128) return lb ? launch_bwd_d<128, true>(a, st, why) : launch_bwd_d<128, false>(a, st, why);
    if (a.d == 64) return lb ? launch_bwd_d<64, true>(a, st, why) : launch_bwd_d<64, false>(a, st, why);
    *why = "unsupported head width";
    return (int)cudaErrorInvalidValue;
}

}  // namespace cpattn
