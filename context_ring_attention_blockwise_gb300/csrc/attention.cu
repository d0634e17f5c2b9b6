// attention.cu -- the ring-step attention kernel for sm_103a.
//
// One CTA owns one work unit: 128 query rows of one (batch element, query head) on one virtual
// rank r. It walks the key/value blocks in ring order ("Context and expert parallelism",
// "Pass them around a ring": at step s rank r holds the block of rank (r - s) mod n_cp), skips
// key tiles that no query of the unit can see and masks the partly visible ones ("The causal
// mask unbalances the sequence"), and keeps the online-softmax state of the paragraph after it
// (running max, running sum of exponentials, running weighted sum of values, rescaled when a
// larger score arrives) on chip across every step.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q tile once, then K and V tiles through an NS-deep stage ring.
//   warp 1      owns tensor memory; one lane issues tcgen05.mma: S = Q K^T into one of two
//               TMEM score buffers, O += P V into the TMEM output accumulator.
//   warps 2..5  one thread per query row: read S from TMEM, mask, row max, exp2, row sum,
//               write P (bf16) to shared memory, rescale O lazily, and the epilogue.
// Tensor memory (512 columns): S0 at 0, S1 at 128, O at 256 (d_k columns of fp32).
//
// Rescaling is lazy: the row keeps using a stale maximum m_used until a tile raises the row
// maximum by more than 8 (in log2 units), so P stays below 2^8 and the final O / l is unchanged.
// Every wait is bounded by a global-timer limit; on expiry the kernel records the wait site in
// the workspace header, lets every role leave its loop, waits for its own copies and MMAs, and
// frees tensor memory before returning.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace cpattn {
namespace {

using namespace ptx;

struct Params {
    int B, h, n_kv, g, n_cp, n_qt, causal, fused, step, kv_by_holder, layout;
    int64_t n, m, T;
    float scale_log2;
    const int32_t* posL;
    const int2* tile_mm;
    const int32_t* order;
    unsigned long long* counts;
    uint16_t* o;
    float* lse;
    float* o_run;
    float* lse_run;
    uint32_t* header;
    uint64_t timeout_ns;
};

template <int D>
struct Cfg {
    static constexpr int NS = (D == 128) ? 2 : 3;         // K/V stage depth
    static constexpr int PANELS = D / 64;                 // 64-column (128-byte) swizzle panels
    static constexpr int PANEL_BYTES = 128 * 128;         // 128 rows x 128 bytes
    static constexpr int Q_BYTES = 128 * D * 2;
    static constexpr int KV_BYTES = 128 * D * 2;
    static constexpr int P_BYTES = 128 * 128 * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + NS * KV_BYTES;
    static constexpr int OFF_P = OFF_V + NS * KV_BYTES;
    static constexpr int OFF_BAR = OFF_P + P_BYTES;
    static constexpr int NBAR = 1 + 4 * NS + 2 + 2 + 1 + 1 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t O_COL = 256;
};

// Barrier addresses in shared memory.
template <int D>
struct Bars {
    uint32_t q_full, k_full[Cfg<D>::NS], v_full[Cfg<D>::NS], k_empty[Cfg<D>::NS], v_empty[Cfg<D>::NS];
    uint32_t s_full[2], s_free[2], p_full, pv_done, mma_done;
    __device__ void setup(uint32_t base) {
        uint32_t a = base;
        auto next = [&]() { uint32_t r = a; a += 8; return r; };
        q_full = next();
        for (int i = 0; i < Cfg<D>::NS; ++i) k_full[i] = next();
        for (int i = 0; i < Cfg<D>::NS; ++i) v_full[i] = next();
        for (int i = 0; i < Cfg<D>::NS; ++i) k_empty[i] = next();
        for (int i = 0; i < Cfg<D>::NS; ++i) v_empty[i] = next();
        s_full[0] = next(); s_full[1] = next();
        s_free[0] = next(); s_free[1] = next();
        p_full = next(); pv_done = next(); mma_done = next();
    }
    __device__ void init() {
        mbar_init(q_full, 1);
        for (int i = 0; i < Cfg<D>::NS; ++i) {
            mbar_init(k_full[i], 1); mbar_init(v_full[i], 1);
            mbar_init(k_empty[i], 1); mbar_init(v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) { mbar_init(s_full[i], 1); mbar_init(s_free[i], 128); }
        mbar_init(p_full, 128);
        mbar_init(pv_done, 1);
        mbar_init(mma_done, 1);
    }
};

// Wait sites reported through the header on a timeout.
enum Site : int { kSiteQ = 1, kSiteKFull, kSiteVFull, kSiteKEmpty, kSiteVEmpty, kSiteSFull, kSiteSFree,
                  kSitePFull, kSitePvDone, kSiteDrain, kSiteSelfTest };

struct Waiter {
    volatile int* abort_flag;
    uint32_t* header;
    uint64_t timeout_ns;
    // Spin on (bar, parity). Returns false on abort or timeout (then recorded in the header).
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

// The key tiles one unit visits, in ring order, with SKIP tiles left out. Every role walks the
// same sequence. mask = 1 when the tile is partly visible or shorter than 128 keys.
struct TileWalk {
    const Params* p;
    int r, qmin, qmax, s, s_end, kt, src, mask, diag;
    __device__ void init(const Params& P, int r_, int2 qmm) {
        p = &P; r = r_; qmin = qmm.x; qmax = qmm.y;
        s = P.fused ? 0 : P.step;
        s_end = P.fused ? P.n_cp : P.step + 1;
        kt = -1;
    }
    __device__ bool next() {
        const Params& P = *p;
        for (;;) {
            if (++kt >= P.n_qt) {
                kt = 0;
                if (++s >= s_end) return false;
            }
            src = r - s;
            if (src < 0) src += P.n_cp;
            const bool short_tile = (kt == P.n_qt - 1) && (P.n % 128) != 0;
            if (!P.causal) { diag = 0; mask = short_tile; return true; }
            const int2 kmm = __ldg(P.tile_mm + src * P.n_qt + kt);
            if (kmm.x > qmax) continue;                 // every key after every query: skip
            diag = kmm.y > qmin;                        // some key after some query
            mask = diag || short_tile;                  // partly visible: element mask
            return true;
        }
    }
};

template <int D>
__device__ void producer(const Params& P, const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                         uint32_t sQ, uint32_t sK, uint32_t sV, const Bars<D>& bars, const Waiter& wait, int r,
                         int qt, int b, int head, int kvh, int2 qmm) {
    using C = Cfg<D>;
    TileWalk w;
    w.init(P, r, qmm);
    const int qrow = (int)((((int64_t)r * P.B + b) * P.h + head) * P.n + (int64_t)qt * 128);
    int nk = 0, nv = 0;            // K and V tiles issued
    int prev_row = 0;
    bool ok = true, q_issued = false;
    auto load_v = [&](int i, int row) -> bool {
        const int st = i % C::NS;
        if (i >= C::NS && !wait(bars.v_empty[st], ((i / C::NS) - 1) & 1, kSiteVEmpty)) return false;
        mbar_arrive_expect_tx(bars.v_full[st], C::KV_BYTES);
        for (int pn = 0; pn < C::PANELS; ++pn)
            tma_load_2d(sV + st * C::KV_BYTES + pn * C::PANEL_BYTES, tmV, bars.v_full[st], pn * 64, row);
        ++nv;
        return true;
    };
    while (w.next()) {
        const int holder = P.kv_by_holder ? r : w.src;
        const int krow = (int)((((int64_t)holder * P.B + b) * P.n_kv + kvh) * P.n + (int64_t)w.kt * 128);
        if (!q_issued) {
            mbar_arrive_expect_tx(bars.q_full, C::Q_BYTES);
            for (int pn = 0; pn < C::PANELS; ++pn) tma_load_2d(sQ + pn * C::PANEL_BYTES, tmQ, bars.q_full, pn * 64, qrow);
            q_issued = true;
        }
        const int st = nk % C::NS;
        if (nk >= C::NS && !wait(bars.k_empty[st], ((nk / C::NS) - 1) & 1, kSiteKEmpty)) { ok = false; break; }
        mbar_arrive_expect_tx(bars.k_full[st], C::KV_BYTES);
        for (int pn = 0; pn < C::PANELS; ++pn)
            tma_load_2d(sK + st * C::KV_BYTES + pn * C::PANEL_BYTES, tmK, bars.k_full[st], pn * 64, krow);
        ++nk;
        if (nk >= 2 && !load_v(nk - 2, prev_row)) { ok = false; break; }   // V runs one tile behind K
        prev_row = krow;
    }
    if (ok && nk >= 1) ok = load_v(nk - 1, prev_row);
    if (ok) {
        // Normal tail: the last arrivals of the tensor core on the stage barriers have landed.
        for (int i = (nk > C::NS ? nk - C::NS : 0); i < nk; ++i) wait(bars.k_empty[i % C::NS], (i / C::NS) & 1, kSiteKEmpty);
        for (int i = (nv > C::NS ? nv - C::NS : 0); i < nv; ++i) wait(bars.v_empty[i % C::NS], (i / C::NS) & 1, kSiteVEmpty);
    } else {
        // Aborted: still wait (bounded) until our own copies in flight have landed.
        if (q_issued) wait(bars.q_full, 0, kSiteQ, false);
        for (int i = (nk > C::NS ? nk - C::NS : 0); i < nk; ++i) wait(bars.k_full[i % C::NS], (i / C::NS) & 1, kSiteKFull, false);
        for (int i = (nv > C::NS ? nv - C::NS : 0); i < nv; ++i) wait(bars.v_full[i % C::NS], (i / C::NS) & 1, kSiteVFull, false);
    }
}

template <int D>
__device__ void mma_issuer(const Params& P, uint32_t tmem, uint32_t sQ, uint32_t sK, uint32_t sV, uint32_t sP,
                           const Bars<D>& bars, const Waiter& wait, int r, int2 qmm) {
    using C = Cfg<D>;
    constexpr uint32_t kIdescQK = idesc_bf16(128, 128, 0, 0);   // A = Q (K-major), B = K (K-major)
    constexpr uint32_t kIdescPV = idesc_bf16(128, D, 0, 1);     // A = P (K-major), B = V (MN-major)
    TileWalk w;
    w.init(P, r, qmm);
    auto issue_pv = [&](int i) -> bool {
        const int st = i % C::NS;
        if (!wait(bars.p_full, i & 1, kSitePFull)) return false;
        if (!wait(bars.v_full[st], (i / C::NS) & 1, kSiteVFull)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {      // 128 keys, 16 per MMA
            const uint64_t a = desc_sw128(sP + (kk >> 2) * C::PANEL_BYTES + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = desc_sw128(sV + st * C::KV_BYTES + kk * 2048, C::PANEL_BYTES, 1024);
            mma_bf16_ss(tmem + C::O_COL, a, bd, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bars.v_empty[st]);
        mma_commit(bars.pv_done);
        return true;
    };
    int j = 0;
    bool ok = true;
    while (w.next()) {
        if (j == 0 && !wait(bars.q_full, 0, kSiteQ)) { ok = false; break; }
        const int st = j % C::NS, sb = j & 1;
        if (!wait(bars.k_full[st], (j / C::NS) & 1, kSiteKFull)) { ok = false; break; }
        if (j >= 2 && !wait(bars.s_free[sb], ((j >> 1) - 1) & 1, kSiteSFree)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL_BYTES + (kk & 3) * 32;
            mma_bf16_ss(tmem + (sb ? 128u : 0u), desc_sw128(sQ + off, 16, 1024),
                        desc_sw128(sK + st * C::KV_BYTES + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(bars.s_full[sb]);
        mma_commit(bars.k_empty[st]);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
        ++j;
    }
    if (ok && j >= 1) issue_pv(j - 1);
    // Drain: every MMA this thread issued has completed before tensor memory is freed.
    mma_commit(bars.mma_done);
    wait(bars.mma_done, 0, kSiteDrain, false);
}

template <int D>
__device__ void softmax_epilogue(const Params& P, uint32_t tmem, uint32_t sP, const Bars<D>& bars,
                                 const Waiter& wait, int r, int qt, int b, int head, int2 qmm) {
    using C = Cfg<D>;
    const int quarter = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
    const int row = quarter * 32 + lane;                 // TMEM lane = query row of the tile
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int64_t jl = (int64_t)qt * 128 + row;          // local index on rank r
    const bool row_valid = jl < P.n;
    const int qpos = row_valid ? __ldg(P.posL + (int64_t)r * P.n + jl) : 0;
    // l: sum of the fp32 exponentials (for lse); lr: sum of the same values rounded to bf16 as the
    // PV product sees them (for the normalisation of O, so its weights sum to one exactly).
    float m_used = -INFINITY, l = 0.f, lr = 0.f;
    TileWalk w;
    w.init(P, r, qmm);
    int j = 0;
    bool ok = true;
    float x[128];
    const bool counter = (row == 0);                    // one thread tallies computed tiles
    int cnt_s = -1;
    unsigned long long cnt_full = 0, cnt_diag = 0;
    auto flush = [&]() {
        if (counter && cnt_s >= 0) {
            unsigned long long* c = P.counts + ((size_t)r * P.n_cp + cnt_s) * 2;
            if (cnt_full) atomicAdd(c, cnt_full);
            if (cnt_diag) atomicAdd(c + 1, cnt_diag);
        }
        cnt_full = cnt_diag = 0;
    };
    while (w.next()) {
        const int sb = j & 1;
        if (w.s != cnt_s) { flush(); cnt_s = w.s; }
        if (w.diag) ++cnt_diag; else ++cnt_full;
        ok = __all_sync(0xffffffffu, wait(bars.s_full[sb], (j >> 1) & 1, kSiteSFull));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t t[32];
            tmem_ld32(tmem + lane_base + (sb ? 128u : 0u) + c * 32, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(t[i]);
        }
        tc_fence_before();
        mbar_arrive(bars.s_free[sb]);
        if (w.mask) {
            const int64_t kbase = (int64_t)w.src * P.n + (int64_t)w.kt * 128;
            const int64_t left = P.n - (int64_t)w.kt * 128;
            const int kvalid = left < 128 ? (int)left : 128;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                bool vis = row_valid && c < kvalid;
                if (vis && P.causal) vis = __ldg(P.posL + kbase + c) <= qpos;
                if (!vis) x[c] = -INFINITY;
            }
        }
        float mx = x[0];
#pragma unroll
        for (int c = 1; c < 128; ++c) mx = fmaxf(mx, x[c]);
        const float mt = (mx == -INFINITY) ? -INFINITY : mx * P.scale_log2;
        const float m_new = fmaxf(m_used, mt);
        const bool resc = m_new > m_used + 8.0f;
        float alpha = 1.0f;
        if (resc) {
            alpha = ex2(m_used - m_new);
            l *= alpha;
            lr *= alpha;
            m_used = m_new;
        }
        const float msub = (m_used == -INFINITY) ? 0.f : m_used;
        // P is rounded to bf16 for the PV product; the row sum adds the same rounded values, so
        // the weights O / l applies are exactly the ones the tensor core multiplied.
        uint32_t pk[64];
        float rs = 0.f, rsr = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const float p0 = ex2(fmaf(x[2 * c], P.scale_log2, -msub));
            const float p1 = ex2(fmaf(x[2 * c + 1], P.scale_log2, -msub));
            pk[c] = pack_bf16(p0, p1);
            rs += p0 + p1;
            rsr += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xFFFF0000u);
        }
        l += rs;
        lr += rsr;
        if (j > 0) {   // PV of the previous tile done: the P buffer is free and O is stable
            ok = __all_sync(0xffffffffu, wait(bars.pv_done, (j - 1) & 1, kSitePvDone));
            if (!ok) break;
            tc_fence_after();
            if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t t[32];
                    const uint32_t ta = tmem + lane_base + C::O_COL + c * 32;
                    tmem_ld32(ta, t);
#pragma unroll
                    for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
                    tmem_st32(ta, t);
                }
                tmem_st_wait();
            }
        }
        // P as bf16, K-major with the 128-byte swizzle: two panels of 64 keys, row = 128 bytes.
#pragma unroll
        for (int g8 = 0; g8 < 16; ++g8) {
            const int pn = g8 >> 3, cc = g8 & 7;
            const uint32_t addr = sP + pn * C::PANEL_BYTES + row * 128 + (((cc ^ (row & 7)) & 7) << 4);
            st_shared_v4(addr, pk[4 * g8 + 0], pk[4 * g8 + 1], pk[4 * g8 + 2], pk[4 * g8 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bars.p_full);
        ++j;
    }
    flush();
    if (!ok) return;
    if (j > 0) {
        ok = __all_sync(0xffffffffu, wait(bars.pv_done, (j - 1) & 1, kSitePvDone));
        if (!ok) return;
        tc_fence_after();
    } else if (!P.fused && P.step > 0) {
        return;   // nothing visible at this step: the running state is unchanged
    }
    const float inv_l = lr > 0.f ? 1.0f / lr : 0.f;
    const float lse_v = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
    if (P.fused) {
        int64_t tn = 0;
        if (P.layout == CPATTN_CONTIGUOUS) tn = (int64_t)r * P.n + jl;
        else if (P.layout == CPATTN_ZIGZAG) tn = jl < P.m ? (int64_t)r * P.m + jl : (int64_t)(2 * P.n_cp - 1 - r) * P.m + (jl - P.m);
        else tn = jl * P.n_cp + r;
        uint4* dst = reinterpret_cast<uint4*>(P.o + (((int64_t)b * P.T + tn) * P.h + head) * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t t[32];
            if (j > 0) tmem_ld32(tmem + lane_base + C::O_COL + c * 32, t);
            else {
#pragma unroll
                for (int i = 0; i < 32; ++i) t[i] = 0u;
            }
            if (row_valid) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 v;
                    v.x = pack_bf16(__uint_as_float(t[8 * q4 + 0]) * inv_l, __uint_as_float(t[8 * q4 + 1]) * inv_l);
                    v.y = pack_bf16(__uint_as_float(t[8 * q4 + 2]) * inv_l, __uint_as_float(t[8 * q4 + 3]) * inv_l);
                    v.z = pack_bf16(__uint_as_float(t[8 * q4 + 4]) * inv_l, __uint_as_float(t[8 * q4 + 5]) * inv_l);
                    v.w = pack_bf16(__uint_as_float(t[8 * q4 + 6]) * inv_l, __uint_as_float(t[8 * q4 + 7]) * inv_l);
                    dst[c * 4 + q4] = v;
                }
            }
        }
        if (row_valid) P.lse[((int64_t)b * P.h + head) * P.T + tn] = lse_v;
    } else {
        const int64_t base = (((int64_t)r * P.B + b) * P.h + head) * P.n + jl;
        float4* orun = reinterpret_cast<float4*>(P.o_run + base * D);
        float wa = 0.f, wb = 1.f, L = lse_v;
        const bool first = (P.step == 0);
        if (row_valid && !first) {
            const float la = P.lse_run[base];
            const float M = fmaxf(la, lse_v);
            if (M == -INFINITY) { wa = 0.f; wb = 0.f; L = -INFINITY; }
            else {
                L = M + logf(expf(la - M) + expf(lse_v - M));
                wa = expf(la - L);
                wb = expf(lse_v - L);
            }
        }
        wb *= inv_l;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t t[32];
            if (j > 0) tmem_ld32(tmem + lane_base + C::O_COL + c * 32, t);
            else {
#pragma unroll
                for (int i = 0; i < 32; ++i) t[i] = 0u;
            }
            if (row_valid) {
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    float4 ob = make_float4(__uint_as_float(t[4 * q4]) * wb, __uint_as_float(t[4 * q4 + 1]) * wb,
                                            __uint_as_float(t[4 * q4 + 2]) * wb, __uint_as_float(t[4 * q4 + 3]) * wb);
                    if (!first) {
                        const float4 oa = orun[c * 8 + q4];
                        ob.x += wa * oa.x; ob.y += wa * oa.y; ob.z += wa * oa.z; ob.w += wa * oa.w;
                    }
                    orun[c * 8 + q4] = ob;
                }
            }
        }
        if (row_valid) P.lse_run[base] = L;
    }
}

template <int D>
__global__ void __launch_bounds__(192, 1)
    ring_attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const Params P) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sP = sbase + C::OFF_P;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    Bars<D> bars;
    bars.setup(sbase + C::OFF_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int bhn = P.B * P.h;
    const int rq = __ldg(P.order + blockIdx.x / bhn);
    const int r = rq / P.n_qt, qt = rq % P.n_qt;
    const int bh = blockIdx.x % bhn, b = bh / P.h, head = bh % P.h, kvh = head / P.g;
    const int2 qmm = __ldg(P.tile_mm + rq);
    // A unit that starts after another one recorded a device error does no work (the decision
    // is taken by one thread and shared, so the whole block leaves together).
    volatile int* skip_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
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
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Waiter wait{abort_flag, P.header, P.timeout_ns};

    if (warp == 0) {
        if (lane == 0) producer<D>(P, &tmQ, &tmK, &tmV, sQ, sK, sV, bars, wait, r, qt, b, head, kvh, qmm);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<D>(P, tmem, sQ, sK, sV, sP, bars, wait, r, qmm);
    } else {
        softmax_epilogue<D>(P, tmem, sP, bars, wait, r, qt, b, head, qmm);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Failure-detection self test: one thread waits on a barrier nothing will complete.
__global__ void wait_selftest_kernel(uint32_t* header, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const Waiter wait{&abort_flag, header, timeout_ns};
    wait(b, 0, kSiteSelfTest);
}

// ---- host side -------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// rows x d bf16, row-major; tiles of 128 rows x 64 columns with the 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, int d) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch_d(const AttnLaunch& a, cudaStream_t st, std::string* why) {
    using C = Cfg<D>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(ring_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return (int)e;
        attr_set = true;
    }
    CUtensorMap tq, tk, tv;
    const uint64_t qrows = (uint64_t)a.n_cp * a.B * a.h * a.n, kvrows = (uint64_t)a.n_cp * a.B * a.n_kv * a.n;
    if (!make_map(&tq, a.qL, qrows, D) || !make_map(&tk, a.kv_k, kvrows, D) || !make_map(&tv, a.kv_v, kvrows, D)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point unavailable or bad tensor shape)";
        return (int)cudaErrorInvalidValue;
    }
    Params P{};
    P.B = a.B; P.h = a.h; P.n_kv = a.n_kv; P.g = a.h / a.n_kv; P.n_cp = a.n_cp; P.n_qt = a.n_qt; P.causal = a.causal;
    P.fused = a.fused; P.step = a.step; P.kv_by_holder = a.kv_by_holder; P.layout = a.layout;
    P.n = a.n; P.m = a.m; P.T = a.T; P.scale_log2 = a.scale_log2;
    P.posL = a.posL; P.tile_mm = reinterpret_cast<const int2*>(a.tile_mm); P.order = a.order;
    P.counts = a.counts;
    P.o = static_cast<uint16_t*>(a.o); P.lse = a.lse; P.o_run = a.o_run; P.lse_run = a.lse_run;
    P.header = a.header; P.timeout_ns = a.timeout_ns;
    const int64_t units = (int64_t)a.n_cp * a.n_qt * a.B * a.h;
    ring_attention_kernel<D><<<(unsigned)units, 192, C::SMEM_BYTES, st>>>(tq, tk, tv, P);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_attention(const AttnLaunch& a, void* stream, std::string* why) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (a.d == 128) return launch_d<128>(a, st, why);
    if (a.d == 64) return launch_d<64>(a, st, why);
    *why = "unsupported head width";
    return (int)cudaErrorInvalidValue;
}

int launch_wait_selftest(uint32_t* header, uint64_t timeout_ns, void* stream) {
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(header, timeout_ns);
    return (int)cudaGetLastError();
}

}  // namespace cpattn
