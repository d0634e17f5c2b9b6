// attention.cu -- the ring-step attention kernel for sm_103a.
//
// A persistent kernel. Each CTA repeatedly takes a work unit from a global counter, in the
// longest-first order the plan computed. A unit is two 128-row query tiles on one virtual rank r
// that share every key/value tile: two heads of one KV group (the group size is even), or two
// adjacent query tiles of one head (otherwise). The unit walks the key/value blocks in ring order
// ("Context and expert parallelism", "Pass them around a ring": at step s rank r holds the block
// of rank (r - s) mod n_cp). It skips key tiles no query of the unit can see and masks the partly
// visible ones ("The causal mask unbalances the sequence"). With document masks for packed
// sequences ("What context parallelism communicates") every query also has a lowest visible key
// position; a key is visible iff lo[t] <= pos[u] <= pos[t]. With document ids (the same section:
// "arbitrary masks, such as document masks for packed sequences") a key is visible iff it has the
// query's id (and, causally, pos[u] <= pos[t]); documents need not be contiguous, and a small kernel
// records per row group and ring step a bitmask of the key tiles some query can see, which the
// walkers follow. It keeps the online-softmax state of
// the paragraph after the ring one on chip across every step: running max, running sum of
// exponentials, running weighted sum of values, rescaled when a larger score arrives.
//
// Warp roles (384 threads; registers move from warpgroup 0 to the softmax warpgroups with
// setmaxnreg: 128 x 112 + 256 x 192 <= the 384 x 168 the block is launched with, checked on the
// host before the first launch):
//   warp 0      scheduler + TMA producer: the next unit index into a 2-slot ring; both Q tiles
//               once per unit; K and V tiles through an NS-deep stage ring, V one tile behind K.
//   warp 1      owns tensor memory; one lane issues tcgen05.mma. S_i = Q_i K^T (SS form), then
//               O_i += P_i V with P_i read from tensor memory (TS form). It takes the number of
//               key tiles of each unit from a table a small kernel writes before the launch, so
//               no table lookup of the key walk sits between two of its MMA groups.
//   warps 2, 3  idle, except in a ring step with the hop in the kernel: they copy every rank's
//               K and V block into the next rank's slot of the stage while the attention runs.
//   warps 4..7  softmax warpgroup 0 (query tile 0), one thread per row.
//   warps 8..11 softmax warpgroup 1 (query tile 1). Each thread reads its row of S from TMEM,
//               masks, takes the max, exponentiates with exp2, sums, writes P (fp16) back over
//               S in TMEM, rescales O lazily, and writes the unit's output.
// Tensor memory (512 columns): S0 at 0, S1 at 128 (P_i packed fp16x2 over the first 64 columns
// of S_i), O0 at 256, O1 at 256 + d_k.
//
// MMAs from the issuing thread execute in order. So QK_i of the next tile, which overwrites
// S_i / P_i, is issued only after PV_i of this tile, which reads P_i.
//
// One ring step (instead of every step at once) merges each unit's output into a running state
// in HBM: O unnormalised against a running maximum, with its sum (the online softmax carried
// across launches; the finalize kernel divides). Those launches take 32 KB more shared memory,
// through which the epilogue's stores and reductions move whole row segments.
//
// Rescaling is lazy: a row keeps a stale maximum until a tile raises it by more than 8 (log2
// units). P then stays below 2^8 and the final O / l is unchanged. Every wait is bounded by a
// global-timer limit. On expiry the kernel records the wait site in the workspace header, every
// role leaves its loop, the kernel waits for its own copies and MMAs, and frees tensor memory.
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
// Registers per thread of warps 0..3 (producer, MMA issue) and of the softmax warpgroups after
// setmaxnreg: 120 / 184 (128 * 120 + 256 * 184 = 62464 <= 384 * 168); the document-mask walk
// keeps 192 in the softmax warps (112 / 192, 63488), where 184 spills more. Measured: 120 / 184
// is 0.4 % faster than 112 / 192 on the plain kernel, 128 / 176 and 104 / 200 are slower.
// Mask modes of the kernel: causal (or none) from positions alone; a per-query lower bound on the
// key positions; document ids.
enum MaskMode : int { kMaskPos = 0, kMaskLower = 1, kMaskDoc = 2 };

template <int M>
struct RegSplit {
    static constexpr int low = M != kMaskPos ? 112 : 120, high = M != kMaskPos ? 192 : 184;
};

struct Params {
    int B, h, n_kv, g, n_cp, n_qt, n_grp, pair_heads, causal, fused, step, kv_by_holder, layout;
    int num_units;
    int64_t n, m, T;
    float scale_log2;
    const int32_t* posL;
    const int4* tile_mm;
    const int32_t* kposL;   // key-side positions [.][n] and tiles [.][n_qt], indexed by the rank whose
    const int4* ktile_mm;   // block is read (posL / tile_mm except in a multi-process ring)
    const int32_t* order;
    const int32_t* loL;    // [n_cp][n] lowest visible key position per query, or NULL
    const int4* tile_lo;   // [n_cp][n_qt] (min, max) of loL over a query tile, or NULL
    int32_t* unit_tiles;   // [n_cp * n_grp]: key tiles of a unit of row group r * n_grp + group
    // document masks only, written by unit_tiles_kernel: per row group and ring step, the key
    // tiles its walk visits lie in [begin, end) (begin | end << 16), and a bit per non-empty step
    int32_t* walk_tab;               // [n_cp * n_grp][n_cp]
    unsigned long long* walk_nz;     // [n_cp * n_grp], for n_cp <= 64
    // document ids only, written by unit_tiles_kernel: per row group and ring step, a bit per key
    // tile that some query of the row group may see ([n_cp * n_grp][n_cp][words], 64 tiles a word)
    unsigned long long* walk_bits;
    int words;                       // ceil(n_qt / 64)
    unsigned long long* counts;
    uint32_t* sched;
    uint16_t* o;
    float* lse;
    float* o_run;
    float* lse_run;         // ring step: running maximum m_run (log2 units)
    float* l_run;           // ring step: running sum l_run
    uint32_t* header;
    uint64_t timeout_ns;
    int first;              // ring step: write the running state instead of merging into it
    int64_t kv_rank_rows;   // all-gather: K/V rows between consecutive ranks' gathered copies (else 0)
    // ring step with the hop in this kernel: each rank's key/value block moves into the next
    // rank's slot (rank-major blocks of hop_blk 16-byte words; hop_words per tensor, 0: no hop)
    const uint4* hop_src_k;
    const uint4* hop_src_v;
    uint4* hop_dst_k;
    uint4* hop_dst_v;
    int64_t hop_words, hop_blk;
    int hop_wrap;           // the last rank's block wraps to rank 0 (else rank 0's is left alone)
};

template <int D>
struct Cfg {
    static constexpr int NS = (D == 128) ? 2 : 4;         // K/V stage depth
    static constexpr int PANELS = D / 64;                 // 64-column (128-byte) swizzle panels
    static constexpr int PANEL_BYTES = 128 * 128;         // 128 rows x 128 bytes
    static constexpr int Q_BYTES = 128 * D * 2;           // one query tile
    static constexpr int KV_BYTES = 128 * D * 2;          // one key (or value) tile
    static constexpr int OFF_Q = 0;                       // two query tiles
    static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + NS * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + NS * KV_BYTES;
    static constexpr int NBAR = 15 + 4 * NS;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 32 + 1024;
    // Ring steps only (launched with SMEM_BYTES_RING; the other launches keep that shared memory as
    // L1): each softmax warp's 32 rows x 128 bytes, through which the epilogue's stores and
    // reductions into the running output move whole row segments.
    static constexpr int STG_WARP_BYTES = 32 * 128;
    static constexpr int OFF_STG = (OFF_MISC + 32 + 127) & ~127;
    static constexpr int SMEM_BYTES_RING = OFF_STG + 8 * STG_WARP_BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL0 = 256, O_COL1 = 256 + D;
};

// Barrier addresses are computed from the base on use (fixed offsets), so no role keeps a
// register per barrier.
template <int D>
struct Bars {
    static constexpr int NS = Cfg<D>::NS;
    uint32_t base;
    __device__ uint32_t at(int i) const { return base + 8u * (uint32_t)i; }
    __device__ uint32_t unit_full(int s) const { return at(s); }
    __device__ uint32_t unit_empty(int s) const { return at(2 + s); }
    __device__ uint32_t q_full() const { return at(4); }
    __device__ uint32_t q_empty() const { return at(5); }
    __device__ uint32_t k_full(int st) const { return at(6 + st); }
    __device__ uint32_t v_full(int st) const { return at(6 + NS + st); }
    __device__ uint32_t k_empty(int st) const { return at(6 + 2 * NS + st); }
    __device__ uint32_t v_empty(int st) const { return at(6 + 3 * NS + st); }
    __device__ uint32_t s_full(int i) const { return at(6 + 4 * NS + i); }
    __device__ uint32_t p_full(int i) const { return at(8 + 4 * NS + i); }
    __device__ uint32_t pv_done(int i) const { return at(10 + 4 * NS + i); }
    __device__ uint32_t o_free(int i) const { return at(12 + 4 * NS + i); }
    __device__ uint32_t mma_done() const { return at(14 + 4 * NS); }
    static constexpr int kCount = 15 + 4 * NS;
    __device__ void init() const {
        for (int i = 0; i < 2; ++i) {
            mbar_init(unit_full(i), 1);
            mbar_init(unit_empty(i), 1 + 8);          // the MMA lane and one lane per softmax warp
            mbar_init(s_full(i), 1);
            mbar_init(p_full(i), 4);                  // one lane per softmax warp
            mbar_init(pv_done(i), 1);
            mbar_init(o_free(i), 4);
        }
        mbar_init(q_full(), 1);
        mbar_init(q_empty(), 1);
        for (int i = 0; i < NS; ++i) {
            mbar_init(k_full(i), 1); mbar_init(v_full(i), 1);
            mbar_init(k_empty(i), 1); mbar_init(v_empty(i), 1);
        }
        mbar_init(mma_done(), 1);
    }
};
static_assert(Bars<64>::kCount == Cfg<64>::NBAR && Bars<128>::kCount == Cfg<128>::NBAR,
              "the shared-memory barrier region holds every barrier");

enum Site : int { kSiteQ = 1, kSiteKFull, kSiteVFull, kSiteKEmpty, kSiteVEmpty, kSiteSFull, kSiteQEmpty,
                  kSitePFull, kSitePvDone, kSiteDrain, kSiteSelfTest, kSiteUnitFull, kSiteUnitEmpty, kSiteOFree };

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

// One work unit: rank r, batch element b, and two query tiles (head_i, qt_i) sharing KV head kvh.
struct Unit {
    int r, b, kvh, rg;   // rank, batch element, KV head, row group r * n_grp + group
    int head[2], qt[2], valid[2];
    int2 qmm[2];   // position range of each query tile; (INT_MAX, INT_MIN) for a missing tile
    int2 qlo[2];   // range of the tile's lowest visible key positions (document ids: range of its ids);
                   // (INT_MIN, INT_MIN) without one
    unsigned long long qbits[2];   // document ids: a bit per id modulo 64 in the tile; 0 without one
};

// The query tiles' position ranges and (with a per-query lower bound or document ids) the range of
// the bounds or ids.
template <int M>
__device__ __forceinline__ void unit_ranges(const Params& P, Unit& U) {
    for (int i = 0; i < 2; ++i) {
        if (U.valid[i]) {
            const int4 t4 = __ldg(P.tile_mm + U.r * P.n_qt + U.qt[i]);
            U.qmm[i] = make_int2(t4.x, t4.y);
            if (M != kMaskPos) {
                const int4 l4 = __ldg(P.tile_lo + U.r * P.n_qt + U.qt[i]);
                U.qlo[i] = make_int2(l4.x, l4.y);
                U.qbits[i] = (unsigned long long)(unsigned)l4.z | ((unsigned long long)(unsigned)l4.w << 32);
            } else {
                U.qlo[i] = make_int2(INT_MIN, INT_MIN);
                U.qbits[i] = 0ull;
            }
        } else {
            U.qmm[i] = make_int2(INT_MAX, INT_MIN);
            U.qlo[i] = make_int2(INT_MIN, INT_MIN);
            U.qbits[i] = 0ull;
        }
    }
}

// Units are numbered KV-head-major: all units of one (batch element, KV head) come before the
// next, so the CTAs running at any moment read the keys and values of one or two KV heads and
// those stay in L2. Within a KV head, (rank, row group) follow the plan's longest-first order,
// then the query heads of the group.
template <int M>
__device__ __forceinline__ Unit decode_unit(const Params& P, int u) {
    Unit U;
    const int per = P.pair_heads ? P.g / 2 : P.g;        // units per (b, kvh, row group)
    const int n_rg = P.n_cp * P.n_grp;
    const int pp = u % per;
    const int t = u / per;
    const int rgi = t % n_rg;
    const int bk = t / n_rg;
    U.kvh = bk % P.n_kv;
    U.b = bk / P.n_kv;
    const int rg = __ldg(P.order + rgi);
    U.rg = rg;
    U.r = rg / P.n_grp;
    const int grp = rg % P.n_grp;
    if (P.pair_heads) {
        U.head[0] = U.kvh * P.g + 2 * pp;
        U.head[1] = U.head[0] + 1;
        U.qt[0] = U.qt[1] = grp;
        U.valid[0] = U.valid[1] = 1;
    } else {
        U.head[0] = U.head[1] = U.kvh * P.g + pp;
        U.qt[0] = 2 * grp;
        U.qt[1] = 2 * grp + 1;
        U.valid[0] = 1;
        U.valid[1] = U.qt[1] < P.n_qt;
    }
    unit_ranges<M>(P, U);
    return U;
}

// Block class of a key tile for one query tile under document ids: SKIP when no id can be shared (the
// id ranges are disjoint, or no id modulo 64 is in both tiles) or (causal) every key follows every
// query; FULL when both tiles hold one id, the same, and every key precedes every query; otherwise
// partly visible (the element mask decides).
__device__ __forceinline__ int doc_class(int causal, int qmin, int qmax, int dqmin, int dqmax,
                                         unsigned long long qbits, const int4& t4, const int4& d4) {
    if (d4.y < dqmin || d4.x > dqmax) return CPATTN_TILE_SKIP;
    const unsigned long long kbits = (unsigned long long)(unsigned)d4.z | ((unsigned long long)(unsigned)d4.w << 32);
    if ((qbits & kbits) == 0ull) return CPATTN_TILE_SKIP;
    const int pc = !causal ? CPATTN_TILE_FULL : (t4.x > qmax) ? CPATTN_TILE_SKIP
                                              : (t4.y > qmin) ? CPATTN_TILE_DIAG : CPATTN_TILE_FULL;
    if (pc == CPATTN_TILE_SKIP) return CPATTN_TILE_SKIP;
    const bool one_id = dqmin == dqmax && d4.x == d4.y && d4.x == dqmin;
    return (pc == CPATTN_TILE_FULL && one_id) ? CPATTN_TILE_FULL : CPATTN_TILE_DIAG;
}

// The key tiles a unit visits, in ring order, leaving out tiles that both query tiles skip.
// cls(i): FULL / DIAG / SKIP for query tile i; mask(i): the tile needs the element mask for
// query tile i (partly visible, skipped by this tile only, or shorter than 128 keys). A block
// whose remaining tiles all start after every query of the unit is left in one step. LB: the
// queries also have a lowest visible key position (document masks). DOC: document ids; the walk
// follows the per-step bitmask of visited key tiles.
template <int M>
struct TileWalk {
    static constexpr bool LB = M == kMaskLower, DOC = M == kMaskDoc;
    const Params* p;
    int r, s, s_end, kt, src;
    int qmin0, qmax0, qmin1, qmax1, qmax, cls0, cls1, mask0, mask1;
    int lmin0, lmax0, lmin1, lmax1;   // lower-bound ranges of the two query tiles
    unsigned long long qbits0, qbits1;   // document ids: the query tiles' id-bit masks
    __device__ int cls(int i) const { return i ? cls1 : cls0; }
    __device__ int mask(int i) const { return i ? mask1 : mask0; }
    __device__ void init(const Params& P, const Unit& U) {
        p = &P;
        r = U.r;
        qmin0 = U.qmm[0].x; qmax0 = U.qmm[0].y;
        qmin1 = U.qmm[1].x; qmax1 = U.qmm[1].y;
        lmin0 = U.qlo[0].x; lmax0 = U.qlo[0].y;
        lmin1 = U.qlo[1].x; lmax1 = U.qlo[1].y;
        qbits0 = U.qbits[0]; qbits1 = U.qbits[1];
        qmax = max(qmax0, qmax1);
        s = P.fused ? 0 : P.step;
        s_end = P.fused ? P.n_cp : P.step + 1;
        kt = -1;
        rg = U.rg;
        if (LB && P.causal) {
            // the table walk starts before its first step: kt >= kend moves to the next one
            s -= 1;
            kt = kend = 0;
            nz = P.n_cp <= 64 ? __ldg(P.walk_nz + rg) : 0ull;
            if (!P.fused && P.n_cp <= 64) nz &= 1ull << P.step;   // one step: only its own bit
        }
        if (DOC) {
            // the bitmask walk starts on the last word before its first step
            s -= 1;
            wi = P.words - 1;
            bits = 0ull;
        }
    }
    int wi;
    unsigned long long bits;
    // Document ids: the next set bit of the row group's bitmask, step by step.
    __device__ bool next_bits() {
        const Params& P = *p;
        for (;;) {
            while (bits == 0ull) {
                if (++wi >= P.words) {
                    wi = 0;
                    if (++s >= s_end) return false;
                }
                bits = __ldg(P.walk_bits + ((int64_t)rg * P.n_cp + s) * P.words + wi);
            }
            kt = wi * 64 + (__ffsll((long long)bits) - 1);
            bits &= bits - 1ull;
            src = r - s;
            if (src < 0) src += P.n_cp;
            const int short_tile = (kt == P.n_qt - 1) && (P.n % 128) != 0;
            const int4 t4 = __ldg(P.ktile_mm + src * P.n_qt + kt);
            const int4 d4 = __ldg(P.tile_lo + src * P.n_qt + kt);
            cls0 = doc_class(P.causal, qmin0, qmax0, lmin0, lmax0, qbits0, t4, d4);
            cls1 = doc_class(P.causal, qmin1, qmax1, lmin1, lmax1, qbits1, t4, d4);
            if (cls0 == CPATTN_TILE_SKIP && cls1 == CPATTN_TILE_SKIP) continue;
            mask0 = (cls0 != CPATTN_TILE_FULL) || short_tile;
            mask1 = (cls1 != CPATTN_TILE_FULL) || short_tile;
            return true;
        }
    }
    // Document masks: the walk of a row group is the same for all its units, and the kernel
    // before this one recorded it per step as a key-tile range (next_scan below): jump from one
    // non-empty step to the next with one table load, instead of a chain of dependent loads
    // (a running-maximum test and a binary search) per step.
    int rg, kend;
    unsigned long long nz;
    __device__ bool next() {
        if (DOC) return next_bits();
        if (!LB || !p->causal) return next_scan();
        const Params& P = *p;
        for (;;) {
            if (++kt >= kend) {
                int sn = s + 1;
                if (P.n_cp <= 64) {
                    const unsigned long long rest = sn < 64 ? (nz >> sn) : 0ull;
                    if (rest == 0ull) return false;
                    sn += __ffsll((long long)rest) - 1;
                }
                if (sn >= s_end) return false;
                s = sn;
                const int e = __ldg(P.walk_tab + (int64_t)rg * P.n_cp + s);
                kt = e & 0xFFFF;
                kend = e >> 16;
                if (kt >= kend) { kt = kend; continue; }   // (n_cp > 64: empty steps are visited)
                src = r - s;
                if (src < 0) src += P.n_cp;
            }
            const int short_tile = (kt == P.n_qt - 1) && (P.n % 128) != 0;
            const int4 t4 = __ldg(P.ktile_mm + src * P.n_qt + kt);
            cls0 = (t4.x > qmax0 || t4.y < lmin0) ? CPATTN_TILE_SKIP
                   : (t4.y > qmin0 || t4.x < lmax0) ? CPATTN_TILE_DIAG : CPATTN_TILE_FULL;
            cls1 = (t4.x > qmax1 || t4.y < lmin1) ? CPATTN_TILE_SKIP
                   : (t4.y > qmin1 || t4.x < lmax1) ? CPATTN_TILE_DIAG : CPATTN_TILE_FULL;
            if (cls0 == CPATTN_TILE_SKIP && cls1 == CPATTN_TILE_SKIP) continue;
            mask0 = (cls0 != CPATTN_TILE_FULL) || short_tile;
            mask1 = (cls1 != CPATTN_TILE_FULL) || short_tile;
            return true;
        }
    }
    // The walk from the position tables alone (every step, every layout and mask).
    __device__ bool next_scan() {
        const Params& P = *p;
        for (;;) {
            if (++kt >= P.n_qt) {
                kt = 0;
                if (++s >= s_end) return false;
            }
            src = r - s;
            if (src < 0) src += P.n_cp;
            if (LB && kt == 0 && P.causal) {
                // Entering a block: its tiles below every query's lower bound come first in the
                // non-decreasing running maximum (.w); skip the block, or start at its first tile
                // whose running maximum reaches the smallest bound.
                const int lmin = min(lmin0, lmin1);
                const int* mm = reinterpret_cast<const int*>(P.ktile_mm + src * P.n_qt);
                if (__ldg(mm + 4 * (P.n_qt - 1) + 3) < lmin) {
                    kt = P.n_qt - 1;
                    continue;
                }
                int lo = 0, hi = P.n_qt - 1;              // first kt with running max >= lmin
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (__ldg(mm + 4 * mid + 3) < lmin) lo = mid + 1;
                    else hi = mid;
                }
                kt = lo;
            }
            const int short_tile = (kt == P.n_qt - 1) && (P.n % 128) != 0;
            if (!P.causal) {
                cls0 = cls1 = CPATTN_TILE_FULL;
                mask0 = mask1 = short_tile;
                return true;
            }
            const int4 t4 = __ldg(P.ktile_mm + src * P.n_qt + kt);
            if (t4.z > qmax) {           // this tile and every later one of the block: skipped
                kt = P.n_qt - 1;
                continue;
            }
            if (LB) {
                // SKIP: every key after every query, or below every query's lower bound; FULL: every
                // key at or before every query and at or above every lower bound
                cls0 = (t4.x > qmax0 || t4.y < lmin0) ? CPATTN_TILE_SKIP
                       : (t4.y > qmin0 || t4.x < lmax0) ? CPATTN_TILE_DIAG : CPATTN_TILE_FULL;
                cls1 = (t4.x > qmax1 || t4.y < lmin1) ? CPATTN_TILE_SKIP
                       : (t4.y > qmin1 || t4.x < lmax1) ? CPATTN_TILE_DIAG : CPATTN_TILE_FULL;
            } else {
                cls0 = (t4.x > qmax0) ? CPATTN_TILE_SKIP : (t4.y > qmin0) ? CPATTN_TILE_DIAG : CPATTN_TILE_FULL;
                cls1 = (t4.x > qmax1) ? CPATTN_TILE_SKIP : (t4.y > qmin1) ? CPATTN_TILE_DIAG : CPATTN_TILE_FULL;
            }
            if (cls0 == CPATTN_TILE_SKIP && cls1 == CPATTN_TILE_SKIP) continue;
            mask0 = (cls0 != CPATTN_TILE_FULL) || short_tile;
            mask1 = (cls1 != CPATTN_TILE_FULL) || short_tile;
            return true;
        }
    }
};

// ---------------------------------------------------------------------------------------------
// warp 0: scheduler and TMA producer
// ---------------------------------------------------------------------------------------------
template <int D, int M>
__device__ void producer(const Params& P, const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                         uint32_t sQ, uint32_t sK, uint32_t sV, volatile int* unit_slot, const Bars<D>& bars,
                         const Waiter& wait) {
    using C = Cfg<D>;
    int nk = 0, nv = 0, nq = 0;   // K tiles, V tiles, Q pairs issued by this CTA
    bool ok = true;
    // Q tiles are read once per unit; the K/V tiles of one KV head are re-read by every unit in
    // flight, so they are the lines L2 should keep.
    const uint64_t pol_q = l2_evict_first(), pol_kv = l2_evict_last();
    auto load_v = [&](int row) -> bool {
        const int st = nv % C::NS;
        if (nv >= C::NS && !wait(bars.v_empty(st), ((nv / C::NS) - 1) & 1, kSiteVEmpty)) return false;
        mbar_arrive_expect_tx(bars.v_full(st), C::KV_BYTES);
        for (int pn = 0; pn < C::PANELS; ++pn)
            tma_load_2d_hint(sV + st * C::KV_BYTES + pn * C::PANEL_BYTES, tmV, bars.v_full(st), pn * 64, row, pol_kv);
        ++nv;
        return true;
    };
    for (int it = 0; ok; ++it) {
        const int slot = it & 1;
        const int u = (int)atomicAdd(P.sched, 1u);
        if (it >= 2 && !wait(bars.unit_empty(slot), ((it >> 1) - 1) & 1, kSiteUnitEmpty)) { ok = false; break; }
        unit_slot[slot] = (u < P.num_units) ? u : -1;
        mbar_arrive(bars.unit_full(slot));
        if (u >= P.num_units) break;
        const Unit U = decode_unit<M>(P, u);
        TileWalk<M> w;
        w.init(P, U);
        int j = 0, prev_row = 0;
        while (w.next()) {
            const int holder = P.kv_by_holder ? U.r : w.src;
            const int krow = (int)((int64_t)U.r * P.kv_rank_rows +
                                   (((int64_t)holder * P.B + U.b) * P.n_kv + U.kvh) * P.n + (int64_t)w.kt * 128);
            if (j == 0) {
                if (nq >= 1 && !wait(bars.q_empty(), (nq - 1) & 1, kSiteQEmpty)) { ok = false; break; }
                mbar_arrive_expect_tx(bars.q_full(), 2 * C::Q_BYTES);
                for (int i = 0; i < 2; ++i) {
                    const int qrow = (int)((((int64_t)U.r * P.B + U.b) * P.h + U.head[i]) * P.n + (int64_t)U.qt[i] * 128);
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_2d_hint(sQ + i * C::Q_BYTES + pn * C::PANEL_BYTES, tmQ, bars.q_full(), pn * 64, qrow,
                                         pol_q);
                }
                ++nq;
            }
            const int st = nk % C::NS;
            if (nk >= C::NS && !wait(bars.k_empty(st), ((nk / C::NS) - 1) & 1, kSiteKEmpty)) { ok = false; break; }
            mbar_arrive_expect_tx(bars.k_full(st), C::KV_BYTES);
            for (int pn = 0; pn < C::PANELS; ++pn)
                tma_load_2d_hint(sK + st * C::KV_BYTES + pn * C::PANEL_BYTES, tmK, bars.k_full(st), pn * 64, krow, pol_kv);
            ++nk;
            if (j >= 1 && !load_v(prev_row)) { ok = false; break; }     // V runs one tile behind K
            prev_row = krow;
            ++j;
        }
        if (ok && j >= 1) ok = load_v(prev_row);
    }
    if (ok) {
        // The tensor core's last arrivals on the stage barriers have landed before the CTA exits.
        for (int i = (nk > C::NS ? nk - C::NS : 0); i < nk; ++i) wait(bars.k_empty(i % C::NS), (i / C::NS) & 1, kSiteKEmpty);
        for (int i = (nv > C::NS ? nv - C::NS : 0); i < nv; ++i) wait(bars.v_empty(i % C::NS), (i / C::NS) & 1, kSiteVEmpty);
        if (nq >= 1) wait(bars.q_empty(), (nq - 1) & 1, kSiteQEmpty);
    } else {
        // Aborted: still wait (bounded) until our own copies in flight have landed.
        if (nq >= 1) wait(bars.q_full(), (nq - 1) & 1, kSiteQ, false);
        for (int i = (nk > C::NS ? nk - C::NS : 0); i < nk; ++i) wait(bars.k_full(i % C::NS), (i / C::NS) & 1, kSiteKFull, false);
        for (int i = (nv > C::NS ? nv - C::NS : 0); i < nv; ++i) wait(bars.v_full(i % C::NS), (i / C::NS) & 1, kSiteVFull, false);
    }
}

// ---------------------------------------------------------------------------------------------
// warp 1, lane 0: MMA issue
// ---------------------------------------------------------------------------------------------
template <int D>
__device__ void mma_issuer(const Params& P, uint32_t tmem, uint32_t sQ, uint32_t sK, uint32_t sV,
                           volatile int* unit_slot, const Bars<D>& bars, const Waiter& wait) {
    using C = Cfg<D>;
    constexpr uint32_t kIdescQK = idesc_bf16(128, 128, 0, 0);   // A = Q (K-major), B = K (K-major)
    constexpr uint32_t kIdescPV = idesc_f16(128, D, 0, 1);      // A = P (TMEM, fp16), B = V (MN-major, fp16)
    int nk = 0, nv = 0, nq = 0, npv = 0, nunits = 0;   // K, V, Q consumed; PV tiles; units with tiles
    bool ok = true;
    auto issue_qk = [&](int i, int kst) {
        const uint32_t qb = sQ + i * C::Q_BYTES, kb = sK + kst * C::KV_BYTES;
        const uint32_t d = tmem + (i ? C::S_COL1 : C::S_COL0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::PANEL_BYTES + (kk & 3) * 32;
            mma_bf16_ss(d, desc_sw128(qb + off, 16, 1024), desc_sw128(kb + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(bars.s_full(i));
    };
    auto issue_pv = [&](int i, int vst, bool first) {
        const uint32_t vb = sV + vst * C::KV_BYTES;
        const uint32_t d = tmem + (i ? C::O_COL1 : C::O_COL0), a = tmem + (i ? C::S_COL1 : C::S_COL0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)       // 128 keys, 16 per MMA; P_i packs 2 keys per column
            mma_bf16_ts(d, a + kk * 8, desc_sw128(vb + kk * 2048, C::PANEL_BYTES, 1024), kIdescPV,
                        (!first || kk > 0) ? 1u : 0u);
        mma_commit(bars.pv_done(i));
    };
    for (int it = 0; ok; ++it) {
        const int slot = it & 1;
        if (!wait(bars.unit_full(slot), (it >> 1) & 1, kSiteUnitFull)) { ok = false; break; }
        const int u = unit_slot[slot];
        mbar_arrive(bars.unit_empty(slot));
        if (u < 0) break;
        const Unit U = decode_unit<false>(P, u);
        const int n_tiles = __ldg(P.unit_tiles + U.rg);
        if (n_tiles == 0) continue;                    // nothing visible for this unit
        if (!wait(bars.q_full(), nq & 1, kSiteQ)) { ok = false; break; }
        int kst = nk % C::NS;
        if (!wait(bars.k_full(kst), (nk / C::NS) & 1, kSiteKFull)) { ok = false; break; }
        tc_fence_after();
        issue_qk(0, kst);
        issue_qk(1, kst);
        mma_commit(bars.k_empty(kst));
        ++nk;
        for (int j = 0; ok; ++j) {
            const bool nxt = j + 1 < n_tiles;
            const int vst = nv % C::NS;
            // query tile 0: PV_0(j), then QK_0(j+1)
            if (!wait(bars.p_full(0), npv & 1, kSitePFull)) { ok = false; break; }
            if (j == 0 && nunits >= 1 && !wait(bars.o_free(0), (nunits - 1) & 1, kSiteOFree)) { ok = false; break; }
            if (!wait(bars.v_full(vst), (nv / C::NS) & 1, kSiteVFull)) { ok = false; break; }
            tc_fence_after();
            issue_pv(0, vst, j == 0);
            if (nxt) {
                kst = nk % C::NS;
                if (!wait(bars.k_full(kst), (nk / C::NS) & 1, kSiteKFull)) { ok = false; break; }
                tc_fence_after();
                issue_qk(0, kst);
            }
            // query tile 1: PV_1(j), then QK_1(j+1)
            if (!wait(bars.p_full(1), npv & 1, kSitePFull)) { ok = false; break; }
            if (j == 0 && nunits >= 1 && !wait(bars.o_free(1), (nunits - 1) & 1, kSiteOFree)) { ok = false; break; }
            tc_fence_after();
            issue_pv(1, vst, j == 0);
            mma_commit(bars.v_empty(vst));
            ++nv;
            if (nxt) {
                issue_qk(1, kst);
                mma_commit(bars.k_empty(kst));
                ++nk;
            }
            ++npv;
            if (!nxt) break;
        }
        if (!ok) break;
        mma_commit(bars.q_empty());        // every QK of this unit has been issued
        ++nq;
        ++nunits;
    }
    // Drain: every MMA this thread issued has completed before tensor memory is freed.
    mma_commit(bars.mma_done());
    wait(bars.mma_done(), 0, kSiteDrain, false);
}

// ---------------------------------------------------------------------------------------------
// warps 2..3 of a ring step (otherwise idle): the hop to the next step ("Pass them around a ring":
// send right, receive left). Word w of a tensor's rank-major blocks moves to w + hop_blk, the
// last rank's block wrapping to rank 0 (or, in a process holding only part of the ring, left
// for the transport that brings the previous process's block). The CTAs split the two tensors' words evenly; the 64
// threads of a CTA take consecutive words (coalesced), four loads in flight per thread. The
// source is read-only in this launch and the destination slot is read only by the next step.
// ---------------------------------------------------------------------------------------------
__device__ void ring_hop_copy(const Params& P, int t) {
    const int64_t total = 2 * P.hop_words;
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    const int64_t beg = (int64_t)blockIdx.x * per;
    const int64_t end = beg + per < total ? beg + per : total;
    const uint64_t pol = l2_evict_first();       // the next step reads the slot long after this one
    for (int64_t w0 = beg + t; w0 < end; w0 += 4 * 64) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t w = w0 + u * 64;
            if (w < end) {
                const bool isv = w >= P.hop_words;
                v[u] = __ldg((isv ? P.hop_src_v : P.hop_src_k) + (isv ? w - P.hop_words : w));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t w = w0 + u * 64;
            if (w < end) {
                const bool isv = w >= P.hop_words;
                int64_t o = (isv ? w - P.hop_words : w) + P.hop_blk;
                const bool wraps = o >= P.hop_words;
                if (wraps) o -= P.hop_words;
                if (!wraps || P.hop_wrap) st_global_v4_hint((isv ? P.hop_dst_v : P.hop_dst_k) + o, v[u], pol);
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// warps 4..11: softmax and epilogue, warpgroup i for query tile i, one thread per row
// ---------------------------------------------------------------------------------------------
template <int D, int M>
__device__ void softmax_epilogue(const Params& P, uint32_t tmem, volatile int* unit_slot, const Bars<D>& bars,
                                 const Waiter& wait, uint32_t stg) {
    using C = Cfg<D>;
    const int wg = (threadIdx.x >> 5) >= 8 ? 1 : 0;
    const int quarter = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
    const int row = quarter * 32 + lane;                        // TMEM lane = query row of the tile
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_col = wg ? C::S_COL1 : C::S_COL0, o_col = wg ? C::O_COL1 : C::O_COL0;
    const uint64_t scale2 = f2_pack(P.scale_log2, P.scale_log2);
    const uint64_t pol_o = l2_evict_first();          // O rows are written once: keep K/V in L2 instead
    int ntile = 0;   // tiles processed by this warpgroup
    bool ok = true;
    for (int it = 0; ok; ++it) {
        const int slot = it & 1;
        ok = __all_sync(0xffffffffu, wait(bars.unit_full(slot), (it >> 1) & 1, kSiteUnitFull));
        if (!ok) break;
        const int u = unit_slot[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.unit_empty(slot));
        if (u < 0) break;
        constexpr bool LB = M == kMaskLower, DOC = M == kMaskDoc;
        const Unit U = decode_unit<M>(P, u);
        const int head = wg ? U.head[1] : U.head[0];
        const int qt = wg ? U.qt[1] : U.qt[0];
        const int member_valid = wg ? U.valid[1] : U.valid[0];
        const int64_t jl = (int64_t)qt * 128 + row;             // local index on rank r
        const bool row_valid = member_valid && jl < P.n;
        const int qpos = row_valid ? __ldg(P.posL + (int64_t)U.r * P.n + jl) : 0;
        // the query's lowest visible key position, or its document id
        const int qlo = ((LB || DOC) && row_valid) ? __ldg(P.loL + (int64_t)U.r * P.n + jl) : INT_MIN;
        // l: sum of the fp32 exponentials (for lse and the normaliser of O)
        float m_used = -INFINITY, l = 0.f;
        const bool counter = (row == 0) && member_valid;       // one thread tallies computed tiles
        int cnt_s = -1;
        unsigned long long cnt_full = 0, cnt_diag = 0;
        auto flush = [&]() {
            if (counter && cnt_s >= 0) {
                unsigned long long* c = P.counts + ((size_t)U.r * P.n_cp + cnt_s) * 2;
                if (cnt_full) atomicAdd(c, cnt_full);
                if (cnt_diag) atomicAdd(c + 1, cnt_diag);
            }
            cnt_full = cnt_diag = 0;
        };
        TileWalk<M> w;
        w.init(P, U);
        int j = 0;
        bool have = w.next();
        while (have) {
            // This tile's walk state; the walk moves on to the next tile right away so its table
            // load overlaps the work below.
            const int cls = w.cls(wg), tmask = w.mask(wg), tsrc = w.src, tkt = w.kt;
            if (w.s != cnt_s) { flush(); cnt_s = w.s; }
            if (cls == CPATTN_TILE_DIAG) ++cnt_diag;
            else if (cls == CPATTN_TILE_FULL) ++cnt_full;
            have = w.next();
            ok = __all_sync(0xffffffffu, wait(bars.s_full(wg), ntile & 1, kSiteSFull));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld128(tmem + lane_base + s_col, sr);
            float x[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c]);
            if (tmask) {
                const int64_t kbase = (int64_t)tsrc * P.n + (int64_t)tkt * 128;
                const int64_t left = P.n - (int64_t)tkt * 128;
                const int kvalid = (cls == CPATTN_TILE_SKIP) ? 0 : (left < 128 ? (int)left : 128);
                // 16 keys at a time; the empty asm keeps the position loads of later chunks from
                // being hoisted (128 live loads would double the register footprint).
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    int kp[16], kd[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        kp[c] = (c0 + c < kvalid && P.causal) ? __ldg(P.kposL + kbase + c0 + c) : INT_MIN;
                        if (DOC) kd[c] = (c0 + c < kvalid) ? __ldg(P.loL + kbase + c0 + c) : qlo;
                    }
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const bool vis = row_valid && (c0 + c < kvalid) && kp[c] <= qpos && (!LB || kp[c] >= qlo) &&
                                         (!DOC || kd[c] == qlo);
                        if (!vis) x[c0 + c] = -INFINITY;
                    }
                    asm volatile("" ::: "memory");
                }
            }
            // Row max over four independent chains (short dependency chains).
            float mq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) mq[q] = x[q];
#pragma unroll
            for (int c = 4; c < 124; c += 8) {
#pragma unroll
                for (int q = 0; q < 4; ++q) mq[q] = max3(mq[q], x[c + 2 * q], x[c + 2 * q + 1]);
            }
            mq[0] = max3(mq[0], x[124], x[125]);
            mq[1] = max3(mq[1], x[126], x[127]);
            const float mx = max3(fmaxf(mq[0], mq[1]), mq[2], mq[3]);
            const float mt = (mx == -INFINITY) ? -INFINITY : mx * P.scale_log2;
            const float m_new = fmaxf(m_used, mt);
            const bool resc = m_new > m_used + 8.0f;
            float alpha = 1.0f;
            if (resc) {
                alpha = ex2(m_used - m_new);
                l *= alpha;
                m_used = m_new;
            }
            const float msub = (m_used == -INFINITY) ? 0.f : -m_used;
            const uint64_t neg_m2 = f2_pack(msub, msub);
            uint32_t pk[64];
            uint64_t sum2[4] = {0, 0, 0, 0};                          // packed pairs of +0.0f
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                float a0, a1;
                f2_unpack(f2_fma(f2_pack(x[2 * c], x[2 * c + 1]), scale2, neg_m2), a0, a1);
                const float p0 = ex2(a0), p1 = ex2(a1);
                pk[c] = pack_f16(p0, p1);
                sum2[c & 3] = f2_add(sum2[c & 3], f2_pack(p0, p1));
            }
            float s0, s1;
            f2_unpack(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), s0, s1);
            l += s0 + s1;
            // P_i over the first 64 columns of S_i: column c holds keys 2c (low half) and 2c + 1.
            tmem_st64(tmem + lane_base + s_col, pk);
            if (j > 0 && __any_sync(0xffffffffu, resc)) {
                // O_i holds the PVs of earlier tiles: wait for the last one, then rescale in place.
                ok = __all_sync(0xffffffffu, wait(bars.pv_done(wg), (ntile - 1) & 1, kSitePvDone));
                if (!ok) {
                    tmem_st_wait();
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t t[32];
                    const uint32_t ta = tmem + lane_base + o_col + c * 32;
                    tmem_ld32(ta, t);
#pragma unroll
                    for (int q = 0; q < 32; ++q) t[q] = __float_as_uint(__uint_as_float(t[q]) * alpha);
                    tmem_st32(ta, t);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.p_full(wg));
            ++ntile;
            ++j;
        }
        flush();
        if (!ok) break;
        if (j == 0 && !P.fused && !P.first) continue;     // nothing visible at this step
        // ring step: the running row's maximum and sum, loaded before the wait for the last P·V so
        // that their round trip overlaps it
        float mr = -INFINITY, lr = 0.f;
        if (!P.fused && row_valid && P.first == 0 && l > 0.f) {
            const int64_t base = (((int64_t)U.r * P.B + U.b) * P.h + head) * P.n + jl;
            mr = P.lse_run[base];
            lr = P.l_run[base];
        }
        if (j > 0) {
            ok = __all_sync(0xffffffffu, wait(bars.pv_done(wg), (ntile - 1) & 1, kSitePvDone));
            if (!ok) break;
            tc_fence_after();
        }
        const float inv_l = l > 0.f ? 1.0f / l : 0.f;
        const float lse_v = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
        // Fused: O_i / l in bf16 at the row's natural position, and its lse.
        // Ring step: the running row holds O unnormalised relative to its maximum m_run (log2
        // units, like m_used) with the sum l_run; the finalize kernel divides. This step's (O_i,
        // m_used, l) joins it in one of three ways:
        //   write   (the first step, or a running row that has seen no key yet): O_i, m_used, l;
        //   add     (m_used <= m_run + 8): O_run += 2^(m_used - m_run) O_i by fire-and-forget
        //           reductions, no read of O_run; l_run grows by the same weight;
        //   rescale (m_used > m_run + 8, rare once a row has seen its largest scores):
        //           O_run = 2^(m_run - m_used) O_run + O_i, read back, and m_run = m_used.
        // A row none of whose keys this step shows is left as it is.
        uint4* dst = nullptr;                 // fused: bf16 row in natural order
        float* orow = nullptr;                // ring step: fp32 running row in layout order
        enum { kKeep, kWrite, kAdd, kRescale };
        int mode = kKeep;
        float f = 1.f;
        if (P.fused) {
            int64_t tn;
            if (P.layout == CPATTN_CONTIGUOUS) tn = (int64_t)U.r * P.n + jl;
            else if (P.layout == CPATTN_ZIGZAG)
                tn = jl < P.m ? (int64_t)U.r * P.m + jl : (int64_t)(2 * P.n_cp - 1 - U.r) * P.m + (jl - P.m);
            else tn = jl * P.n_cp + U.r;
            if (row_valid) {
                dst = reinterpret_cast<uint4*>(P.o + (((int64_t)U.b * P.T + tn) * P.h + head) * D);
                P.lse[((int64_t)U.b * P.h + head) * P.T + tn] = lse_v;
            }
        } else if (row_valid) {
            const int64_t base = (((int64_t)U.r * P.B + U.b) * P.h + head) * P.n + jl;
            orow = P.o_run + base * D;
            if (P.first != 0 || (l > 0.f && !(lr > 0.f))) {
                mode = kWrite;
                P.lse_run[base] = m_used;
                P.l_run[base] = l;
            } else if (l > 0.f) {
                if (m_used <= mr + 8.0f) {
                    mode = kAdd;
                    f = ex2(m_used - mr);
                    P.l_run[base] = lr + f * l;
                } else {
                    mode = kRescale;
                    f = ex2(mr - m_used);
                    P.lse_run[base] = m_used;
                    P.l_run[base] = lr * f + l;
                }
            }
        }
        // ring step: the warp's 32 rows (consecutive in layout order; row r is lane r's) and which
        // of them are added or written through the staging buffer
        const int64_t run_row0 = (((int64_t)U.r * P.B + U.b) * P.h + head) * P.n;
        const int64_t wrow0 = (int64_t)qt * 128 + quarter * 32;
        const unsigned add_rows = __ballot_sync(0xffffffffu, mode == kAdd);
        const unsigned write_rows = __ballot_sync(0xffffffffu, mode == kWrite);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t ot[32];
            if (j > 0) {
                tmem_ld32(tmem + lane_base + o_col + c * 32, ot);
            } else {
#pragma unroll
                for (int q = 0; q < 32; ++q) ot[q] = 0u;
            }
            if (dst) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 v;
                    v.x = pack_bf16(__uint_as_float(ot[8 * q4 + 0]) * inv_l, __uint_as_float(ot[8 * q4 + 1]) * inv_l);
                    v.y = pack_bf16(__uint_as_float(ot[8 * q4 + 2]) * inv_l, __uint_as_float(ot[8 * q4 + 3]) * inv_l);
                    v.z = pack_bf16(__uint_as_float(ot[8 * q4 + 4]) * inv_l, __uint_as_float(ot[8 * q4 + 5]) * inv_l);
                    v.w = pack_bf16(__uint_as_float(ot[8 * q4 + 6]) * inv_l, __uint_as_float(ot[8 * q4 + 7]) * inv_l);
                    st_global_v4_hint(dst + c * 4 + q4, v, pol_o);
                }
            } else if (!P.fused) {
                // Ring step. A row taking the rescale path merges by itself (read back, rare).
                // The written and added rows go through the warp's staging buffer (16-byte pieces
                // XOR-swizzled by row): the stores and reductions then move whole 128-byte row
                // segments, 8 lanes per row and 4 rows per instruction, instead of 16 bytes of
                // each of 32 rows per instruction.
                if (mode == kRescale) {
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        float4* a = reinterpret_cast<float4*>(orow) + c * 8 + q4;
                        const float4 oa = *a;
                        *a = make_float4(oa.x * f + __uint_as_float(ot[4 * q4]), oa.y * f + __uint_as_float(ot[4 * q4 + 1]),
                                         oa.z * f + __uint_as_float(ot[4 * q4 + 2]),
                                         oa.w * f + __uint_as_float(ot[4 * q4 + 3]));
                    }
                }
                const float mul = mode == kAdd ? f : 1.0f;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    st_shared_v4(stg + (lane * 8 + (q ^ (lane & 7))) * 16, __float_as_uint(__uint_as_float(ot[4 * q]) * mul),
                                 __float_as_uint(__uint_as_float(ot[4 * q + 1]) * mul),
                                 __float_as_uint(__uint_as_float(ot[4 * q + 2]) * mul),
                                 __float_as_uint(__uint_as_float(ot[4 * q + 3]) * mul));
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = i * 4 + (lane >> 3), q = lane & 7;
                    const int4 t = ld_shared_v4(stg + (r * 8 + (q ^ (r & 7))) * 16);
                    float* dst = P.o_run + (run_row0 + wrow0 + r) * D + c * 32 + q * 4;
                    if ((add_rows >> r) & 1u)
                        red_add_v4_f32(dst, __int_as_float(t.x), __int_as_float(t.y), __int_as_float(t.z), __int_as_float(t.w));
                    else if ((write_rows >> r) & 1u)
                        *reinterpret_cast<int4*>(dst) = t;
                }
                __syncwarp();
            }
        }
        if (j > 0) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.o_free(wg));  // O_i has been read: the next unit may overwrite it
        }
    }
}

template <int D, int M>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attention_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const Params P) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* skip_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
    volatile int* unit_slot = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);   // [2]
    const Bars<D> bars{sbase + C::OFF_BAR};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // A CTA that starts after a device error was recorded does no work (one thread decides for
    // the whole block).
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

    if (warp < 4) {
        setmaxnreg_dec<RegSplit<M>::low>();
        if (warp == 0 && lane == 0) producer<D, M>(P, &tmQ, &tmK, &tmV, sQ, sK, sV, unit_slot, bars, wait);
        if (warp == 1 && lane == 0) mma_issuer<D>(P, tmem, sQ, sK, sV, unit_slot, bars, wait);
        if (warp >= 2 && P.hop_words > 0) ring_hop_copy(P, (int)threadIdx.x - 64);
    } else {
        setmaxnreg_inc<RegSplit<M>::high>();
        softmax_epilogue<D, M>(P, tmem, unit_slot, bars, wait, sbase + C::OFF_STG + (warp - 4) * C::STG_WARP_BYTES);
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

// One thread per row group (rank r, group): the number of key tiles a unit of that row group
// visits in this launch, by the same walk the producer and the softmax warps take. Units of one
// row group differ only in batch element and heads, which do not change the walk.
template <int M>
__global__ void unit_tiles_kernel(const Params P) {
    constexpr bool LB = M == kMaskLower, DOC = M == kMaskDoc;
    const int rg = blockIdx.x * blockDim.x + threadIdx.x;
    if (rg >= P.n_cp * P.n_grp) return;
    Unit U;
    U.rg = rg;
    U.r = rg / P.n_grp;
    U.b = 0;
    U.kvh = 0;
    const int grp = rg % P.n_grp;
    if (P.pair_heads) {
        U.qt[0] = U.qt[1] = grp;
        U.valid[0] = U.valid[1] = 1;
    } else {
        U.qt[0] = 2 * grp;
        U.qt[1] = 2 * grp + 1;
        U.valid[0] = 1;
        U.valid[1] = U.qt[1] < P.n_qt;
    }
    unit_ranges<M>(P, U);
    U.head[0] = U.head[1] = 0;
    if (DOC) {
        // one bit per key tile some query of the row group may see, for every step of this launch
        const int s0 = P.fused ? 0 : P.step, s1 = P.fused ? P.n_cp : P.step + 1;
        int c = 0;
        for (int s = s0; s < s1; ++s) {
            int src = U.r - s;
            if (src < 0) src += P.n_cp;
            for (int wi = 0; wi < P.words; ++wi) {
                unsigned long long bits = 0ull;
                for (int b = 0; b < 64; ++b) {
                    const int kt = wi * 64 + b;
                    if (kt >= P.n_qt) break;
                    const int4 t4 = __ldg(P.ktile_mm + src * P.n_qt + kt);
                    const int4 d4 = __ldg(P.tile_lo + src * P.n_qt + kt);
                    const int c0 =
                        doc_class(P.causal, U.qmm[0].x, U.qmm[0].y, U.qlo[0].x, U.qlo[0].y, U.qbits[0], t4, d4);
                    const int c1 =
                        doc_class(P.causal, U.qmm[1].x, U.qmm[1].y, U.qlo[1].x, U.qlo[1].y, U.qbits[1], t4, d4);
                    if (c0 != CPATTN_TILE_SKIP || c1 != CPATTN_TILE_SKIP) {
                        bits |= 1ull << b;
                        ++c;
                    }
                }
                P.walk_bits[((int64_t)rg * P.n_cp + s) * P.words + wi] = bits;
            }
        }
        P.unit_tiles[rg] = c;
        return;
    }
    TileWalk<M> w;
    w.init(P, U);
    if (LB && P.causal) {                 // the scan, as the table walk will replay it
        w.s = P.fused ? 0 : P.step;
        w.kt = -1;
    }
    int c = 0;
    int cur = -1, first = 0, last = 0;
    unsigned long long nz = 0ull;
    while (w.next_scan()) {
        ++c;
        if (LB && P.causal) {
            if (w.s != cur) {
                if (cur >= 0) P.walk_tab[(int64_t)rg * P.n_cp + cur] = first | ((last + 1) << 16);
                for (int t = cur + 1; t < w.s; ++t) P.walk_tab[(int64_t)rg * P.n_cp + t] = 0;
                cur = w.s;
                first = w.kt;
                if (cur < 64) nz |= 1ull << cur;
            }
            last = w.kt;
        }
    }
    if (LB && P.causal) {
        if (cur >= 0) P.walk_tab[(int64_t)rg * P.n_cp + cur] = first | ((last + 1) << 16);
        for (int t = cur + 1; t < P.n_cp; ++t) P.walk_tab[(int64_t)rg * P.n_cp + t] = 0;
        if (cur < 0)
            for (int t = 0; t < P.n_cp; ++t) P.walk_tab[(int64_t)rg * P.n_cp + t] = 0;
        P.walk_nz[rg] = nz;
    }
    P.unit_tiles[rg] = c;
}

// Under a mask the plan's longest-first order (from positions alone) says little about the work of
// a row group: one block sorts the row groups by the tile counts unit_tiles_kernel just wrote,
// most tiles first (ties by index), so the persistent CTAs start the heaviest units first.
constexpr int kSortMax = 8192;
__global__ void __launch_bounds__(1024) order_by_tiles_kernel(const int32_t* __restrict__ tiles,
                                                             int32_t* __restrict__ order, int n) {
    __shared__ int32_t t[kSortMax];
    for (int i = threadIdx.x; i < n; i += blockDim.x) t[i] = tiles[i];
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ti = t[i];
        int rank = 0;
        for (int j = 0; j < n; ++j) rank += (t[j] > ti) || (t[j] == ti && j < i);
        order[rank] = i;
    }
}

// ---- host side -------------------------------------------------------------------------------
template <int D, int M>
int launch_d(const AttnLaunch& a, cudaStream_t st, std::string* why) {
    using C = Cfg<D>;
    static PerDeviceOnce attr_once;
    int dev = 0;
    cudaGetDevice(&dev);
    const int ea = attr_once.run(dev, [&]() -> int {
        cudaError_t e = cudaFuncSetAttribute(ring_attention_kernel<D, M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES_RING);
        if (e != cudaSuccess) return (int)e;
        // setmaxnreg.inc waits until enough registers are free in the block's allocation: the
        // split must fit in what the block is launched with, or the kernel would never proceed.
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, ring_attention_kernel<D, M>);
        if (e != cudaSuccess) return (int)e;
        if ((long)fa.numRegs * kThreads < 128L * RegSplit<M>::low + 256L * RegSplit<M>::high) {
            *why = "attention kernel built with " + std::to_string(fa.numRegs) +
                   " registers per thread, too few for its warpgroup register split";
            return (int)cudaErrorInvalidConfiguration;
        }
        return 0;
    });
    if (ea) return ea;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    CUtensorMap tq, tk, tv;
    const uint64_t qrows = (uint64_t)a.n_cp * a.B * a.h * a.n;
    const uint64_t kvrows = a.kv_rows ? a.kv_rows : (uint64_t)a.n_cp * a.B * a.n_kv * a.n;
    if (!make_map(&tq, a.qL, qrows, D) || !make_map(&tk, a.kv_k, kvrows, D) || !make_map(&tv, a.kv_v, kvrows, D)) {
        *why = "cuTensorMapEncodeTiled failed (driver entry point unavailable or bad tensor shape)";
        return (int)cudaErrorInvalidValue;
    }
    Params P{};
    P.B = a.B; P.h = a.h; P.n_kv = a.n_kv; P.g = a.h / a.n_kv; P.n_cp = a.n_cp; P.n_qt = a.n_qt;
    P.n_grp = a.n_grp; P.pair_heads = a.pair_heads; P.causal = a.causal;
    P.fused = a.fused; P.step = a.step; P.kv_by_holder = a.kv_by_holder; P.layout = a.layout;
    P.n = a.n; P.m = a.m; P.T = a.T; P.scale_log2 = a.scale_log2;
    P.posL = a.posL; P.tile_mm = reinterpret_cast<const int4*>(a.tile_mm); P.order = a.order;
    P.kposL = a.kposL ? a.kposL : a.posL;
    P.ktile_mm = reinterpret_cast<const int4*>(a.ktile_mm ? a.ktile_mm : a.tile_mm);
    P.first = a.first >= 0 ? a.first : (a.step == 0);
    P.kv_rank_rows = a.kv_rank_rows;
    P.hop_src_k = static_cast<const uint4*>(a.hop_src_k); P.hop_src_v = static_cast<const uint4*>(a.hop_src_v);
    P.hop_dst_k = static_cast<uint4*>(a.hop_dst_k); P.hop_dst_v = static_cast<uint4*>(a.hop_dst_v);
    P.hop_words = a.hop_words; P.hop_blk = a.hop_blk; P.hop_wrap = a.hop_wrap;
    P.unit_tiles = a.unit_tiles;
    P.walk_tab = a.walk_tab;
    P.walk_nz = a.walk_nz;
    P.walk_bits = a.walk_bits;
    P.words = (a.n_qt + 63) / 64;
    P.loL = a.loL; P.tile_lo = reinterpret_cast<const int4*>(a.tile_lo);
    P.counts = a.counts; P.sched = a.sched;
    P.o = static_cast<uint16_t*>(a.o); P.lse = a.lse; P.o_run = a.o_run; P.lse_run = a.lse_run; P.l_run = a.l_run;
    P.header = a.header; P.timeout_ns = a.timeout_ns;
    const int64_t units = (int64_t)a.n_cp * a.n_grp * a.B * (a.pair_heads ? a.h / 2 : a.h);
    if (units > INT_MAX) {
        *why = "too many work units";
        return (int)cudaErrorInvalidValue;
    }
    P.num_units = (int)units;
    // one CTA per SM, leaving the reserved SMs free for concurrent transfers
    const int avail = sms - a.reserved_sms > 0 ? sms - a.reserved_sms : 1;
    const int grid = (int)(units < avail ? units : avail);
    const int n_rg = a.n_cp * a.n_grp;
    unit_tiles_kernel<M><<<(n_rg + 127) / 128, 128, 0, st>>>(P);
    if (M != kMaskPos && a.order_scratch && n_rg <= kSortMax) {
        order_by_tiles_kernel<<<1, 1024, 0, st>>>(P.unit_tiles, a.order_scratch, n_rg);
        P.order = a.order_scratch;
    }
    ring_attention_kernel<D, M><<<grid, kThreads, a.fused ? C::SMEM_BYTES : C::SMEM_BYTES_RING, st>>>(tq, tk, tv, P);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_attention(const AttnLaunch& a, void* stream, std::string* why) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // a per-query lower bound or document ids, both read from loL / tile_lo
    const int mode = a.loL == nullptr ? kMaskPos : a.doc_ids ? kMaskDoc : kMaskLower;
    if (mode == kMaskDoc && !a.walk_bits) {
        *why = "document ids need the walk bitmask region";
        return (int)cudaErrorInvalidValue;
    }
    if (a.d == 128)
        return mode == kMaskPos ? launch_d<128, kMaskPos>(a, st, why)
               : mode == kMaskLower ? launch_d<128, kMaskLower>(a, st, why) : launch_d<128, kMaskDoc>(a, st, why);
    if (a.d == 64)
        return mode == kMaskPos ? launch_d<64, kMaskPos>(a, st, why)
               : mode == kMaskLower ? launch_d<64, kMaskLower>(a, st, why) : launch_d<64, kMaskDoc>(a, st, why);
    *why = "unsupported head width";
    return (int)cudaErrorInvalidValue;
}

int launch_wait_selftest(uint32_t* header, uint64_t timeout_ns, void* stream) {
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(header, timeout_ns);
    return (int)cudaGetLastError();
}

}  // namespace cpattn
