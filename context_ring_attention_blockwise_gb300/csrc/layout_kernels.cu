// layout_kernels.cu -- the HBM-bound kernels of the path: token placement (gather Q, K, V and
// position ids into rank-major layout order), the position range of every tile, the final
// scatter of the ring-step paths back to natural order, the backward ring-step path's add of a
// circulating gradient block, and the standalone log-sum-exp merge.
//
// For the forward, placement also writes V in fp16: the attention kernel multiplies fp16 P by fp16
// V (the tensor core wants one type for both operands), so that P carries three more significand
// bits than bf16 and O is normalised by the plain fp32 sum of the exponentials. bf16 to fp16 is
// exact for 2^-14 <= |v| <= 65504; below 2^-14 (fp16 subnormals) the absolute error is at most
// 2^-25, and a value beyond 65504 (or an infinite or NaN one) is recorded in the workspace header
// for cpattn_check to report.
//
// Placement: "Context and expert parallelism", section "The causal mask unbalances the
// sequence" (contiguous, zigzag and round-robin stripes) and section "In PyTorch" (every
// position-indexed tensor is sharded with the sequence, so position ids travel with tokens).
// Merge: same page, online-softmax paragraph of "Pass them around a ring".
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "internal.h"

namespace cpattn {
namespace {

// rank and local index of natural token t
__device__ __forceinline__ void rank_of(int layout, int64_t t, int64_t n, int64_t m, int n_cp, int& r, int64_t& j) {
    if (layout == CPATTN_CONTIGUOUS) {
        r = (int)(t / n);
        j = t - (int64_t)r * n;
    } else if (layout == CPATTN_ZIGZAG) {
        int c = (int)(t / m);
        if (c < n_cp) { r = c; j = t - (int64_t)c * m; }
        else { r = 2 * n_cp - 1 - c; j = m + (t - (int64_t)c * m); }
    } else {
        r = (int)(t % n_cp);
        j = t / n_cp;
    }
}

__device__ __forceinline__ int64_t token_of_dev(int layout, int r, int64_t j, int64_t n, int64_t m, int n_cp) {
    if (layout == CPATTN_CONTIGUOUS) return (int64_t)r * n + j;
    if (layout == CPATTN_ZIGZAG) return j < m ? (int64_t)r * m + j : (int64_t)(2 * n_cp - 1 - r) * m + (j - m);
    return j * n_cp + r;
}

// One 128-thread block per (rank, tile): position ids in layout order and their min/max.
// With a lower-bound array (document masks) the block also writes each token's bound in layout
// order and the min/max bound of the tile.
struct DefaultPos {
    int n_cp, layout, rank0;   // n_cp == 0: a token's default position is its natural index here
    int64_t m;
};

__global__ void __launch_bounds__(128) pos_tiles_kernel(const int32_t* __restrict__ pos, int32_t* __restrict__ posL,
                                                        int4* __restrict__ tile_mm, const int32_t* __restrict__ lob,
                                                        int32_t* __restrict__ loL, int4* __restrict__ tile_lo,
                                                        int64_t n, int64_t m, int n_cp, int layout, int n_qt,
                                                        DefaultPos dp) {
    const int r = blockIdx.x / n_qt, tile = blockIdx.x % n_qt;
    const int64_t j = (int64_t)tile * kBlockQ + threadIdx.x;
    int lo = INT_MAX, hi = INT_MIN, blo = INT_MAX, bhi = INT_MIN;
    unsigned bm_lo = 0u, bm_hi = 0u;   // document ids: a bit per id modulo 64 present in the tile
    if (j < n) {
        int64_t t = token_of_dev(layout, r, j, n, m, n_cp);
        const int dflt = dp.n_cp > 0 ? (int)token_of_dev(dp.layout, dp.rank0 + r, j, n, dp.m, dp.n_cp) : (int)t;
        int pv = pos ? pos[t] : dflt;
        posL[(int64_t)r * n + j] = pv;
        lo = hi = pv;
        if (lob) {
            const int bv = lob[t];
            loL[(int64_t)r * n + j] = bv;
            blo = bhi = bv;
            const unsigned bit = (unsigned)bv & 63u;
            if (bit < 32u) bm_lo = 1u << bit;
            else bm_hi = 1u << (bit - 32u);
        }
    }
    bm_lo = __reduce_or_sync(0xffffffffu, bm_lo);
    bm_hi = __reduce_or_sync(0xffffffffu, bm_hi);
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        blo = min(blo, __shfl_xor_sync(0xffffffffu, blo, o));
        bhi = max(bhi, __shfl_xor_sync(0xffffffffu, bhi, o));
    }
    __shared__ int slo[4], shi[4], sblo[4], sbhi[4];
    __shared__ unsigned sbm[4][2];
    if ((threadIdx.x & 31) == 0) {
        slo[threadIdx.x >> 5] = lo; shi[threadIdx.x >> 5] = hi;
        sblo[threadIdx.x >> 5] = blo; sbhi[threadIdx.x >> 5] = bhi;
        sbm[threadIdx.x >> 5][0] = bm_lo; sbm[threadIdx.x >> 5][1] = bm_hi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < 4; ++w) {
            lo = min(lo, slo[w]); hi = max(hi, shi[w]);
            blo = min(blo, sblo[w]); bhi = max(bhi, sbhi[w]);
            bm_lo |= sbm[w][0]; bm_hi |= sbm[w][1];
        }
        tile_mm[blockIdx.x] = make_int4(lo, hi, lo, 0);
        // (min, max) of the bound or id; with document ids, .z/.w hold the 64-bit id-bit mask
        if (lob) tile_lo[blockIdx.x] = make_int4(blo, bhi, (int)bm_lo, (int)bm_hi);
    }
}

// Per rank block, the minimum position over tiles kt..n_qt-1 (a backward scan): a key walk that
// finds it above every query position skips the rest of the block in one step. And the maximum
// over tiles 0..kt (a forward scan, non-decreasing in kt): under per-query lower bounds a walk
// skips a block whose maximum lies below every bound, or searches for its first tile that does not.
__global__ void tile_suffix_kernel(int4* __restrict__ tile_mm, int n_cp, int n_qt) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n_cp) return;
    int run = INT_MAX;
    for (int kt = n_qt - 1; kt >= 0; --kt) {
        int4 t = tile_mm[(int64_t)r * n_qt + kt];
        run = min(run, t.x);
        t.z = run;
        tile_mm[(int64_t)r * n_qt + kt] = t;
    }
    int pre = INT_MIN;
    for (int kt = 0; kt < n_qt; ++kt) {
        int4 t = tile_mm[(int64_t)r * n_qt + kt];
        pre = max(pre, t.y);
        t.w = pre;
        tile_mm[(int64_t)r * n_qt + kt] = t;
    }
}

// Gather rows of d bf16 from natural [B,T,heads,d] into rank-major [n_cp][B][heads][n][d].
// A block takes one natural token row (b, t) at a time: its h query heads and n_kv key and value
// heads, (h + 2 n_kv) * d / 8 pieces of 16 bytes, contiguous in each source. The rank and local
// index are worked out once per row; each thread then issues up to kUnroll loads before its
// stores, so enough bytes are in flight to keep HBM busy.
constexpr int kPermuteUnroll = 8;

__global__ void __launch_bounds__(256, 4) permute_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k,
                                                      const uint4* __restrict__ v, uint4* __restrict__ qL,
                                                      uint4* __restrict__ kL, uint4* __restrict__ vL, int B, int64_t T,
                                                      int64_t n, int64_t m, int h, int n_kv, int d, int n_cp,
                                                      int layout, int v_f16, uint32_t* __restrict__ header) {
    const int lg = (d == 128) ? 4 : 3;                      // log2 of the 16-byte pieces per head row
    const int cpr = 1 << lg;
    const int per_row = (h + 2 * n_kv) * cpr;
    const int64_t rows = (int64_t)B * T;
    for (int64_t rw = blockIdx.x; rw < rows; rw += gridDim.x) {
        const int64_t t = rw % T;
        const int b = (int)(rw / T);
        int r;
        int64_t j;
        rank_of(layout, t, n, m, n_cp, r, j);
        const int64_t rb = (int64_t)r * B + b;
        for (int e0 = threadIdx.x; e0 < per_row; e0 += kPermuteUnroll * blockDim.x) {
            uint4 x[kPermuteUnroll];
            uint4* dp[kPermuteUnroll];
#pragma unroll
            for (int u = 0; u < kPermuteUnroll; ++u) {
                const int e = e0 + u * blockDim.x;
                dp[u] = nullptr;
                if (e < per_row) {
                    const int hh = e >> lg, c = e & (cpr - 1);
                    const uint4* src;
                    uint4* dst;
                    int heads, hd;
                    if (hh < h) { src = q; dst = qL; heads = h; hd = hh; }
                    else if (hh < h + n_kv) { src = k; dst = kL; heads = n_kv; hd = hh - h; }
                    else { src = v; dst = vL; heads = n_kv; hd = hh - h - n_kv; }
                    x[u] = __ldg(src + (rw * heads + hd) * cpr + c);
                    if (v_f16 && hh >= h + n_kv) {
                        // bf16 -> fp16: exact for |v| <= 65504 (fp16 has more significand bits)
                        uint32_t* w = reinterpret_cast<uint32_t*>(&x[u]);
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {
                            const float lo = __uint_as_float(w[q2] << 16), hi = __uint_as_float(w[q2] & 0xFFFF0000u);
                            uint32_t r;
                            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
                            w[q2] = r;
                            // all-ones exponent: |v| beyond 65504, or an infinite or NaN input
                            if ((r & 0x7C00u) == 0x7C00u || (r & 0x7C000000u) == 0x7C000000u)
                                atomicOr(header + kErrFlags, (uint32_t)kErrRangeFlag);
                        }
                    }
                    dp[u] = dst + ((rb * heads + hd) * n + j) * cpr + c;
                }
            }
#pragma unroll
            for (int u = 0; u < kPermuteUnroll; ++u)
                if (dp[u]) *dp[u] = x[u];
        }
    }
}

// The two kernels below go from layout order [n_cp][B][H][n][d] (fp32) back to natural order
// [B][T][H][d] (bf16). One warp per token (b, t): its rank and local index are found once, then
// the warp walks the token's H rows, d / 4 lanes per row (one float4 each), 32 / (d / 4) rows at a
// time. (Taking the index apart for every float4 cost more instructions than the bytes allowed:
// the kernel ran at half the copy bandwidth.)

// Ring-step path: the running state (O unnormalised over d columns, its maximum m_run in log2
// units and its sum l_run) -> O / l_run in bf16 and lse = (m_run + log2 l_run) ln 2 as [B,h,T]; a
// row that saw no key gets 0 and -inf.
__global__ void __launch_bounds__(256) finalize_kernel(const float4* __restrict__ o_run, const float* __restrict__ m_run,
                                                       const float* __restrict__ l_run, uint2* __restrict__ o,
                                                       float* __restrict__ lse, int B, int64_t T, int64_t n, int64_t m,
                                                       int h, int d, int n_cp, int layout) {
    const int cpr = d / 4, per = 32 / cpr;
    const int lane = threadIdx.x & 31, c = lane % cpr, sub = lane / cpr;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t tok = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); tok < (int64_t)B * T;
         tok += warps) {
        const int b = (int)(tok / T);
        const int64_t t = tok - (int64_t)b * T;
        int r;
        int64_t j;
        rank_of(layout, t, n, m, n_cp, r, j);
        const int64_t row0 = ((int64_t)r * B + b) * h * n + j;      // head hd's row: row0 + hd n
        for (int hd = sub; hd < h; hd += per) {
            const int64_t row = row0 + (int64_t)hd * n;
            const float4 x = o_run[row * cpr + c];
            const float lr = l_run[row];
            const float inv = lr > 0.f ? 1.0f / lr : 0.f;
            __nv_bfloat162 lo = __floats2bfloat162_rn(x.x * inv, x.y * inv), hi = __floats2bfloat162_rn(x.z * inv, x.w * inv);
            uint2 out;
            out.x = *reinterpret_cast<uint32_t*>(&lo);
            out.y = *reinterpret_cast<uint32_t*>(&hi);
            o[(tok * h + hd) * cpr + c] = out;
            if (c == 0) lse[((int64_t)b * h + hd) * T + t] = lr > 0.f ? (m_run[row] + log2f(lr)) * 0.69314718055994531f : -INFINITY;
        }
    }
}

// The backward ring-step path's gradients: fp32 -> bf16, same orders.
__global__ void __launch_bounds__(256) unpermute_f32_kernel(const float4* __restrict__ src, uint2* __restrict__ dst, int B,
                                                            int64_t T, int64_t n, int64_t m, int H, int d, int n_cp,
                                                            int layout) {
    const int cpr = d / 4, per = 32 / cpr;
    const int lane = threadIdx.x & 31, c = lane % cpr, sub = lane / cpr;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t tok = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); tok < (int64_t)B * T;
         tok += warps) {
        const int b = (int)(tok / T);
        const int64_t t = tok - (int64_t)b * T;
        int r;
        int64_t j;
        rank_of(layout, t, n, m, n_cp, r, j);
        const int64_t row0 = ((int64_t)r * B + b) * H * n + j;
        for (int hd = sub; hd < H; hd += per) {
            const float4 x = src[(row0 + (int64_t)hd * n) * cpr + c];
            __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
            uint2 out;
            out.x = *reinterpret_cast<uint32_t*>(&lo);
            out.y = *reinterpret_cast<uint32_t*>(&hi);
            dst[(tok * H + hd) * cpr + c] = out;
        }
    }
}

// S-way merge: o = sum_s exp(lse_s - L) o_s with L = M + ln sum_s exp(lse_s - M), M = max lse_s.
// One thread per 8 consecutive d of one (row, head). One pass over the partials, four at a time:
// the chunk's loads are issued together, then a running maximum, sum and weighted sum are
// updated (rescaled when the maximum rises). An empty partial (lse = -inf) is skipped, whatever
// its O holds.
__global__ void __launch_bounds__(256, 4) merge_kernel(int S, int64_t rows, int h, int d,
                                                       const float4* __restrict__ o_parts,
                                                       const float* __restrict__ lse_parts, uint4* __restrict__ o,
                                                       float* __restrict__ lse) {
    const int cpr = d / 8;
    const int64_t total = rows * h * cpr;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % cpr);
        const int64_t rh = i / cpr;
        const int hd = (int)(rh % h);
        const int64_t row = rh / h;
        float M = -INFINITY, sum = 0.f;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int s0 = 0; s0 < S; s0 += 4) {
            float ls[4];
            float4 x[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s = s0 + u;
                ls[u] = -INFINITY;
                x[u][0] = x[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (s < S) {
                    ls[u] = __ldg(lse_parts + ((int64_t)s * h + hd) * rows + row);
                    const float4* src = o_parts + ((int64_t)s * total + i) * 2;
                    x[u][0] = __ldg(src);
                    x[u][1] = __ldg(src + 1);
                }
            }
            const float mc = fmaxf(fmaxf(ls[0], ls[1]), fmaxf(ls[2], ls[3]));
            if (mc == -INFINITY) continue;
            const float Mn = fmaxf(M, mc);
            const float a = expf(M - Mn);                 // 0 while nothing has been merged
            sum *= a;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] *= a;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (ls[u] == -INFINITY) continue;
                const float w = expf(ls[u] - Mn);
                sum += w;
                acc[0] += w * x[u][0].x; acc[1] += w * x[u][0].y; acc[2] += w * x[u][0].z; acc[3] += w * x[u][0].w;
                acc[4] += w * x[u][1].x; acc[5] += w * x[u][1].y; acc[6] += w * x[u][1].z; acc[7] += w * x[u][1].w;
            }
            M = Mn;
        }
        const float inv = (M == -INFINITY) ? 0.f : 1.0f / sum;
        const float L = (M == -INFINITY) ? -INFINITY : M + logf(sum);
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
            pk[e] = *reinterpret_cast<uint32_t*>(&b2);
        }
        o[i] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        if (c == 0) lse[(int64_t)hd * rows + row] = L;
    }
}

int sm_count() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

int grid_for(int64_t work, int threads) {
    int64_t blocks = (work + threads - 1) / threads;
    int64_t cap = (int64_t)sm_count() * 16;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

// A small int32 table carried to the device inside the kernel's parameter block: the values are
// copied when the launch is enqueued, so the upload needs neither a page-locked host buffer nor a
// host-to-device copy from pageable memory.
constexpr int kParamInts = 960;
struct ParamInts {
    int n;
    int32_t v[kParamInts];
};

__global__ void __launch_bounds__(256) upload_i32_kernel(int32_t* __restrict__ dst, const ParamInts vals) {
    for (int i = threadIdx.x; i < vals.n; i += blockDim.x) dst[i] = vals.v[i];
}

}  // namespace

int launch_upload_i32(int32_t* dst, const int32_t* host, int64_t n, void* stream) {
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int64_t off = 0; off < n; off += kParamInts) {
        ParamInts p;
        p.n = (int)(n - off < kParamInts ? n - off : kParamInts);
        for (int i = 0; i < p.n; ++i) p.v[i] = host[off + i];
        upload_i32_kernel<<<1, 256, 0, st>>>(dst + off, p);
        const int e = (int)cudaGetLastError();
        if (e) return e;
    }
    return 0;
}

// ---- Ulysses all-to-alls ("Ulysses, splitting by heads instead") --------------------------
// Virtual rank r' of n_cp holds, after the first all-to-all, every token of its hp = h / n_cp query
// heads r' hp .. r' hp + hp - 1 and of the nkvp KV heads they use: (r' hp) / g + j' for j' < nkvp,
// with g = h / n_kv (one KV head shared by n_cp / n_kv ranks when n_cp > n_kv). Its buffers are
// the batches b' = b n_cp + r' of a natural-order [B n_cp][T][hp or nkvp][d] problem. One
// natural token row (b, t) per block iteration: the block writes the row's head slices to every
// rank that holds them.
__global__ void __launch_bounds__(256, 4) ulysses_split_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k,
                                                             const uint4* __restrict__ v, uint4* __restrict__ qs,
                                                             uint4* __restrict__ ks, uint4* __restrict__ vs, int B,
                                                             int64_t T, int h, int n_kv, int d, int n_cp, int hp,
                                                             int nkvp) {
    const int lg = (d == 128) ? 4 : 3;                      // log2 of the 16-byte pieces per head row
    const int cpr = 1 << lg;
    const int g = h / n_kv;
    const int slots_kv = n_cp * nkvp;                       // (rank, KV head of the rank) pairs
    const int per_row = (h + 2 * slots_kv) * cpr;
    const int64_t rows = (int64_t)B * T;
    for (int64_t rw = blockIdx.x; rw < rows; rw += gridDim.x) {
        const int64_t t = rw % T;
        const int b = (int)(rw / T);
        for (int e0 = threadIdx.x; e0 < per_row; e0 += kPermuteUnroll * blockDim.x) {
            uint4 x[kPermuteUnroll];
            uint4* dp[kPermuteUnroll];
#pragma unroll
            for (int u = 0; u < kPermuteUnroll; ++u) {
                const int e = e0 + u * blockDim.x;
                dp[u] = nullptr;
                if (e < per_row) {
                    const int sl = e >> lg, c = e & (cpr - 1);
                    if (sl < h) {                           // query head sl -> rank sl / hp
                        const int rr = sl / hp, i = sl - rr * hp;
                        x[u] = __ldg(q + (rw * h + sl) * cpr + c);
                        dp[u] = qs + ((((int64_t)b * n_cp + rr) * T + t) * hp + i) * cpr + c;
                    } else {
                        const bool is_k = sl < h + slots_kv;
                        const int s2 = sl - h - (is_k ? 0 : slots_kv);
                        const int rr = s2 / nkvp, j = s2 - rr * nkvp;
                        const int kvh = (rr * hp) / g + j;
                        x[u] = __ldg((is_k ? k : v) + (rw * n_kv + kvh) * cpr + c);
                        dp[u] = (is_k ? ks : vs) + ((((int64_t)b * n_cp + rr) * T + t) * nkvp + j) * cpr + c;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kPermuteUnroll; ++u)
                if (dp[u]) *dp[u] = x[u];
        }
    }
}

// The second all-to-all: every rank's output rows back to natural order [B][T][h][d].
__global__ void __launch_bounds__(256, 4) ulysses_merge_kernel(const uint4* __restrict__ os, uint4* __restrict__ o,
                                                             int B, int64_t T, int h, int d, int n_cp, int hp) {
    const int lg = (d == 128) ? 4 : 3;
    const int cpr = 1 << lg;
    const int per_row = h * cpr;
    const int64_t rows = (int64_t)B * T;
    for (int64_t rw = blockIdx.x; rw < rows; rw += gridDim.x) {
        const int64_t t = rw % T;
        const int b = (int)(rw / T);
        for (int e0 = threadIdx.x; e0 < per_row; e0 += kPermuteUnroll * blockDim.x) {
            uint4 x[kPermuteUnroll];
            uint4* dp[kPermuteUnroll];
#pragma unroll
            for (int u = 0; u < kPermuteUnroll; ++u) {
                const int e = e0 + u * blockDim.x;
                dp[u] = nullptr;
                if (e < per_row) {
                    const int hh = e >> lg, c = e & (cpr - 1);
                    const int rr = hh / hp, i = hh - rr * hp;
                    x[u] = __ldg(os + ((((int64_t)b * n_cp + rr) * T + t) * hp + i) * cpr + c);
                    dp[u] = o + (rw * h + hh) * cpr + c;
                }
            }
#pragma unroll
            for (int u = 0; u < kPermuteUnroll; ++u)
                if (dp[u]) *dp[u] = x[u];
        }
    }
}

int launch_ulysses_split(const UlyssesArgs& a, void* stream) {
    const int64_t rows = (int64_t)a.B * a.T, cap = (int64_t)sm_count() * 4;
    ulysses_split_kernel<<<(int)(rows < cap ? rows : cap), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(a.q), static_cast<const uint4*>(a.k), static_cast<const uint4*>(a.v),
        static_cast<uint4*>(a.qs), static_cast<uint4*>(a.ks), static_cast<uint4*>(a.vs), a.B, a.T, a.h, a.n_kv, a.d,
        a.n_cp, a.hp, a.nkvp);
    return (int)cudaGetLastError();
}

int launch_ulysses_merge(const UlyssesArgs& a, void* stream) {
    const int64_t rows = (int64_t)a.B * a.T, cap = (int64_t)sm_count() * 4;
    ulysses_merge_kernel<<<(int)(rows < cap ? rows : cap), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(a.os), static_cast<uint4*>(a.o), a.B, a.T, a.h, a.d, a.n_cp, a.hp);
    return (int)cudaGetLastError();
}

int launch_permute(const PermuteArgs& a, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const DefaultPos dp{a.dflt_ncp, a.dflt_layout, a.dflt_rank0, a.dflt_m};
    pos_tiles_kernel<<<a.n_cp * a.n_qt, 128, 0, st>>>(a.pos, a.posL, reinterpret_cast<int4*>(a.tile_mm), a.lo, a.loL,
                                                      reinterpret_cast<int4*>(a.tile_lo), a.n, a.m, a.n_cp, a.layout,
                                                      a.n_qt, dp);
    int e = (int)cudaGetLastError();
    if (e) return e;
    tile_suffix_kernel<<<(a.n_cp + 127) / 128, 128, 0, st>>>(reinterpret_cast<int4*>(a.tile_mm), a.n_cp, a.n_qt);
    e = (int)cudaGetLastError();
    if (e) return e;
    // one token row per block iteration; four resident 256-thread blocks per SM
    const int64_t rows = (int64_t)a.B * a.T, cap = (int64_t)sm_count() * 4;
    permute_kernel<<<(int)(rows < cap ? rows : cap), 256, 0, st>>>(
        static_cast<const uint4*>(a.q), static_cast<const uint4*>(a.k), static_cast<const uint4*>(a.v),
        static_cast<uint4*>(a.qL), static_cast<uint4*>(a.kL), static_cast<uint4*>(a.vL), a.B, a.T, a.n, a.m, a.h,
        a.n_kv, a.d, a.n_cp, a.layout, a.v_f16, a.header);
    return (int)cudaGetLastError();
}

int launch_finalize(const FinalizeArgs& a, void* stream) {
    const int64_t work = (int64_t)a.B * a.T * 32;          // a warp per token
    finalize_kernel<<<grid_for(work, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(a.o_run), a.lse_run, a.l_run, static_cast<uint2*>(a.o), a.lse, a.B, a.T, a.n, a.m,
        a.h, a.d, a.n_cp, a.layout);
    return (int)cudaGetLastError();
}

int launch_unpermute_f32(const float* src, void* dst, int B, int64_t T, int64_t n, int64_t m, int H, int d, int n_cp,
                         int layout, void* stream) {
    const int64_t work = (int64_t)B * T * 32;              // a warp per token
    unpermute_f32_kernel<<<grid_for(work, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(src), static_cast<uint2*>(dst), B, T, n, m, H, d, n_cp, layout);
    return (int)cudaGetLastError();
}

int launch_merge(int S, int64_t rows, int h, int d, const float* o_parts, const float* lse_parts, void* o, float* lse,
                 void* stream) {
    // four resident 256-thread blocks per SM, grid-stride over (row, head, 8 columns)
    const int64_t work = rows * h * (d / 8), cap = (int64_t)sm_count() * 4;
    const int64_t blocks = (work + 255) / 256;
    merge_kernel<<<(int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        S, rows, h, d, reinterpret_cast<const float4*>(o_parts), lse_parts, static_cast<uint4*>(o), lse);
    return (int)cudaGetLastError();
}

}  // namespace cpattn
