// Quantised expert FFN for batches of 3 or more tokens (Q8_0), or any
// batch (Q4_0), one lane per weight row.
//
// Gate/up "Q8_0-quantised SwiGLU experts" and down + weighted combine
// (amalgafy.com/technical-overview, "Warm target path"; the gate/up and down
// geometry of expxa.com/research/reuse-ordering-qualification, "Shape"); the
// 4-bit weights of the next stage, "Q4 expert execution" (same page,
// "Execution architecture"), as Q4_0 blocks.
//
// With several tokens per expert the per-token work is no longer negligible
// next to the weight stream, and a warp-per-row layout (lanes split K) pays
// twice for it: every lane re-reads the activations from shared memory for
// each row it owns (shared-memory bandwidth becomes the bound) and every
// (row, token) sum needs a cross-lane reduction.  Here the roles are
// swapped: a CTA item is 32 rows of one expert (lane = row), every lane
// dequantises its own row once per item, and the activations are read as
// shared-memory broadcasts (all lanes read the same address), so one 16-byte
// activation load feeds 32 rows.  K is split over the CTA's warps; each
// warp streams its K slice of the 32 rows through a private cp.async ring,
// and the per-warp partial sums are added in a fixed order (deterministic)
// through shared memory at the end of the item.
//
//   gate/up item: 32 features r of expert e, pairs p of one bucket chunk:
//       h[p][r] = silu(Wg[e][r] . x_p) * (Wu[e][r] . x_p)
//   down item:    32 output rows o, pairs p of one bucket chunk:
//       out[tok(p)][o] += w(p) * (Wd[e][o] . h[p])      (or ypairs[p][o])
#include <atomic>

#include "common.cuh"
#include "pipeline.cuh"
#include "stream_common.cuh"

namespace moe {

namespace {

using namespace stream;

constexpr int kRowsFT = 32;   // rows per CTA item: one per lane
constexpr int kRowsKS = 64;   // K per warp stage: two 32-wide blocks, 4 bytes of scales per row
constexpr int kRowsG = 8;     // pairs per bucket chunk (down)
constexpr int kRowsNSTG = 4;  // ring stages per warp (down)
constexpr int kScaleBytes = kRowsFT * 4;            // a stage's scales of one matrix: 2 fp16 per row
// Both kernels run several small CTAs per SM rather than one large one: a
// CTA's warps meet at a barrier after every item (to add their K slices), and
// with three independent CTAs per SM one CTA's barrier wait is covered by
// the other two CTAs' work (measured at T = 64: 407 -> 337 us per layer
// against one 12-warp down CTA and two 8-warp gate/up CTAs per SM).
constexpr int kGuNW = 4;                            // gate/up warps (K = d_model split 4 ways)
// gate/up: each CTA holds chunks of at most kGuG pairs and a kGuNSTG-stage
// ring per warp (~71 KB of shared memory), three CTAs per SM
constexpr int kGuG = 4;
constexpr int kGuNSTG = 2;
constexpr int kGuCtasPerSm = 3;
constexpr int kDnNW = 4;                            // down warps (K = d_ff split 4 ways)
constexpr int kDnCtasPerSm = 3;                     // down: ~64 KB of shared memory per CTA

// Format-dependent stage geometry.  FMT 0 (Q8_0): a row's 64 K of a stage
// are 64 bytes (four 16-byte chunks of 16 values); FMT 1 (Q4_0): 32 bytes
// (two 16-byte chunks, each one whole block of 32 nibbles).
template <int FMT>
struct RowsFmt {
    static constexpr int kRowBytes = FMT ? kRowsKS / 2 : kRowsKS;      // bytes of one row per stage
    static constexpr int kChunks = kRowBytes / 16;                     // 16-byte chunks per row
    static constexpr int kTileBytes = kRowsFT * kRowBytes;             // one matrix's [32 rows] of a stage
    static constexpr int kGuStage = 2 * kTileBytes + 2 * kScaleBytes;
    static constexpr int kDnStage = kTileBytes + kScaleBytes;
    // Byte offset of 16-byte chunk c of row r in a tile.  Q8_0: rotated by
    // r/2 over 4 chunks; Q4_0: by r/4 over 2 chunks.  Either way the 8 lanes
    // of one 16-byte shared-memory phase read 8 different bank groups.
    static __device__ __forceinline__ int tile_off(int r, int c) {
        return FMT ? r * kRowBytes + (((c + (r >> 2)) & 1) << 4) : r * kRowBytes + (((c + (r >> 1)) & 3) << 4);
    }
};

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Rows row0 .. row0+31, K range [k0, k0+64) of one matrix (qs row stride
// K bytes for Q8_0, K/2 for Q4_0; scale row stride K/32 halves) into a tile
// and its scales.
template <int FMT>
__device__ __forceinline__ void issue_tile(unsigned char* tile, unsigned char* sc, const int8_t* qs, const uint16_t* d,
                                           size_t row0, int K, int k0, int lane) {
    using F = RowsFmt<FMT>;
    const int rb = FMT ? K / 2 : K;  // bytes per weight row
#pragma unroll
    for (int m = 0; m < F::kChunks; ++m) {
        const int pc = lane + 32 * m, r = pc / F::kChunks, c = pc % F::kChunks;
        cp_async16(tile + F::tile_off(r, c),
                   reinterpret_cast<const unsigned char*>(qs) + (row0 + r) * rb + (FMT ? k0 / 2 : k0) + c * 16);
    }
    cp_async4(sc + lane * 4, d + (row0 + lane) * (K / 32) + k0 / 32);
}

// 16 consecutive weights (values 16u .. 16u+15 of a stage row, u = 0..3) of
// this lane's row, dequantised exactly into 8 fp32 pairs.  Q8_0: chunk u.
// Q4_0: chunk u/2 holds one block; its low nibbles are the block's values
// 0..15, its high nibbles 16..31.
template <int FMT>
__device__ __forceinline__ void stage_w16(const unsigned char* tile, int lane, int u, float d, f32x2 (&w)[8]) {
    using F = RowsFmt<FMT>;
    if (FMT == 0)
        dequant16(*reinterpret_cast<const uint4*>(tile + F::tile_off(lane, u)), d, w);
    else
        dequant16_q4(*reinterpret_cast<const uint4*>(tile + F::tile_off(lane, u >> 1)), u & 1, d, w);
}

// The fp16 scale of 16-byte chunk c (0..3) from a row's 4-byte scale word.
__device__ __forceinline__ float chunk_scale(uint32_t word, int c) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(c < 2 ? word & 0xffffu : word >> 16)));
}

// 16 activations as 8 fp32 pairs: 64-bit shared-memory loads, so the pairs
// land in register pairs with no repacking.  Every lane reads the same
// address (a shared-memory broadcast).
__device__ __forceinline__ ulonglong2 ld_pairs(const float* v) { return *reinterpret_cast<const ulonglong2*>(v); }

// One stage (64 K of the 32 rows) against the NT pairs of the item, NT
// known at compile time (the caller switches on it once per stage), so every
// token's accumulators are registers and nothing is padded.  Each (row,
// token) sum is split in two accumulators (even and odd 4-wide steps), which
// gives at least 4 independent FMA chains even for a single token.
template <int NT, int FMT>
__device__ __forceinline__ void gu_stage(const unsigned char* st, int lane, const float* xk, const int* xoff,
                                         f32x2 (&ag)[2][kGuG], f32x2 (&au)[2][kGuG]) {
    constexpr int TB = RowsFmt<FMT>::kTileBytes;
    const uint32_t sgw = reinterpret_cast<const uint32_t*>(st + 2 * TB)[lane];
    const uint32_t suw = reinterpret_cast<const uint32_t*>(st + 2 * TB + kScaleBytes)[lane];
#pragma unroll
    for (int c = 0; c < kRowsKS / 16; ++c) {
        f32x2 wg[8], wu[8];
        stage_w16<FMT>(st, lane, c, chunk_scale(sgw, c), wg);
        stage_w16<FMT>(st + TB, lane, c, chunk_scale(suw, c), wu);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const ulonglong2 xv = ld_pairs(xk + xoff[t] + c * 16 + 4 * i);
                ag[i & 1][t] = f2_fma(wg[2 * i + 1], xv.y, f2_fma(wg[2 * i], xv.x, ag[i & 1][t]));
                au[i & 1][t] = f2_fma(wu[2 * i + 1], xv.y, f2_fma(wu[2 * i], xv.x, au[i & 1][t]));
            }
    }
}

template <int NT, int FMT>
__device__ __forceinline__ void dn_stage(const unsigned char* st, int lane, const float* hk, int f,
                                         f32x2 (&acc)[2][kRowsG]) {
    const uint32_t sw = reinterpret_cast<const uint32_t*>(st + RowsFmt<FMT>::kTileBytes)[lane];
#pragma unroll
    for (int c = 0; c < kRowsKS / 16; ++c) {
        f32x2 wv[8];
        stage_w16<FMT>(st, lane, c, chunk_scale(sw, c), wv);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const ulonglong2 xv = ld_pairs(hk + t * f + c * 16 + 4 * i);
                acc[i & 1][t] = f2_fma(wv[2 * i + 1], xv.y, f2_fma(wv[2 * i], xv.x, acc[i & 1][t]));
            }
    }
}

#define MOE_GU_SWITCH(n, CALL)     \
    switch (n) {                   \
        case 1: CALL(1); break;    \
        case 2: CALL(2); break;    \
        case 3: CALL(3); break;    \
        default: CALL(4); break;   \
    }

#define MOE_ROWS_SWITCH(n, CALL)   \
    switch (n) {                   \
        case 1: CALL(1); break;    \
        case 2: CALL(2); break;    \
        case 3: CALL(3); break;    \
        case 4: CALL(4); break;    \
        case 5: CALL(5); break;    \
        case 6: CALL(6); break;    \
        case 7: CALL(7); break;    \
        default: CALL(8); break;   \
    }

// ------------------------------------------------------------------ gate/up
// Items: (bucket chunk g, feature tile ft) with f/32 tiles per chunk.  Warp
// w owns K range [w*dm/4, (w+1)*dm/4), SPI = dm/256 stages per item.
// ALLTOK: every token's x staged once (T <= kGuG); else the chunk's x is
// staged per chunk (restaged at chunk changes).  Chunks hold at most kGuG
// pairs; three CTAs share an SM.
template <bool ALLTOK, int FMT>
__global__ void __launch_bounds__(kGuNW * 32, kGuCtasPerSm) gateup_rows_kernel(
    const float* __restrict__ x, int T, int dm, int f, int E, const int8_t* __restrict__ gqs,
    const uint16_t* __restrict__ gd, const int8_t* __restrict__ uqs, const uint16_t* __restrict__ ud,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok, float* __restrict__ h,
    float* __restrict__ out_init, int init_residual, int P, const int32_t* __restrict__ eslot, int nslots) {
    extern __shared__ __align__(128) unsigned char gr_smem[];
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    __shared__ int s_tok[ALLTOK ? kMaxStagedPairs : kGuG];
    constexpr int kThreads = kGuNW * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d4 = dm / 4;
    const int kw = dm / kGuNW, spi = kw / kRowsKS;
    const int ftn = f / kRowsFT;
    constexpr int kGuStage = RowsFmt<FMT>::kGuStage, TB = RowsFmt<FMT>::kTileBytes;
    unsigned char* ring = gr_smem + (size_t)warp * kGuNSTG * kGuStage;
    float* xs = reinterpret_cast<float*>(gr_smem + (size_t)kGuNW * kGuNSTG * kGuStage);  // [kGuG or T][dm]
    float* part = xs + (size_t)kGuG * dm;  // [kGuNW warps][kGuG pairs][gate, up][32]

    pdl_wait();  // routing / bucketing of this layer complete and visible
    if (warp == 0)
        build_active(offsets, E, ALLTOK ? (1 << 30) : kGuG, P, s_act, s_beg, s_end, s_cb, &s_n, eslot, nslots);
    if (ALLTOK) {
        for (int p = threadIdx.x; p < P; p += kThreads) {
            const int t = __ldcg(pair_tok + p);
            s_tok[p] = (t >= 0 && t < T) ? t : 0;
        }
        for (int i = threadIdx.x; i < T * d4; i += kThreads)
            reinterpret_cast<float4*>(xs)[i] = __ldcg(reinterpret_cast<const float4*>(x) + i);
    }
    if (out_init) {  // combine target: (residual ? x : 0), consumed by the down kernel
        const size_t n4 = (size_t)T * d4;
        float4* o4 = reinterpret_cast<float4*>(out_init);
        const float4* x4 = reinterpret_cast<const float4*>(x);
        for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < n4; i += (size_t)gridDim.x * kThreads)
            o4[i] = init_residual ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    pdl_launch_dependents();
    int lo, hi;
    item_range(s_cb[s_n] * ftn, &lo, &hi);
    const int nst = (hi - lo) * spi;

    // issue cursor: stages are issued in order, one per call
    int is_i = lo, is_s = 0, is_g = -1, is_a = 0;
    size_t is_row0 = 0;
    auto issue = [&](int q, int slot) {
        if (q < nst) {
            if (is_s == 0) {
                const int g = is_i / ftn;
                if (g != is_g) {
                    is_g = g;
                    is_a = locate(g, s_cb, s_n);
                }
                is_row0 = (size_t)s_act[is_a] * f + (size_t)(is_i - g * ftn) * kRowsFT;
            }
            const int k0 = warp * kw + is_s * kRowsKS;
            unsigned char* st = ring + (size_t)slot * kGuStage;
            issue_tile<FMT>(st, st + 2 * TB, gqs, gd, is_row0, dm, k0, lane);
            issue_tile<FMT>(st + TB, st + 2 * TB + kScaleBytes, uqs, ud, is_row0, dm, k0, lane);
            if (++is_s == spi) {
                is_s = 0;
                ++is_i;
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int q = 0; q < kGuNSTG - 1; ++q) issue(q, q);

    int staged_chunk = -1;
    int n = 0, pb = 0, ft = 0, s = 0, ci = lo;
    int xoff[kGuG];
    f32x2 ag[2][kGuG], au[2][kGuG];
    for (int q = 0; q < nst; ++q) {
        if (s == 0) {  // a new item: its pairs, and (chunked) its activations
            const int g = ci / ftn;
            ft = ci - g * ftn;
            const int a = locate(g, s_cb, s_n);
            pb = ALLTOK ? s_beg[a] : s_beg[a] + (g - s_cb[a]) * kGuG;
            const int pe = ALLTOK ? s_end[a] : min(s_end[a], pb + kGuG);
            n = pe - pb;
            if (!ALLTOK && g != staged_chunk) {
                for (int j = threadIdx.x; j < n; j += kThreads) s_tok[j] = __ldcg(pair_tok + pb + j);
                __syncthreads();  // also: the previous chunk's x is no longer read
#pragma unroll 4
                for (int e4 = threadIdx.x; e4 < n * d4; e4 += kThreads) {
                    const int j = e4 / d4, qq = e4 - j * d4;
                    const int t = s_tok[j];
                    reinterpret_cast<float4*>(xs)[e4] =
                        (t >= 0 && t < T) ? __ldcg(reinterpret_cast<const float4*>(x) + (size_t)t * d4 + qq)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                __syncthreads();
                staged_chunk = g;
            }
#pragma unroll
            for (int j = 0; j < kGuG; ++j) {
                xoff[j] = (j < n ? (ALLTOK ? s_tok[pb + j] : j) : 0) * dm;
                ag[0][j] = ag[1][j] = 0ull;
                au[0][j] = au[1][j] = 0ull;
            }
        }
        issue(q + kGuNSTG - 1, (q + kGuNSTG - 1) % kGuNSTG);
        cp_async_wait<kGuNSTG - 1>();
        __syncwarp();
        {
            const unsigned char* st = ring + (size_t)(q % kGuNSTG) * kGuStage;
            const float* xk = xs + warp * kw + s * kRowsKS;
#define MOE_GU_STAGE(NT) gu_stage<NT, FMT>(st, lane, xk, xoff, ag, au)
            MOE_GU_SWITCH(n, MOE_GU_STAGE)
#undef MOE_GU_STAGE
        }
        __syncwarp();  // every lane done with this stage before it is refilled
        if (s == spi - 1) {  // item complete: add the warps' K slices in order
#pragma unroll
            for (int j = 0; j < kGuG; ++j) {
                if (j < n) {
                    part[((warp * kGuG + j) * 2 + 0) * 32 + lane] = f2_sum(f2_add(ag[0][j], ag[1][j]));
                    part[((warp * kGuG + j) * 2 + 1) * 32 + lane] = f2_sum(f2_add(au[0][j], au[1][j]));
                }
            }
            __syncthreads();
            {
                const int j = threadIdx.x >> 5, r = threadIdx.x & 31;
                if (j < n) {
                    float gs = 0.f, us = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < kGuNW; ++w2) {
                        gs += part[((w2 * kGuG + j) * 2 + 0) * 32 + r];
                        us += part[((w2 * kGuG + j) * 2 + 1) * 32 + r];
                    }
                    h[(size_t)(pb + j) * f + ft * kRowsFT + r] = silu_f(gs) * us;
                }
            }
            __syncthreads();  // partials read before the next item writes them
        }
        if (++s == spi) {
            s = 0;
            ++ci;
        }
    }
    cp_async_wait<0>();
}

// --------------------------------------------------------------------- down
// Items: (bucket chunk g, output tile ot) with d_model/32 tiles per chunk.
// NW warps split K = d_ff (NW * 64 | d_ff), SPI = d_ff / (NW * 64).  The
// chunk's h rows, tokens and routing weights are staged per chunk.
template <int NW, int FMT>
__global__ void __launch_bounds__(NW * 32, kDnCtasPerSm) down_rows_kernel(
    const float* __restrict__ h, int T, int f, int dm, int E, int k, const int8_t* __restrict__ dqs,
    const uint16_t* __restrict__ dd, const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok,
    const int32_t* __restrict__ pair_slot, const float* __restrict__ wts, int fuse, float* __restrict__ out,
    const int32_t* __restrict__ eslot, int nslots) {
    extern __shared__ __align__(128) unsigned char dr_smem[];
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    __shared__ int s_tok[kRowsG];
    __shared__ float s_w[kRowsG];
    constexpr int kThreads = NW * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int f4 = f / 4;
    const int kw = f / NW, spi = kw / kRowsKS;
    const int otn = dm / kRowsFT;
    constexpr int kDnStage = RowsFmt<FMT>::kDnStage;
    unsigned char* ring = dr_smem + (size_t)warp * kRowsNSTG * kDnStage;
    float* hs = reinterpret_cast<float*>(dr_smem + (size_t)NW * kRowsNSTG * kDnStage);  // [8][f]
    float* part = hs + (size_t)kRowsG * f;                                             // [NW][8][32]

    // Offsets were complete before gate/up released this grid: Wd streams at once.
    if (warp == 0) build_active(offsets, E, kRowsG, T * k, s_act, s_beg, s_end, s_cb, &s_n, eslot, nslots);
    __syncthreads();
    int lo, hi;
    item_range(s_cb[s_n] * otn, &lo, &hi);
    const int nst = (hi - lo) * spi;

    int is_i = lo, is_s = 0, is_g = -1, is_a = 0;
    size_t is_row0 = 0;
    auto issue = [&](int q, int slot) {
        if (q < nst) {
            if (is_s == 0) {
                const int g = is_i / otn;
                if (g != is_g) {
                    is_g = g;
                    is_a = locate(g, s_cb, s_n);
                }
                is_row0 = (size_t)s_act[is_a] * dm + (size_t)(is_i - g * otn) * kRowsFT;
            }
            unsigned char* st = ring + (size_t)slot * kDnStage;
            issue_tile<FMT>(st, st + RowsFmt<FMT>::kTileBytes, dqs, dd, is_row0, f, warp * kw + is_s * kRowsKS, lane);
            if (++is_s == spi) {
                is_s = 0;
                ++is_i;
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int q = 0; q < kRowsNSTG - 1; ++q) issue(q, q);
    pdl_wait();  // gate/up complete: h and the combine target are ready
    pdl_launch_dependents();

    int staged_chunk = -1;
    int n = 0, pb = 0, ot = 0, s = 0, ci = lo;
    f32x2 acc[2][kRowsG];
    for (int q = 0; q < nst; ++q) {
        if (s == 0) {
            const int g = ci / otn;
            ot = ci - g * otn;
            const int a = locate(g, s_cb, s_n);
            pb = s_beg[a] + (g - s_cb[a]) * kRowsG;
            n = min(s_end[a], pb + kRowsG) - pb;
            if (g != staged_chunk) {
                __syncthreads();  // the previous chunk's h is no longer read
#pragma unroll 4
                for (int e4 = threadIdx.x; e4 < n * f4; e4 += kThreads)
                    reinterpret_cast<float4*>(hs)[e4] = __ldcg(reinterpret_cast<const float4*>(h) + (size_t)pb * f4 + e4);
                for (int j = threadIdx.x; j < n; j += kThreads) {
                    const int tok = __ldcg(pair_tok + pb + j), sl = __ldcg(pair_slot + pb + j);
                    const bool ok = tok >= 0 && tok < T && sl >= 0 && sl < k;
                    s_tok[j] = ok ? tok : -1;
                    s_w[j] = ok ? __ldcg(wts + (size_t)tok * k + sl) : 0.f;
                }
                __syncthreads();
                staged_chunk = g;
            }
#pragma unroll
            for (int j = 0; j < kRowsG; ++j) acc[0][j] = acc[1][j] = 0ull;
        }
        issue(q + kRowsNSTG - 1, (q + kRowsNSTG - 1) % kRowsNSTG);
        cp_async_wait<kRowsNSTG - 1>();
        __syncwarp();
        {
            const unsigned char* st = ring + (size_t)(q % kRowsNSTG) * kDnStage;
            const float* hk = hs + warp * kw + s * kRowsKS;
#define MOE_DN_STAGE(NT) dn_stage<NT, FMT>(st, lane, hk, f, acc)
            MOE_ROWS_SWITCH(n, MOE_DN_STAGE)
#undef MOE_DN_STAGE
        }
        __syncwarp();
        if (s == spi - 1) {
#pragma unroll
            for (int j = 0; j < kRowsG; ++j)
                if (j < n) part[(warp * kRowsG + j) * 32 + lane] = f2_sum(f2_add(acc[0][j], acc[1][j]));
            __syncthreads();
            for (int t2 = threadIdx.x; t2 < n * 32; t2 += kThreads) {
                const int j = t2 >> 5, r = t2 & 31;
                float y = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2) y += part[(w2 * kRowsG + j) * 32 + r];
                const int o = ot * kRowsFT + r;
                if (fuse) {
                    if (s_tok[j] >= 0) atomicAdd(out + (size_t)s_tok[j] * dm + o, s_w[j] * y);
                } else {
                    out[(size_t)(pb + j) * dm + o] = y;
                }
            }
            __syncthreads();
        }
        if (++s == spi) {
            s = 0;
            ++ci;
        }
    }
    cp_async_wait<0>();
}

int rows_num_sms() {
    static std::atomic<int> cached[64];  // zero-initialised; racing first calls store the same value
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    int c = cached[dev].load(std::memory_order_relaxed);
    if (!c) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        c = n > 0 ? n : 148;
        cached[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

template <typename K, typename... Args>
cudaError_t launch_rows(K kern, int threads, size_t smem, int ctas_per_sm, cudaStream_t s, Args... args) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows_num_sms() * ctas_per_sm, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Warps of the down kernel: K = d_ff split into kDnNW slices of whole 64-wide stages.
int down_rows_warps(int f) { return f % (kDnNW * kRowsKS) == 0 ? kDnNW : 0; }

size_t gateup_rows_smem(int dm, int fmt) {
    const size_t stage = fmt ? RowsFmt<1>::kGuStage : RowsFmt<0>::kGuStage;
    return (size_t)kGuNW * kGuNSTG * stage + (size_t)kGuG * dm * 4 + (size_t)kGuNW * kGuG * 2 * 32 * 4;
}

size_t down_rows_smem(int f, int nw, int fmt) {
    const size_t stage = fmt ? RowsFmt<1>::kDnStage : RowsFmt<0>::kDnStage;
    return (size_t)nw * kRowsNSTG * stage + (size_t)kRowsG * f * 4 + (size_t)nw * kRowsG * 32 * 4;
}

constexpr size_t kRowsSmemCap = 220 * 1024;

}  // namespace

// Q8_0 from 3 tokens on (1-2 tokens stream faster with a warp per row);
// Q4_0 for every T, these being its only kernels.
bool ffn_rows_supported(const moe_layer_w& w, int T) {
    if (w.wfmt != MOE_WFMT_Q8_0 && w.wfmt != MOE_WFMT_Q4_0) return false;
    if (T < 3 && w.wfmt == MOE_WFMT_Q8_0) return false;
    if (w.d_model % (kGuNW * kRowsKS) != 0 || w.d_ff % kRowsFT != 0 || w.d_model % kRowsFT != 0) return false;
    const int nw = down_rows_warps(w.d_ff);
    return nw != 0 && gateup_rows_smem(w.d_model, w.wfmt) <= kRowsSmemCap &&
           down_rows_smem(w.d_ff, nw, w.wfmt) <= kRowsSmemCap;
}

cudaError_t launch_ffn_rows(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                            const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                            float* out_or_ypairs, int residual, float* h, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int P = T * w.k;
    float* out_init = fuse_combine ? out_or_ypairs : nullptr;
    const bool alltok = T <= kGuG && P <= kMaxStagedPairs;
    const int fmt = w.wfmt;
    const size_t gsm = gateup_rows_smem(w.d_model, fmt);
#define MOE_GU_ROWS(AT, FM)                                                                                       \
    launch_rows(gateup_rows_kernel<AT, FM>, kGuNW * 32, gsm, kGuCtasPerSm, s, x, T, w.d_model, w.d_ff, w.E,       \
                w.gate.qs, w.gate.d,                                                                             \
                w.up.qs, w.up.d, offsets, pair_tok, h, out_init, residual, P, w.expert_slot, weight_slots(w))
    cudaError_t err = fmt ? (alltok ? MOE_GU_ROWS(true, 1) : MOE_GU_ROWS(false, 1))
                          : (alltok ? MOE_GU_ROWS(true, 0) : MOE_GU_ROWS(false, 0));
#undef MOE_GU_ROWS
    if (err != cudaSuccess) return err;
    const int nw = down_rows_warps(w.d_ff);
    const size_t dsm = down_rows_smem(w.d_ff, nw, fmt);
#define MOE_DOWN_ROWS(FM)                                                                                          \
    launch_rows(down_rows_kernel<kDnNW, FM>, kDnNW * 32, dsm, kDnCtasPerSm, s, h, T, w.d_ff, w.d_model, w.E, w.k,  \
                w.down.qs, w.down.d, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, w.expert_slot, \
                weight_slots(w))
    return fmt ? MOE_DOWN_ROWS(1) : MOE_DOWN_ROWS(0);
#undef MOE_DOWN_ROWS
#undef MOE_ROWS_SWITCH
}

}  // namespace moe
