// The whole MoE layer for one or two decode tokens in ONE cooperative launch
// with a single grid-wide exchange: router GEMV -> top-k -> bucketing ->
// gate/up + SwiGLU -> down + weighted combine, Q8_0 or Q4_0 experts ("router ->
// resident expert -> combine -> next layer", amalgafy.com/technical-overview,
// "Warm target path").
//
// At T = 1 a layer moves ~41 MB; beyond streaming it, time goes to the steps
// where every SM must learn something from every other SM.  Here there is
// exactly one such step, the routing:
//
//   1. CTA b computes router logit b (its 8 KB router row is bulk-copied into
//      shared memory at launch) and publishes it as one 64-bit word tagged
//      with this launch, after initialising its slice of the output
//      (out = residual ? x : 0); a CTA without a router row publishes a
//      tagged word with no logit (its presence).  Every CTA reads all the
//      words until each carries its tag -- the logits arrive with them --
//      then ranks the logits itself (top-k, weights, active experts).  The
//      tag is a launch counter in the workspace, read by every CTA once the
//      previous kernel in the stream has completed and bumped by CTA 0 once
//      every word is in (so every CTA has read it): nothing needs clearing
//      between launches, and words of earlier launches carry other tags
//      whatever the workspace held.
//   2. The routed (expert, feature) units are cut into equal 16-aligned
//      ranges, one per CTA; the producer warp derives the active experts
//      and its CTA's range straight from the ranks and starts the weight
//      stream while the other warps finish the weights and the bucketing.
//      A CTA streams the gate and up rows of its
//      features (1-D bulk copies; h = silu(g) * u kept in shared memory) and
//      then the down-projection COLUMNS of the same features (2-D TMA boxes
//      of Wd rows x the CTA's columns, with their scales): the down
//      projection is split along K, so no CTA needs another CTA's h.
//   3. Each CTA adds its partial outputs w * Wd[:, its features] h into out
//      with vector fp32 atomics (out was initialised during step 1, which
//      every CTA has passed).
//
// Every wait is bounded (2 s, then MOE_STATUS_TIMEOUT and invalid outputs).
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "pipeline.cuh"
#include "route_warp.cuh"
#include "stream_common.cuh"
#include "tc.cuh"

namespace moe {

namespace {

using namespace stream;

constexpr int kSpNW = 16;                     // compute warps
constexpr int kSpThreads = (kSpNW + 1) * 32;  // + one producer warp
constexpr int kSpStage = 52224;               // ring stage bytes: 12 gate/up features at d_model 2048
constexpr int kSpNST = 3;                     // ring stages
constexpr int kSpBoxScCols = 16;              // down scale box: fp16 scales per row
constexpr int kSpMaxChunks = 9;               // down window: 16-column chunks (box width 16 * odd)
constexpr int kSpWin = kSpMaxChunks * 16;     // h window per segment
constexpr int kSpMaxT = 2;                    // tokens (the word layout below assumes at most two)
constexpr int kSpMaxP = kSpMaxT * 16;         // pairs: one warp's lanes hold them
constexpr int kSpMaxRows = 2;                 // router rows per CTA (E <= 2 * grid)
constexpr int kSpRankSplit = 4;               // threads per top-k candidate (at most)
constexpr int kSpMaxGrid = 1024;              // CTAs (SMs) a launch may use: presence words in the workspace
constexpr bool kSpEarlyRows = false;          // router rows copied before griddepcontrol.wait

struct SplitParams {
    const float* x;
    int T, dm, f, E, k, residual;
    int W;                        // down box width in bytes (16 * odd, >= every CTA's range)
    int BR;                       // down box rows (a multiple of 32)
    int BRB;                      // rows of one TMA box (BR / BRB boxes per stage; TMA boxes have <= 256 rows)
    int fcap;                     // gate/up features per ring stage
    int ndn;                      // down boxes per segment (d_model / BR)
    // ceil(2^40 / n) for n = d_ff, fcap and 16 * grid: fast_div() divides by
    // them exactly (the serial scheduling step has no integer divisions)
    unsigned long long m_f, m_fcap, m_g16;
    const float* Wr;
    const float* bias;
    const int8_t* gqs;
    const uint16_t* gd;
    const int8_t* uqs;
    const uint16_t* ud;
    float* out;                   // [T][dm]
    unsigned long long* lgw;      // [T][max(E, grid)] words: launch tag << 32 | logit bits (slot e: expert e;
                                  // slots >= E of token 0: presence words of the CTAs without a router row)
    unsigned int* epoch;          // launch counter (workspace; any start value), its value is this launch's tag
    int32_t* idx_out;             // [T][k] or null
    float* wts_out;               // [T][k] or null
    int32_t* offsets_out;         // [E+1] or null
    int32_t* status;
};

// One expert's share of a CTA's range: features [r0, r1) of expert e (16-
// aligned), the CTA-local index of its first feature, its first stage and
// its gate/up stage count.
struct SpSeg {
    int e, a, r0, r1, nch, local0, sbase, ngu;  // a: index of e among the active experts
    float w[kSpMaxT];  // routing weight of each token for this expert (0 if not routed)
};

// Wait for a ring barrier phase, suspended (no issue slots taken) between
// tries; gives up (false) on the 2 s deadline or when another warp has
// already given up (checked every 20 us at most).
__device__ __forceinline__ bool sp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;  // suspended, not spinning
        if (*abort_flag || global_ns() - t0 > kWaitDeadlineNs) return false;
    }
}

// acc[t] += (16 weights (u - c0) * d, exactly) . x_t for 16 unsigned bytes u
// (four words), the weights dequantised four at a time and used at once (few
// live registers): u goes into the mantissa of 2^15 and one fma with
// c = -(2^15 + c0) d gives (u - c0) d exactly (see dequant16; Q8_0: u = q +
// 128, c0 = 128; Q4_0: u = the nibble, c0 = 8).  xt[t][m * st] is the float4
// of x_t matching word m.  acc[t][0] collects the even pairs of every chunk,
// acc[t][1] the odd pairs.
template <int TT>
__device__ __forceinline__ void chunk_fma_u(const uint32_t (&words)[4], float d, float c0,
                                            const float4* const (&xt)[TT], int st, f32x2 (&acc)[TT][2]) {
    const f32x2 dd = f2_pack(d, d);
    const float c = -(32768.0f + c0) * d;
    const f32x2 cc = f2_pack(c, c);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t u = words[m];
        const f32x2 w01 = f2_fma(f2_pack(__uint_as_float(__byte_perm(u, 0x47000000u, 0x7504)),
                                         __uint_as_float(__byte_perm(u, 0x47000000u, 0x7514))),
                                 dd, cc);
        const f32x2 w23 = f2_fma(f2_pack(__uint_as_float(__byte_perm(u, 0x47000000u, 0x7524)),
                                         __uint_as_float(__byte_perm(u, 0x47000000u, 0x7534))),
                                 dd, cc);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const float4 xv = xt[t][m * st];
            acc[t][0] = f2_fma(w01, f2_pack(xv.x, xv.y), acc[t][0]);
            acc[t][1] = f2_fma(w23, f2_pack(xv.z, xv.w), acc[t][1]);
        }
    }
}

// Q8_0: one 16-byte chunk of 16 values (device layout: bytes u = q + 128).
template <int TT>
__device__ __forceinline__ void chunk_fma(const uint4 q, float d, const float4* const (&xt)[TT], int st,
                                          f32x2 (&acc)[TT][2]) {
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};  // bytes u = q + 128 (device layout)
    chunk_fma_u<TT>(u, d, 128.0f, xt, st, acc);
}

// Q4_0: the low (half 0: block values 0..15) or high (half 1: values 16..31)
// nibbles of one 16-byte block.
template <int TT>
__device__ __forceinline__ void chunk_fma_q4(const uint4 q, int half, float d, const float4* const (&xt)[TT], int st,
                                             f32x2 (&acc)[TT][2]) {
    const int sh = 4 * half;
    const uint32_t u[4] = {(q.x >> sh) & 0x0F0F0F0Fu, (q.y >> sh) & 0x0F0F0F0Fu, (q.z >> sh) & 0x0F0F0F0Fu,
                           (q.w >> sh) & 0x0F0F0F0Fu};
    chunk_fma_u<TT>(u, d, 8.0f, xt, st, acc);
}

// x / n for 0 <= x < 2^24 and m = ceil(2^40 / n): with m n = 2^40 + e,
// 0 <= e < n, x m / 2^40 = x / n + x e / (n 2^40) and x e < 2^40, so the
// floor is exact.
__device__ __forceinline__ int fast_div(int x, unsigned long long m) {
    return (int)(((unsigned long long)(unsigned)x * m) >> 40);
}
unsigned long long fast_div_magic(unsigned n) { return ((1ull << 40) + n - 1) / n; }

__device__ __forceinline__ void red_add_v4(float* addr, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

// FMT 0: Q8_0 (a weight row of K values is K bytes); FMT 1: Q4_0 (K / 2
// bytes: 16-byte blocks of 32 values, low nibbles the first 16).
template <int KG, int TT, int FMT>
__global__ void __launch_bounds__(kSpThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dd,
                        SplitParams p) {
    extern __shared__ __align__(1024) unsigned char sp_smem_raw[];
    __shared__ __align__(8) uint64_t full[kSpNST], empty[kSpNST], h_ready[2], rbar;
    __shared__ __align__(16) float s_lg[kSpMaxT][MOE_MAX_EXPERTS];
    __shared__ int s_rank[kSpRankSplit][kSpMaxT * MOE_MAX_EXPERTS];
    __shared__ float s_red[kSpMaxRows][kSpMaxT][kSpNW];
    __shared__ int s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];  // pair range of active expert a
    __shared__ int s_pact[MOE_MAX_EXPERTS];  // active experts in id order (the producer warp's list)
    __shared__ int32_t s_idx[kSpMaxP];
    __shared__ float s_val[kSpMaxP];
    __shared__ int32_t s_ptok[kSpMaxP];
    __shared__ float s_pw[kSpMaxP];
    __shared__ SpSeg s_seg[2];
    __shared__ int s_nst, s_nseg;
    __shared__ volatile int s_abort;
    __shared__ uint32_t s_tag;

    constexpr int kXTok4 = KG * 4 * 32;  // float4 per staged token
    constexpr int kCF4 = FMT ? 8 : 4;    // float4 of x per 16-byte weight chunk (one lane's share)
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(sp_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* ring = smem;                                              // [kSpNST][kSpStage]
    float4* xs = reinterpret_cast<float4*>(ring + kSpNST * kSpStage);         // [TT][kXTok4] chunk layout
    float* ys = reinterpret_cast<float*>(xs + TT * kXTok4);                  // [TT][dm] partial outputs
    float* hw = ys + TT * p.dm;                                             // [2][TT][kSpWin]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.T, dm = p.dm, f = p.f, E = p.E, k = p.k;
    const int P = T * k, d4 = dm / 4;
    const int W = p.W, BR = p.BR;
    const int G = gridDim.x;
    // 0. this CTA's router rows (e = blockIdx.x + G * j) start streaming into
    //    the (still idle) ring at once: they do not depend on the previous
    //    kernel, so the copy overlaps its tail (this kernel is launched as a
    //    programmatic dependent: its CTAs start as the previous kernel's
    //    leave) and the staging of x
    const int nrows = blockIdx.x < E ? (E - blockIdx.x + G - 1) / G : 0;
    auto issue_rows = [&]() {
        mbar_arrive_expect_tx(&rbar, (uint32_t)nrows * dm * 4);
        for (int j = 0; j < nrows; ++j)
            bulk_g2s(ring + (size_t)j * dm * 4, p.Wr + (size_t)(blockIdx.x + G * j) * dm, dm * 4, &rbar);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSpNST; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kSpNW);
        }
        mbar_init(h_ready + 0, kSpNW);
        mbar_init(h_ready + 1, kSpNW);
        mbar_init(&rbar, 1);
        s_abort = 0;
        fence_barrier_init();
        if (kSpEarlyRows) issue_rows();
    }
    if (warp == kSpNW && lane == 0) {
        prefetch_tmap(&tm_dq);
        prefetch_tmap(&tm_dd);
    }
    for (int i = threadIdx.x; i < TT * dm; i += kSpThreads) ys[i] = 0.f;
    for (int i = threadIdx.x; i < 2 * TT * kSpWin; i += kSpThreads) hw[i] = 0.f;
    pdl_wait();  // x (the previous layer's output) and the workspace are ready
    // this launch's tag: the launch counter (bumped below once every CTA has
    // read it), made odd so that zeroed memory never carries it.  Read only
    // after the previous kernel is complete: a previous launch of this kernel
    // on the same workspace bumps it, and this launch may start while that
    // one's last CTAs still run (programmatic dependent launch).
    if (threadIdx.x == 0) {
        s_tag = (__ldcg(p.epoch) << 1) | 1u;
        if (!kSpEarlyRows) issue_rows();
    }
    for (int i = threadIdx.x; i < TT * d4; i += kSpThreads) {
        const int t = i >= d4, q = i - t * d4;  // T <= 2
        xs[t * kXTok4 + stage_idx<32, kCF4>(q)] =
            t < T ? __ldcg(reinterpret_cast<const float4*>(p.x) + (size_t)t * d4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    // 1. the CTAs with a router row initialise out = residual ? x : 0, one
    //    slice each, from the staged x: warp 0 alone writes it and every one
    //    of its lanes fences at once, while the other warps (the producer
    //    warp included) compute the router logits of the CTA's rows (threads
    //    split K).  Warp 0 then publishes the logits -- whoever sees them
    //    sees the initialised slice -- and reads every CTA's words until all
    //    carry this launch's tag, the logits with them.
    const int npub = E < G ? E : G;
    if (warp == 0) {
        if (blockIdx.x < npub) {
            const int n4 = T * d4, per = (n4 + npub - 1) / npub;
            for (int i = blockIdx.x * per + lane; i < min(n4, (blockIdx.x + 1) * per); i += 32) {
                const int t = i >= d4, q = i - t * d4;  // T <= 2
                reinterpret_cast<float4*>(p.out)[i] =
                    p.residual ? xs[t * kXTok4 + stage_idx<32, kCF4>(q)] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        __threadfence();  // every lane: its slice of out is visible before any word of this CTA
    } else if (nrows > 0) {
        if (!sp_wait(&rbar, 0, &s_abort)) {
            if (threadIdx.x == 32) {
                flag_status(p.status, MOE_STATUS_TIMEOUT_BIT);
                s_abort = 1;
            }
        }
        const int gw = warp - 1;  // 0 .. kSpNW - 1 (warps 1 .. kSpNW, the producer warp last)
        for (int j = 0; j < nrows; ++j) {
            const float4* wr = reinterpret_cast<const float4*>(ring) + (size_t)j * d4;
            float acc[TT];
#pragma unroll
            for (int t = 0; t < TT; ++t) acc[t] = 0.f;
            for (int q = threadIdx.x - 32; q < d4; q += kSpNW * 32) {
                const float4 w4 = wr[q];
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    const float4 xv = xs[t * kXTok4 + stage_idx<32, kCF4>(q)];
                    acc[t] = fmaf(w4.x, xv.x, fmaf(w4.y, xv.y, fmaf(w4.z, xv.z, fmaf(w4.w, xv.w, acc[t]))));
                }
            }
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                const float sw = warp_sum(acc[t]);
                if (lane == 0) s_red[j][t][gw] = sw;
            }
        }
    }
    __syncthreads();  // partial sums in
    const int NW = E > G ? E : G;  // word slots per token
    if (warp == 0) {
        const uint32_t tag = s_tag;
        float v = 0.f;
        const bool pub = lane < nrows * T;
        if (pub) {
            const int j = T == 2 ? lane >> 1 : lane, t = lane - j * T;
            for (int w2 = 0; w2 < kSpNW; ++w2) v += s_red[j][t][w2];  // fixed order
            v += p.bias ? __ldg(p.bias + blockIdx.x + G * j) : 0.f;
        }
        if (pub) {
            const int j = T == 2 ? lane >> 1 : lane, t = lane - j * T;
            const unsigned long long word = ((unsigned long long)tag << 32) | __float_as_uint(v);
            asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p.lgw + (size_t)t * NW + blockIdx.x + G * j),
                         "l"(word)
                         : "memory");
        } else if (nrows == 0 && lane == 0) {
            asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p.lgw + blockIdx.x),
                         "l"((unsigned long long)tag << 32)
                         : "memory");
        }
        // token 0: all NW slots (logits, then presence words); tokens >= 1:
        // the E logit slots.  A word carrying this launch's tag holds this
        // launch's logit, so each is stored as soon as it is seen.
        // (T <= 2: word i is slot i of token 0 for i < NW, else slot i - NW of
        // token 1; either way lgw[i].)  Each pass issues a batch of loads
        // before it looks at any of them: one round trip per batch, not one
        // per word.
        const int nwords = NW + (T - 1) * E;
        constexpr int kB = 8;  // words per lane per batch
        const unsigned long long t0 = global_ns();
        for (uint32_t it = 0;; ++it) {
            bool mine = true;
            for (int base = 0; base < nwords; base += 32 * kB) {
                unsigned long long w[kB];
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    const int i = base + 32 * u + lane;
                    w[u] = 0ull;  // tag 0 is never a launch's tag (tags are odd)
                    if (i < nwords)
                        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];"
                                     : "=l"(w[u])
                                     : "l"(p.lgw + i)
                                     : "memory");
                }
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    const int i = base + 32 * u + lane;
                    if (i < nwords) {
                        const int t = i < NW ? 0 : 1, e = i < NW ? i : i - NW;
                        const bool ok = (uint32_t)(w[u] >> 32) == tag;
                        if (ok && e < E) {
                            const float lv = __uint_as_float((uint32_t)w[u]);
                            s_lg[t][e] = lv != lv ? -INFINITY : lv;
                        }
                        mine = mine && ok;
                    }
                }
            }
            if (__all_sync(0xffffffffu, mine)) break;
            __nanosleep(128);  // back off: every CTA polls the same few lines
            if (s_abort || ((it & 15u) == 15u && global_ns() - t0 > kWaitDeadlineNs)) {
                if (lane == 0) {
                    flag_status(p.status, MOE_STATUS_TIMEOUT_BIT);
                    s_abort = 1;
                }
                break;
            }
        }
        __threadfence();  // acquire side: every CTA's out initialisation is visible from here on
        if (blockIdx.x == 0 && lane == 0) __stcg(p.epoch, (tag >> 1) + 1u);
    }
    __syncthreads();
    pdl_launch_dependents();

    // 2. top-k by every CTA.  Rank of candidate (t, e) = #{e2 : l > l_e} +
    //    #{e2 < e : l == l_e}, a permutation (ties to the lower id); each
    //    candidate's scan is split over S threads whose partial counts are
    //    summed in a fixed order.
    // (no integer division on this serial path: T <= 2, S <= 4)
    const int nc = T * E;
    const int S = 4 * nc <= kSpThreads ? 4 : 3 * nc <= kSpThreads ? 3 : 2 * nc <= kSpThreads ? 2 : 1;
    static_assert(kSpRankSplit == 4, "split cases below");
    const int per = S == 4 ? (E + 3) >> 2 : S == 3 ? (E + 2) / 3 : S == 2 ? (E + 1) >> 1 : E;
    const int span = (per + 3) & ~3;  // a multiple of 4 (vector loads)
    for (int id = threadIdx.x; id < nc * S; id += kSpThreads) {
        const int part = (id >= nc) + (id >= 2 * nc) + (id >= 3 * nc);
        const int c = id - part * nc;
        const int t = c >= E, e = c - t * E;
        const float* row = s_lg[t];
        const float v = row[e];
        const int e0 = part * span, e1 = min(E, e0 + span);
        int r = 0;
        if (e1 - e0 == 32 && (e0 & 3) == 0) {  // E = 128 split four ways: eight vector loads, all in flight
            int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
            float4 l[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) l[i] = *reinterpret_cast<const float4*>(row + e0 + 4 * i);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e2 = e0 + 4 * i;
                r0 += (l[i].x > v) | ((l[i].x == v) & (e2 < e));
                r1 += (l[i].y > v) | ((l[i].y == v) & (e2 + 1 < e));
                r2 += (l[i].z > v) | ((l[i].z == v) & (e2 + 2 < e));
                r3 += (l[i].w > v) | ((l[i].w == v) & (e2 + 3 < e));
            }
            r = (r0 + r1) + (r2 + r3);
        } else if (((e0 | e1) & 3) == 0) {  // 16-byte aligned run: vector loads (a broadcast per warp)
            int r0 = 0, r1 = 0, r2 = 0, r3 = 0;  // four independent counts
#pragma unroll 4
            for (int e2 = e0; e2 < e1; e2 += 4) {
                const float4 l4 = *reinterpret_cast<const float4*>(row + e2);
                r0 += (l4.x > v) | ((l4.x == v) & (e2 < e));
                r1 += (l4.y > v) | ((l4.y == v) & (e2 + 1 < e));
                r2 += (l4.z > v) | ((l4.z == v) & (e2 + 2 < e));
                r3 += (l4.w > v) | ((l4.w == v) & (e2 + 3 < e));
            }
            r = (r0 + r1) + (r2 + r3);
        } else {
#pragma unroll 8
            for (int e2 = e0; e2 < e1; ++e2) {
                const float l2 = row[e2];
                r += (l2 > v) | ((l2 == v) & (e2 < e));
            }
        }
        s_rank[part][c] = r;
    }
    __syncthreads();
    const int rowb = FMT ? dm / 2 : dm;  // bytes of one gate / up weight row
    const int fcap = p.fcap, ndn = p.ndn;
    // stage s -> (segment, kind, index within its kind); valid once the
    // producer warp has published the schedule
    auto stage_of = [&](int s, int& seg, int& kind, int& i) {
        seg = (s_nseg > 1 && s >= s_seg[1].sbase) ? 1 : 0;
        i = s - s_seg[seg].sbase;
        kind = i >= s_seg[seg].ngu;
        if (kind) i -= s_seg[seg].ngu;
    };

    if (warp == kSpNW) {
        // ------------------------------------------------------------ producer
        // 3. the active experts in id order straight from the ranks (expert
        //    e is active if some token ranks it below k), this CTA's range of
        //    (active expert, feature) units -- equal ranges of a multiple of
        //    16 features, at most two experts -- and its stage list: seg 0
        //    gate/up, seg 0 down boxes, seg 1 gate/up, seg 1 down boxes.  The
        //    schedule goes to the compute warps through named barrier 1 and
        //    the stream starts at once; the routing weights, the bucketing and
        //    the outputs for the caller are left to the compute warps.
        // (every rank load of the scan issued before any is used: one
        // shared-memory round trip, not one per load)
        constexpr int kJ = MOE_MAX_EXPERTS / 32;
        bool selj[kJ];
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const int e = 32 * j + lane;
            int r[kSpMaxT][kSpRankSplit];
#pragma unroll
            for (int t = 0; t < kSpMaxT; ++t)
#pragma unroll
                for (int part = 0; part < kSpRankSplit; ++part)
                    r[t][part] = (e < E && t < T && part < S) ? s_rank[part][t * E + e] : 0;
            bool sel = false;
#pragma unroll
            for (int t = 0; t < kSpMaxT; ++t)
                sel = sel || (e < E && t < T && (r[t][0] + r[t][1]) + (r[t][2] + r[t][3]) < k);
            selj[j] = sel;
        }
        int n = 0;
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const uint32_t m = __ballot_sync(0xffffffffu, selj[j]);
            if (selj[j]) s_pact[n + __popc(m & ((1u << lane) - 1u))] = 32 * j + lane;
            n += __popc(m);
        }
        __syncwarp();
        if (lane == 0) {
            const int F = n * f;
            const int L = 16 * fast_div(F + 16 * G - 1, p.m_g16);
            const int lo = min(F, (int)blockIdx.x * L), hi = min(F, lo + L);
            int ns = 0, nseg = 0, local = 0;
            const int a_hi = fast_div(hi - 1, p.m_f);
            for (int a = fast_div(lo, p.m_f); lo < hi && a <= a_hi && nseg < 2; ++a) {
                SpSeg sg;
                sg.e = s_pact[a];
                sg.a = a;
                sg.r0 = max(lo, a * f) - a * f;
                sg.r1 = min(hi, (a + 1) * f) - a * f;
                sg.nch = (sg.r1 - sg.r0) / 16;
                sg.local0 = local;
                sg.sbase = ns;
                sg.ngu = fast_div(sg.r1 - sg.r0 + fcap - 1, p.m_fcap);
                s_seg[nseg++] = sg;
                local += sg.r1 - sg.r0;
                ns += sg.ngu + ndn;
            }
            s_nst = s_abort ? 0 : ns;
            s_nseg = nseg;
        }
        __syncwarp();
        asm volatile("bar.arrive 1, %0;" ::"r"(kSpThreads) : "memory");
        const int nst = s_nst;
        if (lane == 0) {
            fence_proxy_async_smem();  // the router rows were read through the generic proxy
            int s = 0;
            for (; s < nst && !s_abort; ++s) {
                const int slot = s % kSpNST;
                if (s >= kSpNST && !sp_wait(empty + slot, ((s / kSpNST) - 1) & 1, &s_abort)) {
                    flag_status(p.status, MOE_STATUS_TIMEOUT_BIT);
                    s_abort = 1;
                    break;
                }
                int seg, kind, i;
                stage_of(s, seg, kind, i);
                const SpSeg& sg = s_seg[seg];
                unsigned char* b = ring + (size_t)slot * kSpStage;
                if (kind == 0) {
                    const int r = sg.r0 + i * fcap, nf = min(fcap, sg.r1 - r);
                    const size_t row = (size_t)sg.e * f + r;
                    const uint32_t qb = (uint32_t)nf * rowb, sb = (uint32_t)nf * (dm / 16);
                    mbar_arrive_expect_tx(full + slot, 2 * (qb + sb));
                    bulk_g2s(b, p.gqs + row * rowb, qb, full + slot);
                    bulk_g2s(b + (size_t)fcap * rowb, p.uqs + row * rowb, qb, full + slot);
                    bulk_g2s(b + (size_t)2 * fcap * rowb,
                             reinterpret_cast<const unsigned char*>(p.gd) + row * (dm / 16), sb, full + slot);
                    bulk_g2s(b + (size_t)2 * fcap * rowb + (size_t)fcap * (dm / 16),
                             reinterpret_cast<const unsigned char*>(p.ud) + row * (dm / 16), sb, full + slot);
                } else {
                    const int y = sg.e * dm + i * BR;
                    mbar_arrive_expect_tx(full + slot, BR * (W + 2 * kSpBoxScCols));
                    // the box starts at the byte of the range's first feature
                    // (Q4_0: of the block that holds it, 16-byte aligned)
                    const int bx = FMT ? 16 * (sg.r0 / 32) : sg.r0;
                    for (int r0 = 0; r0 < BR; r0 += p.BRB) {
                        tma_load_2d(b + r0 * W, &tm_dq, bx, y + r0, full + slot);
                        tma_load_2d(b + BR * W + r0 * 2 * kSpBoxScCols, &tm_dd, (sg.r0 / 32) & ~7, y + r0, full + slot);
                    }
                }
            }
            // every copy issued has landed before the CTA moves on
            for (int c = (s > kSpNST ? s - kSpNST : 0); c < s; ++c) mbar_wait(full + c % kSpNST, (c / kSpNST) & 1);
        }
    } else {
        // select, weights, bucketing (the compute warps, 512 threads)
        constexpr int kCT = kSpNW * 32;
        for (int c = threadIdx.x; c < nc; c += kCT) {
            int r = 0;
            for (int part = 0; part < S; ++part) r += s_rank[part][c];
            if (r < k) {
                const int t = c >= E;  // T <= 2
                s_idx[t * k + r] = c - t * E;
                s_val[t * k + r] = s_lg[t][c - t * E];
            }
        }
        named_bar(2, kCT);
        for (int q = warp; q < P; q += kSpNW) {
            const int e = s_idx[q];
            const int e2 = lane < P ? s_idx[lane] : 0x7fffffff;
            const uint32_t lt = __ballot_sync(0xffffffffu, e2 < e);
            const uint32_t eq = __ballot_sync(0xffffffffu, e2 == e);
            const uint32_t eq_before = eq & ((1u << q) - 1u);
            const uint32_t same = __match_any_sync(0xffffffffu, e2);
            const bool lead = lane < P && __ffs(same) - 1 == lane;
            const uint32_t leads_below = __ballot_sync(0xffffffffu, lead && e2 < e);
            const int t = q >= k;  // T <= 2
            const float v0 = s_val[t * k];
            const float den = warp_sum(lane < k ? expf(s_val[t * k + lane] - v0) : 0.0f);
            const float w = expf(s_val[q] - v0) / den;
            if (lane == 0) {
                const int r = __popc(lt) + __popc(eq_before);
                s_ptok[r] = t;
                s_pw[r] = w;
                if (eq_before == 0) {
                    const int a = __popc(leads_below);
                    s_beg[a] = __popc(lt);
                    s_end[a] = __popc(lt) + __popc(eq);
                }
                if (blockIdx.x == 0) {
                    if (p.idx_out) p.idx_out[q] = e;
                    if (p.wts_out) p.wts_out[q] = w;
                }
            }
        }
        if (blockIdx.x == 0 && p.offsets_out) bucket_offsets(s_idx, P, E, kCT, p.offsets_out);
        named_bar(2, kCT);                            // pairs in (s_beg, s_end, s_ptok, s_pw)
        named_bar(1, kSpThreads);                     // the producer's schedule is in
        if (threadIdx.x == 0) {
            for (int sg = 0; sg < s_nseg; ++sg) {
                const int a = s_seg[sg].a;
#pragma unroll
                for (int t = 0; t < kSpMaxT; ++t) {  // a token routes to an expert at most once
                    float wt = 0.f;
                    for (int r = s_beg[a]; r < s_end[a]; ++r)
                        if (s_ptok[r] == t) wt = s_pw[r];
                    s_seg[sg].w[t] = wt;
                }
            }
        }
        named_bar(2, kCT);
        const int nst = s_nst;
        // -------------------------------------------------------------- compute
        // After a timeout (`ok` false) the warp walks the remaining stages
        // without waiting or computing.
        bool ok = true;
        int cur_seg = -1;
        for (int s = 0; s < nst; ++s) {
            int seg, kind, i;
            stage_of(s, seg, kind, i);
            const SpSeg& sg = s_seg[seg];
            if (kind == 1 && seg != cur_seg) {
                // the segment's h is complete once every warp is past its gate/up stages
                ok = ok && sp_wait(h_ready + seg, 0, &s_abort);
                cur_seg = seg;
            }
            const int slot = s % kSpNST;
            const bool was_ok = ok;
            ok = ok && sp_wait(full + slot, (s / kSpNST) & 1, &s_abort);
            const unsigned char* b = ring + (size_t)slot * kSpStage;
            if (kind == 0 && ok) {
                // gate/up: feature j of the stage belongs to warp (local index) % kSpNW,
                // which computes both of its rows over the whole of K
                const int r = sg.r0 + i * fcap, nf = min(fcap, sg.r1 - r);
                const int a2 = sg.local0 + i * fcap;
                const __half* gsc = reinterpret_cast<const __half*>(b + (size_t)2 * fcap * rowb);
                const __half* usc =
                    reinterpret_cast<const __half*>(b + (size_t)2 * fcap * rowb + (size_t)fcap * (dm / 16));
                for (int j = (warp - a2 % kSpNW + kSpNW) % kSpNW; j < nf; j += kSpNW) {
                    const unsigned char* gq = b + (size_t)j * rowb;
                    const unsigned char* uq = b + (size_t)(fcap + j) * rowb;
                    f32x2 accg[TT][2], accu[TT][2];
#pragma unroll
                    for (int t = 0; t < TT; ++t) accg[t][0] = accg[t][1] = accu[t][0] = accu[t][1] = 0ull;
#pragma unroll
                    for (int m = 0; m < (FMT ? KG / 2 : KG); ++m) {
                        // 16-byte chunk c of the row: Q8_0 16 values (block c / 2),
                        // Q4_0 one whole block of 32 (block c)
                        const int c = lane + 32 * m;
                        const uint4 qg = *reinterpret_cast<const uint4*>(gq + c * 16);
                        const uint4 qu = *reinterpret_cast<const uint4*>(uq + c * 16);
                        const int blk = FMT ? c : c >> 1;
                        const float sgv = __half2float(gsc[j * (dm / 32) + blk]);
                        const float suv = __half2float(usc[j * (dm / 32) + blk]);
                        const float4* xt[TT];
#pragma unroll
                        for (int t = 0; t < TT; ++t) xt[t] = xs + t * kXTok4 + m * kCF4 * 32 + lane;
                        if (FMT == 0) {
                            chunk_fma<TT>(qg, sgv, xt, 32, accg);
                            chunk_fma<TT>(qu, suv, xt, 32, accu);
                        } else {
                            const float4* xh[TT];
#pragma unroll
                            for (int t = 0; t < TT; ++t) xh[t] = xt[t] + 4 * 32;
                            chunk_fma_q4<TT>(qg, 0, sgv, xt, 32, accg);
                            chunk_fma_q4<TT>(qg, 1, sgv, xh, 32, accg);
                            chunk_fma_q4<TT>(qu, 0, suv, xt, 32, accu);
                            chunk_fma_q4<TT>(qu, 1, suv, xh, 32, accu);
                        }
                    }
                    float ga[TT], ua[TT];
#pragma unroll
                    for (int t = 0; t < TT; ++t) {
                        ga[t] = f2_sum(f2_add(accg[t][0], accg[t][1]));
                        ua[t] = f2_sum(f2_add(accu[t][0], accu[t][1]));
                    }
#pragma unroll
                    for (int t = 0; t < TT; ++t) {
                        ga[t] = warp_sum(ga[t]);
                        ua[t] = warp_sum(ua[t]);
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int t = 0; t < TT; ++t) hw[(seg * TT + t) * kSpWin + r + j - sg.r0] = silu_f(ga[t]) * ua[t];
                    }
                }
            } else if (ok) {
                // down box: rows [BR i, BR i + BR) of expert e, the CTA's
                // columns; lane = row, 32-row group g belongs to warp g % kSpNW
                const int g0 = i * (BR / 32);
                for (int gl = (warp - g0 % kSpNW + kSpNW) % kSpNW; gl < BR / 32; gl += kSpNW) {
                    const int rl = gl * 32 + lane;
                    const unsigned char* qrow = b + (size_t)rl * W;
                    const __half* sc = reinterpret_cast<const __half*>(b + BR * W) + rl * kSpBoxScCols;
                    const int sx = (sg.r0 / 32) & ~7;
                    const float* hs = hw + seg * TT * kSpWin;
                    f32x2 acc[TT][2];
#pragma unroll
                    for (int t = 0; t < TT; ++t) acc[t][0] = acc[t][1] = 0ull;
#pragma unroll
                    for (int c = 0; c < kSpMaxChunks; ++c) {
                        if (c < sg.nch) {
                            // features f0 .. f0 + 15 of the range (Q4_0: one half
                            // of the block that holds them)
                            const int f0 = sg.r0 + 16 * c;
                            const float4* ht[TT];
#pragma unroll
                            for (int t = 0; t < TT; ++t) ht[t] = reinterpret_cast<const float4*>(hs + t * kSpWin + 16 * c);
                            const float dv = __half2float(sc[f0 / 32 - sx]);
                            if (FMT == 0) {
                                chunk_fma<TT>(*reinterpret_cast<const uint4*>(qrow + 16 * c), dv, ht, 1, acc);
                            } else {
                                const uint4 qv = *reinterpret_cast<const uint4*>(qrow + 16 * (f0 / 32 - sg.r0 / 32));
                                chunk_fma_q4<TT>(qv, (f0 >> 4) & 1, dv, ht, 1, acc);
                            }
                        }
                    }
                    const int o = i * BR + rl;
#pragma unroll
                    for (int t = 0; t < TT; ++t) ys[t * dm + o] += sg.w[t] * f2_sum(f2_add(acc[t][0], acc[t][1]));
                }
            }
            if (!ok) {
                if (was_ok && lane == 0) {
                    flag_status(p.status, MOE_STATUS_TIMEOUT_BIT);
                    s_abort = 1;
                }
                continue;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(empty + slot);
                // after this warp's last gate/up stage of a segment: its h is in
                if (kind == 0 && i + 1 == sg.ngu) mbar_arrive(h_ready + seg);
            }
        }
    }
    __syncthreads();

    // 4. this CTA's partial outputs into out (vector fp32 atomics; out was
    //    initialised before any CTA could pass step 1)
    if (s_nst > 0) {
        for (int i = threadIdx.x; i < T * d4; i += kSpThreads)
            red_add_v4(p.out + 4 * (size_t)i, reinterpret_cast<const float4*>(ys)[i]);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 sp_encode_fn() {
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 f0 = fn.load(std::memory_order_acquire);
    if (!f0) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f0 = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
            fn.store(f0, std::memory_order_release);
        }
        cudaGetLastError();
    }
    return f0;
}

// 2-D row-major map, no swizzle: inner dimension `inner` elements, `rows` rows.
bool sp_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner, uint64_t rows,
             uint32_t bx, uint32_t by) {
    auto fn = sp_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * (uint64_t)esize};
    const cuuint32_t box[2] = {bx, by};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KG, int TT>
size_t sp_smem_bytes(int dm) {
    return 1024 + (size_t)kSpNST * kSpStage + (size_t)TT * KG * 4 * 32 * 16 + (size_t)TT * dm * 4 +
           (size_t)2 * TT * kSpWin * 4;
}

int sp_num_sms() {
    static std::atomic<int> cached[64];  // zero-initialised; racing first calls store the same value
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = cached[dev].load(std::memory_order_relaxed);
    if (!c) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        c = n;
        cached[dev].store(c, std::memory_order_relaxed);
    }
    return c;
}

template <int KG, int TT, int FMT>
cudaError_t launch_split(const SplitParams& p, int dm, int f, const moe_layer_w& w, cudaStream_t s) {
    auto kern = decode_split_kernel<KG, TT, FMT>;
    const size_t smem = sp_smem_bytes<KG, TT>(dm);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSpThreads, smem);
    if (err != cudaSuccess || per_sm < 1) return cudaErrorInvalidConfiguration;
    const int G = sp_num_sms();  // one CTA per SM, all co-resident (cooperative launch)
    if (G < 1 || G > kSpMaxGrid || (w.E + G - 1) / G > kSpMaxRows) return cudaErrorInvalidConfiguration;
    // the widest range a CTA can get (every pair on its own expert); its
    // down box in an odd number of 16-byte chunks so that the lane-per-row
    // reads of a box are free of shared-memory bank conflicts.  Q8_0: a
    // chunk per 16 features; Q4_0: a chunk per 32-feature block the range
    // touches (a 16-aligned range of L features touches at most
    // L / 32 + 1 blocks).  The range must not exceed d_ff (at most two
    // experts per range) nor the h window.
    const long long Fmax = (long long)p.T * p.k * f;
    const int Lmax = (int)(16 * ((Fmax + 16LL * G - 1) / (16LL * G)));
    if (Lmax / 16 > kSpMaxChunks || Lmax > f) return cudaErrorInvalidConfiguration;
    int nch = FMT ? Lmax / 32 + 1 : Lmax / 16;
    if ((nch & 1) == 0) ++nch;
    if (nch > kSpMaxChunks) return cudaErrorInvalidConfiguration;
    SplitParams q = p;
    q.W = 16 * nch;
    // down box rows: the most 32-row groups (at most one per compute warp)
    // that fit a stage and divide d_model; each box is loaded as BR / BRB
    // TMA boxes of BRB <= 256 rows (a multiple of 16: 128-byte aligned)
    const int cap = min(kSpNW, kSpStage / (32 * (q.W + 2 * kSpBoxScCols)));
    if (cap < 1) return cudaErrorInvalidConfiguration;
    q.BR = 32;
    for (int m = cap; m >= 1; --m)
        if (dm % (32 * m) == 0) {
            q.BR = 32 * m;
            break;
        }
    q.BRB = 0;
    for (int n = (q.BR + 255) / 256; n <= q.BR / 16; ++n)
        if (q.BR % n == 0 && (q.BR / n) % 16 == 0) {
            q.BRB = q.BR / n;
            break;
        }
    if (q.BRB == 0) return cudaErrorInvalidConfiguration;
    // gate/up features per stage (Q4_0: a multiple of the compute warps, so
    // that every warp gets the same number of features)
    const int rowb = FMT ? dm / 2 : dm;
    const int fcap0 = kSpStage / (2 * rowb + dm / 8);
    q.fcap = (FMT && fcap0 > kSpNW) ? fcap0 - fcap0 % kSpNW : fcap0;
    q.ndn = dm / q.BR;
    if (q.fcap < 1 || (long long)w.E * f + 16LL * G >= (1LL << 24)) return cudaErrorInvalidConfiguration;
    q.m_f = fast_div_magic((unsigned)f);
    q.m_fcap = fast_div_magic((unsigned)q.fcap);
    q.m_g16 = fast_div_magic(16u * (unsigned)G);
    CUtensorMap tq, td;
    if (!sp_tmap(&tq, w.down.qs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, FMT ? f / 2 : f, (uint64_t)w.E * dm, q.W, q.BRB) ||
        !sp_tmap(&td, w.down.d, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, f / 32, (uint64_t)w.E * dm, kSpBoxScCols, q.BRB))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G, 1, 1);
    cfg.blockDim = dim3(kSpThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // cooperative (every CTA resident: the exchange waits on all of them) and
    // a programmatic dependent of the previous kernel in the stream (its
    // prologue -- barriers, the router row copy -- overlaps that kernel's
    // tail; everything that reads what the previous kernel wrote comes after
    // griddepcontrol.wait).  Where the pair of attributes is refused, the
    // launch is made cooperative only, and that answer is kept.
    static std::atomic<int> pdl_ok{1};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_ok.load(std::memory_order_relaxed) ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tq, td, q);
    if (e != cudaSuccess && cfg.numAttrs == 2 && e != cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();
        pdl_ok.store(0, std::memory_order_relaxed);
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, tq, td, q);
    }
    return e;
}

}  // namespace

size_t decode_split_words(int T, int E) { return (size_t)T * (E > kSpMaxGrid ? E : kSpMaxGrid); }

bool decode_split_supported(const moe_layer_w& w, int T) {
    if ((w.wfmt != MOE_WFMT_Q8_0 && w.wfmt != MOE_WFMT_Q4_0) || w.expert_slot) return false;
    // Q4_0: a lane's 16-byte chunk of a gate/up row holds 32 values, so
    // d_model is a multiple of 1024 (32 lanes x 32)
    const int dmul = w.wfmt == MOE_WFMT_Q4_0 ? 1024 : 512;
    return T >= 1 && T <= kSpMaxT && T * w.k <= kSpMaxP && w.d_model % dmul == 0 && w.d_model <= 2048 &&
           w.d_ff % 256 == 0 && w.d_ff <= 8192 && w.E <= MOE_MAX_EXPERTS && sp_encode_fn() != nullptr;
}

cudaError_t launch_decode_split(const float* x, int T, const moe_layer_w& w, int residual, float* out,
                                int32_t* idx_out, float* wts_out, int32_t* offsets_out, unsigned long long* lgw,
                                unsigned int* epoch, int32_t* status, cudaStream_t s) {
    SplitParams p = {};
    p.x = x;
    p.T = T;
    p.dm = w.d_model;
    p.f = w.d_ff;
    p.E = w.E;
    p.k = w.k;
    p.residual = residual;
    p.Wr = w.router_w;
    p.bias = w.router_bias;
    p.gqs = w.gate.qs;
    p.gd = w.gate.d;
    p.uqs = w.up.qs;
    p.ud = w.up.d;
    p.out = out;
    p.lgw = lgw;
    p.epoch = epoch;
    p.idx_out = idx_out;
    p.wts_out = wts_out;
    p.offsets_out = offsets_out;
    p.status = status;
    const int dm = w.d_model, f = w.d_ff;
#define MOE_SPLIT_GO(KG, FMT)                                                                             \
    return T == 1 ? launch_split<KG, 1, FMT>(p, dm, f, w, s) : launch_split<KG, 2, FMT>(p, dm, f, w, s)
    if (w.wfmt == MOE_WFMT_Q4_0) {
        switch (dm / 512) {
            case 2: MOE_SPLIT_GO(2, 1);
            case 4: MOE_SPLIT_GO(4, 1);
            default: return cudaErrorInvalidConfiguration;
        }
    }
    switch (dm / 512) {
        case 1: MOE_SPLIT_GO(1, 0);
        case 2: MOE_SPLIT_GO(2, 0);
        case 3: MOE_SPLIT_GO(3, 0);
        case 4: MOE_SPLIT_GO(4, 0);
        default: return cudaErrorInvalidConfiguration;
    }
#undef MOE_SPLIT_GO
}

}  // namespace moe
