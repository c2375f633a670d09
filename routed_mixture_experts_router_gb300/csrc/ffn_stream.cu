// Expert SwiGLU FFNs with fp32 activations, streaming design (decode path).
//
//   gate/up  h[p][r] = silu(Wg_e[r] . x[t]) * (Wu_e[r] . x[t])   pair p = (t, slot) in bucket e
//   down     y[p][o] = Wd_e[o] . h[p];  out[t][o] += w[t][slot] * y[p][o]  (combine fused)
// Q8_0 weights w = q * d (amalgafy.com/technical-overview, "Validated GPU
// foundation"); down projection K=768 -> 2048 rows (expxa.com
// reuse-ordering-qualification, "What changed from the first experiment");
// weighted combine ("Execution architecture", amalgafy.com/technical-overview).
//
// HBM-bound design for GB300.  A persistent grid of one CTA per SM walks a
// contiguous range of work items: one output feature (its gate row and up
// row) for gate/up, four rows for down, always of one expert.  Every warp owns
// a private ring of NSTG shared-memory stages and streams its items into it
// with 16-byte asynchronous copies (cp.async.cg: L2 -> shared, no registers),
// NSTG - 1 items ahead of the one it computes, so 100+ KB per SM stay in
// flight -- the bandwidth-latency product GB300's HBM needs.  (A ring fed by
// 1-D bulk copies was measured slower: each bulk copy has a fixed cost that
// small Q8_0 rows cannot amortise.)  The activations of the tokens routed to
// the expert sit in shared memory.  Each weight byte is read from HBM once per
// layer.
//
// Arithmetic: int8 -> fp32 exactly (byte placed in the mantissa of 2^23, then
// 2^23 + 128 subtracted), products and sums in fp32 with Blackwell's paired
// fp32 FMA (fma.rn.f32x2), the fp16 block scale applied once per 16-value half
// block.  The down kernel is a programmatic dependent of gate/up: it starts
// streaming Wd before gate/up finishes and waits only before reading h.
#include "common.cuh"
#include "pipeline.cuh"

namespace moe {

namespace {

constexpr int kMaxStagedPairs = 256;  // pair metadata staged in shared memory
constexpr int kDnRowsPerItem = 4;     // down item: 4 rows, 2 per half-warp

typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float a, float b) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float f2_sum(f32x2 v) {
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
    return a + b;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// One word of four int8 -> (q0, q1), (q2, q3) as exact fp32 pairs.
__device__ __forceinline__ void i8x4_to_f2(uint32_t w, f32x2& lo, f32x2& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const f32x2 bias = 0xCB000080CB000080ull;  // (-(2^23 + 128), -(2^23 + 128))
    lo = f2_add(f2_pack(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)),
                        __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541))),
                bias);
    hi = f2_add(f2_pack(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)),
                        __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543))),
                bias);
}

// sum over 16 values of q * x: one 16-byte weight chunk, four float4 of x at stride `st`.
__device__ __forceinline__ float chunk_dot(const uint4 q, const float4* xv4, int st) {
    f32x2 acc = 0ull;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        f32x2 lo, hi;
        i8x4_to_f2(w[m], lo, hi);
        const float4 xv = xv4[m * st];
        acc = f2_fma(lo, f2_pack(xv.x, xv.y), acc);
        acc = f2_fma(hi, f2_pack(xv.z, xv.w), acc);
    }
    return f2_sum(acc);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared-memory layout of one staged activation vector for LPR lanes that
// split K in 16-value chunks c = hl + LPR*m: float4 j of chunk c sits at
// (m*4 + j)*LPR + hl, so one load instruction reads consecutive float4s.
template <int LPR>
__device__ __forceinline__ int stage_idx(int q) {
    const int c = q >> 2, j = q & 3;
    return ((c / LPR) * 4 + j) * LPR + (c % LPR);
}

// Active experts (non-empty buckets) in id order, by warp 0, and the work
// list they imply: expert a's bucket is cut into chunks of at most `chunk`
// pairs (the activations one pass stages in shared memory); s_cb[a] is the
// index of a's first chunk and s_cb[n] the total.  All offsets are fetched in
// one round trip, through L2 (they were written by an earlier kernel).
__device__ void build_active(const int32_t* offsets, int E, int chunk, int* s_act, int* s_beg, int* s_end,
                             int* s_cb, int* s_n) {
    const int lane = threadIdx.x & 31;
    int lo[MOE_MAX_EXPERTS / 32], hi[MOE_MAX_EXPERTS / 32];
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
        const int e = 32 * j + lane;
        lo[j] = e < E ? __ldcg(offsets + e) : 0;
        hi[j] = e < E ? __ldcg(offsets + e + 1) : 0;
    }
    int n = 0, nc = 0;
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
        const bool a = hi[j] > lo[j];
        const uint32_t m = __ballot_sync(0xffffffffu, a);
        const int my_c = a ? (hi[j] - lo[j] + chunk - 1) / chunk : 0;
        int incl = my_c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (a) {
            const int jj = n + __popc(m & ((1u << lane) - 1u));
            s_act[jj] = 32 * j + lane;
            s_beg[jj] = lo[j];
            s_end[jj] = hi[j];
            s_cb[jj] = nc + incl - my_c;
        }
        n += __popc(m);
        nc += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        *s_n = n;
        s_cb[n] = nc;
    }
}

// Global chunk g -> active expert index a (largest a with s_cb[a] <= g).
__device__ __forceinline__ int locate(int g, const int* s_cb, int n) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_cb[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ void item_range(int n_items, int* lo, int* hi) {
    const long long b = blockIdx.x, G = gridDim.x;
    *lo = (int)(b * n_items / G);
    *hi = (int)((b + 1) * n_items / G);
}

// A warp walks items lo + warp, lo + warp + NW, ... of [lo, hi) that share a
// segment (same bucket chunk).  issue(i, stage) starts the copies of item i
// and commits them; compute(i, stage) runs once they have landed.  NSTG - 1
// items are always in flight ahead of the one being computed.
template <int NSTG, typename Issue, typename Compute>
__device__ __forceinline__ void warp_stream(int first, int end, int step, Issue issue, Compute compute) {
    int n = first < end ? (end - first + step - 1) / step : 0;
#pragma unroll
    for (int j = 0; j < NSTG - 1; ++j) {
        if (j < n) issue(first + j * step, j);
        else cp_async_commit();
    }
    for (int j = 0; j < n; ++j) {
        const int jn = j + NSTG - 1;
        if (jn < n) issue(first + jn * step, jn % NSTG);
        else cp_async_commit();
        cp_async_wait<NSTG - 1>();
        __syncwarp();
        compute(first + j * step, j % NSTG);
        __syncwarp();  // every lane done with this stage before it is refilled
    }
}

// ============================================================== gate / up ==
// One warp per output feature r (its gate row and up row); lanes split
// K = d_model in 16-byte chunks c = lane + 32*m, m < KCH.  G: tokens per
// register block; ALLTOK: every token's x staged once (T small), else per
// bucket chunk of at most tca pairs.
template <int KCH, int G, bool ALLTOK, int NW, int NSTG>
__global__ void __launch_bounds__(NW * 32, 1) gateup_cp_kernel(
    const float* __restrict__ x, int T, int dm, int f, int E, const int8_t* __restrict__ gqs,
    const uint16_t* __restrict__ gd, const int8_t* __restrict__ uqs, const uint16_t* __restrict__ ud,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok, float* __restrict__ h,
    float* __restrict__ out_init, int init_residual, int tca, int P) {
    extern __shared__ __align__(128) unsigned char gu_smem[];
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    __shared__ int s_tok[ALLTOK ? kMaxStagedPairs : 1];
    constexpr int kThreads = NW * 32;
    constexpr int kTok4 = KCH * 4 * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d4 = dm / 4, nch = dm / 16;
    const int item_bytes = 2 * dm + 2 * (dm / 16);  // gate qs, up qs, gate d, up d
    unsigned char* ring = gu_smem + (size_t)warp * NSTG * item_bytes;
    float4* xs = reinterpret_cast<float4*>(gu_smem + (size_t)NW * NSTG * item_bytes);

    pdl_wait();  // routing / bucketing of this layer complete and visible
    if (warp == 0) build_active(offsets, E, ALLTOK ? (1 << 30) : tca, s_act, s_beg, s_end, s_cb, &s_n);
    if (ALLTOK) {
        for (int p = threadIdx.x; p < P; p += kThreads) {
            const int t = __ldcg(pair_tok + p);
            s_tok[p] = (t >= 0 && t < T) ? t : 0;
        }
        for (int i = threadIdx.x; i < T * d4; i += kThreads) {
            const int t = i / d4, q = i - t * d4;
            xs[t * kTok4 + stage_idx<32>(q)] = __ldcg(reinterpret_cast<const float4*>(x) + (size_t)t * d4 + q);
        }
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
    item_range(s_cb[s_n] * f, &lo, &hi);

    // item i = (global chunk i / f, feature i % f)
    auto issue = [&](int i, int st) {
        const int g = i / f, r = i - g * f;
        const size_t row = (size_t)s_act[locate(g, s_cb, s_n)] * f + r;
        unsigned char* b = ring + (size_t)st * item_bytes;
#pragma unroll
        for (int m = 0; m < KCH; ++m) {
            const int c = lane + 32 * m;
            if (c < nch) {
                cp_async16(b + c * 16, gqs + row * dm + c * 16);
                cp_async16(b + dm + c * 16, uqs + row * dm + c * 16);
            }
        }
        const int sp = dm / 256;  // 16-byte pieces of one row's scales
        if (lane < sp) cp_async16(b + 2 * dm + lane * 16, reinterpret_cast<const unsigned char*>(gd) + row * (dm / 16) + lane * 16);
        else if (lane < 2 * sp)
            cp_async16(b + 2 * dm + dm / 16 + (lane - sp) * 16,
                       reinterpret_cast<const unsigned char*>(ud) + row * (dm / 16) + (lane - sp) * 16);
        cp_async_commit();
    };
    auto compute = [&](int i, int st) {
        const int g = i / f, r = i - g * f;
        const int a = locate(g, s_cb, s_n);
        const int c0 = g - s_cb[a];
        const int pb = ALLTOK ? s_beg[a] : s_beg[a] + c0 * tca;
        const int pe = ALLTOK ? s_end[a] : min(s_end[a], pb + tca);
        const unsigned char* b = ring + (size_t)st * item_bytes;
        const __half* gsc = reinterpret_cast<const __half*>(b + 2 * dm);
        const __half* usc = reinterpret_cast<const __half*>(b + 2 * dm + dm / 16);
        for (int pp = pb; pp < pe; pp += G) {
            const int ng = min(G, pe - pp);
            int toff[G];
#pragma unroll
            for (int g2 = 0; g2 < G; ++g2)
                toff[g2] = (g2 < ng ? (ALLTOK ? s_tok[pp + g2] : (pp + g2 - pb)) : 0) * kTok4;
            float ga[G], ua[G];
#pragma unroll
            for (int g2 = 0; g2 < G; ++g2) {
                ga[g2] = 0.f;
                ua[g2] = 0.f;
            }
#pragma unroll
            for (int m = 0; m < KCH; ++m) {
                const int c = lane + 32 * m;
                if (c < nch) {
                    const uint4 qg = *reinterpret_cast<const uint4*>(b + c * 16);
                    const uint4 qu = *reinterpret_cast<const uint4*>(b + dm + c * 16);
                    const float sg = __half2float(gsc[c >> 1]), su = __half2float(usc[c >> 1]);
#pragma unroll
                    for (int g2 = 0; g2 < G; ++g2) {
                        if (g2 < ng) {
                            const float4* xv = xs + toff[g2] + m * 4 * 32 + lane;
                            ga[g2] = fmaf(sg, chunk_dot(qg, xv, 32), ga[g2]);
                            ua[g2] = fmaf(su, chunk_dot(qu, xv, 32), ua[g2]);
                        }
                    }
                }
            }
#pragma unroll
            for (int g2 = 0; g2 < G; ++g2) {
                ga[g2] = warp_sum(ga[g2]);
                ua[g2] = warp_sum(ua[g2]);
            }
#pragma unroll
            for (int g2 = 0; g2 < G; ++g2)
                if (lane == g2 && g2 < ng) h[(size_t)(pp + g2) * f + r] = silu_f(ga[g2]) * ua[g2];
        }
    };

    if (ALLTOK) {
        warp_stream<NSTG>(lo + warp, hi, NW, issue, compute);
    } else {
        for (int seg = lo; seg < hi;) {
            const int g = seg / f;
            const int seg_end = min(hi, (g + 1) * f);
            const int a = locate(g, s_cb, s_n);
            const int pb = s_beg[a] + (g - s_cb[a]) * tca;
            const int pe = min(s_end[a], pb + tca);
            __syncthreads();  // the previous segment's activations are no longer read
            for (int q = threadIdx.x; q < (pe - pb) * d4; q += kThreads) {
                const int jj = q / d4, qq = q - jj * d4;
                const int t = __ldcg(pair_tok + pb + jj);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t >= 0 && t < T) v = __ldcg(reinterpret_cast<const float4*>(x) + (size_t)t * d4 + qq);
                xs[jj * kTok4 + stage_idx<32>(qq)] = v;
            }
            __syncthreads();
            warp_stream<NSTG>(seg + warp, seg_end, NW, issue, compute);
            seg = seg_end;
        }
    }
    cp_async_wait<0>();
}

// =================================================================== down ==
// An item is 4 consecutive rows (2 per half-warp, LPR = 16 lanes per row);
// lanes split K = d_ff in 16-byte chunks c = hl + 16*m, m < KCH.
// ALLP: every pair's h staged once, else per bucket chunk of at most tcp.
template <int KCH, int G, bool ALLP, int NW, int NSTG>
__global__ void __launch_bounds__(NW * 32, 1) down_cp_kernel(
    const float* __restrict__ h, int T, int f, int dm, int E, int k, const int8_t* __restrict__ dqs,
    const uint16_t* __restrict__ dd, const int32_t* __restrict__ offsets, const int32_t* __restrict__ pair_tok,
    const int32_t* __restrict__ pair_slot, const float* __restrict__ wts, int fuse, float* __restrict__ out,
    int tcp) {
    extern __shared__ __align__(128) unsigned char dn_smem[];
    __shared__ int s_act[MOE_MAX_EXPERTS], s_beg[MOE_MAX_EXPERTS], s_end[MOE_MAX_EXPERTS];
    __shared__ int s_cb[MOE_MAX_EXPERTS + 1], s_n;
    __shared__ int s_ptok[ALLP ? kMaxStagedPairs : 1];
    __shared__ float s_pw[ALLP ? kMaxStagedPairs : 1];
    constexpr int kThreads = NW * 32;
    constexpr int LPR = 16;
    constexpr int kTok4 = KCH * 4 * LPR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hl = lane & 15, sub = lane >> 4;
    const int f4 = f / 4, nch = f / 16;
    const int P = T * k;
    const int nq = dm / kDnRowsPerItem;
    const int item_bytes = kDnRowsPerItem * f + kDnRowsPerItem * (f / 16);  // qs rows, then their scales
    unsigned char* ring = dn_smem + (size_t)warp * NSTG * item_bytes;
    float4* hs = reinterpret_cast<float4*>(dn_smem + (size_t)NW * NSTG * item_bytes);

    // Offsets were written two kernels back (routing/bucketing) and were
    // complete before gate/up released this grid: Wd can stream at once.
    if (warp == 0) build_active(offsets, E, ALLP ? (1 << 30) : tcp, s_act, s_beg, s_end, s_cb, &s_n);
    __syncthreads();
    int lo, hi;
    item_range(s_cb[s_n] * nq, &lo, &hi);

    auto issue = [&](int i, int st) {
        const int g = i / nq, qd = i - g * nq;
        const size_t row0 = (size_t)s_act[locate(g, s_cb, s_n)] * dm + (size_t)qd * kDnRowsPerItem;
        unsigned char* b = ring + (size_t)st * item_bytes;
        const int qpieces = kDnRowsPerItem * f / 16;  // contiguous qs of the 4 rows
        const unsigned char* qsrc = reinterpret_cast<const unsigned char*>(dqs) + row0 * f;
        for (int pc = lane; pc < qpieces; pc += 32) cp_async16(b + pc * 16, qsrc + pc * 16);
        const int spieces = kDnRowsPerItem * f / 256;  // their scales
        const unsigned char* ssrc = reinterpret_cast<const unsigned char*>(dd) + row0 * (f / 16);
        if (lane < spieces) cp_async16(b + kDnRowsPerItem * f + lane * 16, ssrc + lane * 16);
        cp_async_commit();
    };
    auto compute = [&](int i, int st) {
        const int g = i / nq, qd = i - g * nq;
        const int a = locate(g, s_cb, s_n);
        const int c0 = g - s_cb[a];
        const int pb = ALLP ? s_beg[a] : s_beg[a] + c0 * tcp;
        const int pe = ALLP ? s_end[a] : min(s_end[a], pb + tcp);
        const unsigned char* b = ring + (size_t)st * item_bytes;
        const __half* sc = reinterpret_cast<const __half*>(b + kDnRowsPerItem * f);
        for (int pp = pb; pp < pe; pp += G) {
            const int ng = min(G, pe - pp);
            int hoff[G];
#pragma unroll
            for (int g2 = 0; g2 < G; ++g2) hoff[g2] = (g2 < ng ? (ALLP ? (pp + g2) : (pp + g2 - pb)) : 0) * kTok4;
            float acc[2][G];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int g2 = 0; g2 < G; ++g2) acc[rr][g2] = 0.f;
#pragma unroll
            for (int m = 0; m < KCH; ++m) {
                const int c = hl + LPR * m;
                if (c < nch) {
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const int rl = sub * 2 + rr;
                        const uint4 q = *reinterpret_cast<const uint4*>(b + (size_t)rl * f + c * 16);
                        const float s = __half2float(sc[rl * (f / 32) + (c >> 1)]);
#pragma unroll
                        for (int g2 = 0; g2 < G; ++g2)
                            if (g2 < ng)
                                acc[rr][g2] = fmaf(s, chunk_dot(q, hs + hoff[g2] + m * 4 * LPR + hl, LPR), acc[rr][g2]);
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int g2 = 0; g2 < G; ++g2) acc[rr][g2] = group_sum<LPR>(acc[rr][g2]);
#pragma unroll
            for (int g2 = 0; g2 < G; ++g2) {
                if (g2 < ng && hl < 2) {
                    const int o = qd * kDnRowsPerItem + sub * 2 + hl;  // lane 0 / 1 of the half: row 0 / 1
                    const float y = hl == 0 ? acc[0][g2] : acc[1][g2];
                    const int p = pp + g2;
                    if (fuse) {
                        int tok;
                        float wgt;
                        if (ALLP) {
                            tok = s_ptok[p];
                            wgt = s_pw[p];
                        } else {
                            tok = __ldcg(pair_tok + p);
                            const int sl = __ldcg(pair_slot + p);
                            const bool ok = tok >= 0 && tok < T && sl >= 0 && sl < k;
                            wgt = ok ? __ldcg(wts + (size_t)tok * k + sl) : 0.f;
                            tok = ok ? tok : -1;
                        }
                        if (tok >= 0) atomicAdd(out + (size_t)tok * dm + o, wgt * y);
                    } else {
                        out[(size_t)p * dm + o] = y;
                    }
                }
            }
        }
    };

    if (ALLP) {
        // start the weight stream, then wait for gate/up before staging h
        const int first = lo + warp;
        const int n = first < hi ? (hi - first + NW - 1) / NW : 0;
#pragma unroll
        for (int j = 0; j < NSTG - 1; ++j) {
            if (j < n) issue(first + j * NW, j);
            else cp_async_commit();
        }
        pdl_wait();  // gate/up complete: h and the combine target are ready
        pdl_launch_dependents();
        for (int q = threadIdx.x; q < P * f4; q += kThreads) {
            const int p = q / f4, qq = q - p * f4;
            hs[p * kTok4 + stage_idx<LPR>(qq)] = __ldcg(reinterpret_cast<const float4*>(h) + (size_t)p * f4 + qq);
        }
        for (int p = threadIdx.x; p < P; p += kThreads) {
            const int tok = __ldcg(pair_tok + p), sl = __ldcg(pair_slot + p);
            const bool ok = tok >= 0 && tok < T && sl >= 0 && sl < k;
            s_ptok[p] = ok ? tok : -1;
            s_pw[p] = ok ? __ldcg(wts + (size_t)tok * k + sl) : 0.f;
        }
        __syncthreads();
        for (int j = 0; j < n; ++j) {
            const int jn = j + NSTG - 1;
            if (jn < n) issue(first + jn * NW, jn % NSTG);
            else cp_async_commit();
            cp_async_wait<NSTG - 1>();
            __syncwarp();
            compute(first + j * NW, j % NSTG);
            __syncwarp();
        }
    } else {
        pdl_wait();
        pdl_launch_dependents();
        for (int seg = lo; seg < hi;) {
            const int g = seg / nq;
            const int seg_end = min(hi, (g + 1) * nq);
            const int a = locate(g, s_cb, s_n);
            const int pb = s_beg[a] + (g - s_cb[a]) * tcp;
            const int pe = min(s_end[a], pb + tcp);
            __syncthreads();
            for (int q = threadIdx.x; q < (pe - pb) * f4; q += kThreads) {
                const int jj = q / f4, qq = q - jj * f4;
                hs[jj * kTok4 + stage_idx<LPR>(qq)] =
                    __ldcg(reinterpret_cast<const float4*>(h) + (size_t)(pb + jj) * f4 + qq);
            }
            __syncthreads();
            warp_stream<NSTG>(seg + warp, seg_end, NW, issue, compute);
            seg = seg_end;
        }
    }
    cp_async_wait<0>();
}

int g_num_sms[64] = {0};

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!g_num_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_num_sms[dev] = n > 0 ? n : 148;
    }
    return g_num_sms[dev];
}

template <typename K, typename... Args>
cudaError_t launch_pdl(K kern, int grid, int threads, size_t smem, cudaStream_t s, Args... args) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
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

constexpr size_t kSmemCap = 220 * 1024;  // dynamic shared memory per CTA we allow ourselves

template <int KCH, int G, bool ALLTOK, int NW, int NSTG>
cudaError_t gateup_go(const float* x, int T, const moe_layer_w& w, const int32_t* offsets, const int32_t* pair_tok,
                      float* h, float* out_init, int residual, int tca, cudaStream_t s) {
    const int dm = w.d_model;
    const size_t ring = (size_t)NW * NSTG * (2 * dm + 2 * (dm / 16));
    const size_t smem = ring + (size_t)tca * KCH * 4 * 32 * 16;
    if (smem > kSmemCap) return cudaErrorInvalidConfiguration;
    return launch_pdl(gateup_cp_kernel<KCH, G, ALLTOK, NW, NSTG>, num_sms(), NW * 32, smem, s, x, T, dm, w.d_ff,
                      w.E, w.gate.qs, w.gate.d, w.up.qs, w.up.d, offsets, pair_tok, h, out_init, residual, tca,
                      T * w.k);
}

template <int KCH>
cudaError_t gateup_dispatch(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                            const int32_t* pair_tok, float* h, float* out_init, int residual, cudaStream_t s) {
    const int P = T * w.k;
    const int tca = T <= 8 ? T : 8;
    const bool alltok = T <= 8 && P <= kMaxStagedPairs;
    // ring: 16 warps x 3 stages of one feature (gate + up rows) when the
    // activations are small, 12 warps otherwise
    if (T == 1 && alltok) return gateup_go<KCH, 1, true, 16, 3>(x, T, w, offsets, pair_tok, h, out_init, residual, tca, s);
    if (T <= 2 && alltok) return gateup_go<KCH, 2, true, 16, 3>(x, T, w, offsets, pair_tok, h, out_init, residual, tca, s);
    if (alltok) return gateup_go<KCH, 4, true, 12, 3>(x, T, w, offsets, pair_tok, h, out_init, residual, tca, s);
    return gateup_go<KCH, 4, false, 12, 3>(x, T, w, offsets, pair_tok, h, out_init, residual, tca, s);
}

template <int KCH, int G, bool ALLP, int NW, int NSTG>
cudaError_t down_go(const float* h, int T, const moe_layer_w& w, const int32_t* offsets, const int32_t* pair_tok,
                    const int32_t* pair_slot, const float* wts, int fuse, float* out, int tcp, cudaStream_t s) {
    const int f = w.d_ff;
    const size_t ring = (size_t)NW * NSTG * (kDnRowsPerItem * f + kDnRowsPerItem * (f / 16));
    const size_t smem = ring + (size_t)tcp * KCH * 4 * 16 * 16;
    if (smem > kSmemCap) return cudaErrorInvalidConfiguration;
    return launch_pdl(down_cp_kernel<KCH, G, ALLP, NW, NSTG>, num_sms(), NW * 32, smem, s, h, T, f, w.d_model, w.E,
                      w.k, w.down.qs, w.down.d, offsets, pair_tok, pair_slot, wts, fuse, out, tcp);
}

template <int KCH>
cudaError_t down_dispatch(const float* h, int T, const moe_layer_w& w, const int32_t* offsets,
                          const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse, float* out,
                          cudaStream_t s) {
    const int P = T * w.k;
    const size_t tok_bytes = (size_t)KCH * 4 * 16 * 16;
    const bool allp = (size_t)P * tok_bytes <= 48 * 1024 && P <= kMaxStagedPairs;
    if (T == 1 && allp)
        return down_go<KCH, 1, true, 16, 3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, P, s);
    if (allp) return down_go<KCH, 4, true, 16, 3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, P, s);
    return down_go<KCH, 4, false, 16, 3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse, out, 8, s);
}

}  // namespace

bool ffn_stream_supported(const moe_layer_w& w) {
    // whole 16-byte pieces of weights and of each row's scales: K % 256 == 0;
    // down items are 4 whole rows; at most 4 chunks per lane.
    return w.d_model % 256 == 0 && w.d_ff % 256 == 0 && w.d_model % kDnRowsPerItem == 0 && w.d_model <= 2048 &&
           w.d_ff <= 1024;
}

cudaError_t launch_ffn_stream(const float* x, int T, const moe_layer_w& w, const int32_t* offsets,
                              const int32_t* pair_tok, const int32_t* pair_slot, const float* wts, int fuse_combine,
                              float* out_or_ypairs, int residual, float* h, int32_t* status, cudaStream_t s) {
    (void)status;
    if (T == 0) return cudaSuccess;
    float* out_init = fuse_combine ? out_or_ypairs : nullptr;
    const int kg = (w.d_model / 16 + 31) / 32;
    cudaError_t err;
    switch (kg) {
        case 1: err = gateup_dispatch<1>(x, T, w, offsets, pair_tok, h, out_init, residual, s); break;
        case 2: err = gateup_dispatch<2>(x, T, w, offsets, pair_tok, h, out_init, residual, s); break;
        default: err = gateup_dispatch<4>(x, T, w, offsets, pair_tok, h, out_init, residual, s); break;
    }
    if (err != cudaSuccess) return err;
    const int kd = (w.d_ff / 16 + 15) / 16;
    switch (kd) {
        case 1: return down_dispatch<1>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
        case 2: return down_dispatch<2>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
        case 3: return down_dispatch<3>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
        default: return down_dispatch<4>(h, T, w, offsets, pair_tok, pair_slot, wts, fuse_combine, out_or_ypairs, s);
    }
}

}  // namespace moe
