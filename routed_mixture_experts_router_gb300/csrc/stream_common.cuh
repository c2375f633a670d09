// Streaming helpers of the fp32 (decode) expert path: exact int8 -> fp32,
// paired fp32 FMA dot products, per-warp cp.async rings, the active-expert
// work list and the gate/up and down work items.  Shared by the separate
// gate/up and down kernels and the fused single-launch decode kernel.
#pragma once

#include "common.cuh"
#include "pipeline.cuh"

namespace moe {
namespace stream {

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

// The 16 weights of a chunk times their block scale d, exactly, as 8 fp32
// pairs.  Byte u = q + 128 goes into the mantissa of 2^15 (v = 2^15 + u), and
// fma(v, d, -(2^15 + 128) d) = q d: the constant is exact (9 x 11 significant
// bits) and so is the result (q d has at most 19), so the one rounding of
// the fma changes nothing.
__device__ __forceinline__ void dequant16(const uint4 q, float d, f32x2 (&w)[8]) {
    const f32x2 dd = f2_pack(d, d);
    const float c = -32896.0f * d;
    const f32x2 cc = f2_pack(c, c);
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t u = words[m];  // bytes u = q + 128 (device layout)
        w[2 * m] = f2_fma(f2_pack(__uint_as_float(__byte_perm(u, 0x47000000u, 0x7504)),
                                  __uint_as_float(__byte_perm(u, 0x47000000u, 0x7514))),
                          dd, cc);
        w[2 * m + 1] = f2_fma(f2_pack(__uint_as_float(__byte_perm(u, 0x47000000u, 0x7524)),
                                      __uint_as_float(__byte_perm(u, 0x47000000u, 0x7534))),
                              dd, cc);
    }
}

// 16 Q4_0 weights times their block scale d, exactly, as 8 fp32 pairs: the
// low (half 0) or high (half 1) nibbles of a 16-byte block, values n in
// 0..15.  As above, v = 2^15 + n and fma(v, d, -(2^15 + 8) d) = (n - 8) d:
// the constant has 13 x 11 significant bits (exact in fp32) and the result
// at most 15, so the fma's one rounding changes nothing.
__device__ __forceinline__ void dequant16_q4(const uint4 q, int half, float d, f32x2 (&w)[8]) {
    const f32x2 dd = f2_pack(d, d);
    const float c = -32776.0f * d;
    const f32x2 cc = f2_pack(c, c);
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint32_t u = (half ? words[m] >> 4 : words[m]) & 0x0f0f0f0fu;
        w[2 * m] = f2_fma(f2_pack(__uint_as_float(__byte_perm(u, 0x47000000u, 0x7504)),
                                  __uint_as_float(__byte_perm(u, 0x47000000u, 0x7514))),
                          dd, cc);
        w[2 * m + 1] = f2_fma(f2_pack(__uint_as_float(__byte_perm(u, 0x47000000u, 0x7524)),
                                      __uint_as_float(__byte_perm(u, 0x47000000u, 0x7534))),
                              dd, cc);
    }
}

// sum over 16 values of (q * d) * x: one 16-byte weight chunk dequantised
// with its block scale d (exactly), four float4 of x at stride `st`.
__device__ __forceinline__ float chunk_dot_scaled(const uint4 q, float d, const float4* xv4, int st) {
    f32x2 w[8];
    dequant16(q, d, w);
    f32x2 acc0 = 0ull, acc1 = 0ull;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 xv = xv4[m * st];
        acc0 = f2_fma(w[2 * m], f2_pack(xv.x, xv.y), acc0);
        acc1 = f2_fma(w[2 * m + 1], f2_pack(xv.z, xv.w), acc1);
    }
    return f2_sum(f2_add(acc0, acc1));
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
// split K in chunks of CF4 float4 (16 values for Q8_0 chunks, 32 for Q4_0
// blocks), chunk c = hl + LPR*m: float4 j of chunk c sits at
// (m*CF4 + j)*LPR + hl, so one load instruction reads consecutive float4s.
template <int LPR, int CF4 = 4>
__device__ __forceinline__ int stage_idx(int q) {
    const int c = q / CF4, j = q % CF4;
    return ((c / LPR) * CF4 + j) * LPR + (c % LPR);
}

// Active experts (non-empty buckets) in id order, by warp 0, and the work
// list they imply: expert a's bucket is cut into chunks of at most `chunk`
// pairs (the activations one pass stages in shared memory); s_cb[a] is the
// index of a's first chunk and s_cb[n] the total.  All offsets are fetched in
// one round trip, through L2 (they were written by an earlier kernel, or come
// from the caller).  Every bucket is clamped into [0, P]: offsets that are
// not a valid bucketing give wrong sums, never an out-of-range pair.
// s_act holds each active expert's index into the weight arrays (its arena
// slot when expert_slot is given); an expert without a slot is left out.
__device__ inline void build_active(const int32_t* offsets, int E, int chunk, int P, int* s_act, int* s_beg, int* s_end,
                             int* s_cb, int* s_n, const int32_t* expert_slot, int n_slots) {
    const int lane = threadIdx.x & 31;
    int lo[MOE_MAX_EXPERTS / 32], hi[MOE_MAX_EXPERTS / 32], wi[MOE_MAX_EXPERTS / 32];
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
        const int e = 32 * j + lane;
        const int a = e < E ? __ldcg(offsets + e) : 0;
        const int b = e < E ? __ldcg(offsets + e + 1) : 0;
        wi[j] = e < E ? weight_index(expert_slot, n_slots, e) : -1;
        lo[j] = min(max(a, 0), P);
        hi[j] = wi[j] < 0 ? lo[j] : min(max(b, lo[j]), P);
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
            s_act[jj] = wi[j];
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


// ---- work items ------------------------------------------------------------
// gate/up item: one output feature `row` (global row index e*d_ff + r) -- its
// gate row and up row, then their fp16 scales -- copied into stage buffer b.
template <int KCH>
__device__ __forceinline__ void gu_issue_item(unsigned char* b, const int8_t* gqs, const int8_t* uqs,
                                              const uint16_t* gd, const uint16_t* ud, size_t row, int dm, int lane) {
    const int nch = dm / 16;
#pragma unroll
    for (int m = 0; m < KCH; ++m) {
        const int c = lane + 32 * m;
        if (c < nch) {
            cp_async16(b + c * 16, gqs + row * dm + c * 16);
            cp_async16(b + dm + c * 16, uqs + row * dm + c * 16);
        }
    }
    const int sp = dm / 256;  // 16-byte pieces of one row's scales
    const unsigned char* gsrc = reinterpret_cast<const unsigned char*>(gd) + row * (dm / 16);
    const unsigned char* usrc = reinterpret_cast<const unsigned char*>(ud) + row * (dm / 16);
    if (lane < sp) cp_async16(b + 2 * dm + lane * 16, gsrc + lane * 16);
    else if (lane < 2 * sp) cp_async16(b + 2 * dm + dm / 16 + (lane - sp) * 16, usrc + (lane - sp) * 16);
    cp_async_commit();
}

// h[p][r] = silu(g) * u for the pairs p in [pb, pe) of one feature r, from a
// landed gate/up item.  xs: staged activations (ALLTOK: indexed by token
// through s_tok; else by p - pb).
template <int KCH, int G, bool ALLTOK>
__device__ __forceinline__ void gu_compute_item(const unsigned char* b, int r, int pb, int pe, int dm, int f,
                                                int lane, const float4* xs, const int* s_tok, float* h) {
    constexpr int kTok4 = KCH * 4 * 32;
    const int nch = dm / 16;
    const __half* gsc = reinterpret_cast<const __half*>(b + 2 * dm);
    const __half* usc = reinterpret_cast<const __half*>(b + 2 * dm + dm / 16);
    for (int pp = pb; pp < pe; pp += G) {
        const int ng = min(G, pe - pp);
        int toff[G];
#pragma unroll
        for (int g2 = 0; g2 < G; ++g2) toff[g2] = (g2 < ng ? (ALLTOK ? s_tok[pp + g2] : (pp + g2 - pb)) : 0) * kTok4;
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
                        ga[g2] += chunk_dot_scaled(qg, sg, xv, 32);
                        ua[g2] += chunk_dot_scaled(qu, su, xv, 32);
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
}

// down item: rows row0 .. row0+3 of Wd (contiguous), then their scales.
__device__ __forceinline__ void dn_issue_item(unsigned char* b, const int8_t* dqs, const uint16_t* dd, size_t row0,
                                              int f, int lane) {
    const int qpieces = kDnRowsPerItem * f / 16;
    const unsigned char* qsrc = reinterpret_cast<const unsigned char*>(dqs) + row0 * f;
    for (int pc = lane; pc < qpieces; pc += 32) cp_async16(b + pc * 16, qsrc + pc * 16);
    const int spieces = kDnRowsPerItem * f / 256;
    const unsigned char* ssrc = reinterpret_cast<const unsigned char*>(dd) + row0 * (f / 16);
    if (lane < spieces) cp_async16(b + kDnRowsPerItem * f + lane * 16, ssrc + lane * 16);
    cp_async_commit();
}

// y = Wd[o] . h[p] for the 4 rows o = 4*qd.. of a landed down item and the
// pairs p in [pb, pe); combined into out (fuse) or written to ypairs.  Half
// warp `sub` owns rows 2*sub, 2*sub+1; hs: staged h (ALLP: by p, else p - pb).
template <int KCH, int G, bool ALLP>
__device__ __forceinline__ void dn_compute_item(const unsigned char* b, int qd, int pb, int pe, int f, int dm, int k,
                                                int T, int hl, int sub, const float4* hs, const int* s_ptok,
                                                const float* s_pw, const int32_t* pair_tok,
                                                const int32_t* pair_slot, const float* wts, int fuse, float* out) {
    constexpr int LPR = 16;
    constexpr int kTok4 = KCH * 4 * LPR;
    const int nch = f / 16;
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
                            acc[rr][g2] += chunk_dot_scaled(q, s, hs + hoff[g2] + m * 4 * LPR + hl, LPR);
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
}

// ---- Q4_0 work items (the fused decode kernel) -------------------------------
// A 16-byte chunk is one whole Q4_0 block (32 values, one scale).  Down items
// are 8 rows, two per quarter-warp, so that a row's d_ff/32 blocks spread over
// 8 lanes as evenly as a Q8_0 row's d_ff/16 chunks over 16.
constexpr int kDnRowsPerItemQ4 = 8;

// sum over the 32 values of one Q4_0 block of w * x: low nibbles against
// float4 0..3 of the chunk, high nibbles against float4 4..7 (stride st).
__device__ __forceinline__ float chunk_dot_q4(const uint4 q, float d, const float4* xv4, int st) {
    f32x2 w[8];
    f32x2 acc0 = 0ull, acc1 = 0ull;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        dequant16_q4(q, half, d, w);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 xv = xv4[(4 * half + m) * st];
            acc0 = f2_fma(w[2 * m], f2_pack(xv.x, xv.y), acc0);
            acc1 = f2_fma(w[2 * m + 1], f2_pack(xv.z, xv.w), acc1);
        }
    }
    return f2_sum(f2_add(acc0, acc1));
}

// gate/up item of feature `row`: its Q4_0 gate row and up row (dm/2 bytes
// each), then their fp16 scales (dm/32 each).
template <int KCH>
__device__ __forceinline__ void gu_issue_item_q4(unsigned char* b, const int8_t* gqs, const int8_t* uqs,
                                                 const uint16_t* gd, const uint16_t* ud, size_t row, int dm,
                                                 int lane) {
    const int nch = dm / 32, rb = dm / 2;
    const unsigned char* g = reinterpret_cast<const unsigned char*>(gqs) + row * rb;
    const unsigned char* u = reinterpret_cast<const unsigned char*>(uqs) + row * rb;
#pragma unroll
    for (int m = 0; m < KCH; ++m) {
        const int c = lane + 32 * m;
        if (c < nch) {
            cp_async16(b + c * 16, g + c * 16);
            cp_async16(b + rb + c * 16, u + c * 16);
        }
    }
    const int sp = dm / 256;  // 16-byte pieces of one row's scales
    const unsigned char* gsrc = reinterpret_cast<const unsigned char*>(gd) + row * (dm / 16);
    const unsigned char* usrc = reinterpret_cast<const unsigned char*>(ud) + row * (dm / 16);
    if (lane < sp) cp_async16(b + dm + lane * 16, gsrc + lane * 16);
    else if (lane < 2 * sp) cp_async16(b + dm + dm / 16 + (lane - sp) * 16, usrc + (lane - sp) * 16);
    cp_async_commit();
}

// h[p][r] = silu(g) * u for the pairs p in [pb, pe) of feature r; xs holds
// every token's activations in the 32-value chunk layout (stage_idx<32, 8>).
template <int KCH, int G>
__device__ __forceinline__ void gu_compute_item_q4(const unsigned char* b, int r, int pb, int pe, int dm, int f,
                                                   int lane, const float4* xs, const int* s_tok, float* h) {
    constexpr int kTok4 = KCH * 8 * 32;
    const int nch = dm / 32, rb = dm / 2;
    const __half* gsc = reinterpret_cast<const __half*>(b + dm);
    const __half* usc = gsc + dm / 32;
    for (int pp = pb; pp < pe; pp += G) {
        const int ng = min(G, pe - pp);
        int toff[G];
#pragma unroll
        for (int g2 = 0; g2 < G; ++g2) toff[g2] = (g2 < ng ? s_tok[pp + g2] : 0) * kTok4;
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
                const uint4 qu = *reinterpret_cast<const uint4*>(b + rb + c * 16);
                const float sg = __half2float(gsc[c]), su = __half2float(usc[c]);
#pragma unroll
                for (int g2 = 0; g2 < G; ++g2) {
                    if (g2 < ng) {
                        const float4* xv = xs + toff[g2] + m * 8 * 32 + lane;
                        ga[g2] += chunk_dot_q4(qg, sg, xv, 32);
                        ua[g2] += chunk_dot_q4(qu, su, xv, 32);
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
}

// down item: Q4_0 rows row0 .. row0+7 of Wd (contiguous, f/2 bytes each),
// then their scales (f/32 each).
__device__ __forceinline__ void dn_issue_item_q4(unsigned char* b, const int8_t* dqs, const uint16_t* dd,
                                                 size_t row0, int f, int lane) {
    const int qbytes = kDnRowsPerItemQ4 * f / 2;
    const unsigned char* qsrc = reinterpret_cast<const unsigned char*>(dqs) + row0 * (f / 2);
    for (int pc = lane; pc < qbytes / 16; pc += 32) cp_async16(b + pc * 16, qsrc + pc * 16);
    const int spieces = kDnRowsPerItemQ4 * f / 256;  // 8 rows x f/32 fp16 scales, in 16-byte pieces
    const unsigned char* ssrc = reinterpret_cast<const unsigned char*>(dd) + row0 * (f / 16);
    if (lane < spieces) cp_async16(b + qbytes + lane * 16, ssrc + lane * 16);
    cp_async_commit();
}

// y = Wd[o] . h[p] for the 8 rows o = 8*qd.. of a landed Q4_0 down item and
// the pairs p in [pb, pe), combined into out with the staged pair tokens and
// weights.  Quarter warp `sub` owns rows 2*sub, 2*sub+1; hs: every pair's h
// in the 32-value chunk layout for 8 lanes (stage_idx<8, 8>).
template <int KCH, int G>
__device__ __forceinline__ void dn_compute_item_q4(const unsigned char* b, int qd, int pb, int pe, int f, int dm,
                                                   int hl, int sub, const float4* hs, const int* s_ptok,
                                                   const float* s_pw, float* out) {
    constexpr int LPR = 8;
    constexpr int kTok4 = KCH * 8 * LPR;
    const int nch = f / 32, rb = f / 2;
    const __half* sc = reinterpret_cast<const __half*>(b + kDnRowsPerItemQ4 * rb);
    for (int pp = pb; pp < pe; pp += G) {
        const int ng = min(G, pe - pp);
        int hoff[G];
#pragma unroll
        for (int g2 = 0; g2 < G; ++g2) hoff[g2] = (g2 < ng ? pp + g2 : 0) * kTok4;
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
                    const uint4 q = *reinterpret_cast<const uint4*>(b + (size_t)rl * rb + c * 16);
                    const float s = __half2float(sc[rl * nch + c]);
#pragma unroll
                    for (int g2 = 0; g2 < G; ++g2)
                        if (g2 < ng) acc[rr][g2] += chunk_dot_q4(q, s, hs + hoff[g2] + m * 8 * LPR + hl, LPR);
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
                const int o = qd * kDnRowsPerItemQ4 + sub * 2 + hl;  // lane 0 / 1 of the quarter: row 0 / 1
                const float y = hl == 0 ? acc[0][g2] : acc[1][g2];
                const int tok = s_ptok[pp + g2];
                if (tok >= 0) atomicAdd(out + (size_t)tok * dm + o, s_pw[pp + g2] * y);
            }
        }
    }
}

// ---- items of up to kMultiG tokens (batches of 3 or more tokens) ------------
// Each 16-byte weight chunk is dequantised once per item (not once per token)
// and reused for every token of the item; the per-token partial sums are
// reduced across lanes with one butterfly reduce-scatter.
constexpr int kMultiG = 8;

// One reduce-scatter step over lane pairs (L, L ^ o): N values in, N/2 out.
// The lane with (L & o) set keeps the upper half.  After steps o = W/2, ...,
// the lane holds the cross-lane sum of value index sum(upper_s * N_s / 2).
template <int N>
__device__ __forceinline__ void rs_step(float (&v)[16], int o, bool upper) {
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = upper ? v[i] : v[i + N / 2];
        const float keep = upper ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
}

// Gate/up item of one feature r for the n = pe - pb <= kMultiG pairs of a
// bucket chunk.  xs holds the activations: ALLTOK, by token (s_tok[p]);
// else by position p - pb.  Writes h[p][r] = silu(g) * u.
template <int KCH, bool ALLTOK>
__device__ __forceinline__ void gu_compute_multi(const unsigned char* b, int r, int pb, int pe, int dm, int f,
                                                 int lane, const float4* xs, const int* s_tok, float* h) {
    constexpr int kTok4 = KCH * 4 * 32;
    const int nch = dm / 16;
    const int n = pe - pb;
    const __half* gsc = reinterpret_cast<const __half*>(b + 2 * dm);
    const __half* usc = reinterpret_cast<const __half*>(b + 2 * dm + dm / 16);
    int toff[kMultiG];
    f32x2 ag[kMultiG], au[kMultiG];
#pragma unroll
    for (int j = 0; j < kMultiG; ++j) {
        toff[j] = (j < n ? (ALLTOK ? s_tok[pb + j] : j) : 0) * kTok4;
        ag[j] = 0ull;
        au[j] = 0ull;
    }
#pragma unroll
    for (int m = 0; m < KCH; ++m) {
        const int c = lane + 32 * m;
        if (c < nch) {
            f32x2 wg[8], wu[8];
            dequant16(*reinterpret_cast<const uint4*>(b + c * 16), __half2float(gsc[c >> 1]), wg);
            dequant16(*reinterpret_cast<const uint4*>(b + dm + c * 16), __half2float(usc[c >> 1]), wu);
#pragma unroll
            for (int j = 0; j < kMultiG; ++j) {
                if (j < n) {
                    const float4* xv = xs + toff[j] + m * 4 * 32 + lane;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 x = xv[i * 32];
                        const f32x2 xl = f2_pack(x.x, x.y), xh = f2_pack(x.z, x.w);
                        ag[j] = f2_fma(wg[2 * i + 1], xh, f2_fma(wg[2 * i], xl, ag[j]));
                        au[j] = f2_fma(wu[2 * i + 1], xh, f2_fma(wu[2 * i], xl, au[j]));
                    }
                }
            }
        }
    }
    float v[16];
#pragma unroll
    for (int j = 0; j < kMultiG; ++j) {
        v[2 * j] = f2_sum(ag[j]);
        v[2 * j + 1] = f2_sum(au[j]);
    }
    rs_step<16>(v, 16, lane & 16);
    rs_step<8>(v, 8, lane & 8);
    rs_step<4>(v, 4, lane & 4);
    rs_step<2>(v, 2, lane & 2);
    // value index lane >> 1: token lane >> 2, gate (bit 1 clear) or up
    const float s = v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
    const float u = __shfl_xor_sync(0xffffffffu, s, 2);
    const int j = lane >> 2;
    if ((lane & 3) == 0 && j < n) h[(size_t)(pb + j) * f + r] = silu_f(s) * u;
}

// Down item (4 rows from o = 4*qd) for n = pe - pb <= kMultiG pairs.  Half
// warp `sub` owns rows 2*sub, 2*sub + 1; hs row of pair j at hrow0 + j.
// tok_of[j] / w_of[j]: the pair's token (-1: skip) and routing weight.
// fuse: out[tok][o] += w * y (fp32 atomics); else ypairs[pb + j][o] = y.
template <int KCH>
__device__ __forceinline__ void dn_compute_multi(const unsigned char* b, int qd, int pb, int pe, int f, int dm,
                                                 int hl, int sub, const float4* hs, int hrow0, const int* tok_of,
                                                 const float* w_of, int fuse, float* out) {
    constexpr int LPR = 16;
    constexpr int kTok4 = KCH * 4 * LPR;
    const int nch = f / 16;
    const int n = pe - pb;
    const __half* sc = reinterpret_cast<const __half*>(b + kDnRowsPerItem * f);
    f32x2 acc[2][kMultiG];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int j = 0; j < kMultiG; ++j) acc[rr][j] = 0ull;
#pragma unroll
    for (int m = 0; m < KCH; ++m) {
        const int c = hl + LPR * m;
        if (c < nch) {
            f32x2 w0[8], w1[8];
            const int r0 = sub * 2;
            dequant16(*reinterpret_cast<const uint4*>(b + (size_t)r0 * f + c * 16),
                      __half2float(sc[r0 * (f / 32) + (c >> 1)]), w0);
            dequant16(*reinterpret_cast<const uint4*>(b + (size_t)(r0 + 1) * f + c * 16),
                      __half2float(sc[(r0 + 1) * (f / 32) + (c >> 1)]), w1);
#pragma unroll
            for (int j = 0; j < kMultiG; ++j) {
                if (j < n) {
                    const float4* hv = hs + (size_t)(hrow0 + j) * kTok4 + m * 4 * LPR + hl;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 x = hv[i * LPR];
                        const f32x2 xl = f2_pack(x.x, x.y), xh = f2_pack(x.z, x.w);
                        acc[0][j] = f2_fma(w0[2 * i + 1], xh, f2_fma(w0[2 * i], xl, acc[0][j]));
                        acc[1][j] = f2_fma(w1[2 * i + 1], xh, f2_fma(w1[2 * i], xl, acc[1][j]));
                    }
                }
            }
        }
    }
    float v[16];
#pragma unroll
    for (int j = 0; j < kMultiG; ++j) {
        v[j] = f2_sum(acc[0][j]);
        v[kMultiG + j] = f2_sum(acc[1][j]);
    }
    // within the half warp: value index hl = row (hl >> 3), pair (hl & 7)
    rs_step<16>(v, 8, hl & 8);
    rs_step<8>(v, 4, hl & 4);
    rs_step<4>(v, 2, hl & 2);
    rs_step<2>(v, 1, hl & 1);
    const int j = hl & 7;
    if (j < n) {
        const int o = qd * kDnRowsPerItem + sub * 2 + (hl >> 3);
        if (fuse) {
            const int tok = tok_of[j];
            if (tok >= 0) atomicAdd(out + (size_t)tok * dm + o, w_of[j] * v[0]);
        } else {
            out[(size_t)(pb + j) * dm + o] = v[0];
        }
    }
}

}  // namespace stream
}  // namespace moe
