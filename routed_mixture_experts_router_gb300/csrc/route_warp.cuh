// Top-k selection, routing weights and small-batch bucketing by a whole
// thread block, shared by the router kernels and the fused decode kernel.
//
// Everything here is a rank computed by independent comparisons: the slot of
// a selected expert is its rank under a strict total order of the logits, and
// the bucket position of a pair is its rank in (expert, token, slot) order.
// Each thread counts for its own candidates, so there are no dependent
// shuffle or ballot chains (a one-warp selection loop over 128 experts costs
// microseconds of latency), and the result is the one a sequential
// "take the best remaining" loop or a stable counting sort would give.
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

// Add the bias (if any) to nt rows of E logits in shared memory (row t at
// lg + t*ld) and map NaN to -inf, so that the order below is total.
__device__ __forceinline__ void prep_logits(float* lg, int ld, int nt, int E, const float* bias, int nthreads) {
    for (int c = threadIdx.x; c < nt * E; c += nthreads) {
        const int t = c / E, e = c - t * E;
        const float v = lg[t * ld + e] + (bias ? __ldg(bias + e) : 0.0f);
        lg[t * ld + e] = v != v ? -INFINITY : v;
    }
}

// Top-k of nt rows of E prepared logits (ld a multiple of 4, lg 16-byte
// aligned).  Order: descending logit, ties to the lower expert id, so the
// rank of expert e in row t is #{e2 : l2 > l} + #{e2 < e : l2 == l}, a
// permutation of 0..E-1.  Ranks below k land in sel[t*k + rank] (expert id)
// and val[t*k + rank] (its logit).
__device__ __forceinline__ void topk_rank_block(const float* lg, int ld, int nt, int E, int k, int nthreads,
                                                int32_t* sel, float* val) {
    for (int c = threadIdx.x; c < nt * E; c += nthreads) {
        const int t = c / E, e = c - t * E;
        const float* row = lg + t * ld;
        const float v = row[e];
        int gt0 = 0, gt1 = 0, eq0 = 0, eq1 = 0;
        int e2 = 0;
#pragma unroll 4
        for (; e2 + 4 <= E; e2 += 4) {
            const float4 l = *reinterpret_cast<const float4*>(row + e2);
            gt0 += (l.x > v) + (l.y > v);
            gt1 += (l.z > v) + (l.w > v);
            eq0 += (l.x == v) + (l.y == v);
            eq1 += (l.z == v) + (l.w == v);
        }
        for (; e2 < E; ++e2) {
            gt0 += row[e2] > v;
            eq0 += row[e2] == v;
        }
        int r = gt0 + gt1;
        if (eq0 + eq1 > 1)  // exact ties: the lower ids come first
            for (int e3 = 0; e3 < e; ++e3) r += row[e3] == v;
        if (r < k) {
            sel[t * k + r] = e;
            val[t * k + r] = v;
        }
    }
}

// Routing weight of pair q = (t, s) from the selected logits:
// w = exp(l_s - l_0) / sum_{s' < k} exp(l_s' - l_0) (softmax over the top-k,
// the same as the full softmax renormalised over the selection).
__device__ __forceinline__ float topk_weight(const float* val, int q, int k) {
    const int t = q / k;
    const float* v = val + t * k;
    float den = 0.0f;
#pragma unroll 8
    for (int s = 0; s < k; ++s) den += expf(v[s] - v[0]);
    return expf(val[q] - v[0]) / den;
}

// Bucket position of pair q among the P pairs with experts sel[0..P):
// #{q2 : e2 < e or (e2 == e and q2 < q)} -- grouped by expert, stable in
// (token, slot) order.
__device__ __forceinline__ int pair_rank(const int32_t* sel, int P, int q) {
    const int e = sel[q];
    int r = 0;
#pragma unroll 8
    for (int q2 = 0; q2 < P; ++q2) {
        const int e2 = sel[q2];
        r += (e2 < e) | ((e2 == e) & (q2 < q));
    }
    return r;
}

// offsets[e] = #{q : sel[q] < e} for e = 0..E (the exclusive scan of the
// bucket sizes), by all threads of the block.
__device__ __forceinline__ void bucket_offsets(const int32_t* sel, int P, int E, int nthreads, int32_t* offsets) {
    for (int e = threadIdx.x; e <= E; e += nthreads) {
        int c = 0;
#pragma unroll 8
        for (int q = 0; q < P; ++q) c += sel[q] < e;
        offsets[e] = c;
    }
}

}  // namespace moe
