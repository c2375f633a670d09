// Compact expert grouping: a stable counting sort of the T*k (token, slot)
// pairs by expert id ("compact expert grouping", expxa.com
// reuse-ordering-qualification, "What changed from the first experiment").
//
// The pages report shared-memory race warnings in their grouping helper
// ("Why it was not adopted"); this one decides every position without
// atomics, so it is deterministic and race-free by construction:
//   1. counts per expert (shared-memory atomics: order-free integer adds),
//      exclusive scan -> offsets;
//   2. tokens in chunks of 1024, one token per thread.  A token's experts
//      form a bitmap over E; warp ballots transpose the bitmaps so that lane
//      b of warp w holds M[w][e] = the set of lanes (tokens) of warp w that
//      picked expert e.  The rank of token t in bucket e is
//        (pairs of e in earlier chunks) + (popcounts of M[w'][e], w' < w)
//        + popc(M[w][e] & lanes below t).
//      Since one token picks each expert at most once, ascending token order
//      is ascending (token, slot) order within a bucket.
// Single CTA: the work is T*k integers; latency, not bandwidth, matters.
#include "common.cuh"
#include "pipeline.cuh"

namespace moe {

namespace {

// Token t's k expert ids, each valid id (in [0, E)) kept at its first
// occurrence: keep(s, e) for every kept slot s; *bad set when an id is out of
// range or repeats.  k <= 8 (the common top-k): the ids in registers (two
// 16-byte loads when aligned), each compared with the token's earlier slots;
// larger k: a bitmap over the experts.
template <class Keep>
__device__ __forceinline__ void token_ids(const int32_t* __restrict__ idx, int t, int k, int E, int* bad,
                                          Keep keep) {
    if (k <= 8) {
        int ids[8];
        const int32_t* row = idx + (size_t)t * k;
        if (k == 8 && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
            const int4 a = __ldcg(reinterpret_cast<const int4*>(row)), b = __ldcg(reinterpret_cast<const int4*>(row) + 1);
            ids[0] = a.x, ids[1] = a.y, ids[2] = a.z, ids[3] = a.w, ids[4] = b.x, ids[5] = b.y, ids[6] = b.z, ids[7] = b.w;
        } else {
#pragma unroll
            for (int s = 0; s < 8; ++s) ids[s] = s < k ? __ldcg(row + s) : -1;
        }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            if (s >= k) break;
            const int e = ids[s];
            bool ok = e >= 0 && e < E;
#pragma unroll
            for (int s3 = 0; s3 < s; ++s3) ok = ok && ids[s3] != e;
            if (!ok) {
                *bad = 1;
                continue;
            }
            keep(s, e);
        }
        return;
    }
    uint32_t seen[MOE_MAX_EXPERTS / 32];
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) seen[j] = 0;
    for (int s = 0; s < k; ++s) {
        const int e = __ldcg(idx + (size_t)t * k + s);
        bool ok = e >= 0 && e < E;
        if (ok) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j)
                if (j == (e >> 5)) word = seen[j];
            ok = !(word & (1u << (e & 31)));
#pragma unroll
            for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j)
                if (j == (e >> 5)) seen[j] |= 1u << (e & 31);
        }
        if (!ok) {
            *bad = 1;
            continue;
        }
        keep(s, e);
    }
}

constexpr int kBucketThreads = 1024;
constexpr int kBucketWarps = kBucketThreads / kWarp;

__global__ void __launch_bounds__(kBucketThreads) bucket_kernel(const int32_t* __restrict__ idx, int T, int k, int E,
                                                                int32_t* __restrict__ offsets,
                                                                int32_t* __restrict__ pair_tok,
                                                                int32_t* __restrict__ pair_slot,
                                                                int32_t* __restrict__ pos, int32_t* status) {
    __shared__ int s_cnt[MOE_MAX_EXPERTS];
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ int s_run[MOE_MAX_EXPERTS];   // pairs placed by earlier chunks
    __shared__ int s_scan[MOE_MAX_EXPERTS];
    __shared__ int s_bad;
    extern __shared__ uint32_t bucket_dyn[];
    const int words = (E + 31) >> 5;
    const int ep = words * 32;
    uint32_t* s_mask = bucket_dyn;                                   // M[w][e], [32][ep]
    int* s_base = reinterpret_cast<int*>(bucket_dyn + kBucketWarps * ep);  // rank base of warp w in bucket e

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();  // idx written by the router
    pdl_launch_dependents();
    if (tid < MOE_MAX_EXPERTS) {
        s_cnt[tid] = 0;
        s_run[tid] = 0;
    }
    if (tid == 0) s_bad = 0;
    __syncthreads();

    // 1. counts (valid ids only; a repeated id within a token is dropped below
    //    and not counted: rows with repeats are detected per token)
    int bad = 0;
    for (int t = tid; t < T; t += kBucketThreads)
        token_ids(idx, t, k, E, &bad, [&](int, int e) { atomicAdd(&s_cnt[e], 1); });
    if (bad) s_bad = 1;
    __syncthreads();
    // exclusive scan over E <= 256 counts: warps 0..7 scan 32 each, then fix up
    if (tid < MOE_MAX_EXPERTS) {
        int v = tid < E ? s_cnt[tid] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        s_scan[tid] = incl;  // inclusive within its warp
    }
    __syncthreads();
    if (tid < MOE_MAX_EXPERTS) {
        int add = 0;
        for (int w = 0; w < (tid >> 5); ++w) add += s_scan[w * 32 + 31];
        const int incl = s_scan[tid] + add;
        const int v = tid < E ? s_cnt[tid] : 0;
        if (tid < E) s_off[tid] = incl - v;
        if (tid == E - 1) s_off[E] = incl;
    }
    __syncthreads();
    for (int e = tid; e <= E; e += kBucketThreads) offsets[e] = s_off[e];

    // 2. stable scatter, 1024 tokens per chunk
    for (int c0 = 0; c0 < T; c0 += kBucketThreads) {
        const int t = c0 + tid;
        const bool valid = t < T;
        uint32_t bm[MOE_MAX_EXPERTS / 32];
#pragma unroll
        for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) bm[j] = 0;
        int es[MOE_MAX_TOPK];
#pragma unroll
        for (int s = 0; s < MOE_MAX_TOPK; ++s) es[s] = (valid && s < k) ? __ldcg(idx + (size_t)t * k + s) : -1;
#pragma unroll
        for (int s = 0; s < MOE_MAX_TOPK; ++s) {
            if (s >= k) break;
            int e = es[s];
            if (e >= 0 && e < E) {
                uint32_t word = 0;
#pragma unroll
                for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j)
                    if (j == (e >> 5)) word = bm[j];
                if (word & (1u << (e & 31))) {
                    e = -1;  // repeat within the token: dropped
                } else {
#pragma unroll
                    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j)
                        if (j == (e >> 5)) bm[j] |= 1u << (e & 31);
                }
            } else {
                e = -1;
            }
            es[s] = e;
        }
        // transpose: lane b of warp w keeps M[w][32j + b]
#pragma unroll
        for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
            if (j < words) {
                uint32_t mine = 0;
#pragma unroll 4
                for (int b = 0; b < 32; ++b) {
                    const uint32_t m = __ballot_sync(0xffffffffu, (bm[j] >> b) & 1u);
                    if (lane == b) mine = m;
                }
                s_mask[warp * ep + j * 32 + lane] = mine;
            }
        }
        __syncthreads();
        if (tid < E) {
            int run = s_run[tid];
            for (int w = 0; w < kBucketWarps; ++w) {
                s_base[w * ep + tid] = run;
                run += __popc(s_mask[w * ep + tid]);
            }
            s_run[tid] = run;
        }
        __syncthreads();
        if (valid) {
            const uint32_t below = (1u << lane) - 1u;
#pragma unroll
            for (int s = 0; s < MOE_MAX_TOPK; ++s) {
                if (s >= k) break;
                const int e = es[s];
                if (e < 0) {
                    pos[(size_t)t * k + s] = -1;
                    continue;
                }
                const int p = s_off[e] + s_base[warp * ep + e] + __popc(s_mask[warp * ep + e] & below);
                pair_tok[p] = t;
                pair_slot[p] = s;
                pos[(size_t)t * k + s] = p;
            }
        }
        __syncthreads();
    }
    if (tid == 0 && s_bad) flag_status(status, MOE_STATUS_BAD_INDEX);
}

// Same result, for batches whose per-expert pair bitmaps fit in shared
// memory: pair p = t*k + s sets bit p of its expert's bitmap M[e]; one warp
// per expert turns the bitmap into word prefix counts (popcount + warp scan)
// and the bucket size; pair p then lands at
//   offsets[e] + (pairs of e in words below p/32) + popc(M[e][p/32] & bits below p).
// Every phase is parallel over pairs, words or experts (no serial ballot
// transposes), and the order is the same stable (token, slot) order.
__global__ void __launch_bounds__(kBucketThreads) bucket_mask_kernel(const int32_t* __restrict__ idx, int T, int k,
                                                                     int E, int32_t* __restrict__ offsets,
                                                                     int32_t* __restrict__ pair_tok,
                                                                     int32_t* __restrict__ pair_slot,
                                                                     int32_t* __restrict__ pos, int32_t* status) {
    __shared__ int s_cnt[MOE_MAX_EXPERTS];
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ int s_wsum[kBucketWarps];
    __shared__ int s_bad;
    extern __shared__ uint32_t bucket_dyn[];
    const int P = T * k;
    const int W = (P + 31) >> 5;
    uint32_t* s_mask = bucket_dyn;                                          // [E][W]
    uint16_t* s_pre = reinterpret_cast<uint16_t*>(bucket_dyn + (size_t)E * W);  // [E][W] pairs in earlier words
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();  // idx written by the router
    pdl_launch_dependents();
    for (int i = tid; i < E * W; i += kBucketThreads) s_mask[i] = 0;
    if (tid == 0) s_bad = 0;
    __syncthreads();

    // 1. one token per thread: validate its ids, drop repeats, set the bits
    int bad = 0;
    for (int t = tid; t < T; t += kBucketThreads)
        token_ids(idx, t, k, E, &bad, [&](int s, int e) {
            const int p = t * k + s;
            atomicOr(&s_mask[(size_t)e * W + (p >> 5)], 1u << (p & 31));
        });
    if (bad) s_bad = 1;
    __syncthreads();
    // 2. per expert (one warp each): word prefix counts and the bucket size
    for (int e = warp; e < E; e += kBucketWarps) {
        int carry = 0;
        for (int w0 = 0; w0 < W; w0 += 32) {
            const int w = w0 + lane;
            const int c = w < W ? __popc(s_mask[(size_t)e * W + w]) : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (w < W) s_pre[(size_t)e * W + w] = static_cast<uint16_t>(carry + incl - c);
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_cnt[e] = carry;
    }
    __syncthreads();
    // 3. offsets: exclusive scan of the bucket sizes (E <= 256: 8 warps + fix-up)
    if (tid < MOE_MAX_EXPERTS) {
        const int v = tid < E ? s_cnt[tid] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) s_wsum[warp] = incl;
        s_off[tid] = incl - v;  // exclusive within the warp for now
    }
    __syncthreads();
    if (tid < MOE_MAX_EXPERTS) {
        int add = 0;
        for (int w = 0; w < (tid >> 5); ++w) add += s_wsum[w];
        if (tid < E) s_off[tid] += add;
        if (tid == E - 1) s_off[E] = s_off[tid] + s_cnt[tid];
    }
    __syncthreads();
    for (int e = tid; e <= E; e += kBucketThreads) offsets[e] = s_off[e];
    // 4. positions: one pair per thread (unrolled: the id loads overlap)
#pragma unroll 8
    for (int p = tid; p < P; p += kBucketThreads) {
        const int e = __ldcg(idx + p);
        int ps = -1;
        if (e >= 0 && e < E) {
            const uint32_t m = s_mask[(size_t)e * W + (p >> 5)];
            if (m & (1u << (p & 31)))  // kept (not an invalid or repeated id)
                ps = s_off[e] + s_pre[(size_t)e * W + (p >> 5)] + __popc(m & ((1u << (p & 31)) - 1u));
        }
        pos[p] = ps;
        if (ps >= 0) {
            pair_tok[ps] = p / k;
            pair_slot[ps] = p - (p / k) * k;
        }
    }
    if (tid == 0 && s_bad) flag_status(status, MOE_STATUS_BAD_INDEX);
}

// Large batches over many CTAs, no inter-CTA communication: CTA c owns the
// tokens of pair tile c (kTilePairs pairs).  Every CTA reads all the ids
// (a few tens of KB, from L2) to count, per expert, all kept pairs and the
// kept pairs of earlier tiles; it scans the totals into offsets itself and
// ranks its own pairs with per-expert bitmaps of its tile.  A pair's position
// is offsets[e] + (pairs of e in earlier tiles) + (its rank in the tile), the
// same stable (token, slot) order as the single-CTA kernels.
constexpr int kTilePairs = 1024;
constexpr int kTileWords = kTilePairs / 32;

__global__ void __launch_bounds__(kBucketThreads) bucket_tiles_kernel(const int32_t* __restrict__ idx, int T, int k,
                                                                      int E, int32_t* __restrict__ offsets,
                                                                      int32_t* __restrict__ pair_tok,
                                                                      int32_t* __restrict__ pair_slot,
                                                                      int32_t* __restrict__ pos, int32_t* status) {
    __shared__ int s_total[MOE_MAX_EXPERTS], s_before[MOE_MAX_EXPERTS];
    __shared__ int s_off[MOE_MAX_EXPERTS + 1];
    __shared__ int s_wsum[kBucketWarps];
    __shared__ int s_bad;
    extern __shared__ uint32_t bucket_dyn[];
    uint32_t* s_mask = bucket_dyn;                                   // [E][kTileWords], bit = pair - tile start
    int* s_pre = reinterpret_cast<int*>(bucket_dyn + E * kTileWords);  // [E][kTileWords] pairs in earlier words
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tpt = kTilePairs / k;  // tokens per tile
    const int t0 = blockIdx.x * tpt, t1 = min(T, t0 + tpt);
    pdl_wait();  // idx written by the router
    pdl_launch_dependents();
    for (int i = tid; i < E * kTileWords; i += kBucketThreads) s_mask[i] = 0;
    if (tid < MOE_MAX_EXPERTS) {
        s_total[tid] = 0;
        s_before[tid] = 0;
    }
    if (tid == 0) s_bad = 0;
    __syncthreads();

    // 1. every token: validate, drop repeats; count; set this tile's bits
    int bad = 0;
    for (int t = tid; t < T; t += kBucketThreads)
        token_ids(idx, t, k, E, &bad, [&](int s2, int e) {
            atomicAdd(&s_total[e], 1);
            if (t < t0) {
                atomicAdd(&s_before[e], 1);
            } else if (t < t1) {
                const int q = (t - t0) * k + s2;
                atomicOr(&s_mask[e * kTileWords + (q >> 5)], 1u << (q & 31));
            }
        });
    if (bad) s_bad = 1;
    __syncthreads();
    // 2. offsets (exclusive scan of the totals) and the tile's word prefixes
    if (tid < MOE_MAX_EXPERTS) {
        const int v = tid < E ? s_total[tid] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) s_wsum[warp] = incl;
        s_off[tid] = incl - v;
    }
    for (int e = warp; e < E; e += kBucketWarps) {  // kTileWords == 32: one word per lane
        const int c = __popc(s_mask[e * kTileWords + lane]);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        s_pre[e * kTileWords + lane] = incl - c;
    }
    __syncthreads();
    if (tid < MOE_MAX_EXPERTS) {
        int add = 0;
        for (int w = 0; w < (tid >> 5); ++w) add += s_wsum[w];
        if (tid < E) s_off[tid] += add;
        if (tid == E - 1) s_off[E] = s_off[tid] + s_total[tid];
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int e = tid; e <= E; e += kBucketThreads) offsets[e] = s_off[e];
    // 3. this tile's pairs
    const int np = (t1 - t0) * k;
    for (int q = tid; q < np; q += kBucketThreads) {
        const int p = t0 * k + q;
        const int e = __ldcg(idx + p);
        int ps = -1;
        if (e >= 0 && e < E) {
            const uint32_t m = s_mask[e * kTileWords + (q >> 5)];
            if (m & (1u << (q & 31)))
                ps = s_off[e] + s_before[e] + s_pre[e * kTileWords + (q >> 5)] + __popc(m & ((1u << (q & 31)) - 1u));
        }
        pos[p] = ps;
        if (ps >= 0) {
            pair_tok[ps] = p / k;
            pair_slot[ps] = p - (p / k) * k;
        }
    }
    if (blockIdx.x == 0 && tid == 0 && s_bad) flag_status(status, MOE_STATUS_BAD_INDEX);
}

size_t bucket_mask_smem(int T, int k, int E) {
    const size_t W = ((size_t)T * k + 31) / 32;
    return (size_t)E * W * (sizeof(uint32_t) + sizeof(uint16_t));
}

constexpr size_t kBucketMaskCap = 200 * 1024;

}  // namespace

cudaError_t launch_bucket(const int32_t* idx, int T, int k, int E, int32_t* offsets, int32_t* pair_tok,
                          int32_t* pair_slot, int32_t* pos, int32_t* status, cudaStream_t s) {
    const long long P = (long long)T * k;
    const size_t msmem = bucket_mask_smem(T, k, E);
    // 2048+ pairs: tiles of 1024 pairs on as many CTAs (every CTA re-reads all
    // ids, so very large batches keep the single-CTA kernels)
    const bool use_tiles = P >= 2048 && T <= 16384;
    const bool use_mask = !use_tiles && P <= 65535 && msmem <= kBucketMaskCap;  // word prefixes fit 16 bits
    const size_t tsmem = (size_t)E * kTileWords * 2 * sizeof(uint32_t);
    const size_t smem = use_tiles ? tsmem
                                  : (use_mask ? msmem : (size_t)2 * kBucketWarps * ((E + 31) & ~31) * sizeof(uint32_t));
    auto kern = use_tiles ? bucket_tiles_kernel : (use_mask ? bucket_mask_kernel : bucket_kernel);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(use_tiles ? (unsigned)((T + kTilePairs / k - 1) / (kTilePairs / k)) : 1u, 1, 1);
    cfg.blockDim = dim3(kBucketThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, idx, T, k, E, offsets, pair_tok, pair_slot, pos, status);
}

}  // namespace moe
