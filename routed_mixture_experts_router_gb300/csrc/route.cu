// Router: logits x . Wr^T (+ bias) in fp32, top-k with ties to the lower id,
// renormalised softmax weights.
//
// "LinearGate" routing (amalgafy.com/evidence, "Layer-qualified experts") and
// "GPU router/top-k" (amalgafy.com/technical-overview, "Not complete today").
//
// Design: one thread-block cluster per tile of TT tokens.  The cluster's CTAs
// split the experts; inside a CTA each warp owns one router row at a time and
// its lanes split K with coalesced 16-byte loads, so the 1 MiB router matrix
// streams through 16 SMs in parallel even at T = 1.  Logits land in the
// leader CTA's shared memory (distributed shared memory), and after one
// cluster barrier the leader's warps run a warp-shuffle top-k, one warp per
// token.  No global scratch, no atomics, no inter-CTA spin: deterministic.
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "pipeline.cuh"

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / kWarp;
constexpr int kRouteUnroll = 8;  // float4 loads in flight per lane per step

// Top-k over E (<= 256) logits of one token by one warp.  Lane l holds the
// logits of experts l, l+32, ...  Each round takes the warp-wide maximum,
// ties to the lower expert id; the winner is marked taken.  Round s's winner
// goes to slot s.  Weights: exp(l_s - l_0) / sum over the selection.
__device__ void topk_warp(const float* lg, const float* bias, int E, int k, int32_t* idx_out, float* w_out,
                          int32_t* s_idx) {
    const int lane = threadIdx.x & 31;
    float v[MOE_MAX_EXPERTS / 32];
    uint32_t taken = 0;
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
        const int e = lane + 32 * j;
        if (e < E) {
            v[j] = lg[e] + (bias ? __ldg(bias + e) : 0.0f);
        } else {
            v[j] = -INFINITY;
            taken |= 1u << j;
        }
    }
    float my_v = 0.0f, vmax = 0.0f;
    int my_e = 0;
    for (int s = 0; s < k; ++s) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
            // experts grow with j inside a lane, so strict > keeps the lower id
            if (!((taken >> j) & 1u) && (be == 0x7fffffff || v[j] > bv)) {
                bv = v[j];
                be = lane + 32 * j;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if (lane == (be & 31)) taken |= 1u << (be >> 5);
        if (lane == s) {
            my_v = bv;
            my_e = be;
        }
        if (s == 0) vmax = bv;
    }
    const float num = (lane < k) ? expf(my_v - vmax) : 0.0f;
    const float den = warp_sum(num);
    if (lane < k) {
        idx_out[lane] = my_e;
        w_out[lane] = num / den;
        if (s_idx) s_idx[lane] = my_e;
    }
}

// Compact expert grouping of T <= 32 tokens by one warp (fused into the
// router when one cluster holds every token).  Lane t owns token t; ballots
// over the tokens' expert bitmaps give, for each expert e, the set M[e] of
// tokens that picked it; offsets are the exclusive scan of |M[e]| and pair
// (t, s) lands at offsets[e] + |M[e] & tokens below t|: stable in
// (token, slot) order, no atomics.
__device__ void bucket_warp(const int32_t* s_idx, int T, int k, int E, int* s_off, uint32_t* s_m,
                            int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot, int32_t* pos) {
    const int lane = threadIdx.x & 31;
    uint32_t bm[MOE_MAX_EXPERTS / 32];
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) bm[j] = 0;
    if (lane < T) {
        for (int s = 0; s < k; ++s) {
            const int e = s_idx[lane * k + s];
#pragma unroll
            for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j)
                if (j == (e >> 5)) bm[j] |= 1u << (e & 31);
        }
    }
    const int words = (E + 31) >> 5;
    int run = 0;
#pragma unroll
    for (int j = 0; j < MOE_MAX_EXPERTS / 32; ++j) {
        if (j < words) {
            uint32_t mine = 0;
#pragma unroll 8
            for (int b = 0; b < 32; ++b) {
                const uint32_t m = __ballot_sync(0xffffffffu, (bm[j] >> b) & 1u);
                if (lane == b) mine = m;
            }
            const int e = 32 * j + lane;
            const int cnt = (e < E) ? __popc(mine) : 0;
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            s_off[e] = run + incl - cnt;
            s_m[e] = mine;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    __syncwarp();
    for (int e = lane; e < E; e += 32) offsets[e] = s_off[e];
    if (lane == 0) offsets[E] = run;
    if (lane < T) {
        const uint32_t below = (1u << lane) - 1u;
        for (int s = 0; s < k; ++s) {
            const int e = s_idx[lane * k + s];
            const int p = s_off[e] + __popc(s_m[e] & below);
            pair_tok[p] = lane;
            pair_slot[p] = s;
            pos[lane * k + s] = p;
        }
    }
}

template <int TT>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const float* __restrict__ x,
                                                              const float* __restrict__ Wr,
                                                              const float* __restrict__ bias, int T, int dm, int E,
                                                              int k, int epc, int e_stride,
                                                              int32_t* __restrict__ idx, float* __restrict__ wts,
                                                              int32_t* offsets, int32_t* pair_tok,
                                                              int32_t* pair_slot, int32_t* pos) {
    __shared__ int32_t s_idx[TT * MOE_MAX_TOPK];
    __shared__ int s_off[MOE_MAX_EXPERTS];
    __shared__ uint32_t s_m[MOE_MAX_EXPERTS];
    extern __shared__ float4 route_smem[];
    float4* xs = route_smem;                                   // [TT][dm/4]
    float* lg = reinterpret_cast<float*>(route_smem + TT * (dm / 4));  // [TT][e_stride]

    cg::cluster_group cluster = cg::this_cluster();
    const int c = static_cast<int>(cluster.block_rank());
    const int t0 = blockIdx.y * TT;
    const int nt = min(TT, T - t0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d4 = dm / 4;

    // Start this warp's first router row before staging x, so both streams overlap.
    int el = warp;
    int e = c * epc + el;
    float4 wbuf[kRouteUnroll];
    const float4* wr = reinterpret_cast<const float4*>(Wr) + (size_t)e * d4;
    if (el < epc && e < E) {
#pragma unroll
        for (int u = 0; u < kRouteUnroll; ++u) {
            const int q = lane + 32 * u;
            wbuf[u] = q < d4 ? __ldg(wr + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    pdl_wait();  // x is written by earlier kernels (a previous layer)
    const float4* xg = reinterpret_cast<const float4*>(x) + (size_t)t0 * d4;
    for (int i = threadIdx.x; i < nt * d4; i += kRouteThreads) xs[i] = __ldcg(xg + i);
    __syncthreads();
    pdl_launch_dependents();

    float* lg_leader = cluster.map_shared_rank(lg, 0);
    for (; el < epc; el += kRouteWarps) {
        e = c * epc + el;
        if (e >= E) break;
        wr = reinterpret_cast<const float4*>(Wr) + (size_t)e * d4;
        float acc[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[t] = 0.0f;
        for (int q0 = 0; q0 < d4; q0 += 32 * kRouteUnroll) {
            if (q0 > 0 || el != warp) {
#pragma unroll
                for (int u = 0; u < kRouteUnroll; ++u) {
                    const int q = q0 + lane + 32 * u;
                    wbuf[u] = q < d4 ? __ldg(wr + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int u = 0; u < kRouteUnroll; ++u) {
                const int q = q0 + lane + 32 * u;
                if (q < d4) {
#pragma unroll
                    for (int t = 0; t < TT; ++t) acc[t] = dot4(wbuf[u], xs[t * d4 + q], acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[t] = warp_sum(acc[t]);
        if (lane == 0) {
#pragma unroll
            for (int t = 0; t < TT; ++t)
                if (t < nt) lg_leader[t * e_stride + e] = acc[t];
        }
    }
    cluster.sync();  // all logits of the tile are in the leader's shared memory
    if (c == 0) {
        const bool fuse_bucket = offsets != nullptr && gridDim.y == 1;
        for (int t = warp; t < nt; t += kRouteWarps)
            topk_warp(lg + t * e_stride, bias, E, k, idx + (size_t)(t0 + t) * k, wts + (size_t)(t0 + t) * k,
                      fuse_bucket ? s_idx + t * k : nullptr);
        if (fuse_bucket) {
            __syncthreads();
            if (warp == 0) bucket_warp(s_idx, nt, k, E, s_off, s_m, offsets, pair_tok, pair_slot, pos);
        }
    }
}

template <int TT>
cudaError_t launch_route_tt(const float* x, int T, const moe_layer_w& w, int32_t* idx, float* wts, int cl,
                            int32_t* offsets, int32_t* pair_tok, int32_t* pair_slot, int32_t* pos,
                            cudaStream_t s) {
    const int E = w.E, dm = w.d_model;
    const int epc = (E + cl - 1) / cl;
    const int e_stride = (E + 3) & ~3;
    const size_t smem = (size_t)TT * dm * sizeof(float) + (size_t)TT * e_stride * sizeof(float);
    auto kern = route_kernel<TT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    if (cl > 8) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl, (T + TT - 1) / TT, 1);
    cfg.blockDim = dim3(kRouteThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, x, w.router_w, w.router_bias, T, dm, E, w.k, epc, e_stride, idx, wts,
                              offsets, pair_tok, pair_slot, pos);
}

// Largest cluster size (16, else 8) that the device can co-schedule for this
// kernel shape; probed once per process and device.
int route_cluster_size(int E, size_t smem) {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
    int want = E >= 128 ? 16 : 8;
    if (want == 16) {
        if (cached[dev] == 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(16, 1, 1);
            cfg.blockDim = dim3(kRouteThreads, 1, 1);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 16;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            auto kern = route_kernel<8>;
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            cudaError_t err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            cached[dev] = (err == cudaSuccess && n > 0) ? 16 : 8;
            cudaGetLastError();
        }
        want = cached[dev];
    }
    return want;
}

}  // namespace

cudaError_t launch_route(const float* x, int T, const moe_layer_w& w, int32_t* idx, float* wts, int32_t* offsets,
                         int32_t* pair_tok, int32_t* pair_slot, int32_t* pos, bool* bucketed, cudaStream_t s) {
    if (bucketed) *bucketed = false;
    if (T == 0) return cudaSuccess;
    // tokens per tile: bounded so the x tile stays within 96 KB of shared memory
    int tt = T >= 8 ? 8 : (T >= 4 ? 4 : (T >= 2 ? 2 : 1));
    while (tt > 1 && (size_t)tt * w.d_model * sizeof(float) > 96 * 1024) tt >>= 1;
    if (T > tt || !bucketed) offsets = pair_tok = pair_slot = pos = nullptr;  // several tiles: separate bucketing
    if (offsets && bucketed) *bucketed = true;
    const size_t smem8 = (size_t)8 * w.d_model * sizeof(float) + (size_t)8 * ((w.E + 3) & ~3) * sizeof(float);
    const int cl = route_cluster_size(w.E, smem8);
    switch (tt) {
        case 8: return launch_route_tt<8>(x, T, w, idx, wts, cl, offsets, pair_tok, pair_slot, pos, s);
        case 4: return launch_route_tt<4>(x, T, w, idx, wts, cl, offsets, pair_tok, pair_slot, pos, s);
        case 2: return launch_route_tt<2>(x, T, w, idx, wts, cl, offsets, pair_tok, pair_slot, pos, s);
        default: return launch_route_tt<1>(x, T, w, idx, wts, cl, offsets, pair_tok, pair_slot, pos, s);
    }
}

}  // namespace moe
