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
// cluster barrier the leader's threads rank the logits (top-k by rank, one
// thread per (token, expert) candidate).  No global scratch, no atomics, no
// inter-CTA spin: deterministic.
#include <atomic>
#include <climits>
#include <cooperative_groups.h>
#include <math.h>

#include "common.cuh"
#include "pipeline.cuh"
#include "route_warp.cuh"

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / kWarp;
constexpr int kRouteUnroll = 8;  // float4 loads in flight per lane per step

template <int TT>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const float* __restrict__ x,
                                                              const float* __restrict__ Wr,
                                                              const float* __restrict__ bias, int T, int dm, int E,
                                                              int k, int epc, int e_stride,
                                                              int32_t* __restrict__ idx, float* __restrict__ wts,
                                                              int32_t* offsets, int32_t* pair_tok,
                                                              int32_t* pair_slot, int32_t* pos) {
    __shared__ int32_t s_idx[TT * MOE_MAX_TOPK];
    __shared__ float s_val[TT * MOE_MAX_TOPK];
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
        // top-k by rank over the whole CTA; with one tile holding every token
        // the bucketing is fused (pair positions and offsets, also by rank)
        const bool fuse_bucket = offsets != nullptr && gridDim.y == 1;
        prep_logits(lg, e_stride, nt, E, bias, kRouteThreads);
        __syncthreads();
        topk_rank_block(lg, e_stride, nt, E, k, kRouteThreads, s_idx, s_val);
        __syncthreads();
        const int P = nt * k;
        for (int q = threadIdx.x; q < P; q += kRouteThreads) {
            idx[(size_t)t0 * k + q] = s_idx[q];
            wts[(size_t)t0 * k + q] = topk_weight(s_val, q, k);
            if (fuse_bucket) {
                const int r = pair_rank(s_idx, P, q);
                pair_tok[r] = q / k;
                pair_slot[r] = q - (q / k) * k;
                pos[q] = r;
            }
        }
        if (fuse_bucket) bucket_offsets(s_idx, P, E, kRouteThreads, offsets);
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
    static std::atomic<int> cached[64];  // zero-initialised; racing first calls store the same value
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
    int want = E >= 128 ? 16 : 8;
    if (want == 16) {
        if (cached[dev].load(std::memory_order_relaxed) == 0) {
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
            cached[dev].store((err == cudaSuccess && n > 0) ? 16 : 8, std::memory_order_relaxed);
            cudaGetLastError();
        }
        want = cached[dev].load(std::memory_order_relaxed);
    }
    return want;
}

}  // namespace

// ------------------------------------------------------------ large batches
// Router logits as a split-K fp32 GEMM: one cluster of CL CTAs per tile
// of kGemmTok tokens; CTA c accumulates K slice c for all experts with 4x EPT
// register tiles over transposed shared-memory chunks of x and Wr, then
// pushes each token's slice into the shared memory of the CTA that owns the
// token (distributed shared memory, one cluster barrier); the owner sums the
// slices in a fixed order (deterministic) and runs the top-k of its tokens.
constexpr int kGemmTok = 32;
// CL = 16 (a non-portable cluster size, used where the device can
// co-schedule it): twice the CTAs of CL = 8 over the same tiles, 4-6% off a
// prefill layer at T = 768-1024
constexpr int kGemmKc = 32;
constexpr int kGemmThreads = 256;

template <int EPT, int CL>
__global__ void __launch_bounds__(kGemmThreads) route_gemm_kernel(const float* __restrict__ x,
                                                                  const float* __restrict__ Wr,
                                                                  const float* __restrict__ bias, int T, int dm,
                                                                  int E, int k, int32_t* __restrict__ idx,
                                                                  float* __restrict__ wts) {
    constexpr int EP = 32 * EPT;  // padded expert count
    __shared__ __align__(16) float xs[kGemmKc][kGemmTok];
    __shared__ __align__(16) float ws[kGemmKc][EP];
    __shared__ __align__(16) float part[kGemmTok][EP];
    cg::cluster_group cluster = cg::this_cluster();
    const int c = static_cast<int>(cluster.block_rank());
    const int t0 = blockIdx.y * kGemmTok;
    const int tid = threadIdx.x;
    const int tg = tid & 7, eg = tid >> 3;  // tokens 4tg..4tg+3, experts EPT*eg..
    const int kslice = dm / CL;
    const int kbeg = c * kslice;
    const int nch = kslice / kGemmKc;

    // Loaders, coalesced: 8 lanes read one 128-byte row segment (token or
    // expert row, 32 k), so a warp reads 4 whole segments per instruction.
    // The chunks are stored transposed (xs[k][token], ws[k][expert]) with the
    // 16-byte groups of a k row XOR-rotated by k/4: the transposing stores and
    // the float4 reads of the FMA loop are both free of bank conflicts.
    const int lr = tid >> 3, lq = tid & 7;  // row within the chunk, k quad
    float4 xr = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 wr[EPT];
    auto load = [&](int ch) {
        const int kk = kbeg + ch * kGemmKc;
        const int t = t0 + lr;
        xr = (t < T) ? __ldcg(reinterpret_cast<const float4*>(x + (size_t)t * dm + kk) + lq)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const int e = lr + 32 * j;
            const float4* src = reinterpret_cast<const float4*>(Wr + (size_t)e * dm + kk) + lq;
            wr[j] = (e < E) ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    // column `col` of k row `kr` lives at swz(col, kr)
    auto swz = [](int col, int kr) { return (((col >> 2) ^ ((kr >> 2) & 7)) << 2) | (col & 3); };
    // this CTA has started: its receive buffer may be written by the others
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    pdl_wait();  // x is written by earlier kernels
    load(0);
    float acc[4][EPT];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < EPT; ++j) acc[i][j] = 0.f;
    for (int ch = 0; ch < nch; ++ch) {
        __syncthreads();  // previous chunk consumed
        {
            const float xv4[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) xs[lq * 4 + i][swz(lr, lq * 4 + i)] = xv4[i];
        }
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const int e = lr + 32 * j;
            const float wv4[4] = {wr[j].x, wr[j].y, wr[j].z, wr[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) ws[lq * 4 + i][swz(e, lq * 4 + i)] = wv4[i];
        }
        __syncthreads();
        if (ch + 1 < nch) load(ch + 1);  // next chunk in flight during the FMAs
#pragma unroll 8
        for (int kk = 0; kk < kGemmKc; ++kk) {
            const int rot = (kk >> 2) & 7;
            const float4 xv = *reinterpret_cast<const float4*>(&xs[kk][(tg ^ rot) << 2]);
            float wv[EPT];
#pragma unroll
            for (int j = 0; j < EPT; j += 4) {
                const float4 q = *reinterpret_cast<const float4*>(&ws[kk][((eg * EPT + j) >> 2 ^ rot) << 2]);
                wv[j] = q.x;
                wv[j + 1] = q.y;
                wv[j + 2] = q.z;
                wv[j + 3] = q.w;
            }
            const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < EPT; ++j) acc[i][j] = fmaf(xa[i], wv[j], acc[i][j]);
        }
    }
    // CTA c owns tokens c*kOwn .. c*kOwn+kOwn-1 of the tile; part, in the
    // owner, receives slice r of its token tl at row r*kOwn + tl
    constexpr int kOwn = kGemmTok / CL;
    static_assert(EPT % 4 == 0, "vector pushes");
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA of the cluster has started
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int tt = tg * 4 + i, owner = tt / kOwn, tl = tt - owner * kOwn;
#pragma unroll
        for (int j = 0; j < EPT; j += 4) {
            uint32_t a;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                         : "=r"(a)
                         : "r"(smem_u32(&part[c * kOwn + tl][eg * EPT + j])), "r"(owner));
            asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(acc[i][j]),
                         "f"(acc[i][j + 1]), "f"(acc[i][j + 2]), "f"(acc[i][j + 3])
                         : "memory");
        }
    }
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // every slice of this CTA's tokens is in
    // sum the owned tokens' logits over the K slices in a fixed order
    // (deterministic), then rank them
    __shared__ int32_t s_sel[kOwn * MOE_MAX_TOPK];
    __shared__ float s_val[kOwn * MOE_MAX_TOPK];
    float* lg = &xs[0][0];  // reuse: [kOwn][EP] logits (kOwn * EP <= kGemmKc * kGemmTok)
    const int tb = t0 + c * kOwn;
    const int nt = min(kOwn, max(0, T - tb));
    for (int i = tid; i < kOwn * EP; i += kGemmThreads) {
        const int tl = c * kOwn + i / EP, e = i % EP;
        float s = 0.f;
        for (int r = 0; r < CL; ++r) s += part[r * kOwn + (tl - c * kOwn)][e];
        lg[i] = s;
    }
    __syncthreads();
    prep_logits(lg, EP, nt, E, bias, kGemmThreads);
    __syncthreads();
    topk_rank_block(lg, EP, nt, E, k, kGemmThreads, s_sel, s_val);
    __syncthreads();
    for (int q = tid; q < nt * k; q += kGemmThreads) {
        idx[(size_t)tb * k + q] = s_sel[q];
        wts[(size_t)tb * k + q] = topk_weight(s_val, q, k);
    }
}

template <int EPT, int CL>
cudaError_t launch_route_gemm(const float* x, int T, const moe_layer_w& w, int32_t* idx, float* wts,
                              cudaStream_t s) {
    if (CL > 8) {  // clusters above the portable size must be allowed explicitly
        const cudaError_t e =
            cudaFuncSetAttribute(route_gemm_kernel<EPT, CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, (T + kGemmTok - 1) / kGemmTok, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, route_gemm_kernel<EPT, CL>, x, w.router_w, w.router_bias, T, w.d_model, w.E, w.k,
                              idx, wts);
}

// How many clusters of CL CTAs of the router GEMM the device co-schedules
// (0: none); probed once per process, device and cluster size (racing first
// calls store the same answer).
template <int CL>
static int gemm_max_clusters() {
    static std::atomic<int> cached[64];  // count + 1; 0 = not probed
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = cached[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        auto kern = route_gemm_kernel<4, CL>;
        int n = 0;
        cudaError_t err =
            CL > 8 ? cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) : cudaSuccess;
        if (err == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(CL, 1, 1);
            cfg.blockDim = dim3(kGemmThreads, 1, 1);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = CL;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        }
        cudaGetLastError();
        c = (err == cudaSuccess && n > 0 ? n : 0) + 1;
        cached[dev].store(c, std::memory_order_relaxed);
    }
    return c - 1;
}

cudaError_t launch_route(const float* x, int T, const moe_layer_w& w, int32_t* idx, float* wts, int32_t* offsets,
                         int32_t* pair_tok, int32_t* pair_slot, int32_t* pos, bool* bucketed, cudaStream_t s) {
    if (bucketed) *bucketed = false;
    if (T == 0) return cudaSuccess;
    // 16-CTA clusters (twice the CTAs per token tile) where every tile's
    // cluster is resident at once; else 8-CTA clusters, which fit twice as
    // many at a time (T = 2048: 46.5 instead of 50.3 us)
    if (T >= 64 && w.E <= 128 && w.d_model % (16 * kGemmKc) == 0) {
        const int tiles = (T + kGemmTok - 1) / kGemmTok;
        const int n16 = gemm_max_clusters<16>(), n8 = gemm_max_clusters<8>();
        const int waves16 = n16 > 0 ? (tiles + n16 - 1) / n16 : INT_MAX;
        const int waves8 = n8 > 0 ? (tiles + n8 - 1) / n8 : INT_MAX;
        if (n16 > 0 && waves16 <= waves8) return launch_route_gemm<4, 16>(x, T, w, idx, wts, s);
    }
    if (T >= 64 && w.E <= 128 && w.d_model % (8 * kGemmKc) == 0)
        return launch_route_gemm<4, 8>(x, T, w, idx, wts, s);
    // tokens per tile: bounded so the x tile stays within 96 KB of shared
    // memory; several tiles of 4 rather than 8 tokens (twice the clusters
    // streaming the router rows: 1.4% off a T = 64 layer)
    int tt = T > 8 ? 4 : (T >= 8 ? 8 : (T >= 4 ? 4 : (T >= 2 ? 2 : 1)));
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
